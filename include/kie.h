/*
 * kie.h -- C ABI of the GB300 (sm_103a) persistent decode monokernel.
 *
 * The library runs batch-1 greedy decode of a dense Llama-style decoder (fp16 weights and KV cache, fp32
 * arithmetic) as ONE persistent cooperative kernel per call, one CTA per SM, that loops over all requested
 * tokens and all layers without returning to the host. This is the "monokernel" of the Kog Inference
 * Engine pages ("Inside the monokernel: a single resident GPU program that never returns control"): the
 * host launches once, the device embeds, projects, attends, samples and feeds the next token back itself.
 *
 * Where the calls come from: the pages define no programming interface (the creeta article, section "Before
 * adopting", only says the engine can stand in for a vLLM deployment). The create / prefill / decode / destroy
 * shape below is this library's own statement of the batch-1 decode problem; each declaration names the part
 * of the pages its work follows, or says that it has none.
 *
 * Conventions for every entry point:
 *   - Return value: KIE_OK (0) or a negative KIE_ERR_* code. kie_last_error() gives a message.
 *   - Weights are IEEE binary16 bit patterns (uint16_t), row-major [out_features, in_features].
 *   - Pointers are HOST pointers unless the name or comment says "_dev" / "device".
 *   - A kie_ctx is not thread-safe: calls on one ctx must be serialised by the caller. All GPU work of a
 *     ctx is issued on the stream given at creation (NULL = the legacy default stream).
 *   - Positions are 0-based; the first prompt token is at position 0.
 */
#ifndef KIE_H
#define KIE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  KIE_OK = 0,
  KIE_ERR_INVALID = -1,  /* bad argument, unsupported dimension, or call out of order */
  KIE_ERR_OOM = -2,      /* a device allocation failed */
  KIE_ERR_CAPACITY = -3, /* position + n would exceed max_seq */
  KIE_ERR_CUDA = -4,     /* a CUDA runtime call failed (message in kie_last_error) */
  KIE_ERR_LAUNCH = -5,   /* the cooperative grid (one CTA per SM) could not be made co-resident */
  KIE_ERR_TIMEOUT = -6   /* a device-side wait gave up; the kernel exited cleanly, the ctx is reset */
};

/* Model shape. Supported: head_dim in {64, 128}; n_heads % n_kv_heads == 0; d_model, ffn_dim and
 * n_heads*head_dim multiples of 8; n_layers >= 1; vocab >= 2. rope_theta is the RoPE base, rms_eps the
 * RMSNorm epsilon. */
typedef struct {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, max_seq;
  float rope_theta, rms_eps;
} kie_config;

/* Host weights (fp16 bits). Per-layer fields are arrays of n_layers host pointers. Shapes:
 * embed, lm_head [vocab, d_model]; final_norm, attn_norm[l], ffn_norm[l] [d_model];
 * wq [n_heads*head_dim, d_model]; wk, wv [n_kv_heads*head_dim, d_model]; wo [d_model, n_heads*head_dim];
 * w_gate, w_up [ffn_dim, d_model]; w_down [d_model, ffn_dim].
 * Ownership: read during kie_create only; the caller may free them afterwards. */
typedef struct {
  const uint16_t *embed, *lm_head, *final_norm;
  const uint16_t *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo;
  const uint16_t *const *ffn_norm, *const *w_gate, *const *w_up, *const *w_down;
} kie_weights;

typedef struct kie_ctx kie_ctx;

/* Device buffer sizes a ctx needs (bytes), for callers that allocate device memory themselves. */
typedef struct {
  size_t weights_bytes;   /* repacked weights + embedding table (+ the prefill's tensor-core tiles, dense models) */
  size_t kv_bytes;        /* K/V cache [n_layers][2][n_kv_heads][max_seq][head_dim] fp16 */
  size_t workspace_bytes; /* activations, split-attention partials, RoPE table, logits, control words */
  int n_cta;              /* CTAs of the persistent grid the layout was planned for */
} kie_buffer_sizes;

/* Sizes for `cfg` on the current device (n_cta = its SM count when the argument is 0).
 * Errors: KIE_ERR_INVALID for an unsupported cfg; KIE_ERR_CUDA if the device cannot be queried. */
int kie_query_buffers(const kie_config *cfg, int n_cta, kie_buffer_sizes *out);

/* Create a ctx: validates cfg, repacks the weights (QKV fused with RoPE pairs made adjacent, gate/up
 * interleaved, RMSNorm gains folded into the next matrix, rows tiled per CTA -- the fusion list of the
 * "inside the monokernel" section of the monokernel pages), uploads them, builds the RoPE table and
 * zeroes the KV cache. `stream` is a cudaStream_t or NULL. The ctx allocates its own device memory
 * (cudaMalloc) and frees it in kie_destroy. On error *out is NULL. */
int kie_create(const kie_config *cfg, const kie_weights *w, void *stream, kie_ctx **out);

/* As kie_create, but the device memory is provided by the caller (e.g. allocated with PyTorch) and stays
 * owned by the caller: it must outlive the ctx. Each buffer must be 256-byte aligned and at least the size
 * kie_query_buffers returned (for n_cta = 0). kie_create_with_buffers still allocates one temporary
 * staging buffer of the largest repacked matrix while it runs, and frees it before returning. */
int kie_create_with_buffers(const kie_config *cfg, const kie_weights *w, void *stream, void *weights_dev,
                            size_t weights_bytes, void *kv_dev, size_t kv_bytes, void *workspace_dev,
                            size_t workspace_bytes, kie_ctx **out);

/* Prompt ingestion. The pages do not describe prefill (their measurements start at decode); this call exists
 * so that decode has a KV cache and current logits to start from.
 * Append n prompt tokens (host int32 ids in [0, vocab)) to the KV cache at positions pos..pos+n-1 and keep the
 * logits of the last one (so the next decode can start). The tokens go through each layer together, in chunks
 * of up to 128: the projections are tensor-core GEMMs (tcgen05) over a second copy of the dense weights in the
 * tensor cores' tile layout, with each fp32 activation split into fp16 high and low parts (fp32-class results);
 * the causal attention over the cache runs on the tensor cores too, in 512-position pieces. The result does not depend on
 * how a prompt is split over calls (bit for bit). Synchronous. Errors: INVALID (n < 1, bad id), CAPACITY, CUDA,
 * TIMEOUT (a bounded device wait of the GEMM ran out; the sequence is reset). */
int kie_prefill(kie_ctx *ctx, const int32_t *tokens, int n);

/* The monokernel's token loop ("Inside the monokernel", creeta: one resident launch embeds, runs every layer,
 * samples greedily on the device and feeds the token back, with no host round trip between tokens).
 * Greedy decode of n tokens in ONE launch (the hot path). Token i is the argmax of the current logits
 * (lowest id on ties); the kernel then runs the forward of that token at the next position, whose logits
 * are the current ones for token i+1. So n tokens cost n forwards, and decode(a) then decode(b) gives the
 * same tokens as decode(a+b). Requires a prior prefill (INVALID otherwise). `out_tokens` is a host array of
 * n int32; the call synchronises the stream. Errors: INVALID, CAPACITY, CUDA, LAUNCH, TIMEOUT. */
int kie_decode(kie_ctx *ctx, int n, int32_t *out_tokens);

/* As kie_decode, but writes the n tokens to DEVICE memory `out_tokens_dev` and returns right after the
 * launch is enqueued on the ctx stream (no synchronisation). Device-side errors are reported by the next
 * kie_sync(). */
int kie_decode_async(kie_ctx *ctx, int n, int32_t *out_tokens_dev);

/* Wait for the ctx stream and report the status word of the last launch (KIE_OK or KIE_ERR_TIMEOUT). */
int kie_sync(kie_ctx *ctx);

/* No counterpart on the pages: a testing aid of this library (teacher forcing keeps one permitted divergence
 * of a near-tied greedy choice from cascading when the GPU is compared with a CPU reference).
 * Teacher forcing, for tests: for i in [0, n): out_tokens[i] = argmax of the current logits (what greedy
 * decode would emit), then the forward consumes forced[i] (not the argmax) at the next position; if
 * out_logits is not NULL it receives the logits of that forward ([n, vocab] fp32, host). Synchronous.
 * Requires a prior prefill. */
int kie_decode_forced(kie_ctx *ctx, int n, const int32_t *forced, int32_t *out_tokens, float *out_logits);

/* No counterpart on the pages: a testing aid for sparse-MoE models (below). The expert selection is itself a
 * floating-point decision (a top_k over router logits) that a CPU reference and the GPU take from logits rounded
 * differently; to compare every step, the reference's own selections can be imposed on the GPU.
 * As kie_decode_forced, plus: forced_experts (host int32 [n][n_layers][top_k], or NULL) replaces the selection
 * of every layer of every forward by the given expert ids (the routing weights stay the softmax of the GPU's
 * router logits over the given experts, in the given order); out_experts (host int32 [n][n_layers][top_k], or
 * NULL) receives the GPU's own selection (descending router logit, the lowest id first among equal ones; ranked
 * on the logits before their common positive RMS factor, so sums whose scaled values round to the same float may
 * rank either way), computed whether or not it is overridden. It may also start a sequence (no prior prefill: the forwards then
 * ingest the forced tokens like a prompt, and out_tokens[0] is -1). Errors: INVALID (a dense model with
 * non-NULL expert arguments, an expert id outside [0, n_experts)), and those of kie_decode_forced. */
int kie_decode_forced_routed(kie_ctx *ctx, int n, const int32_t *forced, const int32_t *forced_experts,
                             int32_t *out_tokens, float *out_logits, int32_t *out_experts);

/* No counterpart on the pages (they sample on the device and never return logits): an inspection call.
 * Copy the current logits (those the next emitted token is the argmax of) to host float[vocab]. */
int kie_get_logits(kie_ctx *ctx, float *out);

/* No counterpart on the pages: sequence bookkeeping of this library.
 * Number of tokens in the KV cache (the position the next forward writes). */
int kie_position(const kie_ctx *ctx);

/* No counterpart on the pages: sequence bookkeeping of this library.
 * Forget the sequence: position 0, no current logits. The KV cache is not cleared (it is overwritten). */
int kie_reset(kie_ctx *ctx);

/* Device-side wait limit in nanoseconds for grid barriers and ring waits (default 1e9). */
int kie_set_timeout_ns(kie_ctx *ctx, uint64_t ns);

/* Barrier timing of the last launch, from %globaltimer stamps taken by every CTA:
 * barriers = grid barriers the launch passed; mean_wait_ns = mean over CTAs and barriers of the time a CTA
 * spent waiting in a barrier (idle time); mean_latency_ns = mean over barriers of the SHORTEST wait among
 * CTAs (the last CTA to arrive waits only for the barrier's own latency); total_ns = launch duration seen
 * by CTA 0. */
typedef struct {
  int64_t barriers;
  double mean_wait_ns, mean_latency_ns, total_ns;
} kie_barrier_stats;
int kie_get_barrier_stats(kie_ctx *ctx, kie_barrier_stats *out);

/* Raw barrier trace of the last launch (the first 4096 grid barriers): for barrier b in
 * [first, first + count) and CTA i, arrive_ns[(b - first) * n_cta + i] is the %globaltimer value when CTA i
 * arrived and wait_ns[...] how long it waited. Host arrays of count * n_cta entries. Returns the number of
 * barriers copied (>= 0) or a negative error code. */
int kie_get_barrier_trace(kie_ctx *ctx, int first, int count, uint64_t *arrive_ns, uint32_t *wait_ns);

/* Test hook (fault injection on the host side of the contract): if cta >= 0, that CTA skips its arrival
 * at grid barrier number `barrier` of the next launch, so every other CTA's wait runs out and the launch
 * returns KIE_ERR_TIMEOUT after the configured limit. No GPU fault, trap or unbounded wait is involved. */
int kie_debug_skip_arrival(kie_ctx *ctx, int cta, int barrier);

/* No counterpart on the pages: a profiling aid. Runs the decode kernel's split-KV attention step alone (the same
 * device function and grid barrier, one cooperative launch) for layers [0, n_layers) over c cached positions,
 * with the q vector and K/V cache the ctx currently holds, so that a profiler can measure that phase's DRAM bytes
 * and time in isolation. Writes only the attention outputs and split-KV partials of the workspace; the sequence
 * (position, current logits, KV cache) is left as it was. Synchronous. Errors: INVALID (c outside [1, max_seq],
 * n_layers outside [1, n_layers]), CUDA, LAUNCH, TIMEOUT. */
int kie_profile_attention(kie_ctx *ctx, int c, int n_layers);

int kie_n_cta(const kie_ctx *ctx);
const char *kie_last_error(const kie_ctx *ctx); /* ctx may be NULL: last error of a failed create */
void kie_destroy(kie_ctx *ctx);

/* ---- standalone GEMV (the same device code as the monokernel's projections) -------------------------
 * y[M] (fp32) = W[M, K] (fp16) . x[K] (fp16), fp32 accumulation, weights streamed through the same
 * shared-memory ring. W must first be packed into the per-CTA tile layout (kie_gemv_pack), as the
 * decoder's weights are at creation. Requirements: M even, K a multiple of 8, M, K >= 2. */

/* Bytes of the packed matrix (= 2*M*K). */
size_t kie_gemv_packed_bytes(int M, int K);

/* Pack row-major W_dev [M, K] into packed_dev for an n_cta-CTA grid (0 = SM count), on `stream`.
 * Both are device pointers, 16-byte aligned, not overlapping. Asynchronous. */
int kie_gemv_pack(const uint16_t *W_dev, int M, int K, int n_cta, uint16_t *packed_dev, void *stream);

/* y_dev = W . x_dev with W packed for the same n_cta. One launch of n_cta CTAs on `stream`; asynchronous. */
int kie_gemv(const uint16_t *packed_dev, const uint16_t *x_dev, float *y_dev, int M, int K, int n_cta,
             void *stream);

/* ---- decode without device allocation ---------------------------------------------------------------
 * No counterpart on the monokernel pages: this entry point exists for callers of this library that cannot
 * call cudaMalloc once they are running -- for example code whose device memory is owned and capped by a
 * host framework's allocator, or loops that must not hit cudaMalloc/cudaFree because those calls can
 * synchronise the device and stall other streams.
 *
 * kie_decode_noalloc(ctx, n, out_tokens_dev) has the semantics of kie_decode (n greedy tokens, one launch,
 * state carried in ctx), but allocates nothing: the per-launch scratch (activations, split-KV partials and
 * the control block) lives in one static device array of KIE_NOALLOC_SCRATCH_BYTES that every GPU loading
 * the library holds until the process exits. The caller passes the output: out_tokens_dev, n int32 in
 * DEVICE memory. The device the ctx was created on must be the current device (KIE_ERR_INVALID otherwise).
 * The call is synchronous (it waits for the ctx stream) and returns KIE_OK, KIE_ERR_TIMEOUT, or the errors of
 * kie_decode; a model whose scratch exceeds the array is rejected with KIE_ERR_INVALID (the message gives both
 * sizes). It takes the same launch path as kie_decode, so a kie_debug_skip_arrival armed before it applies to
 * it. The first call on a device looks up the array's device address (with that device current), so make that
 * first call before any stream capture. All calls share the one array and it keeps the last call's contents
 * (the control block is cleared by every call): calls that overlap on the GPU, from any ctx on the same
 * device, race with each other and must be serialised by the caller. */
#define KIE_NOALLOC_SCRATCH_BYTES (512u * 1024u)
int kie_decode_noalloc(kie_ctx *ctx, int n, int32_t *out_tokens_dev);

/* ---- sparse-MoE models with FP8 experts ----------------------------------------------------------------
 * The "Extending to frontier MoE models" section of the Kog blog post ("the 2B demo vs frontier scale" in the
 * Creeta write-up) projects the monokernel onto sparse mixture-of-experts models with FP8 weights; the pages
 * give no kernel for it. This library reads it as: the FFN of every layer is n_experts SwiGLU experts of width
 * cfg->ffn_dim; a router (fp16 [n_experts, d_model]) scores the FFN-normalised vector u, the top_k experts are
 * taken (largest logit first, the lowest id among equal logits) and weighted by the softmax of their logits;
 * expert weights are OCP FP8 E4M3 ("fn": no infinities, max 448) codes, one fp32 scale per row, the weight
 * being code value * row scale. out = sum over the routed experts j of w_j * Wd_j (silu(Wg_j u) * (Wu_j u)).
 * Attention, norms, embedding and LM head are those of the dense model. Decode runs the same monokernel with
 * the router folded by linearity into the QKV and WO phases (its logits are inv_rms(h) * (R diag(g) x +
 * R diag(g) Wo o), the two products precomputed in fp32 at creation), the top_k selection right after the WO
 * barrier (ranked on the unnormalised sums, whose order the positive factor inv_rms(h) does not change, so the
 * experts are known before h is staged; the routing weights follow once inv_rms(h) is), and the two expert
 * projections as grid phases: after the selection the producer streams only the routed experts' FP8 tiles, the
 * down projection's once the gate/up tiles have landed.
 *
 * Requirements: 1 <= n_experts <= 256, 1 <= top_k <= min(8, n_experts), d_model and ffn_dim multiples of 16.
 * Prefill of a MoE ctx runs the prompt through the decode kernel one position after another (teacher forcing,
 * LM head at the last position only), in one launch per call. kie_decode_noalloc serves MoE ctxs too. */
typedef struct {
  int n_experts, top_k;
} kie_moe_config;

/* Host MoE weights: arrays of n_layers host pointers. router[l] fp16 bits [n_experts, d_model];
 * gate_q[l], up_q[l] E4M3 codes [n_experts, ffn_dim, d_model]; down_q[l] codes [n_experts, d_model, ffn_dim];
 * gate_s[l], up_s[l] fp32 row scales [n_experts, ffn_dim]; down_s[l] [n_experts, d_model]. The kie_weights
 * passed alongside supply everything else; its w_gate, w_up and w_down are not read (may be NULL).
 * Ownership: read during creation only. */
typedef struct {
  const uint16_t *const *router;
  const uint8_t *const *gate_q, *const *up_q, *const *down_q;
  const float *const *gate_s, *const *up_s, *const *down_s;
} kie_moe_weights;

/* kie_query_buffers for a sparse-MoE model (errors: INVALID for an unsupported cfg or moe, CUDA). */
int kie_query_buffers_moe(const kie_config *cfg, const kie_moe_config *moe, int n_cta, kie_buffer_sizes *out);

/* kie_create / kie_create_with_buffers for a sparse-MoE model: the expert matrices are packed per CTA in
 * 512-code column blocks (kie_packed_offset_fp8), gate and up rows interleaved; the router is stored folded
 * (R diag(g) and R diag(g) Wo, fp32, the second product accumulated in fp64 on the device) and the FFN gains
 * as given (the gain multiplies the staged vector, not the FP8 weights). */
int kie_create_moe(const kie_config *cfg, const kie_moe_config *moe, const kie_weights *w, const kie_moe_weights *mw,
                   void *stream, kie_ctx **out);
int kie_create_moe_with_buffers(const kie_config *cfg, const kie_moe_config *moe, const kie_weights *w,
                                const kie_moe_weights *mw, void *stream, void *weights_dev, size_t weights_bytes,
                                void *kv_dev, size_t kv_bytes, void *workspace_dev, size_t workspace_bytes,
                                kie_ctx **out);

/* Host-side layout query (no GPU needed): byte offset of code Q[r][c] inside a packed FP8 matrix [M, K]
 * (column blocks of 512 codes, each CTA's rows in tiles of up to 32 rows; within a full 512-code block the
 * 16-code chunk q of an odd row r is stored at chunk q ^ 4). M even, K a multiple of 16; -1 for bad
 * arguments. */
int64_t kie_packed_offset_fp8(int M, int K, int n_cta, int r, int c);

/* Host-side layout query (no GPU needed): byte offset of W[r][c] inside the prefill's tensor-core copy of an
 * [M, K] fp16 matrix: 128-row x 64-column tiles of 16 KB (rows padded to 128, columns to 64), tile (i, j) at
 * (i * ceil(K / 64) + j) * 16 KB, inside a tile 8 x 8 core matrices of 128 contiguous bytes (the canonical
 * K-major layout the tensor-core instructions read without swizzle). -1 for bad arguments. */
int64_t kie_tc_tile_offset(int M, int K, int r, int c);

/* Host-side layout query (no GPU needed): element offset of W[r][c] inside the packed matrix. */
int64_t kie_packed_offset(int M, int K, int n_cta, int r, int c);

/* Host-side layout query: first and one-past-last row owned by CTA `cta` (pairs of rows are never split). */
int kie_rows_of_cta(int M, int n_cta, int cta, int *r0, int *r1);

#ifdef __cplusplus
}
#endif
#endif /* KIE_H */
