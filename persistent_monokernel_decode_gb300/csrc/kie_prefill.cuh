// Batched prefill (kie_prefill.cu): buffers and entry point shared with the C ABI.
#pragma once
#include <cuda_runtime.h>

#include "kie_decode.cuh"

namespace kie {

constexpr int PF_TOKENS = 128;  // prompt tokens per chunk

constexpr int PF_PART_SLICES = 6;  // K slices of a split projection, at most

// fp32 activations of one chunk (device): x, h [PF_TOKENS][d]; q, o [PF_TOKENS][Hq*dh]; a [PF_TOKENS][F];
// scale [PF_TOKENS] (per-token RMS scale); part [PF_PART_SLICES][PF_TOKENS][max rows of a split projection]
// (partial sums of K slices).
struct PrefillBufs {
  float *x, *h, *q, *o, *a, *scale, *part;
  int part_rows;  // rows of part: a projection is split only if it has at most this many
};

}  // namespace kie

// Enqueue the prefill of n tokens (device ids) at positions pos0 .. pos0+n-1 on `st`: the K/V cache rows, the
// logits of the last token (p.logits) and the next token to emit (p.persist->next_token).
cudaError_t kie_run_prefill(const kie::DecodeParams &p, const kie::PrefillBufs &b, const int *tok_dev, int pos0,
                            int n, cudaStream_t st);
