// sparse_attn_ot.cuh -- the one-CTA sparse_attn kernel for up to 64 heads of width 512
// (sparse_attn_ot.cu), as dispatched from sparse_attn_tc.cu.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace dsattn {

// The shapes the kernel is built for: head_dim 512, at most 64 heads, bf16 rows, one query per
// work unit (with or without the fused inverse RoPE of the output).
bool sparse_attn_ot_supports(int h, int d, bool fp8, bool pair);
// Whether it is the choice for ntok work units: wherever it is built for the shape (measured
// faster than the cluster kernel on decode batches and on a 4096-query prefill chunk).
bool sparse_attn_ot_preferred(int64_t ntok);
// Kernels a launch enqueues: 1, or 2 when a combine kernel merges tokens cut across CTAs.
int sparse_attn_ot_launches(int64_t ntok, int topk);
// Workspace for its partials (0 when no token is cut).
size_t sparse_attn_ot_workspace_bytes(int64_t ntok, int topk);
int launch_sparse_attn_ot(const AttnArgs &a, cudaStream_t stream, bool stall_first_tile);
// Test switch (ds_test_set_kernel): 0 automatic, 1 always the cluster kernel, 2 this kernel
// wherever it is built for the shape.
void set_test_kernel(int which);
// The kernels ds_sparse_attn runs for a bf16 call of this shape: returns how many it launches,
// stores 1 (cluster kernel) or 2 (one-CTA kernel) to *which and the workspace that kernel needs to
// *workspace (either pointer may be null).
int sparse_attn_plan(int b, int m, int h, int d, int topk, int *which, size_t *workspace);

}  // namespace dsattn
