// sparse_attn_ot.cuh -- the one-CTA sparse_attn kernel for up to 64 heads of width 512
// (sparse_attn_ot.cu), as dispatched from sparse_attn_tc.cu.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace dsattn {

// The shapes the kernel is built for: head_dim 512, at most 64 heads, bf16 rows, plain output,
// one query per work unit.
bool sparse_attn_ot_supports(int h, int d, bool fp8, bool pair, bool rope);
// Whether it is the faster choice for ntok work units (fewer tokens than SMs: decode batches).
bool sparse_attn_ot_preferred(int64_t ntok);
// Workspace for its partials (0 when no token is cut).
size_t sparse_attn_ot_workspace_bytes(int64_t ntok, int topk);
int launch_sparse_attn_ot(const AttnArgs &a, cudaStream_t stream, bool stall_first_tile);
// Test switch (ds_test_set_kernel): 0 automatic, 1 always the cluster kernel, 2 this kernel
// wherever it is built for the shape.
void set_test_kernel(int which);

}  // namespace dsattn
