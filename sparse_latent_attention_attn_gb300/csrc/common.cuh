// common.cuh -- shared device helpers of libdsattn (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsattn.h"

namespace dsattn {

// Launch helpers return DS_OK / DS_ECUDA.
inline int launch_status() { return cudaGetLastError() == cudaSuccess ? DS_OK : DS_ECUDA; }

__device__ __forceinline__ void flag_status(unsigned int *status, unsigned int bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// RoPE of one pair of bf16 values (low half first) by the table entry cs = (cos, sin), negated
// angle when inverse ("Module attn", apply_rotary: adjacent pairs as complex numbers, f32 products,
// bf16 result): a' = a c - b s, b' = a s + b c, each product and sum rounded to f32 on its own
// (no fused multiply-add), then each result rounded to bf16, nearest even.
__device__ __forceinline__ uint32_t rope_rotate_bf16x2(uint32_t w, float2 cs, bool inverse) {
    const float a = bf16_lo(w), b = bf16_hi(w);
    const float sn = inverse ? -cs.y : cs.y;
    const float re = __fsub_rn(__fmul_rn(a, cs.x), __fmul_rn(b, sn));
    const float im = __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, cs.x));
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(re)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(im)) << 16);
}

// ------------------------------------------------------------------------------------------
// Kernel entry points (defined in the per-kernel translation units).
// ------------------------------------------------------------------------------------------
int launch_window_idx(int32_t *idx, int64_t ld, int b, int rows, int cols, int64_t start_pos, int window,
                      cudaStream_t stream);
int launch_kv_quant_ring(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride, int b, int s,
                         int d, int64_t start_pos, int window, cudaStream_t stream);
int launch_kv_quant_ring_fp8(uint16_t *kv, int64_t kv_bstride, uint8_t *codes, int8_t *exps, int64_t ring_bstride,
                             int b, int s, int d, int64_t start_pos, int window, cudaStream_t stream);
int launch_kv_quantize_fp8(const uint16_t *x, int64_t rows, int d, uint8_t *codes, int8_t *exps,
                           cudaStream_t stream);
int launch_kv_rope_quant_ring(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride, int b,
                              int s, int d, int64_t start_pos, int window, int rd, const float *table,
                              cudaStream_t stream);
int launch_apply_rotary(uint16_t *x, int64_t rows, int row_len, int rd, int64_t rows_per_pos,
                        int64_t positions_per_seq, int64_t start_pos, const float *table, bool inverse,
                        cudaStream_t stream);

struct AttnArgs {
    const uint16_t *q;
    const uint16_t *kv;
    const uint8_t *kv8;    // non-null: gather from the fp8 row store (codes + exponents) instead
    const int8_t *kexp;
    int64_t n;
    const float *sink;
    const int32_t *idx;
    int topk;
    float scale;
    uint16_t *o;
    int b, m, h, d;
    void *workspace;
    size_t workspace_bytes;
    unsigned int *status;
    // inverse RoPE of the output, fused (rope == nullptr: none): the last rd values of o[bi][t][hh]
    // rotated back by the angle of position rope_pos0 + t, table rows of rd / 2 (cos, sin) pairs
    const float *rope = nullptr;
    int rd = 0;
    int64_t rope_pos0 = 0;
    // pair mode (prefill): idx holds the union rows of the query pairs (2j, 2j + 1), each 2 topk
    // wide with the listing queries in bits 29-30 of every entry (launch_pair_union); topk is
    // that width
    bool pair = false;
};

int launch_sparse_attn_tc(const AttnArgs &a, cudaStream_t stream);

struct IndexerArgs {
    const uint16_t *q;     // [b][s][H][D] bf16
    const uint16_t *k;     // [b][T][D] bf16
    const float *w;        // [b][s][H]
    int b, s, H, D;
    int64_t T;
    int64_t start_pos;
    int ratio;
    int topk;
    int64_t offset;
    unsigned int *status;
};
int launch_indexer_scores(const IndexerArgs &a, float *scores, int64_t ld, cudaStream_t stream);
int launch_indexer_select(const float *scores, int64_t ld, const IndexerArgs &a, int32_t *idx, cudaStream_t stream);
void set_test_stall(bool on);
size_t sparse_attn_tc_workspace_bytes(int b, int m, int h, int d, int topk, bool pair = false);
int pair_union_cap(int topk);
int launch_pair_union(const int32_t *idx, int b, int m, int topk, int64_t n, int32_t *uidx, unsigned int *status,
                      cudaStream_t stream);

}  // namespace dsattn
