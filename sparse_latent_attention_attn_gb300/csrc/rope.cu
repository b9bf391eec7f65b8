// rope.cu -- the rotation of the last rope_dim values of rows of bf16 values (RoPE and its
// inverse), as an elementwise kernel.
//
// "Module attn": apply_rotary (rotate the last rope_dim elements of each row at its position,
// adjacent pairs as complex numbers, f32 products, bf16 result; negated angle for the inverse),
// freqs_cis (the ratio-0 table of (cos, sin)) and the Precision paragraph; "DeepSeek V4.1",
// attention/query-latent, Attention.forward (RoPE on q and on the kv row, the inverse rotation
// on the attention output).
//
// One thread rotates 4 pairs (16 bytes of x): products and sums rounded one by one in f32 (no
// fused multiply-add), then rounded to bf16.  The (cos, sin) rows are shared by all rows at one
// position (all heads of a token) and stay in cache.  Memory-bound: 16 B read, 16 B written and
// 32 B of table read (mostly cached) per thread.
#include "common.cuh"

namespace dsattn {
namespace {

__global__ void __launch_bounds__(256) apply_rotary_kernel(uint16_t *__restrict__ x, int64_t rows, int row_len,
                                                           int rd, int64_t rows_per_pos, int64_t positions_per_seq,
                                                           int64_t start_pos, const float2 *__restrict__ table,
                                                           bool inverse) {
    const int per_row = rd / 8;                      // threads per row (4 pairs each)
    const int64_t total = rows * per_row;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / per_row;
        const int q = (int)(e % per_row);
        const int64_t pos = start_pos + (r / rows_per_pos) % positions_per_seq;
        uint4 *p4 = reinterpret_cast<uint4 *>(x + r * row_len + (row_len - rd) + q * 8);
        const uint4 v = *p4;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const float2 *cs = table + pos * (rd / 2) + q * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = rope_rotate_bf16x2(w[i], cs[i], inverse);
        *p4 = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

int launch_apply_rotary(uint16_t *x, int64_t rows, int row_len, int rd, int64_t rows_per_pos,
                        int64_t positions_per_seq, int64_t start_pos, const float *table, bool inverse,
                        cudaStream_t stream) {
    const int64_t total = rows * (rd / 8);
    if (total == 0) return DS_OK;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    apply_rotary_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, rows, row_len, rd, rows_per_pos, positions_per_seq,
                                                              start_pos, reinterpret_cast<const float2 *>(table),
                                                              inverse);
    return launch_status();
}

}  // namespace dsattn
