// kv_quant.cu -- fp8 round trip of new KV rows in place, fused with the ring-slot store.
//
// "Module attn": FP8_BLOCK (32 values per scale), pow2_ceil (power-of-two ceiling from the IEEE
// fields of an f32), act_quant_inplace (amax floored at 1e-4, scale = pow2_ceil(amax / 448),
// e4m3 with round-to-nearest-even and clamping, dequantised and rounded to bf16), the Precision
// paragraph (the round trip is bf16-exact) and the ring-cache paragraph (token at position p
// lives in slot p % window; a prefill keeps the last `window` tokens of the chunk).
//
// One thread owns one 32-value block (64 contiguous bytes): it loads the block once, decides
// the scale in f32 exactly as defined, converts pairs with the documented PTX conversion
// cvt.rn.satfinite.e4m3x2.f32 (round to nearest even, saturating at +-448) and widens back with
// cvt.rn.f16x2.e4m3x2 (exact), then stores the block in place and, when the token is among the
// last `window` of the chunk, into its ring slot.  Memory-bound: 64 B read, 64-128 B written.
//
// The fp8 row store keeps the same quantisation as its codes: the 32 e4m3 bytes of a block and
// the scale's exponent k (scale = 2^k), which decode to exactly the round-tripped bf16 values.
// The same block pass writes them to a ring held in such a store, or quantises plain rows.
#include "common.cuh"

namespace dsattn {
namespace {

__device__ __forceinline__ uint16_t e4m3x2_from_f32(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half((unsigned short)h));
}

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// One 32-value block (16 bf16 pairs, w in column order): the scale exactly as defined, then per
// pair the e4m3 codes (cvt.rn.satfinite.e4m3x2.f32: round to nearest even, saturating at
// +-448) and their exact widening back, multiplied by the scale and rounded to bf16 (exact).
// rt: the round-tripped pairs; codes: the 32 codes as bytes in column order; k: log2 of the scale.
__device__ __forceinline__ void quant_block32(const uint32_t (&w)[16], uint32_t (&rt)[16], uint32_t (&codes)[8],
                                              int &k) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    amax = fmaxf(amax, 1e-4f);
    // power-of-two ceiling of amax / 448 from its IEEE fields (positive, normal)
    const uint32_t rb = __float_as_uint(__fdiv_rn(amax, 448.0f));
    const uint32_t se = (rb >> 23) + ((rb & 0x7fffffu) ? 1u : 0u);   // biased exponent of scale
    const float scale = __uint_as_float(se << 23);
    const float inv_scale = __uint_as_float((254u - se) << 23);     // exact reciprocal
    k = (int)se - 127;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float y0 = fminf(fmaxf(bf16_lo(w[i]) * inv_scale, -448.0f), 448.0f);
        const float y1 = fminf(fmaxf(bf16_hi(w[i]) * inv_scale, -448.0f), 448.0f);
        const uint16_t c2 = e4m3x2_from_f32(y1, y0);                 // low byte: column 2i
        if (i % 2 == 0) codes[i / 2] = c2;
        else codes[i / 2] |= (uint32_t)c2 << 16;
        const uint32_t h2 = f16x2_from_e4m3x2(c2);
        const float q0 = f16_bits_to_f32(h2 & 0xffffu) * scale;
        const float q1 = f16_bits_to_f32(h2 >> 16) * scale;
        rt[i] = f32_to_bf16_bits(q0) | (f32_to_bf16_bits(q1) << 16);
    }
}

__device__ __forceinline__ void load_block32(const uint16_t *src, uint32_t (&w)[16]) {
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 v = s4[k];
        w[4 * k + 0] = v.x;
        w[4 * k + 1] = v.y;
        w[4 * k + 2] = v.z;
        w[4 * k + 3] = v.w;
    }
}

__device__ __forceinline__ void store_block32(uint16_t *dst, const uint32_t (&w)[16]) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int k = 0; k < 4; ++k) d4[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

// One row piece of 16 bf16 pairs rotated by the (cos, sin) pairs at cs: each pair a + ib times
// c + is in f32 with every product and sum rounded on its own (no fused multiply-add), then
// rounded to bf16 -- the order the RoPE definition writes.
__device__ __forceinline__ void rotate16(uint32_t (&w)[16], const float2 *__restrict__ cs, bool inverse) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = bf16_lo(w[i]), b = bf16_hi(w[i]);
        const float2 t = cs[i];
        const float sn = inverse ? -t.y : t.y;
        const float re = __fsub_rn(__fmul_rn(a, t.x), __fmul_rn(b, sn));
        const float im = __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, t.x));
        w[i] = f32_to_bf16_bits(re) | (f32_to_bf16_bits(im) << 16);
    }
}

// FP8RING: the ring is an fp8 row store (codes + exponents, ring_bstride in rows); otherwise a
// bf16 tensor (ring_bstride in elements) that receives the round-tripped row.  ROPE: the blocks
// of the last rd values of row t are first rotated to position start_pos + t (table: rows of
// rd / 2 (cos, sin) pairs), as the ratio-0 layer does before the round trip.
template <bool FP8RING, bool ROPE = false>
__global__ void __launch_bounds__(256) kv_quant_ring_kernel(uint16_t *__restrict__ kv, int64_t kv_bstride,
                                                            uint16_t *__restrict__ ring, uint8_t *__restrict__ codes,
                                                            int8_t *__restrict__ exps, int64_t ring_bstride,
                                                            int b, int s, int d, int64_t start_pos, int window,
                                                            int rd = 0, const float2 *__restrict__ table = nullptr) {
    // a kernel launched after this one as a programmatic dependent (the attention kernel) may be
    // scheduled as soon as every block of this grid is running; it still waits for this grid to
    // finish (griddepcontrol.wait) before it reads the ring
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int nblk = d / 32;
    const int64_t total = (int64_t)b * s * nblk;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(e % nblk);
        const int64_t r = e / nblk;
        const int t = (int)(r % s);
        const int64_t bi = r / s;
        uint16_t *src = kv + bi * kv_bstride + (int64_t)t * d + c * 32;
        uint32_t w[16], rt[16], cd[8];
        int k;
        load_block32(src, w);
        if constexpr (ROPE) {
            if (c * 32 >= d - rd)
                rotate16(w, table + (start_pos + t) * (rd / 2) + (c * 32 - (d - rd)) / 2, false);
        }
        quant_block32(w, rt, cd, k);
        store_block32(src, rt);
        if (t >= s - window) {
            const int64_t slot = (start_pos + t) % window;
            if constexpr (FP8RING) {
                const int64_t row = bi * ring_bstride + slot;
                uint4 *c4 = reinterpret_cast<uint4 *>(codes + row * d + c * 32);
                c4[0] = make_uint4(cd[0], cd[1], cd[2], cd[3]);
                c4[1] = make_uint4(cd[4], cd[5], cd[6], cd[7]);
                exps[row * nblk + c] = (int8_t)k;
            } else if (ring != nullptr) {
                store_block32(ring + bi * ring_bstride + slot * d + c * 32, rt);
            }
        }
    }
}

// rows x d values (row-major) into the fp8 row store: codes[rows][d], exps[rows][d / 32].
__global__ void __launch_bounds__(256) kv_quantize_fp8_kernel(const uint16_t *__restrict__ x, int64_t rows, int d,
                                                              uint8_t *__restrict__ codes, int8_t *__restrict__ exps) {
    const int nblk = d / 32;
    const int64_t total = rows * nblk;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        uint32_t w[16], rt[16], cd[8];
        int k;
        load_block32(x + e * 32, w);
        quant_block32(w, rt, cd, k);
        uint4 *c4 = reinterpret_cast<uint4 *>(codes + e * 32);
        c4[0] = make_uint4(cd[0], cd[1], cd[2], cd[3]);
        c4[1] = make_uint4(cd[4], cd[5], cd[6], cd[7]);
        exps[e] = (int8_t)k;
    }
}

int grid_for(int64_t total) {
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    return (int)blocks;
}

}  // namespace

int launch_kv_quant_ring(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride, int b, int s,
                         int d, int64_t start_pos, int window, cudaStream_t stream) {
    const int64_t total = (int64_t)b * s * (d / 32);
    if (total == 0) return DS_OK;
    kv_quant_ring_kernel<false><<<(unsigned)grid_for(total), 256, 0, stream>>>(
        kv, kv_bstride, ring, nullptr, nullptr, ring_bstride, b, s, d, start_pos, window);
    return launch_status();
}

int launch_kv_quant_ring_fp8(uint16_t *kv, int64_t kv_bstride, uint8_t *codes, int8_t *exps, int64_t ring_bstride,
                             int b, int s, int d, int64_t start_pos, int window, cudaStream_t stream) {
    const int64_t total = (int64_t)b * s * (d / 32);
    if (total == 0) return DS_OK;
    kv_quant_ring_kernel<true><<<(unsigned)grid_for(total), 256, 0, stream>>>(
        kv, kv_bstride, nullptr, codes, exps, ring_bstride, b, s, d, start_pos, window);
    return launch_status();
}

int launch_kv_rope_quant_ring(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride, int b,
                              int s, int d, int64_t start_pos, int window, int rd, const float *table,
                              cudaStream_t stream) {
    const int64_t total = (int64_t)b * s * (d / 32);
    if (total == 0) return DS_OK;
    kv_quant_ring_kernel<false, true><<<(unsigned)grid_for(total), 256, 0, stream>>>(
        kv, kv_bstride, ring, nullptr, nullptr, ring_bstride, b, s, d, start_pos, window, rd,
        reinterpret_cast<const float2 *>(table));
    return launch_status();
}

int launch_kv_quantize_fp8(const uint16_t *x, int64_t rows, int d, uint8_t *codes, int8_t *exps,
                           cudaStream_t stream) {
    const int64_t total = rows * (d / 32);
    if (total == 0) return DS_OK;
    kv_quantize_fp8_kernel<<<(unsigned)grid_for(total), 256, 0, stream>>>(x, rows, d, codes, exps);
    return launch_status();
}

}  // namespace dsattn
