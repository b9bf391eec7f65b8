// sparse_attn_simt.cu -- CUDA-core sparse_attn: one warp per (query, head), online softmax.
//
// "Module attn", sparse_attn (softmax over the gathered rows plus the sink, the sink in the
// denominator only, f32, bf16 out); "DeepSeek V4.1", attention/attend, sparse_attn_kernel (rows
// gathered by index, -1 skipped, running max and sum, the same rows reused as values).
//
// Each warp owns one (sequence, query, head).  A lane holds D/32 contiguous elements of q and of
// the running output, so every gathered row is one coalesced D*2-byte warp load.  The CTA's 8
// warps are 8 heads of the same query, so a row fetched by one warp is an L1/L2 hit for the rest.
// This is the simple path for shapes the tensor-core kernel does not take.
#include "common.cuh"

namespace dsattn {
namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 4;

template <int D>
__device__ __forceinline__ void load_slice(const uint16_t *row, float (&x)[D / 32]) {
    constexpr int E = D / 32;  // bf16 elements per lane
    if constexpr (E % 8 == 0) {
#pragma unroll
        for (int k = 0; k < E / 8; ++k) {
            const uint4 v = reinterpret_cast<const uint4 *>(row)[k];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[8 * k + 2 * i] = bf16_lo(w[i]);
                x[8 * k + 2 * i + 1] = bf16_hi(w[i]);
            }
        }
    } else if constexpr (E == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(row);
        x[0] = bf16_lo(v.x);
        x[1] = bf16_hi(v.x);
        x[2] = bf16_lo(v.y);
        x[3] = bf16_hi(v.y);
    } else {
        static_assert(E == 2, "D must be 64, 128, 256 or 512");
        const uint32_t v = *reinterpret_cast<const uint32_t *>(row);
        x[0] = bf16_lo(v);
        x[1] = bf16_hi(v);
    }
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) sparse_attn_simt_kernel(AttnArgs a) {
    constexpr int E = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hh = blockIdx.x * kWarps + warp;
    const int t = blockIdx.y;
    const int64_t bi = blockIdx.z;
    if (hh >= a.h) return;
    const int64_t tok = bi * a.m + t;

    float qf[E];
    load_slice<D>(a.q + (tok * a.h + hh) * D + lane * E, qf);
    const int32_t *irow = a.idx + tok * a.topk;
    const uint16_t *kvb = a.kv + bi * a.n * D + lane * E;

    float run_max = -INFINITY, run_sum = 0.0f, acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.0f;

    for (int j0 = 0; j0 < a.topk; j0 += kUnroll) {
        int v[kUnroll];
        float kf[kUnroll][E];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            v[u] = (j0 + u < a.topk) ? __ldg(irow + j0 + u) : -1;
            if (v[u] >= a.n) {
                if (lane == 0) flag_status(a.status, DS_DEV_BAD_INDEX);
                v[u] = -1;
            }
            if (v[u] >= 0) load_slice<D>(kvb + (int64_t)v[u] * D, kf[u]);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (v[u] < 0) continue;  // warp-uniform
            float dot = 0.0f;
#pragma unroll
            for (int i = 0; i < E; ++i) dot = fmaf(qf[i], kf[u][i], dot);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const float sc = dot * a.scale;
            const float new_max = fmaxf(run_max, sc);
            const float corr = expf(run_max - new_max);  // 0 on the first valid row
            const float p = expf(sc - new_max);
            run_sum = run_sum * corr + p;
#pragma unroll
            for (int i = 0; i < E; ++i) acc[i] = fmaf(p, kf[u][i], acc[i] * corr);
            run_max = new_max;
        }
    }

    // the sink joins the denominator only
    const float sink = a.sink[hh];
    const float top = fmaxf(run_max, sink);
    const float w = (run_max == -INFINITY) ? 0.0f : expf(run_max - top);
    const float inv = w / (run_sum * w + expf(sink - top));
    uint16_t *orow = a.o + (tok * a.h + hh) * D + lane * E;
#pragma unroll
    for (int i = 0; i < E; i += 2) {
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i] * inv));
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i + 1] * inv));
        reinterpret_cast<uint32_t *>(orow)[i / 2] = lo | (hi << 16);
    }
}

}  // namespace

int launch_sparse_attn_simt(const AttnArgs &a, cudaStream_t stream) {
    if ((int64_t)a.b * a.m == 0) return DS_OK;
    const dim3 grid((a.h + kWarps - 1) / kWarps, a.m, a.b);
    switch (a.d) {
        case 64: sparse_attn_simt_kernel<64><<<grid, kWarps * 32, 0, stream>>>(a); break;
        case 128: sparse_attn_simt_kernel<128><<<grid, kWarps * 32, 0, stream>>>(a); break;
        case 256: sparse_attn_simt_kernel<256><<<grid, kWarps * 32, 0, stream>>>(a); break;
        case 512: sparse_attn_simt_kernel<512><<<grid, kWarps * 32, 0, stream>>>(a); break;
        default: return DS_EUNSUPPORTED;
    }
    return launch_status();
}

}  // namespace dsattn
