// pair_union.cu -- the shared row list of two neighbouring queries, for the prefill attention that
// gathers once for both.
//
// In a prefill chunk ("DeepSeek V4.1", attention/attend, get_window_topk_idxs, prefill branch:
// query q sees the causal window max(0, q - W + 1) .. q; attention/query-latent, the Indexer
// re-sorts each query's compressed positions ascending), queries 2j and 2j + 1 of a sequence
// share all but one of their window rows and, once few compressed rows are visible, most of
// their compressed ones.  This kernel writes, for every such pair, the sorted union of the valid
// entries of the two index rows, each entry tagged with the queries that list it:
//     entry = row | (listed by query 2j) << 29 | (listed by query 2j + 1) << 30
// followed by -1 up to the union row's width (twice the index row's).  The attention kernel in
// pair mode then gathers each union row once for both queries and masks, per query, the rows
// that query did not list.
//
// One CTA per pair: the valid entries of each row are collected in shared memory, sorted
// (bitonic), duplicates within a row dropped (and flagged, DS_DEV_BAD_INDEX: this path counts a
// row once per query), then each entry's place in the union comes from a binary search in the
// other row and a prefix count of the rows the two lists share.
#include "common.cuh"
#include "ptx.cuh"

namespace dsattn {
namespace {

using ptx::grid_dependency_wait;

constexpr int UT = 256;                   // threads per pair
constexpr int32_t kBitA = 1 << 29, kBitB = 1 << 30;

// Block-wide exclusive prefix sum of one int per thread (UT threads).
__device__ __forceinline__ int excl_scan(int v, int *warp_sums, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = lane < UT / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < UT / 32) warp_sums[lane] = s;
    }
    __syncthreads();
    total = warp_sums[UT / 32 - 1];
    const int before = warp > 0 ? warp_sums[warp - 1] : 0;
    __syncthreads();
    return before + x - v;
}

// The valid entries (0 <= v < n) of one index row into buf[0..len), in any order; returns len.
// Entries >= n set *bad.
__device__ int collect(const int32_t *row, int topk, int64_t n, int32_t *buf, int *warp_sums, bool &bad) {
    int len = 0;
    for (int j0 = 0; j0 < topk; j0 += UT) {
        const int j = j0 + threadIdx.x;
        const int32_t v = j < topk ? __ldg(row + j) : -1;
        bad |= v >= 0 && (int64_t)v >= n;
        const bool keep = v >= 0 && (int64_t)v < n;
        int total = 0;
        const int pos = excl_scan(keep ? 1 : 0, warp_sums, total);
        if (keep) buf[len + pos] = v;
        len += total;
    }
    return len;
}

// Ascending bitonic sort of buf[0..len) in place, padded to a power of two with INT32_MAX.
__device__ void sort_block(int32_t *buf, int len, int cap) {
    int p2 = 1;
    while (p2 < len) p2 <<= 1;
    for (int i = len + threadIdx.x; i < p2 && i < cap; i += UT) buf[i] = INT32_MAX;
    __syncthreads();
    for (int k = 2; k <= p2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < p2; i += UT) {
                const int l = i ^ j;
                if (l > i) {
                    const int32_t a = buf[i], b = buf[l];
                    const bool up = (i & k) == 0;
                    if ((a > b) == up) {
                        buf[i] = b;
                        buf[l] = a;
                    }
                }
            }
            __syncthreads();
        }
}

// Drop repeated values from the sorted buf[0..len) (stable); returns the new length, sets *dup.
__device__ int dedupe(int32_t *buf, int len, int32_t *tmp, int *warp_sums, bool &dup) {
    int out = 0;
    for (int i0 = 0; i0 < len; i0 += UT) {
        const int i = i0 + threadIdx.x;
        const bool in = i < len;
        const bool first = in && (i == 0 || buf[i] != buf[i - 1]);
        dup |= in && !first;
        int total = 0;
        const int pos = excl_scan(first ? 1 : 0, warp_sums, total);
        if (first) tmp[out + pos] = buf[i];
        out += total;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < out; i += UT) buf[i] = tmp[i];
    __syncthreads();
    return out;
}

// number of values < x in the sorted a[0..len)
__device__ __forceinline__ int lower_bound(const int32_t *a, int len, int32_t x) {
    int lo = 0, hi = len;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(UT) pair_union_kernel(const int32_t *__restrict__ idx, int m, int topk, int64_t n,
                                                        int pairs_per_seq, int32_t *__restrict__ uidx, int cap,
                                                        unsigned int *status) {
    extern __shared__ int32_t sm[];
    int32_t *A = sm, *B = sm + cap, *W = sm + 2 * cap;    // W: scratch, then B's shared-row prefix
    __shared__ int warp_sums[UT / 32];
    grid_dependency_wait();
    const int64_t u = blockIdx.x;
    const int64_t bi = u / pairs_per_seq;
    const int qa = (int)(u % pairs_per_seq) * 2;
    const bool has_b = qa + 1 < m;
    const int32_t *rowa = idx + (bi * m + qa) * (int64_t)topk;
    bool bad = false, dup = false;
    int la = collect(rowa, topk, n, A, warp_sums, bad);
    int lb = has_b ? collect(rowa + topk, topk, n, B, warp_sums, bad) : 0;
    __syncthreads();
    sort_block(A, la, cap);
    sort_block(B, lb, cap);
    la = dedupe(A, la, W, warp_sums, dup);
    lb = dedupe(B, lb, W, warp_sums, dup);
    // DB[j] = rows among B[0..j) that A lists too (exclusive prefix over B)
    int32_t *DB = W;
    int carry = 0;
    for (int j0 = 0; j0 < lb; j0 += UT) {
        const int j = j0 + threadIdx.x;
        int shared_row = 0;
        if (j < lb) {
            const int r = lower_bound(A, la, B[j]);
            shared_row = r < la && A[r] == B[j];
        }
        int total = 0;
        const int pos = excl_scan(shared_row, warp_sums, total);
        if (j < lb) DB[j] = carry + pos;
        carry += total;
    }
    if (threadIdx.x == 0) DB[lb] = carry;
    __syncthreads();
    const int nshared = carry;
    const int U = la + lb - nshared;
    int32_t *out = uidx + u * (int64_t)(2 * topk);
    // A's entries: place = own rank + B's entries below it that A does not list
    for (int i = threadIdx.x; i < la; i += UT) {
        const int r = lower_bound(B, lb, A[i]);
        const bool both = r < lb && B[r] == A[i];
        out[i + r - DB[r]] = A[i] | kBitA | (both ? kBitB : 0);
    }
    // B's entries A does not list: place = A's entries below it + own rank among those not shared
    for (int j = threadIdx.x; j < lb; j += UT) {
        const int r = lower_bound(A, la, B[j]);
        if (!(r < la && A[r] == B[j])) out[r + j - DB[j]] = B[j] | kBitB;
    }
    for (int k = U + threadIdx.x; k < 2 * topk; k += UT) out[k] = -1;
    if (__syncthreads_or(bad || dup) && threadIdx.x == 0) flag_status(status, DS_DEV_BAD_INDEX);
}

}  // namespace

int pair_union_cap(int topk) {
    int cap = 1;
    while (cap < topk) cap <<= 1;
    return cap;
}

int launch_pair_union(const int32_t *idx, int b, int m, int topk, int64_t n, int32_t *uidx, unsigned int *status,
                      cudaStream_t stream) {
    const int pps = (m + 1) / 2;
    const int64_t npairs = (int64_t)b * pps;
    if (npairs == 0) return DS_OK;
    if (npairs > 0x7fffffff) return DS_EUNSUPPORTED;
    const int cap = pair_union_cap(topk);
    const size_t smem = (size_t)(3 * cap + 1) * sizeof(int32_t);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(pair_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DS_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)npairs, 1, 1);
    cfg.blockDim = dim3(UT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pair_union_kernel, idx, m, topk, n, pps, uidx, cap, status) == cudaSuccess
               ? DS_OK
               : DS_ECUDA;
}

}  // namespace dsattn
