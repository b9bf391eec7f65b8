// indexer.cu -- the Indexer's scores and top-k selection of compressed positions.
//
// What it computes ("DeepSeek V4.1", attention/query-latent, Indexer.forward): for query i of
// sequence bi (at position start_pos + i) and every compressed position t it can see,
//     score[t] = sum_h relu(q[bi][i][h] . k[bi][t]) * w[bi][i][h]
// where the query may see t < lens_i = (start_pos + i + 1) / ratio (the other positions score
// -inf).  Then the kk = min(topk, (start_pos + s) / ratio) best positions are kept, re-sorted into
// position order; a kept position >= lens_i becomes -1, the others are shifted by `offset`.
// Scores are f32 (the reading shared with the V3.2 page's index kernel: f32 logits, f32 relu x
// weight, f32 sum over heads); equal scores at the cut go to the smaller position.
//
// How (GB300-first):
//  * Scores are a dense contraction: 128 keys of one sequence form the MMA's M (TMEM lanes) and the
//    index heads of one or more queries of that sequence form N, so one tcgen05 MMA chain of D / 16
//    steps gives a 128 x N tile of dot products in TMEM.  Keys are contiguous rows, so a TMA tile
//    load with 128-byte swizzle lands each 64-column chunk directly in the operand layout; the
//    query block (N rows) is loaded the same way once per CTA.
//  * The epilogue is one thread per key (TMEM lane): it reads its N dot products, applies relu and
//    the head weights and sums over the heads in registers, so the reduction over heads needs no
//    exchange between threads; one coalesced f32 store per key and query.
//  * Selection is a per-query radix select on order-preserving integer keys (four 8-bit digit
//    passes over the row's scores in L2), then one pass that writes the positions above the cut
//    and the first ties at the cut, in position order, through a block-wide scan of per-thread
//    counts.
//  * Warp roles of the score kernel: 0 .. NEPI-1 epilogue (thread = key = TMEM lane; with
//    NEPI = 8 two warps share each lane quarter and split the block's queries), then the TMA
//    producer (one lane) and TMEM allocation + MMA issue (one lane).  Every wait is bounded (2 s), after
//    which the CTA flags DS_DEV_TIMEOUT, lets its issued MMAs finish, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace dsattn {
namespace ix {

using namespace ptx;

constexpr int BM = 128;             // keys per tile: M of the MMA, TMEM lanes
constexpr int NSTAGE_MAX = 4;       // key tiles in flight, at most (barrier slots)
// warps: NEPI epilogue warps (4, or 8 when a query block holds several queries), the TMA producer,
// the MMA warp
template <int NEPI>
struct Roles {
    static constexpr int W_TMA = NEPI, W_MMA = NEPI + 1;
    static constexpr int NTHREADS = (NEPI + 2) * 32;
};
constexpr int CHUNK_TILES_MAX = 16; // key tiles per CTA, at most (2048 keys)
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <int D>
struct Cfg {
    static constexpr int NCH = D / 64;                 // 128-byte column chunks per row
    static constexpr int TILE_BYTES = BM * D * 2;      // one key tile
    static constexpr int SM_K = 0;
    // the query block (N rows) follows the nstage key stages; then its weights and the barriers.
    // Dynamic shared memory for a block of N rows (1024 bytes of slack for the operand alignment).
    static constexpr int smem_bytes(int N, int nstage) { return nstage * TILE_BYTES + N * D * 2 + N * 4 + 256 + 1024; }
};

// Stages for a query block of N rows: blocks of up to 128 rows take two, so two CTAs share an SM
// (shared memory and TMEM both allow it) and one's set-up and latencies overlap the other's work;
// wider blocks take four.
constexpr int stages_for(int N) { return N <= 128 ? 2 : NSTAGE_MAX; }

// barrier slots (8 bytes each)
enum : int { B_FULL = 0, B_EMPTY = B_FULL + NSTAGE_MAX, B_AFULL = B_EMPTY + NSTAGE_MAX, B_AFREE = B_AFULL + 2,
             B_Q = B_AFREE + 2, B_DRAIN = B_Q + 1, B_COUNT = B_DRAIN + 1 };
constexpr int TMEM_ADDR_OFF = 8 * B_COUNT;
constexpr int ABORT_OFF = TMEM_ADDR_OFF + 4;
static_assert(ABORT_OFF + 4 <= 256, "barrier block");

struct ScoreParams {
    const float *w;          // [b][s][H]
    float *scores;           // [b][s] rows of ld floats
    int64_t ld;
    int64_t T;               // key rows per sequence in k
    int64_t Tv;              // positions scored: (start_pos + s) / ratio
    int64_t start_pos;
    int b, s, H, QB, N;      // N = QB * H: MMA N, columns of one accumulator
    int ratio;
    int nchunks;             // CTAs per query block along the keys
    int chunk_tiles;         // key tiles per CTA
    int nstage;              // key stages (stages_for(N))
    uint32_t tmem_cols;
    unsigned int *status;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// tcgen05.ld of 16 consecutive 32-bit columns (32 lanes x 16 columns, thread = lane)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

template <int D, int NEPI>
__global__ void __launch_bounds__(Roles<NEPI>::NTHREADS, 2)
    indexer_scores_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                          const ScoreParams p) {
    using C = Cfg<D>;
    constexpr int W_TMA = Roles<NEPI>::W_TMA, W_MMA = Roles<NEPI>::W_MMA;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);
    const int NSTAGE = p.nstage;
    const uint32_t SM_Q = (uint32_t)(NSTAGE * C::TILE_BYTES);
    float *w_s = reinterpret_cast<float *>(sbase + SM_Q + p.N * D * 2);
    const uint32_t bars = base + SM_Q + p.N * D * 2 + p.N * 4;   // 8-byte aligned (N * 4 multiple of 64)
    uint8_t *bar_p = sbase + (bars - base);
    auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_p + ABORT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA: query block qb (queries i0 .. i0 + QB - 1 of sequence bi), key tiles [j0, j1)
    const int nqb = (p.s + p.QB - 1) / p.QB;
    const int64_t qb = blockIdx.x / p.nchunks;
    const int chunk = (int)(blockIdx.x % p.nchunks);
    const int bi = (int)(qb / nqb);
    const int i0 = (int)(qb % nqb) * p.QB;
    const int nq = min(p.QB, p.s - i0);
    const int64_t ntiles = (p.Tv + BM - 1) / BM;
    const int64_t j0 = (int64_t)chunk * p.chunk_tiles;
    const int64_t j1 = min(j0 + p.chunk_tiles, ntiles);
    // keys the block's last query can see: tiles from there on are all -inf
    int64_t lens_max = (p.start_pos + i0 + nq) / p.ratio;
    if (lens_max > p.Tv) lens_max = p.Tv;
    const int64_t jl = max(j0, min(j1, (lens_max + BM - 1) / BM));   // live tiles: [j0, jl)
    const int nlive = (int)(jl - j0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(BAR(B_FULL + i), 1);
            mbar_init(BAR(B_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(B_AFULL + i), 1);
            mbar_init(BAR(B_AFREE + i), NEPI);  // one arrival per epilogue warp
        }
        mbar_init(BAR(B_Q), 1);
        mbar_init(BAR(B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA && nlive > 0) {
        tmem_alloc(bars + TMEM_ADDR_OFF, p.tmem_cols);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(bar_p + TMEM_ADDR_OFF);
    grid_dependency_wait();

    if (warp == W_TMA) {
        if (lane == 0 && nlive > 0) {
            // the query block: rows (bi, i0 .. i0 + QB - 1, every head), chunk c at SM_Q + c * N * 128
            mbar_arrive_expect_tx(BAR(B_Q), (uint32_t)(p.N * D * 2));
            const int32_t qrow = (int32_t)(((int64_t)bi * p.s + i0) * p.H);
            for (int c = 0; c < C::NCH; ++c) tma_load_2d(base + SM_Q + c * p.N * 128, &qmap, c * 64, qrow, BAR(B_Q));
            for (int it = 0; it < nlive; ++it) {
                const int st = it % NSTAGE;
                if (!mbar_wait(BAR(B_EMPTY + st), ((it / NSTAGE) & 1) ^ 1, abort_flag, kWaitLimitNs)) break;
                mbar_arrive_expect_tx(BAR(B_FULL + st), (uint32_t)C::TILE_BYTES);
                const int32_t krow = (int32_t)((int64_t)bi * p.T + (j0 + it) * BM);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_2d(base + C::SM_K + st * C::TILE_BYTES + c * BM * 128, &kmap, c * 64, krow, BAR(B_FULL + st));
            }
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        if (lane == 0 && nlive > 0) {
            const uint32_t idesc = idesc_bf16_f32(BM, p.N, false);
            bool ok = mbar_wait(BAR(B_Q), 0, abort_flag, kWaitLimitNs);
            for (int it = 0; ok && it < nlive; ++it) {
                const int st = it % NSTAGE, acc = it & 1;
                if (!mbar_wait(BAR(B_FULL + st), (it / NSTAGE) & 1, abort_flag, kWaitLimitNs)) break;
                if (!mbar_wait(BAR(B_AFREE + acc), ((it >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs)) break;
                tc_fence_after();
                const uint32_t kb = base + C::SM_K + st * C::TILE_BYTES;
                const uint32_t qbase = base + SM_Q;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    // 16 columns = 32 bytes inside the 128-byte swizzle atom of chunk k / 4
                    const uint64_t adesc = smem_desc_sw128(kb + (k >> 2) * BM * 128 + (k & 3) * 32, 16, 1024);
                    const uint64_t bdesc = smem_desc_sw128(qbase + (k >> 2) * p.N * 128 + (k & 3) * 32, 16, 1024);
                    mma_bf16_ss(tmem + (uint32_t)(acc * p.N), adesc, bdesc, idesc, k > 0 ? 1u : 0u);
                }
                mma_commit(BAR(B_EMPTY + st));
                mma_commit(BAR(B_AFULL + acc));
            }
            if (*abort_flag) {   // let issued MMAs finish before TMEM is freed
                mma_commit(BAR(B_DRAIN));
                mbar_wait_drain(BAR(B_DRAIN), 0, 100000000ull);
            }
        }
        __syncwarp();
    } else if (warp < NEPI) {
        // ===================================== epilogue =====================================
        const int tid = (warp & 3) * 32 + lane;           // key within the tile = TMEM lane
        for (int e = threadIdx.x; e < nq * p.H; e += 32 * NEPI) w_s[e] = p.w[((int64_t)bi * p.s + i0) * p.H + e];
        named_bar_sync(1, 32 * NEPI);
        // the warps of a lane quarter split the block's queries: warp w takes qi = w / 4 + k NEPI / 4
        constexpr int QSTEP = NEPI / 4;
        const int qg = warp / 4;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        float *srow = p.scores + ((int64_t)bi * p.s + i0) * p.ld;
        for (int it = 0; it < nlive; ++it) {
            const int acc = it & 1;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_AFULL + acc), (it >> 1) & 1, abort_flag, kWaitLimitNs));
            if (!ok) break;
            tc_fence_after();
            const int64_t t = (j0 + it) * BM + tid;
            for (int qi = qg; qi < nq; qi += QSTEP) {
                float sum = 0.0f;
                // up to 64 heads per wait: four 16-column loads in flight, then one wait
                for (int h0 = 0; h0 < p.H; h0 += 64) {
                    uint32_t r[4][16];
                    const uint32_t col = tmem + lane_off + (uint32_t)(acc * p.N + qi * p.H + h0);
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (h0 + 16 * g < p.H) tmem_ld16(col + 16 * g, r[g]);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int j = 0; j < 16; ++j) asm volatile("" : "+r"(r[g][j]));
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (h0 + 16 * g >= p.H) break;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float dot = __uint_as_float(r[g][j]);
                            sum = __fadd_rn(sum, __fmul_rn(dot > 0.0f ? dot : 0.0f, w_s[qi * p.H + h0 + 16 * g + j]));
                        }
                    }
                }
                const int64_t lens = (p.start_pos + i0 + qi + 1) / p.ratio;
                if (t < p.Tv) srow[qi * p.ld + t] = t < lens ? sum : -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_AFREE + acc));
        }
        // tiles no query of the block can see yet
        for (int64_t t = jl * BM + tid; t < min(j1 * BM, p.Tv); t += 128)
            for (int qi = qg; qi < nq; qi += QSTEP) srow[qi * p.ld + t] = -INFINITY;
    }

    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, DS_DEV_TIMEOUT);
    if (warp == W_MMA && nlive > 0) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

// ------------------------------------------------------------------------------------------------
// selection
// ------------------------------------------------------------------------------------------------
// Order-preserving key of an f32 score: larger score, larger key; -0 and +0 are one value.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum of one int per thread (NT threads); also returns the total.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int *warp_sums, int &total) {
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
        int s = lane < NT / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < NT / 32) warp_sums[lane] = s;   // inclusive
    }
    __syncthreads();
    total = warp_sums[NT / 32 - 1];
    const int before = warp > 0 ? warp_sums[warp - 1] : 0;
    __syncthreads();                                 // warp_sums may be reused right after
    return before + x - v;
}

// The digit of the rem-th largest key from a histogram of NBINS digits (digit NBINS - 1 largest):
// each thread sums NBINS / NT bins from the top, a block scan finds the thread whose bins hold the
// rank, and that thread walks them.  Writes the digit and the rank within it to *digit, *rank.
template <int NT, int NBINS>
__device__ __forceinline__ void find_digit(const int *hist, int rem, int *warp_sums, uint32_t *digit, int *rank) {
    constexpr int B = NBINS / NT;
    static_assert(B >= 1 && NBINS % NT == 0, "bins per thread");
    const int top = NBINS - 1 - threadIdx.x * B;     // this thread's bins: top, top - 1, ..., top - B + 1
    int c[B], sum = 0;
#pragma unroll
    for (int k = 0; k < B; ++k) {
        c[k] = hist[top - k];
        sum += c[k];
    }
    int total = 0;
    const int above = block_excl_scan<NT>(sum, warp_sums, total);
    if (above < rem && rem <= above + sum) {
        int acc = above;
#pragma unroll
        for (int k = 0; k < B; ++k) {
            if (acc + c[k] >= rem) {
                *digit = (uint32_t)(top - k);
                *rank = rem - acc;
                break;
            }
            acc += c[k];
        }
    }
    __syncthreads();
}

struct SelectParams {
    const float *scores;
    int64_t ld;
    int32_t *idx;
    int64_t Tv, start_pos, offset;
    int s, ratio, kk;
};

// Rows up to this many positions keep their order keys in shared memory (192 KB) for every pass;
// longer rows are read again from L2 in each pass.
constexpr int64_t kKeysInSmemMax = 49152;

template <int NT, bool SMEM>
__global__ void __launch_bounds__(NT) indexer_select_kernel(const SelectParams p) {
    extern __shared__ uint32_t keys_s[];   // SMEM: the order keys of positions [0, lens)
    __shared__ int hist[4096];
    __shared__ int warp_sums[NT / 32];
    __shared__ uint32_t s_digit;
    __shared__ int s_rank;
    constexpr int NW = NT / 32;
    grid_dependency_wait();   // the scores come from the previous kernel on the stream
    const int64_t row = blockIdx.x;
    const int i = (int)(row % p.s);
    int64_t lens = (p.start_pos + i + 1) / p.ratio;
    if (lens > p.Tv) lens = p.Tv;
    const float *sc = p.scores + row * p.ld;
    int32_t *out = p.idx + row * p.kk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (p.kk == 0) return;
    if (lens <= p.kk) {
        // every position the query sees is kept (the others score -inf and become -1)
        for (int j = tid; j < p.kk; j += NT) out[j] = j < lens ? (int32_t)(j + p.offset) : -1;
        return;
    }
    if constexpr (SMEM) {
        // sixteen loads in flight per thread before any store (a store right after its load would
        // make every element wait out a whole L2 round trip)
        constexpr int U = 16;
        for (int64_t t0 = 0; t0 < lens; t0 += (int64_t)NT * U) {
            float v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t t = t0 + (int64_t)u * NT + tid;
                v[u] = t < lens ? __ldg(sc + t) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t t = t0 + (int64_t)u * NT + tid;
                if (t < lens) keys_s[t] = order_key(v[u]);
            }
        }
        __syncthreads();
    }
    auto key_at = [&](int64_t t) -> uint32_t {
        if constexpr (SMEM) return keys_s[t];
        else return order_key(__ldg(sc + t));
    };
    // Radix select of the kk-th largest key among positions [0, lens) in three digits: bits 31-20
    // (sign, exponent and three mantissa bits: enough distinct values that the histogram atomics
    // seldom collide), bits 19-8, bits 7-0.  Only keys that match the digits found so far count.
    // Short rows (NT = 128) take four 8-bit digits instead: zeroing and scanning 4096 bins would
    // cost more than the extra pass over a few hundred keys.
    constexpr bool kWide = NT > 128;
    constexpr int kPasses = kWide ? 3 : 4;
    uint32_t prefix = 0, pmask = 0;
    int rem = p.kk;
#pragma unroll 1
    for (int pass = 0; pass < kPasses; ++pass) {
        const int shift = kWide ? (pass == 0 ? 20 : pass == 1 ? 8 : 0) : 24 - 8 * pass;
        const uint32_t dmask = kWide && pass < 2 ? 4095u : 255u;
        // the digit search reads at least max(NT, 256) bins: the unused ones must be zero too
        const int nbins = (int)dmask + 1 > (NT > 256 ? NT : 256) ? (int)dmask + 1 : (NT > 256 ? NT : 256);
        for (int j = tid; j < nbins; j += NT) hist[j] = 0;
        __syncthreads();
        for (int64_t t = tid; t < lens; t += NT) {
            const uint32_t key = key_at(t);
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1);
        }
        __syncthreads();
        if (dmask == 4095u) find_digit<NT, 4096>(hist, rem, warp_sums, &s_digit, &s_rank);
        else find_digit<NT, (NT > 256 ? NT : 256)>(hist, rem, warp_sums, &s_digit, &s_rank);
        prefix |= s_digit << shift;
        pmask |= dmask << shift;
        rem = s_rank;
        __syncthreads();
    }
    // prefix is the key of the kk-th largest score; rem of the positions with exactly that key
    // are kept, the first ones in position order.  Warp w owns a contiguous range of positions,
    // read 32 at a time (one per lane); ballots give each lane its rank among the kept ones.
    const int64_t segw = ((lens + NW - 1) / NW + 31) / 32 * 32;
    const int64_t a = min((int64_t)warp * segw, lens), z = min(a + segw, lens);
    int gt = 0, eq = 0;
    for (int64_t c = a; c < z; c += 32) {
        const int64_t t = c + lane;
        const uint32_t key = t < z ? key_at(t) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, t < z && key > prefix));
        eq += __popc(__ballot_sync(0xffffffffu, t < z && key == prefix));
    }
    int total = 0;
    // one value per warp (lane 0 carries it, the others 0) through the block scan
    const int tie0 = __shfl_sync(0xffffffffu, block_excl_scan<NT>(lane == 0 ? eq : 0, warp_sums, total), 0);
    const int take_eq = max(0, min(eq, rem - tie0));
    int pos = __shfl_sync(0xffffffffu, block_excl_scan<NT>(lane == 0 ? gt + take_eq : 0, warp_sums, total), 0);
    int tie = tie0;
    const uint32_t lt = (1u << lane) - 1u;
    for (int64_t c = a; c < z; c += 32) {
        const int64_t t = c + lane;
        const uint32_t key = t < z ? key_at(t) : 0u;
        const bool is_gt = t < z && key > prefix, is_eq = t < z && key == prefix;
        const uint32_t eqm = __ballot_sync(0xffffffffu, is_eq);
        const bool keep = is_gt || (is_eq && tie + __popc(eqm & lt) < rem);
        const uint32_t km = __ballot_sync(0xffffffffu, keep);
        if (keep) out[pos + __popc(km & lt)] = (int32_t)(t + p.offset);
        pos += __popc(km);
        tie += __popc(eqm);
    }
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_mutex;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

// A 2-D bf16 tensor map over `rows` rows of D values with 64-column x box_rows boxes, 128-byte
// swizzle (the MMA operand layout), zero fill past the last row.
bool make_map(CUtensorMap *map, const void *ptr, int64_t rows, int D, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t tmem_cols_for(int N) {
    uint32_t c = 32;
    while (c < (uint32_t)(2 * N)) c <<= 1;
    return c;
}

template <int D>
int launch_scores(const IndexerArgs &a, float *scores, int64_t ld, cudaStream_t stream) {
    using C = Cfg<D>;
    // queries per block: up to 128 rows of N (two CTAs per SM), at least one query
    const int qcap = a.H <= 128 ? 128 / a.H : 1;
    const int QB = a.s < qcap ? a.s : qcap;
    const int N = QB * a.H;
    const int64_t Tv = (a.start_pos + a.s) / a.ratio;
    if (Tv <= 0) return DS_OK;
    CUtensorMap kmap, qmap;
    if (!make_map(&kmap, a.k, (int64_t)a.b * a.T, D, BM)) return DS_ECUDA;
    if (!make_map(&qmap, a.q, (int64_t)a.b * a.s * a.H, D, N)) return DS_ECUDA;
    ScoreParams p;
    p.w = a.w;
    p.scores = scores;
    p.ld = ld;
    p.T = a.T;
    p.Tv = Tv;
    p.start_pos = a.start_pos;
    p.b = a.b;
    p.s = a.s;
    p.H = a.H;
    p.QB = QB;
    p.N = N;
    p.ratio = a.ratio;
    const int64_t ntiles = (Tv + BM - 1) / BM;
    // chunks short enough that the grid covers every SM twice (two CTAs share an SM in decode),
    // long enough that a CTA's set-up is spread over several tiles
    const int64_t nqb = (int64_t)a.b * ((a.s + QB - 1) / QB);
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t ct = (nqb * ntiles + 2 * sms - 1) / (2 * sms);
    ct = ct < 2 ? 2 : ct > CHUNK_TILES_MAX ? CHUNK_TILES_MAX : ct;
    p.chunk_tiles = (int)ct;
    p.nchunks = (int)((ntiles + ct - 1) / ct);
    p.tmem_cols = tmem_cols_for(N);
    p.status = a.status;
    const int64_t grid = nqb * p.nchunks;
    if (grid > 0x7fffffff) return DS_EUNSUPPORTED;
    p.nstage = stages_for(N);
    const int smem = C::smem_bytes(N, p.nstage);
    // a block of several queries: eight epilogue warps, two per lane quarter, each taking half the
    // queries (the epilogue's per-tile chain is what paces these shapes); one query: four
    const bool wide = QB >= 2;
    auto kernel = wide ? indexer_scores_kernel<D, 8> : indexer_scores_kernel<D, 4>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DS_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(wide ? Roles<8>::NTHREADS : Roles<4>::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, kmap, qmap, p) != cudaSuccess) return DS_ECUDA;
    return DS_OK;
}

template <int NT, bool SMEM>
int launch_select_variant(const SelectParams &p, int64_t rows, cudaStream_t stream) {
    const size_t smem = SMEM ? (size_t)p.Tv * sizeof(uint32_t) : 0;
    if (SMEM && smem > 48 * 1024 &&
        cudaFuncSetAttribute(indexer_select_kernel<NT, SMEM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kKeysInSmemMax * sizeof(uint32_t))) != cudaSuccess)
        return DS_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, indexer_select_kernel<NT, SMEM>, p) == cudaSuccess ? DS_OK : DS_ECUDA;
}

int launch_select(const float *scores, int64_t ld, const IndexerArgs &a, int32_t *idx, cudaStream_t stream) {
    const int64_t Tv = (a.start_pos + a.s) / a.ratio;
    SelectParams p;
    p.scores = scores;
    p.ld = ld;
    p.idx = idx;
    p.Tv = Tv;
    p.start_pos = a.start_pos;
    p.offset = a.offset;
    p.s = a.s;
    p.ratio = a.ratio;
    p.kk = (int)(a.topk < Tv ? a.topk : Tv);
    const int64_t rows = (int64_t)a.b * a.s;
    if (rows == 0 || p.kk == 0) return DS_OK;
    if (rows > 0x7fffffff) return DS_EUNSUPPORTED;
    // short rows: a small block per row; longer rows: 512 threads, keys in shared memory when they fit
    if (Tv <= 1024) return launch_select_variant<128, true>(p, rows, stream);
    if (Tv <= kKeysInSmemMax) return launch_select_variant<512, true>(p, rows, stream);
    return launch_select_variant<512, false>(p, rows, stream);
}

}  // namespace ix

int launch_indexer_scores(const IndexerArgs &a, float *scores, int64_t ld, cudaStream_t stream) {
    switch (a.D) {
        case 64: return ix::launch_scores<64>(a, scores, ld, stream);
        case 128: return ix::launch_scores<128>(a, scores, ld, stream);
        default: return DS_EUNSUPPORTED;
    }
}

int launch_indexer_select(const float *scores, int64_t ld, const IndexerArgs &a, int32_t *idx, cudaStream_t stream) {
    return ix::launch_select(scores, ld, a, idx, stream);
}

}  // namespace dsattn
