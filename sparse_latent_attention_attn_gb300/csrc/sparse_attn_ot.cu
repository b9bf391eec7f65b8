// sparse_attn_ot.cu -- sparse_attn for up to 64 heads of width 512 on one CTA per work range, with
// the output accumulator transposed in tensor memory.
//
// What it computes is sparse_attn_tc.cu's operation ("Module attn", sparse_attn and the
// Precision paragraph; "DeepSeek V4.1", attention/attend, sparse_attn_kernel): for every query
// token and head, softmax over the index-listed rows of the shared latent KV tensor plus an
// attention sink that counts in the denominator only, the rows reused as values, f32 arithmetic,
// bf16 output; optionally with the inverse RoPE of the output fused in ("DeepSeek V4.1",
// attention/query-latent, Attention.forward).
//
// Why a second kernel: with head_dim 512 an accumulator O[heads x 512] in the usual orientation
// (heads as TMEM lanes) takes all 512 TMEM columns even when only 64 of the 128 lanes hold heads,
// which is why sparse_attn_tc.cu splits d over a 2-CTA cluster and exchanges partial scores.
// With at most 64 heads the transposed accumulator O^T[512 x heads] is dense instead: d is the
// lane (four chunks of 128) and the heads are 64 columns per chunk, 256 columns in all.  One CTA
// then holds the whole accumulator next to its score buffers, so there is no cluster, no score
// exchange and no partial scores; every row is gathered once, whole (1 KB), into one CTA.
//  * S = Q K^T: M = 64 heads (the 64-row MMA, whose rows land on lanes 0-15 of each TMEM lane
//    quarter), N = 64 index entries, K = 512; Q and the rows come from 128-byte-swizzled shared
//    memory (K-major).
//  * O^T += V^T P^T: M = 128 columns of d (one chunk), N = 64 heads, K = 64 entries; V^T is the
//    same row tile read MN-major (d contiguous), P^T is P written K-major by the softmax.
//  * The softmax runs two threads per head (the score layout's lane and, with half the columns
//    handed over by shuffles, the idle lane 16 above it); a rescale of the running max (lazy, as
//    in sparse_attn_tc.cu) multiplies the head's column of O^T, which every softmax thread does
//    for its lane (d) of the accumulator, after a vote among the four softmax warps.
//  * Tiles are 64 consecutive index entries, not compacted: -1 and out-of-range entries are
//    masked in the softmax (their rows are neither loaded nor counted).
//  * Work ranges, the cost line and the cut tokens are those of attn_split.cuh.  When every token
//    is split into the same 2-4 parts, a token's parts run as one cluster and merge their f32
//    accumulators among themselves; otherwise a cut token's parts leave f32 partials (O^T, running
//    max and sum) that a combine kernel merges with the sink.
//  * Warp roles (16 warps): 0-3 softmax, q loads and epilogue; 4-11 row gather (cp.async,
//    swizzled in flight); 12 TMEM allocation and single-thread MMA issue; 13-15 none (they
//    complete the last warpgroup, so the softmax warpgroup can take registers from the others).
//  * Every wait is bounded: past a time limit the kernel flags DS_DEV_TIMEOUT, drains its own
//    copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "attn_split.cuh"
#include "common.cuh"
#include "ptx.cuh"
#include "sparse_attn_ot.cuh"

namespace dsattn {
namespace ot {

using namespace ptx;
using split::kMaxCut;
using split::range_start;
using split::unit_at;

constexpr int D = 512;             // row width (head_dim)
constexpr int HM = 64;             // heads at most: M of Q K^T, N of V^T P^T
constexpr int BN = 64;             // index entries per tile
constexpr int NST = 2;             // row stages (64 KB each)
constexpr int NSB = 2;             // score buffers in TMEM
constexpr int NPB = 2;             // P buffers
constexpr int NCH = D / 64;        // 128-byte column chunks of a row
constexpr int CHUNK = 64 * 128;    // one chunk of 64 rows
constexpr int STAGE_BYTES = NCH * CHUNK;
constexpr int Q_BYTES = NCH * CHUNK;   // 64 head rows
constexpr int P_BYTES = HM * 128;      // P of one tile: 64 head rows of 64 bf16
constexpr int SM_Q = 0;
constexpr int SM_KV = SM_Q + Q_BYTES;
constexpr int SM_P = SM_KV + NST * STAGE_BYTES;
constexpr int SM_BAR = SM_P + NPB * P_BYTES;
constexpr int BAR_BYTES = 2048;
constexpr int SMEM_BYTES = SM_BAR + BAR_BYTES + 1024;   // + alignment of the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// TMEM columns: O^T chunk c (d = 128 c + lane) at columns [64 c, 64 c + 64), one per head; then
// the score buffers (64-row MMA: head r on lane 32 (r / 16) + r % 16, entry j on column j)
constexpr int O_COL = 0;
constexpr int S_COL = 4 * HM;
constexpr int TMEM_COLS = 512;
static_assert(S_COL + NSB * BN <= TMEM_COLS, "TMEM budget");

constexpr int NTHREADS = 512;      // 16 warps = 4 warpgroups (13-15 have no role)
constexpr int W_GATHER = 4;        // warps 4-11
constexpr int NGATHER = 256;
constexpr int W_MMA = 12;
// register split: softmax warpgroup 232, the other three 88 (128 * (232 + 3 * 88) = 63488 <= 65536)
constexpr uint32_t REG_SOFTMAX = 232, REG_OTHER = 88;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;           // log2 units

// A partial slot (f32): O^T of the token's part, element (head h, column d) at
// ((h / 4) * D + d) * 4 + h % 4, so a warp's stores and loads (consecutive d) are 512 contiguous
// bytes; then the running maxima (log2 domain, -inf: no row) and the sums of the 64 heads.
// The cluster merge uses one slot per CTA, chunk by chunk: element (h, 128 c + d) at
// c * 128 * HM + ((h / 4) * 128 + d) * 4 + h % 4.
constexpr int SLOT_O = HM * D;
constexpr size_t SLOT = (size_t)SLOT_O + 2 * HM;

// barrier slots (8 bytes each) in the SM_BAR block
enum : int {
    B_FULL = 0,                 // [NST] gather -> softmax, MMA: columns 0..255 of the rows and the mask landed
    B_FULH = B_FULL + NST,      // [NST] gather -> MMA: columns 256..511 of the rows landed
    B_EMPTY = B_FULH + NST,     // [NST] MMA -> gather: stage free (its P V is done)
    B_QFULL = B_EMPTY + NST,    // TMA -> MMA: q rows of the segment landed
    B_SFULL = B_QFULL + 1,      // [NSB] MMA -> softmax: scores ready
    B_SFREE = B_SFULL + NSB,    // [NSB] softmax -> MMA: score buffer read
    B_PFULL = B_SFREE + NSB,    // [NPB] softmax -> MMA: P of tile J written (slot J % NPB)
    B_PVDONE = B_PFULL + NPB,   // [4] MMA -> softmax: P V of tile J done (slot J % 4)
    B_OFREE = B_PVDONE + 4,     // softmax -> MMA: the epilogue has read O^T
    B_DRAIN = B_OFREE + 1,      // MMA drain on abort
    B_XCH = B_DRAIN + 1,        // cluster merge: the other CTAs' accumulator chunks are in the workspace
    B_COUNT = B_XCH + 1
};
constexpr int MASK_OFF = 256;                      // [NST] uint64: the tile's valid entries
constexpr int TMEM_ADDR_OFF = MASK_OFF + 8 * NST;
constexpr int ABORT_OFF = TMEM_ADDR_OFF + 4;
constexpr int VOTE_OFF = ABORT_OFF + 4;            // [2] int: tile number of a rescale request
constexpr int FAC_OFF = 512;                       // [64] f32: rescale factors
constexpr int INV_OFF = FAC_OFF + 4 * HM;          // [64] f32: 1 / denominator (whole tokens)
constexpr int WGT_OFF = INV_OFF + 4 * HM;          // [KC][64] f32: cluster merge weights (KC <= 4)
static_assert(8 * B_COUNT <= MASK_OFF && VOTE_OFF + 8 <= FAC_OFF && WGT_OFF + 16 * HM <= BAR_BYTES, "barrier block");

struct Params {
    const uint16_t *q;
    const uint16_t *kv;
    const float *sink;
    const int32_t *idx;
    uint16_t *o;
    float *ws;
    int64_t n;
    int64_t ntok;     // b * m tokens
    int topk;
    int m;
    int h;
    int G;            // CTAs (work ranges)
    int seg_cost;     // K of range_start, in entries
    bool interleave;  // unit order (unit_at): several queries per sequence
    float scale_log2; // softmax scale * log2(e)
    unsigned int *status;
    int stall_first_tile;   // test switch (ds_test_set_stall): withhold the first tile's arrivals
    // fused inverse RoPE of the output (ROPE kernels), see AttnArgs
    const float2 *rope;
    int rd;
    int64_t rope_pos0;
};

// Instruction descriptor of kind::f16: bf16 A and B, f32 accumulator, dense; A and B each
// K-major or MN-major (bits 15 and 16), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Named barrier over `n` threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// 16 zero bytes into shared memory through the cp.async path (source size 0: nothing is read), so
// they complete, and are counted, like the row copies beside them.
__device__ __forceinline__ void cp_async_zero16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster with release semantics at cluster scope:
// the arriving thread's earlier writes (and those it has observed) are visible to a thread that
// acquires the phase at cluster scope.
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t remote_bar) {
    asm volatile(
        "fence.acq_rel.cluster;\n\t"
        "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
        : "memory");
}

// TMA load of a 2-D box into shared memory, completing `bar` by the bytes it writes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The bf16 value of output column d (this lane) of one head: with ROPE, the last rd columns are
// rotated back as ds_apply_rotary would rotate the stored bf16 pairs.  Lanes d and d ^ 1 hold a
// pair (2j, 2j + 1); each packs the pair from its own value and its neighbour's (one shuffle, so
// every lane of the warp calls this when `warp_rotates`), rotates it and keeps its own half.
// cs_row: the token's table row (rd / 2 (cos, sin) pairs).
template <bool ROPE>
__device__ __forceinline__ uint16_t out_bf16(float x, int d, const float2 *cs_row, int rd, bool warp_rotates) {
    if constexpr (ROPE) {
        if (warp_rotates) {
            const float y = __shfl_xor_sync(0xffffffffu, x, 1);
            if (d >= D - rd) {
                const bool odd = (d & 1) != 0;
                const uint32_t v = odd ? pack_bf16x2(y, x) : pack_bf16x2(x, y);
                const uint32_t r = rope_rotate_bf16x2(v, __ldg(cs_row + (((d & ~1) - (D - rd)) >> 1)), true);
                return odd ? (uint16_t)(r >> 16) : (uint16_t)(r & 0xffffu);
            }
        }
    }
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort, kWaitLimitNs);
    return __all_sync(0xffffffffu, ok);
}

// The segments (token pieces) of a CTA's range, tile by tile.
struct TileIter {
    int64_t tok;      // position in the unit order
    int a, z;         // entries [a, z) of the token's index row
    int t, ntile;     // tile within the segment
    int seg;          // segment number within the range
    int J;            // tile number within the range
    bool valid;
    __device__ void start(int64_t tok0, int64_t e0, int64_t e1, int T) {
        tok = tok0;
        seg = 0;
        J = 0;
        t = 0;
        load(e0, e1, T);
    }
    __device__ void load(int64_t e0, int64_t e1, int T) {
        valid = T > 0 && e1 > e0 && tok * T < e1;
        if (!valid) return;
        a = (int)((e0 > tok * T ? e0 : tok * T) - tok * T);
        z = (int)((e1 < (tok + 1) * T ? e1 : (tok + 1) * T) - tok * T);
        ntile = (z - a + BN - 1) / BN;
    }
    __device__ void next(int64_t e0, int64_t e1, int T) {
        ++J;
        if (++t < ntile) return;
        t = 0;
        ++tok;
        ++seg;
        load(e0, e1, T);
    }
};

// qmap: q as [b m h rows][512] bf16, boxes of 64 columns x h rows, 128-byte swizzle (the MMA's
// operand layout).
// KC > 1: the grid is a cluster of KC CTAs per token, each taking an equal part of the token's
// index row; they merge their accumulators among themselves (no combine kernel): each CTA writes
// the 128-column chunks of O^T that other CTAs own (chunk c belongs to rank c % KC) with its
// running max and sum, tells the others through their XCH barriers, and finishes its own chunks.
// ROPE: the output's last rd columns are rotated back in the epilogue (ds_sparse_attn_rope).
template <int KC, bool ROPE>
__global__ void __launch_bounds__(NTHREADS, 1) sparse_attn_ot_kernel(const __grid_constant__ CUtensorMap qmap,
                                                                     const Params p) {
    static_assert(KC >= 1 && KC <= 4, "cluster merge of 2 to 4 parts");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);
    const uint32_t bars = base + SM_BAR;
    auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
    uint64_t *tile_mask = reinterpret_cast<uint64_t *>(sbase + SM_BAR + MASK_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + SM_BAR + ABORT_OFF);
    volatile int *vote = reinterpret_cast<volatile int *>(sbase + SM_BAR + VOTE_OFF);
    float *fac = reinterpret_cast<float *>(sbase + SM_BAR + FAC_OFF);
    float *inv_h = reinterpret_cast<float *>(sbase + SM_BAR + INV_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cid = blockIdx.x;
    const int T = p.topk;
    const int64_t e0 = range_start(cid, p.ntok, T, p.seg_cost, p.G);
    const int64_t e1 = range_start(cid + 1, p.ntok, T, p.seg_cost, p.G);
    const int64_t tok_begin = T > 0 ? e0 / T : 0;

    // ---- set-up --------------------------------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(BAR(B_FULL + s), NGATHER + 1);   // every gather thread's copies + the mask writer
            mbar_init(BAR(B_FULH + s), NGATHER);
            mbar_init(BAR(B_EMPTY + s), 1);
        }
        mbar_init(BAR(B_QFULL), 1);                    // armed with the q bytes; the TMA completes it
        for (int i = 0; i < NSB; ++i) {
            mbar_init(BAR(B_SFULL + i), 1);
            mbar_init(BAR(B_SFREE + i), 4);            // one arrival per softmax warp
        }
        for (int i = 0; i < NPB; ++i) mbar_init(BAR(B_PFULL + i), 4);
        for (int i = 0; i < 4; ++i) mbar_init(BAR(B_PVDONE + i), 1);
        mbar_init(BAR(B_OFREE), 128);
        mbar_init(BAR(B_DRAIN), 1);
        mbar_init(BAR(B_XCH), KC > 1 ? KC - 1 : 1);     // one arrival per other CTA of the cluster
        *abort_flag = 0;
        vote[0] = -1;
        vote[1] = -1;
        fence_mbar_init();
    }
    // the combine kernel may be scheduled as soon as SMs free up (it waits for this grid itself)
    if (threadIdx.x == 0) grid_launch_dependents();
    // q rows beyond h are multiplied but never used: zero them once, so they stay finite
    if (p.h < HM) {
        for (int i = threadIdx.x; i < NCH * (HM - p.h) * 8; i += NTHREADS) {
            const int c = i / ((HM - p.h) * 8), rest = i % ((HM - p.h) * 8);
            reinterpret_cast<uint4 *>(sbase + SM_Q + c * CHUNK + p.h * 128)[rest] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == W_MMA) {
        tmem_alloc(base + SM_BAR + TMEM_ADDR_OFF, TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sbase + SM_BAR + TMEM_ADDR_OFF);
    // everything above overlaps the previous kernel on the stream (launched as a programmatic
    // dependent); from here on the inputs it may have written are read, and outputs written
    grid_dependency_wait();
    // warpgroups 1-3 give registers back to the softmax warpgroup before they branch
    if (warp >= 4) setmaxnreg_dec<REG_OTHER>();

    if (warp >= W_GATHER && warp < W_GATHER + 8) {
        // ==================== row gather: cp.async into 128-byte-swizzled stages ====================
        // Warp gw copies rows gw, gw + 8, ..., gw + 56, first their columns 0..255 (16-byte units
        // u = lane), then columns 256..511 (u = 32 + lane), each half behind its own barrier, so
        // the MMA can start on the first half of d while the second is in flight.  Every warp
        // instruction moves half a row (512 contiguous bytes).  Unit u sits in column chunk u / 8,
        // swizzled to unit (u % 8) ^ (row % 8) of the row's 128 bytes.  A row the tile does not
        // load is masked in the softmax (P = 0) but still multiplied, so it must hold finite
        // values: at a stage's first use such rows are zeroed; later they keep an earlier tile's
        // rows.
        const int gw = warp - W_GATHER;
        const int u8 = lane & 7;
        const bool writer = gw == 0 && lane == 0;
        bool ok = true, bad = false;
        TileIter it;
        it.start(tok_begin, e0, e1, T);
        while (it.valid && ok) {
            const int64_t utok = unit_at(it.tok, p.ntok, p.interleave);
            // the tile's 64 index entries (every gather warp reads the same ones)
            const int32_t *irow = p.idx + utok * (int64_t)T;
            const int j0 = it.a + it.t * BN;
            const int cnt = it.z - j0 < BN ? it.z - j0 : BN;
            const int v0 = lane < cnt ? __ldg(irow + j0 + lane) : -1;
            const int v1 = lane + 32 < cnt ? __ldg(irow + j0 + 32 + lane) : -1;
            const bool in0 = v0 >= 0 && (int64_t)v0 < p.n, in1 = v1 >= 0 && (int64_t)v1 < p.n;
            bad |= (v0 >= 0 && !in0) || (v1 >= 0 && !in1);
            const uint32_t m0 = __ballot_sync(0xffffffffu, in0), m1 = __ballot_sync(0xffffffffu, in1);
            const int stage = it.J % NST;
            if (!warp_wait(BAR(B_EMPTY + stage), (uint32_t)((it.J / NST) & 1) ^ 1u, abort_flag)) {
                ok = false;
                break;
            }
            // the row numbers of this warp's 8 rows first (independent shuffles), then the copies
            int vr[BN / 8];
#pragma unroll
            for (int i = 0; i < BN / 8; ++i) {
                const int r = gw + 8 * i;
                vr[i] = __shfl_sync(0xffffffffu, r < 32 ? v0 : v1, r & 31);
            }
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int u = 32 * hf + lane;
                const uint16_t *kvb = p.kv + (utok / p.m) * p.n * (int64_t)D + u * 8;
                const uint32_t dst0 = base + SM_KV + stage * STAGE_BYTES + (u >> 3) * CHUNK;
#pragma unroll
                for (int i = 0; i < BN / 8; ++i) {
                    const int r = gw + 8 * i;
                    const uint32_t mk = r < 32 ? m0 : m1;
                    const uint32_t dst = dst0 + r * 128 + ((u8 ^ (r & 7)) << 4);
                    if ((mk >> (r & 31)) & 1u) cp_async_16(dst, kvb + (int64_t)vr[i] * D);
                    else if (it.J < NST) cp_async_zero16(dst, p.kv);
                }
                if (!(p.stall_first_tile && it.J == 0)) {
                    cp_async_arrive_noinc(BAR((hf == 0 ? B_FULL : B_FULH) + stage));
                    if (hf == 0 && writer) {
                        tile_mask[stage] = ((uint64_t)m1 << 32) | m0;
                        mbar_arrive(BAR(B_FULL + stage));
                    }
                }
            }
            it.next(e0, e1, T);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(p.status, DS_DEV_BAD_INDEX);
        cp_async_wait_all();                              // nothing may land after the CTA exits
    } else if (warp == W_MMA) {
        // ================================= MMA issue (lane 0) =================================
        // Two streams in tile order: S = Q K^T for the next tile whose rows have landed (once its
        // score buffer has been read), and O^T += V^T P^T for the oldest tile whose P is written.
        // Whichever is ready goes first.  S goes in two halves of d, each as soon as its columns
        // have landed; a P V may go between them.
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc(HM, BN, false, false);
            constexpr uint32_t IDESC_PV = idesc(128, HM, true, false);
            TileIter s, v;
            s.start(tok_begin, e0, e1, T);
            v.start(tok_begin, e0, e1, T);
            uint64_t idle_since = 0;
            uint32_t idle = 0;
            bool s_half = false;   // the first half of tile s.J's S is issued
            // S over d columns [16 k0, 16 k1): 16 columns of d = 32 bytes inside the 128-byte
            // swizzle atom of chunk k / 4; 8-row groups 1024 B apart, for Q (A) and the rows (B)
            auto issue_s = [&](int stage, int sb, int k0, int k1) {
                // the rows were written by cp.async (generic proxy), q by TMA; the MMA reads them
                // through the async proxy
                fence_proxy_async_smem();
                tc_fence_after();
                const uint64_t qd0 = smem_desc_sw128(base + SM_Q, 16, 1024);
                const uint64_t kd0 = smem_desc_sw128(base + SM_KV + stage * STAGE_BYTES, 16, 1024);
#pragma unroll
                for (int k = k0; k < k1; ++k) {
                    const uint64_t off = (uint64_t)(((k >> 2) * CHUNK + (k & 3) * 32) >> 4);
                    mma_bf16_ss(tmem + S_COL + sb * BN, qd0 + off, kd0 + off, IDESC_S, k > 0 ? 1u : 0u);
                }
            };
            for (;;) {
                bool progressed = false;
                if (s.valid) {
                    const int stage = s.J % NST, sb = s.J % NSB;
                    if (!s_half && mbar_test_wait(BAR(B_FULL + stage), (uint32_t)(s.J / NST) & 1u) &&
                        mbar_test_wait(BAR(B_SFREE + sb), ((uint32_t)(s.J / NSB) & 1u) ^ 1u) &&
                        (s.t != 0 || mbar_test_wait(BAR(B_QFULL), (uint32_t)s.seg & 1u))) {
                        issue_s(stage, sb, 0, D / 32);
                        s_half = true;
                        progressed = true;
                    }
                    if (s_half && mbar_test_wait(BAR(B_FULH + stage), (uint32_t)(s.J / NST) & 1u)) {
                        issue_s(stage, sb, D / 32, D / 16);
                        mma_commit(BAR(B_SFULL + sb));
                        s.next(e0, e1, T);
                        s_half = false;
                        progressed = true;
                    }
                }
                if (v.valid && v.J < s.J) {
                    const int stage = v.J % NST;
                    if (mbar_test_wait(BAR(B_PFULL + v.J % NPB), (uint32_t)(v.J / NPB) & 1u) &&
                        (v.t != 0 || v.seg == 0 || mbar_test_wait(BAR(B_OFREE), (uint32_t)(v.seg - 1) & 1u))) {
                        // P (and any rescale of O^T) was written by the softmax threads and fenced
                        tc_fence_after();
                        // V^T chunk c: columns 128 c .. 128 c + 127 of the rows as the MN-major A
                        // operand (64-column atoms CHUNK apart, 8-row groups 1024 B apart); rows
                        // 16 k .. 16 k + 15 per step.  P^T: K-major B, 16 entries = 32 bytes per step
                        const uint64_t vd0 = smem_desc_sw128(base + SM_KV + stage * STAGE_BYTES, CHUNK, 1024);
                        const uint64_t pd0 = smem_desc_sw128(base + SM_P + (v.J % NPB) * P_BYTES, 16, 1024);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int k = 0; k < BN / 16; ++k)
                                mma_bf16_ss(tmem + O_COL + c * HM, vd0 + (uint64_t)((2 * c * CHUNK + k * 2048) >> 4),
                                            pd0 + (uint64_t)((k * 32) >> 4), IDESC_PV,
                                            (v.t == 0 && k == 0) ? 0u : 1u);
                        mma_commit(BAR(B_EMPTY + stage));
                        mma_commit(BAR(B_PVDONE + (v.J & 3)));
                        v.next(e0, e1, T);
                        progressed = true;
                    }
                }
                if (!s.valid && !v.valid) break;
                if (progressed) {
                    idle = 0;
                    idle_since = 0;
                    continue;
                }
                __nanosleep(32);
                if ((++idle & 63u) == 0u) {
                    if (*abort_flag) break;
                    const uint64_t now = globaltimer_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > kWaitLimitNs) {
                        *abort_flag = 1;
                        break;
                    }
                }
            }
            if (*abort_flag) {   // let issued MMAs finish before TMEM is freed
                mma_commit(BAR(B_DRAIN));
                mbar_wait_drain(BAR(B_DRAIN), 0, 100000000ull);
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ============================ softmax + epilogue (warps 0-3) ============================
        setmaxnreg_inc<REG_SOFTMAX>();
        // Score layout of the 64-row MMA: head 16 w + i (i < 16) on lane 32 w + i; lanes 16-31 of
        // each warp hold no scores.  So lane i takes columns 0-31 of head 16 w + i and lane i + 16
        // columns 32-63, handed over by one shuffle per value: both lanes serve the head (the same
        // running max, each its own part of the sum and of P).  In the O^T work every thread is one
        // column d = 128 c + 32 w + lane of each chunk c.
        const int hl = 16 * warp + (lane & 15);
        const bool upper = lane >= 16;
        const bool live = hl < p.h;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float sink2 = live ? p.sink[hl] * kLog2e : 0.0f;
        const int dl = 32 * warp + lane;
        // q rows of a token into the Q buffer (K-major, 128-byte swizzle, like the row stages):
        // one TMA load per 64-column chunk, issued by thread 0; the MMA waits on QFULL.
        auto load_q = [&](int64_t utok) {
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(BAR(B_QFULL), (uint32_t)p.h * D * 2);
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                    tma_load_2d(base + SM_Q + c * CHUNK, &qmap, c * 64, (int32_t)(utok * p.h), BAR(B_QFULL));
            }
        };
        TileIter it;
        it.start(tok_begin, e0, e1, T);
        if (it.valid) load_q(unit_at(it.tok, p.ntok, p.interleave));
        bool failed = false;
        while (it.valid && !failed) {
            const int64_t utok = unit_at(it.tok, p.ntok, p.interleave);
            const bool whole = it.a == 0 && it.z == T;
            const int64_t tok = it.tok;
            float m_used = -INFINITY, l = 0.0f;
            bool ok = true;
            for (;;) {
                // tile J: scores from TMEM -> online softmax -> P (bf16) into shared memory
                const int J = it.J;
                const int stage = J % NST, sb = J % NSB;
                ok = !*abort_flag;
                ok = ok && warp_wait(BAR(B_FULL + stage), (uint32_t)(J / NST) & 1u, abort_flag);
                ok = ok && warp_wait(BAR(B_SFULL + sb), (uint32_t)(J / NSB) & 1u, abort_flag);
                float s[32];
                float tmax = -INFINITY;
                if (ok) {
                    tc_fence_after();
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem + lane_off + S_COL + sb * BN, r0);
                    tmem_ld32(tmem + lane_off + S_COL + sb * BN + 32, r1);
                    tmem_ld_wait(r0);
                    tmem_ld_wait(r1);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(B_SFREE + sb));   // the MMA may reuse the buffer
                    // the segment's last scores are ready, so its S products are done with Q: the
                    // next token's q rows may replace it
                    if (it.t == it.ntile - 1 && (it.tok + 1) * T < e1)
                        load_q(unit_at(it.tok + 1, p.ntok, p.interleave));
                    const uint64_t mk = tile_mask[stage];
                    const uint32_t mh = upper ? (uint32_t)(mk >> 32) : (uint32_t)mk;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const uint32_t x = __shfl_sync(0xffffffffu, r1[j], lane & 15);
                        s[j] = ((mh >> j) & 1u) ? __uint_as_float(upper ? x : r0[j]) : -INFINITY;
                    }
                    float mx[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
                    for (int j = 16; j < 32; j += 8)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], s[j + i]);
                    const float half = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                    tmax = fmaxf(half, __shfl_xor_sync(0xffffffffu, half, 16)) * p.scale_log2;
                }
                // a head whose running max moves by more than the threshold asks every softmax
                // thread to rescale O^T (each thread holds one d of every head's column)
                if (ok && live && m_used != -INFINITY && tmax > m_used + kRescaleThreshold) vote[J & 1] = J;
                if (bar_red_or(1, 128, !ok)) {   // a wait gave up: every softmax warp leaves together
                    failed = true;
                    break;
                }
                if (vote[J & 1] == J) {
                    float f = 1.0f;
                    if (live) {
                        const float m_new = fmaxf(m_used, tmax);
                        if (m_used != -INFINITY) f = ex2(m_used - m_new);
                        l *= f;
                        m_used = m_new;
                    }
                    if (!upper) fac[hl] = f;
                    named_bar_sync(2, 128);
                    // O^T holds every P V before this tile (J >= 1: a segment's first tile never
                    // rescales, its running max starts at -inf)
                    ok = warp_wait(BAR(B_PVDONE + ((J - 1) & 3)), (uint32_t)((J - 1) >> 2) & 1u, abort_flag);
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            uint32_t r[2][32];
                            tmem_ld32(tmem + lane_off + O_COL + c * HM, r[0]);
                            tmem_ld32(tmem + lane_off + O_COL + c * HM + 32, r[1]);
                            tmem_ld_wait(r);
#pragma unroll
                            for (int g = 0; g < 2; ++g)
#pragma unroll
                                for (int j = 0; j < 32; j += 4) {
                                    const float4 f4 = *reinterpret_cast<const float4 *>(fac + 32 * g + j);
                                    r[g][j] = __float_as_uint(__uint_as_float(r[g][j]) * f4.x);
                                    r[g][j + 1] = __float_as_uint(__uint_as_float(r[g][j + 1]) * f4.y);
                                    r[g][j + 2] = __float_as_uint(__uint_as_float(r[g][j + 2]) * f4.z);
                                    r[g][j + 3] = __float_as_uint(__uint_as_float(r[g][j + 3]) * f4.w);
                                }
                            tmem_st32(tmem + lane_off + O_COL + c * HM, r[0]);
                            tmem_st32(tmem + lane_off + O_COL + c * HM + 32, r[1]);
                        }
                        tmem_st_wait();
                    }
                } else if (live && m_used == -INFINITY) {
                    m_used = tmax;   // the first rows this head sees (tmax may still be -inf)
                }
                // P buffer J % NPB is free once the P V of tile J - NPB is done
                if (ok && J >= NPB)
                    ok = warp_wait(BAR(B_PVDONE + ((J - NPB) & 3)), (uint32_t)((J - NPB) >> 2) & 1u, abort_flag);
                if (ok) {
                    // p = 2^(s * scale_log2 - m); P goes to the MMA in bf16, the row sum stays f32
                    uint32_t pk[16];
                    if (live) {
                        float ls[4] = {0.f, 0.f, 0.f, 0.f};
                        const float neg_m = m_used == -INFINITY ? 0.0f : -m_used;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float p0 = ex2(fmaf(s[2 * j], p.scale_log2, neg_m));
                            const float p1 = ex2(fmaf(s[2 * j + 1], p.scale_log2, neg_m));
                            ls[j & 3] += p0 + p1;
                            pk[j] = pack_bf16x2(p0, p1);
                        }
                        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) pk[j] = 0u;
                    }
                    // row hl of P (K-major for the P^T operand): 16-byte unit u at u ^ (hl % 8); the
                    // lower lane writes units 0-3 (entries 0-31), the upper lane units 4-7
                    const uint32_t prow = base + SM_P + (J % NPB) * P_BYTES + hl * 128;
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        st_shared_v4(prow + (((u + (upper ? 4 : 0)) ^ (hl & 7)) << 4), pk[4 * u], pk[4 * u + 1],
                                     pk[4 * u + 2], pk[4 * u + 3]);
                    // P stores (and a rescale's TMEM stores) are made visible to the MMA, then one
                    // arrival per warp
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(B_PFULL + J % NPB));
                }
                // a wait that gave up set the abort flag: the next barrier takes every warp out
                const bool last = it.t == it.ntile - 1;
                it.next(e0, e1, T);
                if (last) break;
            }
            if (failed) break;
            // ---- epilogue: O^T is final once the segment's last P V is done.  Its barrier slot's
            // previous phase (four tiles back) is complete: the P buffer waits saw to it.
            const int Jl = it.J - 1;
            ok = ok && !*abort_flag;
            ok = ok && warp_wait(BAR(B_PVDONE + (Jl & 3)), (uint32_t)(Jl >> 2) & 1u, abort_flag);
            if (ok) tc_fence_after();
            const bool any = live && m_used != -INFINITY;
            l += __shfl_xor_sync(0xffffffffu, l, 16);   // the head's sum: both halves of its columns
            if (whole && !upper) {
                float inv = 0.0f;
                if (live) {
                    const float top = fmaxf(m_used, sink2);
                    const float w = any ? ex2(m_used - top) : 0.0f;
                    inv = w / (l * w + ex2(sink2 - top));
                }
                inv_h[hl] = inv;
            }
            if (bar_red_or(1, 128, !ok)) {
                failed = true;
                break;
            }
            if (whole) {
                // normalised O as bf16, straight from the accumulator: thread (lane) d of chunk c
                // holds column 128 c + d of every head, and a warp's 32 lanes store 64 contiguous
                // bytes of one head's row per instruction.  (Measured faster on this path than
                // staging the chunk in shared memory, with or without pairing neighbour lanes, and
                // than TMA stores of the staged chunk.)
                uint16_t *obase = p.o + utok * p.h * (int64_t)D;
                const float2 *cs_row = nullptr;
                if constexpr (ROPE) cs_row = p.rope + (p.rope_pos0 + utok % p.m) * (p.rd / 2);
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[2][32];
                    tmem_ld32(tmem + lane_off + O_COL + c * HM, r[0]);
                    tmem_ld32(tmem + lane_off + O_COL + c * HM + 32, r[1]);
                    tmem_ld_wait(r);
                    const bool rot = ROPE && c * 128 + 32 * warp + 31 >= D - p.rd;
#pragma unroll
                    for (int j = 0; j < HM; j += 4) {
                        const float4 iv = *reinterpret_cast<const float4 *>(inv_h + j);
                        const float xv[4] = {__uint_as_float(r[j >> 5][j & 31]) * iv.x,
                                             __uint_as_float(r[j >> 5][(j + 1) & 31]) * iv.y,
                                             __uint_as_float(r[j >> 5][(j + 2) & 31]) * iv.z,
                                             __uint_as_float(r[j >> 5][(j + 3) & 31]) * iv.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint16_t v = out_bf16<ROPE>(xv[k], c * 128 + dl, cs_row, p.rd, rot);
                            if (j + k < p.h) obase[(int64_t)(j + k) * D + c * 128 + dl] = v;
                        }
                    }
                }
            } else if constexpr (KC > 1) {
                // cluster merge of the token's KC parts (this CTA is part `rank`)
                const int rank = (int)(cid % KC);
                float *wsme = p.ws + (size_t)cid * SLOT;
                if (live && !upper) {
                    wsme[SLOT_O + hl] = any ? m_used : -INFINITY;
                    wsme[SLOT_O + HM + hl] = l;
                }
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    if (c % KC == rank) continue;
                    uint32_t r[2][32];
                    tmem_ld32(tmem + lane_off + O_COL + c * HM, r[0]);
                    tmem_ld32(tmem + lane_off + O_COL + c * HM + 32, r[1]);
                    tmem_ld_wait(r);
                    float4 *dst = reinterpret_cast<float4 *>(wsme + c * 128 * HM) + dl;
#pragma unroll
                    for (int hq = 0; hq < HM / 4; ++hq)
                        if (hq * 4 < p.h)
                            dst[hq * 128] = make_float4(__uint_as_float(r[hq >> 3][4 * (hq & 7)]),
                                                        __uint_as_float(r[hq >> 3][4 * (hq & 7) + 1]),
                                                        __uint_as_float(r[hq >> 3][4 * (hq & 7) + 2]),
                                                        __uint_as_float(r[hq >> 3][4 * (hq & 7) + 3]));
                }
                // every softmax thread's writes are in, then one release per other CTA
                named_bar_sync(2, 128);
                if (threadIdx.x == 0) {
                    const uint32_t me = cluster_ctarank();
                    for (uint32_t j = 0; j < (uint32_t)KC; ++j)
                        if (j != me) mbar_arrive_release_cluster(mapa(BAR(B_XCH), j));
                }
                // the other parts' chunks and statistics
                const bool okx = mbar_wait<true>(BAR(B_XCH), 0u, abort_flag, kWaitLimitNs);
                float *wgt = reinterpret_cast<float *>(sbase + SM_BAR + WGT_OFF);
                if (!upper) {
                    if (live && okx) {
                        const float *part0 = p.ws + (size_t)(cid - rank) * SLOT;
                        float mi[KC], li[KC];
#pragma unroll
                        for (int i = 0; i < KC; ++i) {
                            mi[i] = part0[(size_t)i * SLOT + SLOT_O + hl];
                            li[i] = part0[(size_t)i * SLOT + SLOT_O + HM + hl];
                        }
                        float top = sink2;
#pragma unroll
                        for (int i = 0; i < KC; ++i) top = fmaxf(top, mi[i]);
                        float den = ex2(sink2 - top);
#pragma unroll
                        for (int i = 0; i < KC; ++i)
                            if (mi[i] != -INFINITY) den += ex2(mi[i] - top) * li[i];
                        const float inv = 1.0f / den;
#pragma unroll
                        for (int i = 0; i < KC; ++i)
                            wgt[i * HM + hl] = mi[i] == -INFINITY ? 0.0f : ex2(mi[i] - top) * inv;
                    } else {
#pragma unroll
                        for (int i = 0; i < KC; ++i) wgt[i * HM + hl] = 0.0f;
                    }
                }
                if (bar_red_or(1, 128, !__all_sync(0xffffffffu, okx))) {
                    failed = true;
                    break;
                }
                uint16_t *obase = p.o + utok * p.h * (int64_t)D;
                const float2 *cs_row = nullptr;
                if constexpr (ROPE) cs_row = p.rope + (p.rope_pos0 + utok % p.m) * (p.rd / 2);
#pragma unroll 1
                for (int c = rank; c < 4; c += KC) {
                    const bool rot = ROPE && c * 128 + 32 * warp + 31 >= D - p.rd;
                    uint32_t r[2][32];
                    tmem_ld32(tmem + lane_off + O_COL + c * HM, r[0]);
                    tmem_ld32(tmem + lane_off + O_COL + c * HM + 32, r[1]);
                    tmem_ld_wait(r);
                    float acc[HM];
#pragma unroll
                    for (int j = 0; j < HM; ++j) acc[j] = __uint_as_float(r[j >> 5][j & 31]) * wgt[rank * HM + j];
#pragma unroll 1
                    for (int i = 0; i < KC; ++i) {
                        if (i == rank) continue;
                        const float4 *src =
                            reinterpret_cast<const float4 *>(p.ws + (size_t)(cid - rank + i) * SLOT + c * 128 * HM) + dl;
#pragma unroll
                        for (int hq = 0; hq < HM / 4; ++hq) {
                            if (hq * 4 < p.h) {
                                const float4 v = src[hq * 128];
                                acc[4 * hq] += wgt[i * HM + 4 * hq] * v.x;
                                acc[4 * hq + 1] += wgt[i * HM + 4 * hq + 1] * v.y;
                                acc[4 * hq + 2] += wgt[i * HM + 4 * hq + 2] * v.z;
                                acc[4 * hq + 3] += wgt[i * HM + 4 * hq + 3] * v.w;
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < HM; ++j) {
                        const uint16_t v = out_bf16<ROPE>(acc[j], c * 128 + dl, cs_row, p.rd, rot);
                        if (j < p.h) obase[(int64_t)j * D + c * 128 + dl] = v;
                    }
                }
            } else {
                // partial: unnormalised O^T, running max and sum (log2 domain) for the combine
                const int slot = tok == tok_begin ? 0 : 1;
                float *ws = p.ws + ((size_t)cid * 2 + slot) * SLOT;
                if (live && !upper) {
                    ws[SLOT_O + hl] = any ? m_used : -INFINITY;
                    ws[SLOT_O + HM + hl] = l;
                }
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[2][32];
                    tmem_ld32(tmem + lane_off + O_COL + c * HM, r[0]);
                    tmem_ld32(tmem + lane_off + O_COL + c * HM + 32, r[1]);
                    tmem_ld_wait(r);
                    float4 *dst = reinterpret_cast<float4 *>(ws) + c * 128 + dl;
#pragma unroll
                    for (int hq = 0; hq < HM / 4; ++hq)
                        if (hq * 4 < p.h)
                            dst[(size_t)hq * D] = make_float4(__uint_as_float(r[hq >> 3][4 * (hq & 7)]),
                                                              __uint_as_float(r[hq >> 3][4 * (hq & 7) + 1]),
                                                              __uint_as_float(r[hq >> 3][4 * (hq & 7) + 2]),
                                                              __uint_as_float(r[hq >> 3][4 * (hq & 7) + 3]));
                }
            }
            tc_fence_before();
            mbar_arrive(BAR(B_OFREE));
        }
        cp_async_wait_all();                              // nothing may land after the CTA exits
    }

    // ---- teardown --------------------------------------------------------------------------------
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, DS_DEV_TIMEOUT);
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    // no CTA of a merging cluster leaves while another may still signal its XCH barrier (every
    // wait before this point is bounded, so every CTA gets here)
    if constexpr (KC > 1) cluster_sync();
}

// Merge the partials of every token that a range boundary cut, add the sink once, write bf16.
// Block (i, y) merges columns [32 y, 32 y + 32) of cut token i: thread (g, x) takes column
// 32 y + x of heads 16 g .. 16 g + 15, so each of its loads from a slot is 512 contiguous bytes per
// warp.  The heads' weights per part come first, one thread per head, through shared memory.
constexpr int kCombineCols = 32;

struct CombineParams {
    const float *sink;
    const float *ws;
    uint16_t *o;
    const float2 *rope;           // fused inverse RoPE (ROPE combine), see AttnArgs
    int64_t rope_pos0;
    int rd;
    int m;
    int h;
    int interleave;
    int64_t nunits;
    int ncut;
    int4 cut[kMaxCut];            // {unit, first part, parts, slot bits}
};

template <bool ROPE>
__global__ void __launch_bounds__(128) sparse_attn_ot_combine_kernel(const CombineParams cp) {
    grid_dependency_wait();   // launched as a programmatic dependent of the attention kernel
    __shared__ float wgt[32][HM];
    if ((int)blockIdx.x >= cp.ncut) return;
    const int4 c = cp.cut[blockIdx.x];
    const int64_t utok = unit_at(c.x, cp.nunits, cp.interleave != 0);
    const int kf = c.y, np = c.z;
    const uint32_t slots = (uint32_t)c.w;
    auto part = [&](int i) -> const float * { return cp.ws + ((size_t)(kf + i) * 2 + ((slots >> i) & 1u)) * SLOT; };
    const int t = threadIdx.x;
    if (t < HM) {
        if (t < cp.h) {
            const float sink2 = cp.sink[t] * kLog2e;
            float top = sink2;
            for (int i = 0; i < np; ++i) top = fmaxf(top, part(i)[SLOT_O + t]);
            float den = exp2f(sink2 - top);
            for (int i = 0; i < np; ++i) {
                const float mi = part(i)[SLOT_O + t];
                if (mi != -INFINITY) den += exp2f(mi - top) * part(i)[SLOT_O + HM + t];
            }
            const float inv = 1.0f / den;
            for (int i = 0; i < np; ++i) {
                const float mi = part(i)[SLOT_O + t];
                wgt[i][t] = mi == -INFINITY ? 0.0f : exp2f(mi - top) * inv;
            }
        } else {
            for (int i = 0; i < np; ++i) wgt[i][t] = 0.0f;
        }
    }
    __syncthreads();
    const int x = t & 31, g = t >> 5;
    const int d = blockIdx.y * kCombineCols + x;
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
    for (int i = 0; i < np; ++i) {
        const float4 *src = reinterpret_cast<const float4 *>(part(i)) + d;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int hq = 4 * g + q;
            if (hq * 4 < cp.h) {
                const float4 v = src[(size_t)hq * D];
                acc[4 * q] += wgt[i][4 * hq] * v.x;
                acc[4 * q + 1] += wgt[i][4 * hq + 1] * v.y;
                acc[4 * q + 2] += wgt[i][4 * hq + 2] * v.z;
                acc[4 * q + 3] += wgt[i][4 * hq + 3] * v.w;
            }
        }
    }
    uint16_t *dst = cp.o + utok * cp.h * (int64_t)D + d;
    const float2 *cs_row = nullptr;
    if constexpr (ROPE) cs_row = cp.rope + (cp.rope_pos0 + utok % cp.m) * (cp.rd / 2);
    const bool rot = ROPE && (int)blockIdx.y * kCombineCols + kCombineCols - 1 >= D - cp.rd;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int hh = 16 * g + j;
        const uint16_t v = out_bf16<ROPE>(acc[j], d, cs_row, cp.rd, rot);
        if (hh < cp.h) dst[(int64_t)hh * D] = v;
    }
}

// ---------------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------------

constexpr int kMaxDev = 64;
int g_sms[kMaxDev];
int g_clusters[kMaxDev][5];   // co-resident clusters of 2, 3 and 4 CTAs
bool g_ready[kMaxDev];
std::mutex g_mutex;

// CTAs that can run at once on `dev` (one per SM), 0 when the kernel cannot be configured.
int max_ctas(int dev) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_ready[dev]) return g_sms[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const void *kernels[8] = {(const void *)sparse_attn_ot_kernel<1, false>, (const void *)sparse_attn_ot_kernel<2, false>,
                              (const void *)sparse_attn_ot_kernel<3, false>, (const void *)sparse_attn_ot_kernel<4, false>,
                              (const void *)sparse_attn_ot_kernel<1, true>,  (const void *)sparse_attn_ot_kernel<2, true>,
                              (const void *)sparse_attn_ot_kernel<3, true>,  (const void *)sparse_attn_ot_kernel<4, true>};
    for (const void *k : kernels)
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess) return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sparse_attn_ot_kernel<1, false>, NTHREADS, SMEM_BYTES) !=
            cudaSuccess ||
        per_sm < 1)
        return 0;
    g_sms[dev] = sms * per_sm;
    for (int kc = 2; kc <= 4; ++kc) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(kc * sms), 1, 1);
        cfg.blockDim = dim3(NTHREADS, 1, 1);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)kc;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        auto k = kc == 2   ? sparse_attn_ot_kernel<2, false>
                 : kc == 3 ? sparse_attn_ot_kernel<3, false>
                           : sparse_attn_ot_kernel<4, false>;
        g_clusters[dev][kc] = cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess ? n : 0;
    }
    g_ready[dev] = true;
    return g_sms[dev];
}

int max_clusters(int dev, int kc) {
    if (max_ctas(dev) <= 0) return 0;
    std::lock_guard<std::mutex> lock(g_mutex);
    return g_clusters[dev][kc];
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

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

// q as a 2-D bf16 tensor of `rows` rows of D values, boxes of 64 columns x h rows, 128-byte
// swizzle (the MMA operand layout).
bool make_q_map(CUtensorMap *map, const void *q, int64_t rows, int h) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)h};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Fixed cost of a segment on the cost line (the q rows, the epilogue), in index entries.
constexpr int kSegCost = 2 * BN;

struct Plan {
    int64_t ntok, G, K;
    bool split;
    int kc;           // > 1: the token's parts form a cluster and merge in the kernel
};

bool plan(int64_t ntok, int topk, Plan &pl) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    const int gmax = max_ctas(dev);
    if (gmax <= 0) return false;
    pl.ntok = ntok;
    pl.G = split::choose_ranges(ntok, topk, gmax, BN);
    pl.K = split::seg_cost(ntok, pl.G, kSegCost);
    pl.split = split::splits_units(ntok, topk, pl.G, pl.K);
    // every token split into the same number of parts (2 to 4): those CTAs form a cluster, when
    // all the clusters fit on the GPU at once
    const int64_t k = pl.G > ntok && pl.G % ntok == 0 ? pl.G / ntok : 1;
    pl.kc = pl.split && pl.K == 0 && k >= 2 && k <= 4 && ntok <= max_clusters(dev, (int)k) ? (int)k : 1;
    return true;
}

size_t workspace_bytes(const Plan &pl) {
    if (!pl.split) return 0;
    return (size_t)pl.G * (pl.kc > 1 ? 1 : 2) * SLOT * sizeof(float);
}

}  // namespace ot

bool sparse_attn_ot_supports(int h, int d, bool fp8, bool pair) {
    return d == ot::D && h >= 1 && h <= ot::HM && !fp8 && !pair;
}

bool sparse_attn_ot_preferred(int64_t ntok) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= ot::kMaxDev) return false;
    return ot::max_ctas(dev) > 0 && ntok >= 1;
}

int sparse_attn_ot_launches(int64_t ntok, int topk) {
    ot::Plan pl;
    if (topk <= 0 || !ot::plan(ntok, topk, pl)) return 1;
    return pl.split && pl.kc == 1 ? 2 : 1;
}

size_t sparse_attn_ot_workspace_bytes(int64_t ntok, int topk) {
    ot::Plan pl;
    if (topk <= 0 || !ot::plan(ntok, topk, pl)) return 0;
    return ot::workspace_bytes(pl);
}

int launch_sparse_attn_ot(const AttnArgs &a, cudaStream_t stream, bool stall_first_tile) {
    const int64_t ntok = (int64_t)a.b * a.m;
    ot::Plan pl;
    if (!ot::plan(ntok, a.topk, pl)) return DS_ECUDA;
    if (a.topk > 0 && ntok > (INT64_MAX / (pl.G + 1)) / (a.topk + pl.K)) return DS_EUNSUPPORTED;
    const size_t need = ot::workspace_bytes(pl);
    if (a.workspace_bytes < need || (need && !a.workspace)) return DS_EWORKSPACE;
    const bool combine = pl.split && pl.kc == 1;
    ot::CombineParams cpar;
    if (combine) {
        cpar.sink = a.sink;
        cpar.ws = static_cast<const float *>(a.workspace);
        cpar.o = a.o;
        cpar.rope = reinterpret_cast<const float2 *>(a.rope);
        cpar.rope_pos0 = a.rope_pos0;
        cpar.rd = a.rd;
        cpar.m = a.m;
        cpar.h = a.h;
        cpar.interleave = a.m > 1 ? 1 : 0;
        cpar.nunits = ntok;
        cpar.ncut = split::cut_units(ntok, a.topk, pl.K, pl.G, cpar.cut);
        if (cpar.ncut <= 0) return DS_EUNSUPPORTED;
    }
    ot::Params p;
    p.q = a.q;
    p.kv = a.kv;
    p.sink = a.sink;
    p.idx = a.idx;
    p.o = a.o;
    p.ws = static_cast<float *>(a.workspace);
    p.n = a.n;
    p.ntok = ntok;
    p.topk = a.topk;
    p.m = a.m;
    p.h = a.h;
    p.G = (int)pl.G;
    p.seg_cost = (int)pl.K;
    p.interleave = a.m > 1;
    p.scale_log2 = a.scale * ot::kLog2e;
    p.status = a.status;
    p.stall_first_tile = stall_first_tile ? 1 : 0;
    p.rope = reinterpret_cast<const float2 *>(a.rope);
    p.rd = a.rd;
    p.rope_pos0 = a.rope_pos0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.G, 1, 1);
    cfg.blockDim = dim3(ot::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = ot::SMEM_BYTES;
    cfg.stream = stream;
    // programmatic dependent launch: the set-up overlaps the previous kernel on the stream
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)pl.kc;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pl.kc > 1 ? 2 : 1;
    CUtensorMap qmap;
    if (!ot::make_q_map(&qmap, a.q, ntok * a.h, a.h)) return DS_ECUDA;
    const bool rope = a.rope != nullptr;
    auto kernel = pl.kc == 2   ? (rope ? ot::sparse_attn_ot_kernel<2, true> : ot::sparse_attn_ot_kernel<2, false>)
                  : pl.kc == 3 ? (rope ? ot::sparse_attn_ot_kernel<3, true> : ot::sparse_attn_ot_kernel<3, false>)
                  : pl.kc == 4 ? (rope ? ot::sparse_attn_ot_kernel<4, true> : ot::sparse_attn_ot_kernel<4, false>)
                               : (rope ? ot::sparse_attn_ot_kernel<1, true> : ot::sparse_attn_ot_kernel<1, false>);
    if (cudaLaunchKernelEx(&cfg, kernel, qmap, p) != cudaSuccess) return DS_ECUDA;
    if (combine) {
        cudaLaunchConfig_t ccfg = {};
        ccfg.gridDim = dim3((unsigned)cpar.ncut, (unsigned)(ot::D / ot::kCombineCols), 1);
        ccfg.blockDim = dim3(128, 1, 1);
        ccfg.stream = stream;
        ccfg.attrs = attr;
        ccfg.numAttrs = 1;
        auto comb = rope ? ot::sparse_attn_ot_combine_kernel<true> : ot::sparse_attn_ot_combine_kernel<false>;
        if (cudaLaunchKernelEx(&ccfg, comb, cpar) != cudaSuccess) return DS_ECUDA;
    }
    return DS_OK;
}

}  // namespace dsattn
