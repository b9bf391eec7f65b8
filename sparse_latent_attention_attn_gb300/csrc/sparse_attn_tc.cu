// sparse_attn_tc.cu -- sparse_attn on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes ("Module attn", sparse_attn and the Precision paragraph; "DeepSeek V4.1",
// attention/attend, sparse_attn_kernel): for every query token and head, softmax over the
// index-listed rows of one shared latent KV tensor plus an attention sink that counts in the
// denominator only, the same rows reused as values, f32 arithmetic, bf16 output.
//
// How (GB300-first design; the pages' kernel is prior art only):
//  * Every head of a token shares the same gathered rows, so Q[h x d] K^T and P V are dense bf16
//    contractions with M = heads (padded to 128 = TMEM lanes).  S and O accumulate in TMEM.
//  * Rows are gathered once per (token, tile of 64 valid rows) by cp.async into 128-byte-swizzled
//    shared memory and used by all heads, as the keys (K-major B operand of Q K^T) and as the
//    values (MN-major B operand of P V).  -1 entries are compacted away first, so they cost
//    neither bytes nor MMA work.
//  * Q lives in TMEM (A operand of Q K^T); P is written to shared memory in the swizzled K-major
//    layout (A operand of P V), so a score buffer is free again as soon as it has been read and the
//    MMA can run two tiles ahead of the softmax.
//  * head_dim 512: O[128 x 512] f32 alone would fill TMEM, so a 2-CTA cluster splits the d columns:
//    each CTA gathers and multiplies its own 256 columns and the two partial score tiles are summed
//    through distributed shared memory.  Dedicated exchange warps copy this CTA's partial scores
//    (f32, as the tensor core left them) into a local staging buffer and hand them to the copy
//    engine as one bulk copy per lane quarter into the peer's exchange buffer, while the softmax
//    warps work on the previous tile; both CTAs add the same two f32 halves (addition commutes, so
//    the sums are bit-identical) and run the identical softmax.
//  * Warp roles (16 warps): 0-3 softmax and epilogue (thread = head = TMEM lane); 4-7 and 14-15
//    row gather, plus 8-11 when d is not split; 8-11 score exchange when it is (and the next
//    token's q into TMEM after a segment's last score tile); 12 index compaction; 13 TMEM allocation + single-thread MMA issue, in whatever order its inputs
//    become ready.
//  * Persistent clusters take contiguous ranges of the flattened (token, index entry) space, so
//    the load is balanced whatever the batch; the ranges also charge each token a fixed cost for
//    the work of a segment change (epilogue, next q, pipeline refill), so clusters that start more
//    tokens take fewer entries.  A token cut by a range boundary leaves f32 partials (running max,
//    sum, unnormalised O) in the workspace and a combine kernel merges them with the sink.  Whole
//    tokens are normalised with the sink in the epilogue and written as bf16.
//  * Online softmax in the log2 domain with a lazy rescale: the running max is only moved (and O
//    rescaled) when a tile's max exceeds it by more than 2^8, which keeps the rescale off the hot
//    path while every exponent stays <= 2^8.
//  * Every wait is bounded: past a time limit the kernel flags DS_DEV_TIMEOUT, drains its own
//    copies and MMAs, frees TMEM and returns.
#include <atomic>
#include <mutex>

#include "attn_split.cuh"
#include "common.cuh"
#include "ptx.cuh"
#include "sparse_attn_ot.cuh"

namespace dsattn {
namespace tc {

using namespace ptx;
using split::range_start;
using split::unit_at;
using split::kMaxCut;

constexpr int BN = 64;            // gathered rows per tile: N of Q K^T, K of P V
// compacted indices travel from the compaction warp to the gather warps through a ring of LR
// tiles of BN entries, so the compaction runs a few tiles ahead of the copies.  (Pulling the rows
// of later tiles into L2 ahead of the copies was measured and does not help: with every row
// already in L2 the kernel is no faster, because its pace is set on chip.)
constexpr int LR = 4;
constexpr int NTHREADS = 512;     // 16 warps = 4 warpgroups
constexpr int W_XCH0 = 8;         // warps 8-11: score exchange (split d) or row gather
constexpr int W_LIST = 12;        // index compaction
constexpr int W_MMA = 13;         // TMEM allocation + MMA issue
// register split: softmax warpgroup 232, the other three 88 (128 * (232 + 3 * 88) = 63488 <= 65536)
constexpr uint32_t REG_SOFTMAX = 232, REG_OTHER = 88;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;        // log2 units

constexpr int SLOT_HEADS = 128;   // partial slots are laid out for 128 heads
// A partial slot: O of SLOT_HEADS heads x d (f32, element (h, c) at ((c / 4) * SLOT_HEADS + h) * 4
// + c % 4, so a warp's accesses with one thread per head are 512 contiguous bytes), then the
// running maxima and the sums of the heads.

template <int D>
struct Cfg {
    static constexpr int CL = D == 512 ? 2 : 1;     // CTAs per cluster (d split)
    static constexpr int DH = D / CL;               // columns per CTA
    static constexpr int NCHUNK = DH / 64;          // 128-byte column chunks per row
    static constexpr int CHUNK_BYTES = BN * 128;
    static constexpr int TILE_BYTES = BN * DH * 2;
    // tiles in flight in shared memory; with the d split the fifth stage's 32 KB holds the
    // exchange buffers' share instead
    static constexpr int NSTAGE = CL == 2 ? 4 : 5;
    // With the d split each exchange warp stages its quarter of a score tile in this CTA's shared
    // memory and hands it to the copy engine as one bulk copy into the peer's exchange buffer, so
    // the slow cluster-network traffic never sits in the warps' memory instruction queues
    // (where it delays every shared-memory access of the softmax warps on the same sub-core).
    // Each partial score crosses as its full f32, so the summed score is an f32 evaluation.
    static constexpr int XB = 4;                    // bytes per exchanged score
    // exchange buffers (tiles of the peer's partial scores).  With the d split, P of tile J is
    // written into exchange buffer J % NX once its scores have been read, and the peer may send
    // tile J + NX there once this CTA's P V of tile J is done.
    static constexpr int NX = CL == 2 ? 2 : 0;
    static constexpr int NXD = NX > 0 ? NX : 1;     // divisor for buffer arithmetic
    // separate P buffers (no d split): the softmax writes P of tile J into buffer J % NP without
    // waiting, because the MMA thread issues S(J) only after P V of tile J - NP (so S(J)'s
    // completion covers it)
    static constexpr int NP = CL == 2 ? 0 : 3;
    static constexpr int NPD = NP > 0 ? NP : 1;
    static constexpr int NPROD_WARPS = CL == 2 ? 6 : 10;
    static constexpr int NPROD = NPROD_WARPS * 32;
    // TMEM columns (32-bit): O accumulator, two S buffers, Q (bf16 pairs)
    static constexpr int O_COL = 0;
    static constexpr int S_COL = DH;
    static constexpr int Q_COL = DH + 2 * BN;
    static constexpr int TMEM_COLS = (Q_COL + DH / 2) <= 256 ? 256 : 512;
    // shared memory, offsets from a 1024-aligned base
    static constexpr int P_BYTES = 128 * BN * 2;    // one P tile, bf16, 128-byte rows
    static constexpr int SM_KV = 0;
    static constexpr int SM_P = SM_KV + NSTAGE * TILE_BYTES;
    static constexpr int SM_X = SM_P + NP * P_BYTES;
    // an exchange buffer holds four lane quarters of 32 rows x BN scores (XB bytes each), quarter
    // q at q * XQ, row 32q + i's 16-byte unit k at q * XQ + (k * 32 + i) * 16: every warp access
    // is 512 contiguous bytes.  P of the tile (128 rows of 128 bytes) is later written over it.
    static constexpr int XQ = 32 * BN * XB;
    static constexpr int X_STRIDE = 4 * XQ;         // one exchange buffer
    // shared address of P of tile J (relative to the 1024-aligned base)
    __device__ static uint32_t p_off(int J) {
        return NX > 0 ? (uint32_t)(SM_X + (J % NXD) * X_STRIDE) : (uint32_t)(SM_P + (J % NPD) * P_BYTES);
    }
    static constexpr int SM_XS = SM_X + NX * X_STRIDE;        // staging buffer (d split)
    static constexpr int X_BYTES = NX * X_STRIDE + (CL == 2 ? X_STRIDE : 0);
    static constexpr int SM_LIST = SM_X + X_BYTES;
    static constexpr int LIST_BYTES = LR * BN * 4;  // the index ring
    static constexpr int SM_BAR = SM_LIST + LIST_BYTES;
    static constexpr int SM_END = SM_BAR + 1024;
    static constexpr int SMEM_BYTES = SM_END + 1024;
    static_assert(Q_COL + DH / 2 <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(SM_P % 1024 == 0 && P_BYTES % 1024 == 0, "swizzled operands are 1024-byte aligned");
    static_assert(CL == 1 || (SM_X % 1024 == 0 && X_STRIDE % 1024 == 0 && X_STRIDE >= P_BYTES),
                  "P of a tile is written over its exchange buffer");
    static_assert(NSTAGE <= 5 && NX <= 3, "barrier slots");
};

// Producer index (0..NPROD_WARPS-1) of a gather warp, -1 for other warps.
template <int D>
__device__ __forceinline__ int prod_warp(int warp) {
    if (warp >= 4 && warp < 8) return warp - 4;
    if (Cfg<D>::CL == 1 && warp >= 8 && warp < 12) return warp - 4;
    if (warp >= 14) return Cfg<D>::NPROD_WARPS - 2 + (warp - 14);
    return -1;
}

// barrier slots (8 bytes each) inside the SM_BAR block
enum : int {
    B_FULL = 0,                 // [NSTAGE] producer -> consumers: tile landed
    B_EMPTY = B_FULL + 5,       // [NSTAGE] MMA -> producer: stage free
    B_SFULL = B_EMPTY + 5,      // [2] MMA -> softmax, exchange: S ready (or the end marker)
    B_SFREE = B_SFULL + 2,      // [2] softmax, exchange -> MMA: S buffer read
    // [4] softmax -> MMA: P of tile J written (slot J % 4).  Four slots: with NX (at most three)
    // exchange buffers the softmax can finish tile J + NX - 1 before the MMA thread has seen tile
    // J, but not tile J + NX (its peer scores need the P V of tile J, which frees the buffer)
    B_PFULL = B_SFREE + 2,
    B_PVDONE = B_PFULL + 4,     // [4] MMA -> softmax, exchange: P V of tile J done (slot J % 4)
    B_QREADY = B_PVDONE + 4,    // softmax -> MMA: Q of the segment in TMEM
    B_OFREE = B_QREADY + 1,     // softmax -> MMA: epilogue has read O
    B_XFULL = B_OFREE + 1,      // [NX] peer -> me: peer's partial scores are in my exchange buffer
    B_XFREE = B_XFULL + 3,      // [NX] peer -> me: the peer's buffer for my next send is free
    B_DRAIN = B_XFREE + 3,      // MMA drain on abort
    B_ZREAD = B_DRAIN + 1,      // softmax threads have read the meta of a tile without rows
    B_LTFULL = B_ZREAD + 1,     // [LR] compaction -> producers: index ring tile written
    B_LTFREE = B_LTFULL + LR,   // [LR] producers -> compaction: index ring tile consumed
    B_COUNT = B_LTFREE + LR
};
constexpr int META_OFF = 8 * B_COUNT;      // [NSTAGE] int2 {count, last}
constexpr int LMETA_OFF = (META_OFF + 8 * 5 + 15) & ~15;   // [LR] int4 {count, last, sequence, 0}
constexpr int TMEM_ADDR_OFF = LMETA_OFF + 16 * LR;
constexpr int ABORT_OFF = TMEM_ADDR_OFF + 4;
constexpr int SEND_OFF = ABORT_OFF + 4;
// pair mode: per stage, the 64-bit masks of the tile's rows listed by the pair's first and second
// query {A lo, A hi, B lo, B hi}
constexpr int META2_OFF = 512;
// d split: per score tile J (slot J % 4), the next token's offset from the CTA's first token when
// tile J is the last of its segment and a token follows in the range, else -1.  The MMA thread
// writes it before issuing S(J) and arrives on that tile's S barrier, which the exchange warps
// wait on.
constexpr int SINFO_OFF = META2_OFF + 16 * 5;
static_assert(SEND_OFF + 4 <= META2_OFF && SINFO_OFF + 16 <= 1024, "barrier block");
// pair mode: an index entry carries its row in the low 29 bits and the queries listing it above
constexpr int32_t kRowMask = (1 << 29) - 1, kPairA = 1 << 29, kPairB = 1 << 30;

struct Params {
    const uint16_t *q;
    const uint16_t *kv;
    const uint8_t *kv8;       // fp8 row store (F8 kernels): e4m3fn codes [b][n][d]
    const int8_t *kexp;       //   and per-32 scale exponents [b][n][d / 32]
    const float *sink;
    const int32_t *idx;
    uint16_t *o;
    float *ws;
    int64_t n;
    int64_t ntok;     // work units of topk entries each: b * m tokens, or (pair mode) b * ceil(m / 2) pairs
    int topk;
    int useq;         // work units per sequence (m, or ceil(m / 2) in pair mode)
    int hm;           // TMEM lanes (rows of M) in use: h, or 2 h in pair mode
    bool interleave;  // unit order (unit_at): several units per sequence
    int seg_cost;     // K of range_start, in entries
    int wide;         // q and o 32-byte aligned: their rows move in 32-byte accesses
    int m;
    int h;
    int G;            // clusters
    float scale_log2; // softmax scale * log2(e)
    unsigned int *status;
    // test switch for the timeout path (ds_test_set_stall): the gather warps withhold their
    // arrivals for the first tile, so a bounded wait runs out
    int stall_first_tile;
    // fused inverse RoPE of the output (rope == nullptr: none), see AttnArgs
    const float2 *rope;
    int rd;
    int64_t rope_pos0;
};

// A bf16 pair of output columns (col, col + 1) of token tok: the normalised values, and when the
// inverse RoPE is fused and the pair lies in the last rd columns, rotated back exactly as
// ds_apply_rotary would rotate the stored bf16 pair.  cs_row: the token's table row.  The rotation
// is a separate kernel instantiation (ROPE), so the plain kernel carries none of its code.
template <int D, bool ROPE>
__device__ __forceinline__ uint32_t out_pair(float x0, float x1, int col, const float2 *cs_row, int rd) {
    uint32_t v = pack_bf16x2(x0, x1);
    if constexpr (ROPE) {
        if (col >= D - rd) v = rope_rotate_bf16x2(v, __ldg(cs_row + ((col - (D - rd)) >> 1)), true);
    }
    return v;
}

// Four packed entries kept in registers: a loop over constant indices selects the slot.
struct PvRing {
    uint32_t e[4];
    __device__ __forceinline__ void put(int q, uint32_t v) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (i == q) e[i] = v;
    }
    __device__ __forceinline__ uint32_t get(int q) const {
        uint32_t v = e[0];
#pragma unroll
        for (int i = 1; i < 4; ++i)
            if (i == q) v = e[i];
        return v;
    }
};

// Every lane waits for the phase itself (acquire) and the warp proceeds together or not at all,
// so warp-collective tcgen05 instructions never diverge.  (Measured on this path: one polling
// lane plus a broadcast costs about twice as much per wait, and a wake-up three times as long.)
// kCluster: the phase was completed from the other CTA of the cluster (acquire at cluster scope).
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait<kCluster>(bar, parity, abort, kWaitLimitNs);
    return __all_sync(0xffffffffu, ok);
}

// Lane t of unit u (a token, or in pair mode the queries 2j, 2j + 1 of a sequence): the token it
// serves, its head and whether that token exists.  In pair mode lanes [0, h) serve the first
// query and [h, 2 h) the second.
struct LaneRow {
    int64_t tok;
    int head;
    bool live;
};

template <bool PAIR>
__device__ __forceinline__ LaneRow lane_row(int64_t u, int t, int h, int m, int useq) {
    if constexpr (!PAIR) {
        return LaneRow{u, t, t < h};
    } else {
        const int k = t >= h ? 1 : 0;
        const int64_t bi = u / useq;
        const int qi = (int)(u - bi * useq) * 2 + k;
        return LaneRow{bi * m + qi, t - k * h, t < 2 * h && qi < m};
    }
}

template <int D, bool F8 = false, bool ROPE = false, bool PAIR = false>
__global__ void __launch_bounds__(NTHREADS, 1) sparse_attn_tc_kernel(const Params p) {
    using C = Cfg<D>;
    static_assert(!(PAIR && (F8 || ROPE)), "pair mode reads bf16 rows and writes the plain output");
    static_assert(!F8 || C::CL == 2, "the fp8 row store is read by the d-split (d = 512) kernel");
    constexpr int NSTAGE = C::NSTAGE;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);
    const uint32_t bars = base + C::SM_BAR;
    auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
    int2 *meta = reinterpret_cast<int2 *>(sbase + C::SM_BAR + META_OFF);
    uint4 *meta2 = reinterpret_cast<uint4 *>(sbase + C::SM_BAR + META2_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + C::SM_BAR + ABORT_OFF);
    volatile int *s_end = reinterpret_cast<volatile int *>(sbase + C::SM_BAR + SEND_OFF);
    int *sinfo = reinterpret_cast<int *>(sbase + C::SM_BAR + SINFO_OFF);
    int4 *lmeta = reinterpret_cast<int4 *>(sbase + C::SM_BAR + LMETA_OFF);
    int32_t *list = reinterpret_cast<int32_t *>(sbase + C::SM_LIST);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = C::CL == 2 ? cluster_ctarank() : 0u;
    const uint32_t peer = crank ^ 1u;
    const int64_t cid = blockIdx.x / C::CL;
    const int T = p.topk;
    const int64_t e0 = range_start(cid, p.ntok, T, p.seg_cost, p.G);
    const int64_t e1 = range_start(cid + 1, p.ntok, T, p.seg_cost, p.G);

    // ---- set-up --------------------------------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(BAR(B_FULL + s), C::NPROD + 1);   // every gather thread's copies + the meta writer
            mbar_init(BAR(B_EMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            // the MMA commit; with the d split also the MMA thread's arrival after writing sinfo
            mbar_init(BAR(B_SFULL + i), C::CL == 2 ? 2 : 1);
            mbar_init(BAR(B_SFREE + i), C::CL == 2 ? 8 : 4);   // one arrival per reading warp

        }
        for (int i = 0; i < C::NX; ++i) {
            mbar_init(BAR(B_XFULL + i), 1);     // armed by the receiver; the peer's bytes complete it
            mbar_init(BAR(B_XFREE + i), 4);     // one arrival per exchange warp of the peer
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(BAR(B_PFULL + i), 4);       // one arrival per softmax warp
            mbar_init(BAR(B_PVDONE + i), 1);
        }
        mbar_init(BAR(B_QREADY), 128);
        mbar_init(BAR(B_OFREE), 128);
        mbar_init(BAR(B_DRAIN), 1);
        mbar_init(BAR(B_ZREAD), 128 + 1);     // softmax threads + the MMA thread
        for (int i = 0; i < LR; ++i) {
            mbar_init(BAR(B_LTFULL + i), 32);                // every compaction lane's writes
            mbar_init(BAR(B_LTFREE + i), C::NPROD_WARPS);    // one arrival per gather warp
        }
        *abort_flag = 0;
        *s_end = -1;
        fence_mbar_init();
        if constexpr (C::CL == 2) {
            // the exchange buffers expect the peer's quarters with live rows, tiles 0 .. NX-1
            const uint32_t xbytes = (uint32_t)((p.hm < 128 ? p.hm : 128) + 31) / 32 * C::XQ;
            for (int i = 0; i < C::NX; ++i) mbar_arrive_expect_tx(BAR(B_XFULL + i), xbytes);
        }
    }
    // the combine kernel may be scheduled as soon as SMs free up (it waits for this grid itself)
    if (threadIdx.x == 0) grid_launch_dependents();
    // rows a tile does not load keep finite values: zero every stage once
    for (int i = threadIdx.x; i < NSTAGE * C::TILE_BYTES / 16; i += NTHREADS)
        reinterpret_cast<uint4 *>(sbase + C::SM_KV)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == W_MMA) {
        tmem_alloc(base + C::SM_BAR + TMEM_ADDR_OFF, C::TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (C::CL == 2) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sbase + C::SM_BAR + TMEM_ADDR_OFF);
    // everything above overlaps the previous kernel on the stream (launched as a programmatic
    // dependent); from here on the inputs it may have written are read, and outputs written
    grid_dependency_wait();
    // warpgroups 1-3 give registers back to the softmax warpgroup before they branch
    if (warp >= 4) setmaxnreg_dec<REG_OTHER>();

    const int64_t tok_begin = e0 / (T > 0 ? T : 1);
    const bool has_work = e1 > e0 && T > 0;
    const int pw = prod_warp<D>(warp);

    if (warp == W_LIST) {
        // ======================= index compaction into the ring of tiles =======================
        // The index row of each segment is read 256 entries at a time (8 per lane, coalesced, the
        // next batch in flight while this one is compacted); valid entries go in order into ring
        // tiles of BN.  A full tile is published only once the next valid entry (or the segment's
        // end) shows whether it is the segment's last; a segment without valid entries publishes
        // one empty tile.
        int lt = 0;              // ring tiles published so far (= the gather warps' tile counter)
        int fill = 0;            // entries in the tile being filled
        bool ok = true;
        auto acquire = [&]() -> bool {   // ring slot of tile lt is free again
            return warp_wait(BAR(B_LTFREE + lt % LR), (uint32_t)((lt / LR) & 1) ^ 1u, abort_flag);
        };
        auto publish = [&](int cnt, int last, int seq) {
            if (lane == 0) lmeta[lt % LR] = make_int4(cnt, last, seq, 0);
            mbar_arrive(BAR(B_LTFULL + lt % LR));             // every lane releases its own writes
            ++lt;
        };
        bool bad = false;
        for (int64_t tok = tok_begin; has_work && ok && tok * T < e1; ++tok) {
            const int a = (int)((e0 > tok * T ? e0 : tok * T) - tok * T);
            const int z = (int)((e1 < (tok + 1) * T ? e1 : (tok + 1) * T) - tok * T);
            const int64_t utok = unit_at(tok, p.ntok, p.interleave);
            const int seq = (int)(utok / p.useq);
            const int32_t *irow = p.idx + utok * T;
            {   // warm L2 with the next token's index row
                const int64_t nt = tok + 1;
                if (nt * T < e1)
                    for (int j = lane * 32; j < T; j += 32 * 32)
                        prefetch_l2(p.idx + unit_at(nt, p.ntok, p.interleave) * T + j);
            }
            if (!acquire()) {
                ok = false;
                break;
            }
            fill = 0;
            int vb[8];
            auto load = [&](int j0) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const int j = j0 + g * 32 + lane;
                    vb[g] = j < z ? __ldg(irow + j) : -1;
                }
            };
            load(a);
            for (int j0 = a; j0 < z && ok; j0 += 256) {
                int v8[8];
#pragma unroll
                for (int g = 0; g < 8; ++g) v8[g] = vb[g];
                if (j0 + 256 < z) load(j0 + 256);            // next batch in flight
#pragma unroll 1
                for (int g = 0; g < 8 && ok; ++g) {
                    if (j0 + g * 32 >= z) break;
                    const int v = v8[g];
                    const int64_t row = PAIR ? (int64_t)(v & kRowMask) : (int64_t)v;
                    const bool valid = v >= 0 && row < p.n;
                    bad |= v >= 0 && row >= p.n;
                    const uint32_t bal = __ballot_sync(0xffffffffu, valid);
                    const int c = __popc(bal), pos = __popc(bal & lanemask_lt());
                    const int space = BN - fill;
                    int32_t *tile = list + (lt % LR) * BN;
                    if (valid && pos < space) tile[fill + pos] = v;
                    if (c > space) {
                        // the tile is full and more entries follow: publish it, take the next
                        __syncwarp();
                        publish(BN, 0, seq);
                        if (!acquire()) {
                            ok = false;
                            break;
                        }
                        tile = list + (lt % LR) * BN;
                        if (valid && pos >= space) tile[pos - space] = v;
                        fill = c - space;
                    } else {
                        fill += c;
                    }
                }
            }
            if (!ok) break;
            __syncwarp();
            publish(fill, 1, seq);                            // the segment's last (maybe empty) tile
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(p.status, DS_DEV_BAD_INDEX);
    } else if (F8 && pw >= 0) {
        // ============== row gather from the fp8 row store, decoded into the bf16 ring ==============
        // A row half is DH e4m3 codes (U8 = DH / 16 units of 16 bytes, half a 32-value block each)
        // and DH / 32 scale exponents.  A lane takes one unit of a row: its 16 codes and their
        // block's exponent, loaded as soon as the tile's row numbers are known (before its stage
        // is free, so the loads overlap that wait), then decoded to 32 bytes of bf16 -- exactly
        // the values of the bf16 round trip -- and stored swizzled like the cp.async path's rows.
        constexpr int U8 = C::DH / 16;
        constexpr int RPW8 = 32 / U8;                    // rows per warp instruction
        constexpr int STEP = C::NPROD_WARPS * RPW8;
        constexpr int MAXR = (BN + STEP - 1) / STEP;     // rows per lane and tile, at most
        const int rsub = lane / U8, unit = lane % U8;
        const int chunk = unit / 4, ua = 2 * (unit % 4); // the two bf16 units 2 unit, 2 unit + 1
        const bool writer = pw == 0 && lane == 0;
        int it = 0;
        bool ok = true;
        for (int64_t tok = tok_begin; has_work && ok && tok * T < e1; ++tok) {
            const int64_t row0 = (unit_at(tok, p.ntok, p.interleave) / p.useq) * p.n;
            const uint8_t *cb = p.kv8 + row0 * (int64_t)D + crank * C::DH + unit * 16;
            const int8_t *xb = p.kexp + row0 * (int64_t)(D / 32) + crank * (C::DH / 32) + unit / 2;
            for (;; ++it) {
                if (!warp_wait(BAR(B_LTFULL + it % LR), (uint32_t)(it / LR) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int4 lm = lmeta[it % LR];
                const int cnt = lm.x;
                const int32_t *tile = list + (it % LR) * BN;
                uint4 cv[MAXR];
                int kx[MAXR];
#pragma unroll
                for (int i = 0; i < MAXR; ++i) {
                    const int r = i * STEP + pw * RPW8 + rsub;
                    if (r < cnt) {
                        const int64_t v = tile[r];
                        cv[i] = __ldg(reinterpret_cast<const uint4 *>(cb + v * D));
                        kx[i] = __ldg(xb + v * (D / 32));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_LTFREE + it % LR));   // this warp is done with the tile
                const int stage = it % NSTAGE;
                if (!warp_wait(BAR(B_EMPTY + stage), ((it / NSTAGE) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t dst0 = base + C::SM_KV + stage * C::TILE_BYTES + chunk * C::CHUNK_BYTES;
#pragma unroll
                for (int i = 0; i < MAXR; ++i) {
                    const int r = i * STEP + pw * RPW8 + rsub;
                    if (r < cnt) {
                        uint32_t w[8];
                        dequant_e4m3x16(cv[i], kx[i], w);
                        const uint32_t rowa = dst0 + r * 128;
                        st_shared_v4(rowa + ((ua ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
                        st_shared_v4(rowa + (((ua + 1) ^ (r & 7)) << 4), w[4], w[5], w[6], w[7]);
                    }
                }
                // the MMA reads the stage through the async proxy
                fence_proxy_async_smem();
                if (!(p.stall_first_tile && it == 0)) {
                    mbar_arrive(BAR(B_FULL + stage));
                    if (writer) {
                        meta[stage] = make_int2(cnt, lm.y);
                        mbar_arrive(BAR(B_FULL + stage));
                    }
                }
                if (lm.y) {
                    ++it;
                    break;
                }
            }
        }
    } else if (pw >= 0) {
        // ================== row gather: cp.async into the 128-byte-swizzled ring ==================
        // A row half of DH columns is U = DH / 8 units of 16 bytes; each warp instruction copies
        // 32 / U whole rows, so every global access is a contiguous row piece.  The row numbers
        // come from the index ring, tile by tile, in the compaction warp's order.
        constexpr int U = C::DH / 8;
        constexpr int RPW = 32 / U;                      // rows per warp instruction
        const int rsub = lane / U, unit = lane % U;
        const int chunk = unit / 8, u8 = unit % 8;
        const bool writer = pw == 0 && lane == 0;
        int it = 0;
        bool ok = true;
        for (int64_t tok = tok_begin; has_work && ok && tok * T < e1; ++tok) {
            const uint16_t *kvb =
                p.kv + ((unit_at(tok, p.ntok, p.interleave) / p.useq) * p.n) * (int64_t)D + crank * C::DH + unit * 8;
            for (;; ++it) {
                // index tile it, then its stage
                if (!warp_wait(BAR(B_LTFULL + it % LR), (uint32_t)(it / LR) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int4 lm = lmeta[it % LR];
                const int stage = it % NSTAGE;
                if (!warp_wait(BAR(B_EMPTY + stage), ((it / NSTAGE) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int cnt = lm.x;
                const int32_t *tile = list + (it % LR) * BN;
                const uint32_t dst0 = base + C::SM_KV + stage * C::TILE_BYTES + chunk * C::CHUNK_BYTES;
#pragma unroll 4
                for (int r = pw * RPW + rsub; r < cnt; r += C::NPROD_WARPS * RPW) {
                    // row r, 16-byte unit u8 of its 128-byte chunk: swizzled to unit u8 ^ (r % 8)
                    const int v = PAIR ? (tile[r] & kRowMask) : tile[r];
                    cp_async_16(dst0 + r * 128 + ((u8 ^ (r & 7)) << 4), kvb + (int64_t)v * D);
                }
                if constexpr (PAIR) {
                    // the rows of this tile that each query of the pair listed (warp 0 of the gather)
                    if (pw == 0) {
                        const int e0 = lane < cnt ? tile[lane] : 0, e1 = lane + 32 < cnt ? tile[lane + 32] : 0;
                        const uint32_t alo = __ballot_sync(0xffffffffu, (e0 & kPairA) != 0);
                        const uint32_t ahi = __ballot_sync(0xffffffffu, (e1 & kPairA) != 0);
                        const uint32_t blo = __ballot_sync(0xffffffffu, (e0 & kPairB) != 0);
                        const uint32_t bhi = __ballot_sync(0xffffffffu, (e1 & kPairB) != 0);
                        if (lane == 0) meta2[stage] = make_uint4(alo, ahi, blo, bhi);
                    }
                }
                if (!(p.stall_first_tile && it == 0)) {
                    cp_async_arrive_noinc(BAR(B_FULL + stage));
                    if (writer) {
                        meta[stage] = make_int2(cnt, lm.y);
                        mbar_arrive(BAR(B_FULL + stage));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_LTFREE + it % LR));   // this warp is done with the tile
                if (lm.y) {
                    ++it;
                    break;
                }
            }
        }
        cp_async_wait_all();                              // nothing may land after the CTA exits
    } else if (warp == W_MMA) {
        // ================================= MMA issue (lane 0) =================================
        // Two independent streams, each in tile order: S = Q K^T for the next tile whose rows have
        // landed (once its score buffer has been read), and O += P V for the oldest tile whose P is
        // written.  Whichever is ready goes first, so a slow softmax never holds back the scores
        // of the tiles behind it.
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BN, false);
            constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, C::DH, true);
            int64_t tok = tok_begin;
            int it = 0, J = 0, seg = 0;
            bool first = true, s_more = has_work;
            // pending P V, oldest at pq_head; at most three can be outstanding.  Entry pq_tail holds
            // tile J = pq_tail (every S pushes one); its stage, first flag and segment are packed in
            // a register ring (an indexed array would live in local memory)
            PvRing pq;
            int pq_head = 0, pq_tail = 0;
            uint64_t idle_since = 0;
            uint32_t idle = 0;
            bool ok = true;
            for (;;) {
                bool progressed = false;
                if (s_more) {
                    const int stage = it % NSTAGE;
                    if (mbar_test_wait(BAR(B_FULL + stage), (it / NSTAGE) & 1)) {
                        const int2 mt = meta[stage];
                        if (mt.x == 0 && !mbar_test_wait(BAR(B_QREADY), seg & 1)) {
                            // a segment without a single valid row still waits for the q it was
                            // given (unused), so this thread's QREADY waits follow the segments one
                            // phase at a time: a parity wait is only exact one phase ahead, and a
                            // Q written while S reads it would corrupt the product
                        } else if (mt.x == 0) {
                            // a segment without a single valid row: nothing to multiply; the softmax
                            // warps hand the stage back once this thread has read the meta too
                            mbar_arrive(BAR(B_ZREAD));
                            ++it;
                            ++seg;
                            ++tok;
                            first = true;
                            s_more = tok * T < e1;
                            progressed = true;
                        } else if ((C::NP == 0 || pq_head >= J - C::NP + 1) &&
                                   mbar_test_wait(BAR(B_SFREE + (J & 1)), ((J >> 1) & 1) ^ 1) &&
                                   (!first || mbar_test_wait(BAR(B_QREADY), seg & 1))) {
                            if constexpr (C::CL == 2) {
                                // whether this tile ends its segment, for the exchange warps (they
                                // load the next token's Q once this S is done)
                                sinfo[J & 3] = mt.y && (tok + 1) * T < e1 ? (int)(tok + 1 - tok_begin) : -1;
                                mbar_arrive(BAR(B_SFULL + (J & 1)));
                            }
                            // the rows were written by cp.async (generic proxy); the MMA reads them
                            // through the async proxy
                            fence_proxy_async_smem();
                            tc_fence_after();
                            // S = Q K^T: K rows as the K-major B operand; 16 columns = 32 bytes inside
                            // the 128-byte swizzle atom of chunk k/4; 8-row groups 1024 B apart
                            // the start-address field (address >> 4, 14 bits) takes the K step's
                            // offset directly: every operand lies below 256 KB of shared memory
                            const uint64_t kdesc0 = smem_desc_sw128(base + C::SM_KV + stage * C::TILE_BYTES, 16, 1024);
#pragma unroll
                            for (int k = 0; k < C::DH / 16; ++k) {
                                const uint64_t bdesc =
                                    kdesc0 + (uint64_t)(((k >> 2) * C::CHUNK_BYTES + (k & 3) * 32) >> 4);
                                mma_bf16_ts(tmem + C::S_COL + (J & 1) * BN, tmem + C::Q_COL + k * 8, bdesc, IDESC_S,
                                            k > 0 ? 1u : 0u);
                            }
                            mma_commit(BAR(B_SFULL + (J & 1)));
                            pq.put(pq_tail & 3, (uint32_t)stage | (first ? 8u : 0u) | ((uint32_t)seg << 4));
                            ++pq_tail;
                            ++J;
                            ++it;
                            first = false;
                            if (mt.y) {
                                ++seg;
                                ++tok;
                                first = true;
                                s_more = tok * T < e1;
                            }
                            progressed = true;
                        }
                    }
                }
                if (pq_head != pq_tail) {
                    const uint32_t ent = pq.get(pq_head & 3);
                    const int Jp = pq_head;
                    const int pq_stage = (int)(ent & 7u), pq_seg = (int)(ent >> 4);
                    const bool pq_first = (ent & 8u) != 0;
                    if (mbar_test_wait(BAR(B_PFULL + (Jp & 3)), (Jp >> 2) & 1) &&
                        (!pq_first || pq_seg == 0 || mbar_test_wait(BAR(B_OFREE), (pq_seg - 1) & 1))) {
                        // P was written by st.shared (generic proxy) and fenced by its writers
                        tc_fence_after();
                        const uint64_t pdesc0 = smem_desc_sw128(base + C::p_off(Jp), 16, 1024);
                        const uint64_t vdesc0 =
                            smem_desc_sw128(base + C::SM_KV + pq_stage * C::TILE_BYTES, C::CHUNK_BYTES, 1024);
#pragma unroll
                        for (int k = 0; k < BN / 16; ++k) {
                            // P: K-major A operand, 16 columns = 32 bytes of each 128-byte row.
                            // V rows 16k..16k+15 as the MN-major B operand (d contiguous): 8-row
                            // groups 1024 B apart, 64-column chunks CHUNK_BYTES apart
                            const uint64_t adesc = pdesc0 + (uint64_t)((k * 32) >> 4);
                            const uint64_t bdesc = vdesc0 + (uint64_t)((k * 2048) >> 4);
                            mma_bf16_ss(tmem + C::O_COL, adesc, bdesc, IDESC_PV, (pq_first && k == 0) ? 0u : 1u);
                        }
                        mma_commit(BAR(B_EMPTY + pq_stage));
                        mma_commit(BAR(B_PVDONE + (Jp & 3)));
                        ++pq_head;
                        progressed = true;
                    }
                }
                if (!s_more && pq_head == pq_tail) break;
                if (progressed) {
                    idle = 0;
                    idle_since = 0;
                    continue;
                }
                // nothing ready: sleep briefly so the polling does not take issue slots from the
                // softmax warp that shares this warp's scheduler
                __nanosleep(32);
                if ((++idle & 63u) == 0u) {
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    const uint64_t now = globaltimer_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > kWaitLimitNs) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                }
            }
            (void)ok;
            if constexpr (C::CL == 2) {
                // end marker for the exchange warps: no score tile J follows (both arrivals the
                // barrier expects)
                *s_end = J;
                mbar_arrive(BAR(B_SFULL + (J & 1)));
                mbar_arrive(BAR(B_SFULL + (J & 1)));
            }
            if (*abort_flag) {   // let issued MMAs finish before TMEM is freed
                mma_commit(BAR(B_DRAIN));
                mbar_wait_drain(BAR(B_DRAIN), 0, 100000000ull);
            }
        }
        __syncwarp();
    } else if (C::CL == 2 && warp >= W_XCH0 && warp < W_XCH0 + 4) {
        // ======================= score exchange (d split across the cluster) =======================
        // Warp w reads TMEM lane quarter w % 4 of each finished score tile and sends it to the
        // peer's exchange buffer, so the softmax warps never wait on the cluster network to send.
        // Quarters without a live head are not sent (the receiver expects only the others).
        // After the last score tile of a segment these warps also put the next token's q into
        // TMEM (its S products are done with the current one), while the softmax warps finish the
        // segment and write its output.
        const int quarter = warp & 3;
        const int qt = quarter * 32 + lane;               // head row = TMEM lane
        const bool live_q = quarter * 32 < p.hm;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        constexpr uint32_t XSTRIDE = C::X_STRIDE;
        const uint32_t xpeer = mapa(base + C::SM_X, peer) + quarter * C::XQ;
        const uint32_t xfull_peer = mapa(BAR(B_XFULL), peer);   // counts the bytes of each copy
        const uint32_t xfree_peer = mapa(BAR(B_XFREE), peer);
        const uint32_t stage_q = base + C::SM_XS + quarter * C::XQ;   // this warp's staging quarter
        for (int J = 0; has_work; ++J) {
            const int sb = J & 1;
            const uint32_t ph = (J >> 1) & 1;
            const int xs = J % C::NXD;
            const uint32_t xph = (uint32_t)(J / C::NXD) & 1u;
            if (J >= C::NX) {
                // this CTA's P V of tile J - NX is done, so the exchange buffer that held its P may
                // take the peer's scores of tile J (the P V four tiles earlier on the same barrier
                // was waited for at tile J - 4, so this parity wait is exact)
                const int Jo = J - C::NX;
                if (!warp_wait(BAR(B_PVDONE + (Jo & 3)), (Jo >> 2) & 1, abort_flag)) break;
                if (lane == 0) mbar_arrive_cluster_relaxed(xfree_peer + 8u * xs);
            }
            if (!warp_wait(BAR(B_SFULL + sb), ph, abort_flag)) break;
            if (*s_end == J) break;
            const int next_tok = sinfo[J & 3];
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane_off + C::S_COL + sb * BN, r0);
            tmem_ld32(tmem + lane_off + C::S_COL + sb * BN + 32, r1);
            tmem_ld_wait(r0);
            tmem_ld_wait(r1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_SFREE + sb));
            // the staging quarter is free once the copy of the previous tile has read it
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            if (live_q) {
                // row i of the quarter: 16-byte unit k at (k * 32 + i) * 16
                const uint32_t srow = stage_q + lane * 16;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    st_shared_v4(srow + k * 512, r0[4 * k], r0[4 * k + 1], r0[4 * k + 2], r0[4 * k + 3]);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    st_shared_v4(srow + (8 + k) * 512, r1[4 * k], r1[4 * k + 1], r1[4 * k + 2], r1[4 * k + 3]);
                fence_proxy_async_smem();                // the copy engine reads what was written here
            }
            // the peer's exchange buffer for tile J is free (its P V of tile J - NX is done)
            if (!warp_wait<true>(BAR(B_XFREE + xs), xph ^ 1, abort_flag)) break;
            if (live_q && lane == 0) {
                bulk_copy_to_peer(xpeer + xs * XSTRIDE, stage_q, C::XQ, xfull_peer + 8u * xs);
                bulk_commit_group();
            }
            if (next_tok >= 0) {
                // the next token's q: this CTA's DH columns of row qt into TMEM columns
                // [Q_COL, Q_COL + DH / 2) of lane qt, 32 columns per round (these warps have few
                // registers), zeros for rows that are not a live head
                const LaneRow lr =
                    lane_row<PAIR>(unit_at(tok_begin + next_tok, p.ntok, p.interleave), qt, p.h, p.m, p.useq);
                const uint4 *src =
                    reinterpret_cast<const uint4 *>(p.q + (lr.tok * p.h + lr.head) * (int64_t)D + crank * C::DH);
#pragma unroll 1
                for (int c = 0; c < C::NCHUNK; ++c) {
                    uint32_t r[32];
                    if (p.wide) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t w8[8];
                            if (lr.live) ld_global_nc_v8(src + c * 8 + 2 * k, w8);
#pragma unroll
                            for (int i = 0; i < 8; ++i) r[8 * k + i] = lr.live ? w8[i] : 0u;
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint4 v = lr.live ? __ldg(src + c * 8 + k) : make_uint4(0, 0, 0, 0);
                            r[4 * k] = v.x;
                            r[4 * k + 1] = v.y;
                            r[4 * k + 2] = v.z;
                            r[4 * k + 3] = v.w;
                        }
                    }
                    tmem_st32(tmem + lane_off + C::Q_COL + c * 32, r);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(BAR(B_QREADY));
            }
        }
        // every copy to the peer must have landed before either CTA of the cluster may exit (the
        // final cluster barrier comes after this), and the staging buffer must stay valid until
        // the copy engine has read it: wait for the bulk group to complete, not just its reads
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else if (warp < 4) {
        // ============================ softmax + epilogue (warps 0-3) ============================
        setmaxnreg_inc<REG_SOFTMAX>();
        const int t = threadIdx.x;                       // head row = TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        // live: this lane is a row of the MMA (a head of the token, or of one query of the pair);
        // whether that query exists is per unit (lane_row)
        const bool live = t < p.hm;
        const int head = PAIR && t >= p.h ? t - p.h : t;
        const float sink2 = live ? p.sink[head] * kLog2e : 0.0f;
        constexpr uint32_t XSTRIDE = C::X_STRIDE;
        auto q_row = [&](const LaneRow &lr) {
            return reinterpret_cast<const uint4 *>(p.q + (lr.tok * p.h + lr.head) * (int64_t)D + crank * C::DH);
        };
        auto load_q = [&](int64_t tok) {
            // this CTA's DH columns of q[tok][t] into TMEM columns [Q_COL, Q_COL + DH/2) of lane t.
            // Every load of the row is in flight at once (DH <= 256: at most 128 registers), so a
            // token change costs one memory latency, not one per 64 columns.  These loads queue
            // behind the row gathers in the SM's memory pipeline, so fewer, wider ones issue sooner.
            const LaneRow lr = lane_row<PAIR>(unit_at(tok, p.ntok, p.interleave), t, p.h, p.m, p.useq);
            const bool live = lr.live;
            const uint4 *src = q_row(lr);
            uint32_t r[C::NCHUNK][32];
            if (p.wide) {
#pragma unroll
                for (int c = 0; c < C::NCHUNK; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t w8[8];
                        if (live) ld_global_nc_v8(src + c * 8 + 2 * k, w8);
#pragma unroll
                        for (int i = 0; i < 8; ++i) r[c][8 * k + i] = live ? w8[i] : 0u;
                    }
            } else {
#pragma unroll
                for (int c = 0; c < C::NCHUNK; ++c)
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 v = live ? __ldg(src + c * 8 + k) : make_uint4(0, 0, 0, 0);
                        r[c][4 * k] = v.x;
                        r[c][4 * k + 1] = v.y;
                        r[c][4 * k + 2] = v.z;
                        r[c][4 * k + 3] = v.w;
                    }
            }
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c) tmem_st32(tmem + lane_off + C::Q_COL + c * 32, r[c]);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(BAR(B_QREADY));
        };
        int it = 0, J = 0, nzero = 0, seg = 0;
        bool ok = true;
        if (has_work) load_q(tok_begin);
        for (int64_t tok = tok_begin; has_work && ok && tok * T < e1; ++tok, ++seg) {
            const int a = (int)((e0 > tok * T ? e0 : tok * T) - tok * T);
            const int z = (int)((e1 < (tok + 1) * T ? e1 : (tok + 1) * T) - tok * T);
            const LaneRow next = lane_row<PAIR>(unit_at(tok + 1, p.ntok, p.interleave), t, p.h, p.m, p.useq);
            if (next.live && (tok + 1) * T < e1) {
                // the next token's q row is read as soon as this segment's scores are all read:
                // ask for it in L2 now, so that read does not wait on HBM
                const char *nq = reinterpret_cast<const char *>(q_row(next));
#pragma unroll
                for (int i = 0; i < C::DH * 2 / 128; ++i) prefetch_l2(nq + i * 128);
            }
            float m_used = -INFINITY, l = 0.0f;
            bool any = false;
            // each tile's row count and last flag come with its rows (the producers' meta)
            if (!warp_wait(BAR(B_FULL + it % NSTAGE), (it / NSTAGE) & 1, abort_flag)) {
                ok = false;
                break;
            }
            int2 cur = meta[it % NSTAGE];
            uint4 cur2 = make_uint4(0, 0, 0, 0);
            if constexpr (PAIR) cur2 = meta2[it % NSTAGE];
            const bool seg_empty = cur.x == 0;
            if (cur.x == 0) {
                // a segment without a single valid row: its only tile loads nothing; once all
                // 128 threads and the MMA thread have seen it, thread 0 hands the stage back
                mbar_arrive(BAR(B_ZREAD));
                if (t == 0) {
                    if (!mbar_wait(BAR(B_ZREAD), nzero & 1, abort_flag, kWaitLimitNs)) ok = false;
                    else mbar_arrive(BAR(B_EMPTY + it % NSTAGE));
                }
                ++nzero;
                ++it;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            } else {
                for (;;) {
                    // tile J: own scores from TMEM (+ the peer's partial scores) -> online softmax
                    // -> P (bf16) into shared memory
                    const int sb = J & 1;
                    const uint32_t ph = (J >> 1) & 1;
                    // A warp that gives up on a wait below, before the named barrier of this tile,
                    // still arrives there, so the other softmax warps are never left waiting on it
                    // (their own next wait then sees the abort flag).
                    auto leave = [&]() {
                        if constexpr (C::CL == 2) named_bar_arrive(1, 128);
                        ok = false;
                    };
                    if (!warp_wait(BAR(B_SFULL + sb), ph, abort_flag)) {
                        leave();
                        break;
                    }
                    tc_fence_after();
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem + lane_off + C::S_COL + sb * BN, r0);
                    tmem_ld32(tmem + lane_off + C::S_COL + sb * BN + 32, r1);
                    tmem_ld_wait(r0);
                    tmem_ld_wait(r1);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(B_SFREE + sb));   // the MMA may reuse the buffer
                    float s[BN];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        s[j] = __uint_as_float(r0[j]);
                        s[32 + j] = __uint_as_float(r1[j]);
                    }
                    if constexpr (C::CL == 2) {
                        const int xs = J % C::NXD;
                        if (!warp_wait<true>(BAR(B_XFULL + xs), (uint32_t)(J / C::NXD) & 1u, abort_flag)) {
                            leave();
                            break;
                        }
                        // arm the buffer for tile J + NX (its bytes cannot come before every
                        // softmax warp has released tile J below)
                        if (t == 0)
                            mbar_arrive_expect_tx(BAR(B_XFULL + xs), (uint32_t)((p.hm < 128 ? p.hm : 128) + 31) / 32 * C::XQ);
                        const uint32_t xbuf = base + C::SM_X + xs * XSTRIDE + warp * C::XQ + lane * 16;
                        if (live) {
                            // own half + peer half: the peer adds the same two f32 values
#pragma unroll
                            for (int k = 0; k < BN / 4; ++k) {
                                const float4 v = ld_shared_v4(xbuf + k * 512);
                                s[4 * k] += v.x;
                                s[4 * k + 1] += v.y;
                                s[4 * k + 2] += v.z;
                                s[4 * k + 3] += v.w;
                            }
                        }
                        // the exchange warps tell the peer when this buffer is free again (after
                        // the P V of this tile, whose P is written here below)
                    }
                    const int cnt = cur.x;
                    if (cnt < BN) {
#pragma unroll
                        for (int j = 0; j < BN; ++j)
                            if (j >= cnt) s[j] = -INFINITY;
                    }
                    if constexpr (PAIR) {
                        // only the rows this lane's query listed (the tile holds the pair's union)
                        const uint32_t mlo = t < p.h ? cur2.x : cur2.z, mhi = t < p.h ? cur2.y : cur2.w;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (!((mlo >> j) & 1u)) s[j] = -INFINITY;
                            if (!((mhi >> j) & 1u)) s[32 + j] = -INFINITY;
                        }
                    }
                    // row max of the raw scores (the scale is positive), as a tree
                    float mx[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
                    for (int j = 16; j < BN; j += 8)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], s[j + i]);
                    const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * p.scale_log2;
                    if (!any) {
                        m_used = tmax;
                    } else if (__any_sync(0xffffffffu, tmax > m_used + kRescaleThreshold)) {
                        // move the running max: wait for the P V in flight, rescale O and l
                        const int Jp = J - 1;
                        if (!warp_wait(BAR(B_PVDONE + (Jp & 3)), (Jp >> 2) & 1, abort_flag)) {
                            leave();
                            break;
                        }
                        tc_fence_after();
                        const float m_new = fmaxf(m_used, tmax);
                        // pair mode: a lane whose query has listed no row yet keeps m = -inf
                        const float f = PAIR && m_new == -INFINITY ? 1.0f : ex2(m_used - m_new);
                        l *= f;
#pragma unroll 1
                        for (int c = 0; c < C::DH / 32; ++c) {
                            uint32_t r[32];
                            tmem_ld32(tmem + lane_off + C::O_COL + c * 32, r);
                            tmem_ld_wait(r);
#pragma unroll
                            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
                            tmem_st32(tmem + lane_off + C::O_COL + c * 32, r);
                        }
                        tmem_st_wait();
                        m_used = m_new;
                    }
                    any = true;
                    // p = 2^(s * scale_log2 - m); P goes to the MMA in bf16, the row sum stays f32
                    uint32_t pk[32];
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
                    // pair mode: with m = -inf every score of the tile is -inf, and p must be 0
                    const float neg_m = PAIR && m_used == -INFINITY ? 0.0f : -m_used;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float p0 = ex2(fmaf(s[2 * j], p.scale_log2, neg_m));
                        const float p1 = ex2(fmaf(s[2 * j + 1], p.scale_log2, neg_m));
                        ls[j & 3] += p0 + p1;
                        pk[j] = pack_bf16x2(p0, p1);
                    }
                    l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    // row t of P, 16-byte unit u at unit u ^ (t % 8) of its 128-byte row.  With the d
                    // split P goes into this tile's exchange buffer, once all four warps have read
                    // the peer's scores from it; otherwise the buffer is free because S(J) was
                    // issued after the P V of tile J - NP and S(J) is complete.
                    if constexpr (C::CL == 2) named_bar_sync(1, 128);
                    const uint32_t prow = base + C::p_off(J) + t * 128;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(prow + ((u ^ (t & 7)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                    // each thread's P stores are made visible to the MMA (async proxy), then one
                    // arrival per warp
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(B_PFULL + (J & 3)));
                    ++J;
                    ++it;
                    if (cur.y) break;
                    if (!warp_wait(BAR(B_FULL + it % NSTAGE), (it / NSTAGE) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    cur = meta[it % NSTAGE];
                    if constexpr (PAIR) cur2 = meta2[it % NSTAGE];
                }
                if (!ok) break;
            }
            // every S of this segment has been read, so the next token's Q may replace this one.
            // With the d split the exchange warps load it after the segment's last score tile; a
            // segment without rows has no score tile, so its successor's q is loaded here, once
            // the q this segment was given has landed (both write the same TMEM columns)
            if ((tok + 1) * T < e1) {
                if constexpr (C::CL == 2) {
                    if (seg_empty) {
                        if (!warp_wait(BAR(B_QREADY), (uint32_t)seg & 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        load_q(tok + 1);
                    }
                } else {
                    load_q(tok + 1);
                }
            }
            if (any) {
                // O is final once the segment's last P V is done.  A parity wait is only exact
                // when the previous completion of the same barrier (four tiles back) has happened,
                // so wait for the P V before the last first (its predecessor is done: the scores
                // or peer scores of the last tile came after it), then for the last one.
                const int Jl = J - 1;
                if (Jl >= 1 && !warp_wait(BAR(B_PVDONE + ((Jl - 1) & 3)), ((Jl - 1) >> 2) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                if (!warp_wait(BAR(B_PVDONE + (Jl & 3)), (Jl >> 2) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            const bool whole = a == 0 && z == T;
            // O leaves TMEM EG x 32 columns per wait (at most 128 registers), not 32 at a time
            constexpr int EG = C::DH / 32 < 4 ? C::DH / 32 : 4;
            if (whole) {
                const float top = fmaxf(m_used, sink2);
                const float w = any ? ex2(m_used - top) : 0.0f;
                const float inv = w / (l * w + ex2(sink2 - top));
                const LaneRow lr = lane_row<PAIR>(unit_at(tok, p.ntok, p.interleave), t, p.h, p.m, p.useq);
                const bool live = lr.live;
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + (lr.tok * p.h + lr.head) * (int64_t)D + crank * C::DH);
                const float2 *cs_row = nullptr;
                if constexpr (ROPE) cs_row = p.rope + (p.rope_pos0 + lr.tok % p.m) * (p.rd / 2);
                const int col0 = (int)crank * C::DH;
#pragma unroll 1
                for (int c0 = 0; c0 < C::DH / 32; c0 += EG) {
                    uint32_t r[EG][32];
                    if (any) {
#pragma unroll
                        for (int g = 0; g < EG; ++g) tmem_ld32(tmem + lane_off + C::O_COL + (c0 + g) * 32, r[g]);
                        tmem_ld_wait(r);
                    } else {
#pragma unroll
                        for (int g = 0; g < EG; ++g)
#pragma unroll
                            for (int i = 0; i < 32; ++i) r[g][i] = 0u;
                    }
                    if (live && p.wide) {
#pragma unroll
                        for (int g = 0; g < EG; ++g)
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                uint32_t w8[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const float x0 = __uint_as_float(r[g][16 * k + 2 * i]) * inv;
                                    const float x1 = __uint_as_float(r[g][16 * k + 2 * i + 1]) * inv;
                                    w8[i] = out_pair<D, ROPE>(x0, x1, col0 + (c0 + g) * 32 + 16 * k + 2 * i, cs_row, p.rd);
                                }
                                st_global_v8(dst + (c0 + g) * 4 + 2 * k, w8);
                            }
                    } else if (live) {
#pragma unroll
                        for (int g = 0; g < EG; ++g)
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                uint32_t w4[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float x0 = __uint_as_float(r[g][8 * k + 2 * i]) * inv;
                                    const float x1 = __uint_as_float(r[g][8 * k + 2 * i + 1]) * inv;
                                    w4[i] = out_pair<D, ROPE>(x0, x1, col0 + (c0 + g) * 32 + 8 * k + 2 * i, cs_row, p.rd);
                                }
                                dst[(c0 + g) * 4 + k] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                    }
                }
            } else {
                // partial: unnormalised O, running max and sum (log2 domain) for the combine kernel
                const int slot = tok == tok_begin ? 0 : 1;
                float *ws = p.ws + ((size_t)cid * 2 + slot) * (size_t)(SLOT_HEADS * D + 2 * SLOT_HEADS);
                if (live && crank == 0) {
                    ws[SLOT_HEADS * D + t] = any ? m_used : -INFINITY;
                    ws[SLOT_HEADS * D + SLOT_HEADS + t] = l;
                }
                float4 *dst = reinterpret_cast<float4 *>(ws) + (size_t)(crank * C::DH / 4) * SLOT_HEADS + t;
#pragma unroll 1
                for (int c0 = 0; c0 < C::DH / 32; c0 += EG) {
                    uint32_t r[EG][32];
                    if (any) {
#pragma unroll
                        for (int g = 0; g < EG; ++g) tmem_ld32(tmem + lane_off + C::O_COL + (c0 + g) * 32, r[g]);
                        tmem_ld_wait(r);
                    } else {
#pragma unroll
                        for (int g = 0; g < EG; ++g)
#pragma unroll
                            for (int i = 0; i < 32; ++i) r[g][i] = 0u;
                    }
                    if (live) {
#pragma unroll
                        for (int g = 0; g < EG; ++g)
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                dst[(size_t)((c0 + g) * 8 + k) * SLOT_HEADS] =
                                    make_float4(__uint_as_float(r[g][4 * k]), __uint_as_float(r[g][4 * k + 1]),
                                                __uint_as_float(r[g][4 * k + 2]), __uint_as_float(r[g][4 * k + 3]));
                            }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(BAR(B_OFREE));
        }
    }

    // ---- teardown --------------------------------------------------------------------------------
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, DS_DEV_TIMEOUT);
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    // the exchange warps of both CTAs have waited for their copies into the peer to complete, so
    // after this barrier nothing is on its way into either CTA's shared memory
    if constexpr (C::CL == 2) cluster_sync();
}

// Merge the partials of every token that a range boundary cut, add the sink once, write bf16.
// The host lists the cut tokens: token, first part (cluster), number of parts and, per part, the
// partial slot it wrote (0: the part's first segment, 1: its last).  Block (i, y) merges columns
// [y * kCombineCols, (y + 1) * kCombineCols) of cut token i for every head, one thread per head,
// so each of its loads from the slots is 512 contiguous bytes per warp.
constexpr int kCombineCols = 16;   // columns per block: many small blocks read the partials in parallel

struct CombineParams {
    const float *sink;
    const float *ws;
    uint16_t *o;
    const float2 *rope;           // fused inverse RoPE (nullptr: none), see AttnArgs
    int64_t rope_pos0;
    int rd;
    int m;
    int h;
    int hm;                       // lanes in use (h, or 2 h in pair mode)
    int useq;                     // work units per sequence
    int interleave;               // unit order (unit_at)
    int64_t nunits;
    int ncut;
    int4 cut[kMaxCut];            // {unit, first part, parts, slot bits}
};

template <int D, bool ROPE, bool PAIR>
__global__ void __launch_bounds__(SLOT_HEADS) sparse_attn_combine_kernel(const CombineParams cp) {
    grid_dependency_wait();   // launched as a programmatic dependent of the attention kernel
    const int hh = threadIdx.x;
    if (hh >= cp.hm || (int)blockIdx.x >= cp.ncut) return;
    const int4 c = cp.cut[blockIdx.x];
    const LaneRow lr = lane_row<PAIR>(unit_at(c.x, cp.nunits, cp.interleave != 0), hh, cp.h, cp.m, cp.useq);
    if (!lr.live) return;
    const int64_t tok = lr.tok;
    const int kf = c.y, np = c.z;
    const uint32_t slots = (uint32_t)c.w;
    constexpr size_t SLOT = (size_t)SLOT_HEADS * D + 2 * SLOT_HEADS;
    constexpr int COLS = D < kCombineCols ? D : kCombineCols;
    auto part = [&](int i) -> const float * {
        return cp.ws + ((size_t)(kf + i) * 2 + ((slots >> i) & 1u)) * SLOT;
    };
    const float sink2 = cp.sink[lr.head] * kLog2e;
    const int c0 = blockIdx.y * (D < kCombineCols ? D : kCombineCols);
    if (np == 2) {
        // two parts (a cut between two neighbouring ranges): every load of both parts in flight
        // at once, the statistics beside the columns
        constexpr int COLS2 = D < kCombineCols ? D : kCombineCols;
        const float *p0 = part(0), *p1 = part(1);
        const float4 *s0 = reinterpret_cast<const float4 *>(p0) + (size_t)(c0 / 4) * SLOT_HEADS + hh;
        const float4 *s1 = reinterpret_cast<const float4 *>(p1) + (size_t)(c0 / 4) * SLOT_HEADS + hh;
        const float m0 = p0[SLOT_HEADS * D + hh], m1 = p1[SLOT_HEADS * D + hh];
        const float l0 = p0[SLOT_HEADS * D + SLOT_HEADS + hh], l1 = p1[SLOT_HEADS * D + SLOT_HEADS + hh];
        float4 x0[COLS2 / 4], x1[COLS2 / 4];
#pragma unroll
        for (int k = 0; k < COLS2 / 4; ++k) {
            x0[k] = s0[(size_t)k * SLOT_HEADS];
            x1[k] = s1[(size_t)k * SLOT_HEADS];
        }
        const float top2 = fmaxf(sink2, fmaxf(m0, m1));
        float den2 = exp2f(sink2 - top2);
        if (m0 != -INFINITY) den2 += exp2f(m0 - top2) * l0;
        if (m1 != -INFINITY) den2 += exp2f(m1 - top2) * l1;
        const float inv2 = 1.0f / den2;
        const float w0 = m0 == -INFINITY ? 0.0f : exp2f(m0 - top2) * inv2;
        const float w1 = m1 == -INFINITY ? 0.0f : exp2f(m1 - top2) * inv2;
        float acc2[COLS2];
#pragma unroll
        for (int k = 0; k < COLS2 / 4; ++k) {
            acc2[4 * k] = 0.0f + w0 * x0[k].x;
            acc2[4 * k + 1] = 0.0f + w0 * x0[k].y;
            acc2[4 * k + 2] = 0.0f + w0 * x0[k].z;
            acc2[4 * k + 3] = 0.0f + w0 * x0[k].w;
            acc2[4 * k] += w1 * x1[k].x;
            acc2[4 * k + 1] += w1 * x1[k].y;
            acc2[4 * k + 2] += w1 * x1[k].z;
            acc2[4 * k + 3] += w1 * x1[k].w;
        }
        uint4 *dst2 = reinterpret_cast<uint4 *>(cp.o + (tok * cp.h + lr.head) * (int64_t)D + c0);
        const float2 *cs_row2 = nullptr;
        if constexpr (ROPE) cs_row2 = cp.rope + (cp.rope_pos0 + tok % cp.m) * (cp.rd / 2);
#pragma unroll
        for (int k = 0; k < COLS2 / 8; ++k)
            dst2[k] = make_uint4(out_pair<D, ROPE>(acc2[8 * k], acc2[8 * k + 1], c0 + 8 * k, cs_row2, cp.rd),
                                 out_pair<D, ROPE>(acc2[8 * k + 2], acc2[8 * k + 3], c0 + 8 * k + 2, cs_row2, cp.rd),
                                 out_pair<D, ROPE>(acc2[8 * k + 4], acc2[8 * k + 5], c0 + 8 * k + 4, cs_row2, cp.rd),
                                 out_pair<D, ROPE>(acc2[8 * k + 6], acc2[8 * k + 7], c0 + 8 * k + 6, cs_row2, cp.rd));
        return;
    }
    float top = sink2;
    for (int i = 0; i < np; ++i) top = fmaxf(top, part(i)[SLOT_HEADS * D + hh]);
    float den = exp2f(sink2 - top);
    for (int i = 0; i < np; ++i) {
        const float mi = part(i)[SLOT_HEADS * D + hh];
        if (mi != -INFINITY) den += exp2f(mi - top) * part(i)[SLOT_HEADS * D + SLOT_HEADS + hh];
    }
    const float inv = 1.0f / den;
    float acc[COLS];
#pragma unroll
    for (int j = 0; j < COLS; ++j) acc[j] = 0.0f;
    for (int i = 0; i < np; ++i) {
        const float mi = part(i)[SLOT_HEADS * D + hh];
        if (mi == -INFINITY) continue;
        const float w = exp2f(mi - top) * inv;
        const float4 *src = reinterpret_cast<const float4 *>(part(i)) + (size_t)(c0 / 4) * SLOT_HEADS + hh;
#pragma unroll
        for (int k = 0; k < COLS / 4; ++k) {
            const float4 x = src[(size_t)k * SLOT_HEADS];
            acc[4 * k] += w * x.x;
            acc[4 * k + 1] += w * x.y;
            acc[4 * k + 2] += w * x.z;
            acc[4 * k + 3] += w * x.w;
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(cp.o + (tok * cp.h + lr.head) * (int64_t)D + c0);
    const float2 *cs_row = nullptr;
    if constexpr (ROPE) cs_row = cp.rope + (cp.rope_pos0 + tok % cp.m) * (cp.rd / 2);
#pragma unroll
    for (int k = 0; k < COLS / 8; ++k)
        dst[k] = make_uint4(out_pair<D, ROPE>(acc[8 * k], acc[8 * k + 1], c0 + 8 * k, cs_row, cp.rd),
                            out_pair<D, ROPE>(acc[8 * k + 2], acc[8 * k + 3], c0 + 8 * k + 2, cs_row, cp.rd),
                            out_pair<D, ROPE>(acc[8 * k + 4], acc[8 * k + 5], c0 + 8 * k + 4, cs_row, cp.rd),
                            out_pair<D, ROPE>(acc[8 * k + 6], acc[8 * k + 7], c0 + 8 * k + 6, cs_row, cp.rd));
}

// ---------------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------------

struct DeviceInfo {
    int sms = 0;
    int max_clusters[5] = {0, 0, 0, 0, 0};   // per kernel variant, co-resident clusters
    bool ready[5] = {false, false, false, false, false};
};
constexpr int kMaxDev = 64;
DeviceInfo g_dev[kMaxDev];
std::mutex g_dev_mutex;
// test switches: the bounded-wait path (ds_test_set_stall) and the kernel choice
// (ds_test_set_kernel: 0 automatic, 1 the cluster kernel, 2 the one-CTA kernel where it applies)
std::atomic<int> g_test_stall{0};
std::atomic<int> g_test_kernel{0};

// pair mode is built for the fixture's and the model's head_dim
template <int D>
constexpr bool kPairBuilt = D == 64 || D == 512;

template <int D, bool F8>
constexpr int dvar() { return F8 ? 4 : D == 64 ? 0 : D == 128 ? 1 : D == 256 ? 2 : 3; }

template <int D, bool F8 = false>
int max_clusters(int dev) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &di = g_dev[dev];
    if (di.ready[dvar<D, F8>()]) return di.max_clusters[dvar<D, F8>()];
    using C = Cfg<D>;
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaFuncSetAttribute(sparse_attn_tc_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
        return 0;
    // the instantiations with the output rotation and in pair mode have the same resources and
    // residency
    if (!F8 && cudaFuncSetAttribute(sparse_attn_tc_kernel<D, F8, !F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::SMEM_BYTES) != cudaSuccess)
        return 0;
    if constexpr (!F8 && kPairBuilt<D>) {
        if (cudaFuncSetAttribute(sparse_attn_tc_kernel<D, false, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
            return 0;
    }
    int nclusters = di.sms;
    if (C::CL > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C::CL * di.sms, 1, 1);
        cfg.blockDim = dim3(NTHREADS, 1, 1);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C::CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&nclusters, sparse_attn_tc_kernel<D, F8>, &cfg) != cudaSuccess ||
            nclusters < 1)
            return 0;
    }
    di.max_clusters[dvar<D, F8>()] = nclusters;
    di.ready[dvar<D, F8>()] = true;
    return nclusters;
}

int64_t choose_clusters(int64_t ntok, int topk, int gmax) { return split::choose_ranges(ntok, topk, gmax, BN); }
int64_t seg_cost(int64_t ntok, int64_t G) { return split::seg_cost(ntok, G, 4 * BN); }
bool splits_tokens(int64_t ntok, int topk, int64_t G) { return split::splits_units(ntok, topk, G, seg_cost(ntok, G)); }

// Workspace of one kernel variant for a problem on `dev` (0 when no token is cut).
template <int D, bool F8>
size_t variant_workspace_bytes(int dev, int64_t ntok, int topk) {
    const int gmax = max_clusters<D, F8>(dev);
    if (gmax <= 0 || ntok == 0 || topk == 0) return 0;
    const int64_t G = choose_clusters(ntok, topk, gmax);
    if (!splits_tokens(ntok, topk, G)) return 0;
    return (size_t)G * 2 * ((size_t)SLOT_HEADS * D + 2 * SLOT_HEADS) * sizeof(float);
}

// The workspace query serves every kernel that reads rows of width D: at d = 512 that is the bf16
// gather and the fp8 row store, whose co-resident cluster counts could differ, so the larger need
// is returned and either call accepts it.
template <int D>
size_t workspace_bytes_for(int64_t ntok, int topk) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    size_t need = variant_workspace_bytes<D, false>(dev, ntok, topk);
    if constexpr (D == 512) {
        const size_t f8 = variant_workspace_bytes<D, true>(dev, ntok, topk);
        if (f8 > need) need = f8;
    }
    return need;
}

template <int D, bool F8 = false>
int launch(const AttnArgs &a, cudaStream_t stream) {
    using C = Cfg<D>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return DS_ECUDA;
    const int gmax = max_clusters<D, F8>(dev);
    if (gmax <= 0) return DS_ECUDA;
    // work units: tokens, or in pair mode the query pairs (2j, 2j + 1) of each sequence, whose
    // index rows (a.idx) are the pairs' union rows
    const int useq = a.pair ? (a.m + 1) / 2 : a.m;
    const int64_t ntok = (int64_t)a.b * useq;
    const int64_t G = choose_clusters(ntok, a.topk, gmax);
    const int64_t K = seg_cost(ntok, G);
    if (a.topk > 0 && ntok > (INT64_MAX / (G + 1)) / (a.topk + K)) return DS_EUNSUPPORTED;   // G * ntok * (T + K) < 2^63
    const bool split = splits_tokens(ntok, a.topk, G);
    const size_t need = split ? (size_t)G * 2 * ((size_t)SLOT_HEADS * D + 2 * SLOT_HEADS) * sizeof(float) : 0;
    if (a.workspace_bytes < need || (need && !a.workspace)) return DS_EWORKSPACE;
    // the combine's table of cut tokens, checked before anything is launched
    CombineParams cpar;
    if (split) {
        cpar.sink = a.sink;
        cpar.ws = static_cast<const float *>(a.workspace);
        cpar.o = a.o;
        cpar.rope = reinterpret_cast<const float2 *>(a.rope);
        cpar.rope_pos0 = a.rope_pos0;
        cpar.rd = a.rd;
        cpar.m = a.m;
        cpar.h = a.h;
        cpar.hm = a.pair ? 2 * a.h : a.h;
        cpar.useq = useq;
        cpar.interleave = useq > 1 ? 1 : 0;
        cpar.nunits = ntok;
        cpar.ncut = split::cut_units(ntok, a.topk, K, G, cpar.cut);
        if (cpar.ncut <= 0) return DS_EUNSUPPORTED;
    }

    Params p;
    p.q = a.q;
    p.kv = a.kv;
    p.kv8 = a.kv8;
    p.kexp = a.kexp;
    p.sink = a.sink;
    p.idx = a.idx;
    p.o = a.o;
    p.ws = static_cast<float *>(a.workspace);
    p.n = a.n;
    p.ntok = ntok;
    p.topk = a.topk;
    p.seg_cost = (int)K;
    p.wide = (((uintptr_t)a.q | (uintptr_t)a.o) & 31u) == 0;
    p.m = a.m;
    p.h = a.h;
    p.useq = useq;
    p.hm = a.pair ? 2 * a.h : a.h;
    p.interleave = useq > 1;
    p.G = (int)G;
    p.scale_log2 = a.scale * kLog2e;
    p.status = a.status;
    p.stall_first_tile = g_test_stall.load(std::memory_order_relaxed) != 0 ? 1 : 0;
    p.rope = reinterpret_cast<const float2 *>(a.rope);
    p.rd = a.rd;
    p.rope_pos0 = a.rope_pos0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(C::CL * G), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    // programmatic dependent launch: the kernel's set-up overlaps the previous kernel on the
    // stream; it waits for that kernel (griddepcontrol.wait) before touching global memory
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C::CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C::CL > 1 ? 2 : 1;
    const bool rope = a.rope != nullptr;
    if ((rope && F8) || (a.pair && (F8 || rope || 2 * a.h > SLOT_HEADS))) return DS_EUNSUPPORTED;
    auto kernel = rope ? sparse_attn_tc_kernel<D, F8, !F8> : sparse_attn_tc_kernel<D, F8, false>;
    auto combine = rope ? sparse_attn_combine_kernel<D, true, false> : sparse_attn_combine_kernel<D, false, false>;
    if (a.pair) {
        if constexpr (!F8 && kPairBuilt<D>) {
            kernel = sparse_attn_tc_kernel<D, false, false, true>;
            combine = sparse_attn_combine_kernel<D, false, true>;
        } else {
            return DS_EUNSUPPORTED;
        }
    }
    if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) return DS_ECUDA;
    if (split) {
        cudaLaunchConfig_t ccfg = {};
        ccfg.gridDim = dim3((unsigned)cpar.ncut, (unsigned)((D + kCombineCols - 1) / kCombineCols), 1);
        ccfg.blockDim = dim3(SLOT_HEADS, 1, 1);
        ccfg.stream = stream;
        ccfg.attrs = attr;   // programmatic serialization only
        ccfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&ccfg, combine, cpar) != cudaSuccess) return DS_ECUDA;
    }
    return DS_OK;
}

}  // namespace tc

size_t sparse_attn_tc_workspace_bytes(int b, int m, int h, int d, int topk, bool pair) {
    const int64_t ntok = pair ? (int64_t)b * ((m + 1) / 2) : (int64_t)b * m;
    if (pair) topk *= 2;
    size_t need = 0;
    switch (d) {
        case 64: need = tc::workspace_bytes_for<64>(ntok, topk); break;
        case 128: need = tc::workspace_bytes_for<128>(ntok, topk); break;
        case 256: need = tc::workspace_bytes_for<256>(ntok, topk); break;
        case 512: need = tc::workspace_bytes_for<512>(ntok, topk); break;
        default: return 0;
    }
    // the one-CTA kernel serves some of the same calls (the query does not know which: it also
    // answers for the fp8 row store), so the larger need is returned
    if (sparse_attn_ot_supports(h, d, false, pair)) {
        const size_t ot = sparse_attn_ot_workspace_bytes(ntok, topk);
        if (ot > need) need = ot;
    }
    return need;
}

void set_test_stall(bool on) { tc::g_test_stall.store(on ? 1 : 0, std::memory_order_relaxed); }

namespace {
template <int D>
int tc_launches(int64_t ntok, int topk, size_t *workspace) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= tc::kMaxDev) return 1;
    const int gmax = tc::max_clusters<D>(dev);
    if (gmax <= 0) return 1;
    if (workspace) *workspace = tc::variant_workspace_bytes<D, false>(dev, ntok, topk);
    return tc::splits_tokens(ntok, topk, tc::choose_clusters(ntok, topk, gmax)) ? 2 : 1;
}
}  // namespace

int sparse_attn_plan(int b, int m, int h, int d, int topk, int *which, size_t *workspace) {
    const int64_t ntok = (int64_t)b * m;
    const int force = tc::g_test_kernel.load(std::memory_order_relaxed);
    const bool ot = force != 1 && sparse_attn_ot_supports(h, d, false, false) && ntok * h <= INT32_MAX &&
                    (force == 2 || sparse_attn_ot_preferred(ntok));
    if (which) *which = ot ? 2 : 1;
    if (workspace) *workspace = 0;
    if (ntok == 0 || topk == 0) return ntok == 0 ? 0 : 1;
    if (ot) {
        if (workspace) *workspace = sparse_attn_ot_workspace_bytes(ntok, topk);
        return sparse_attn_ot_launches(ntok, topk);
    }
    switch (d) {
        case 64: return tc_launches<64>(ntok, topk, workspace);
        case 128: return tc_launches<128>(ntok, topk, workspace);
        case 256: return tc_launches<256>(ntok, topk, workspace);
        case 512: return tc_launches<512>(ntok, topk, workspace);
        default: return 0;
    }
}
void set_test_kernel(int which) { tc::g_test_kernel.store(which, std::memory_order_relaxed); }

int launch_sparse_attn_tc(const AttnArgs &a, cudaStream_t stream) {
    const int force = tc::g_test_kernel.load(std::memory_order_relaxed);
    const int64_t ntok = (int64_t)a.b * a.m;
    if (force != 1 && sparse_attn_ot_supports(a.h, a.d, a.kv8 != nullptr, a.pair) &&
        ntok * a.h <= INT32_MAX && (force == 2 || sparse_attn_ot_preferred(ntok)))
        return launch_sparse_attn_ot(a, stream, tc::g_test_stall.load(std::memory_order_relaxed) != 0);
    if (a.kv8) return a.d == 512 ? tc::launch<512, true>(a, stream) : DS_EUNSUPPORTED;
    switch (a.d) {
        case 64: return tc::launch<64>(a, stream);
        case 128: return tc::launch<128>(a, stream);
        case 256: return tc::launch<256>(a, stream);
        case 512: return tc::launch<512>(a, stream);
        default: return DS_EUNSUPPORTED;
    }
}

}  // namespace dsattn
