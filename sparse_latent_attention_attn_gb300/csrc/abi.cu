// abi.cu -- the extern "C" entry points of libdsattn (declared in include/dsattn.h): argument
// checks, the per-device status word, NVTX ranges, and dispatch to the kernels.
#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "common.cuh"
#include "sparse_attn_ot.cuh"

namespace dsattn {
namespace {

// One status word per device; kernels OR DS_DEV_* bits into it.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_status_mutex;
unsigned int *g_status_ptr[kMaxDevices];

// Device address of this device's status word (host code may not take &g_status_word).
unsigned int *status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    return g_status_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_head_dim(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }

// An NVTX range around each entry point, named after it, so a timeline tool shows where each
// call's host work (checks, launch) starts and ends.  Without a tool attached it costs a check.
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
};

}  // namespace

// ds_sparse_attn and ds_sparse_attn_rope (rope == nullptr: no rotation of the output).
int sparse_attn_bf16(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink, const int32_t *idx, int topk,
                     float scale, uint16_t *o, int b, int m, int h, int d, void *workspace, size_t workspace_bytes,
                     const float *rope, int rd, int64_t rope_pos0, int64_t table_rows, ds_stream_t stream) {
    if (b < 0 || m < 0 || n < 0 || topk < 0 || h < 1) return DS_EINVAL;
    if (!supported_head_dim(d) || h > 128) return DS_EUNSUPPORTED;
    if ((int64_t)b * m == 0) return DS_OK;
    if (!q || !o || !sink || (topk > 0 && (!idx || !kv))) return DS_EINVAL;
    if (!aligned16(q) || !aligned16(o) || (kv && !aligned16(kv))) return DS_EINVAL;
    // The workspace is checked against the need of the kernel that will run (each launch checks
    // it before enqueueing anything); ds_sparse_attn_workspace_bytes, the larger need of the two
    // attention kernels, always suffices.
    AttnArgs a{q, kv, nullptr, nullptr, n, sink, idx, topk, scale, o, b, m, h, d, workspace, workspace_bytes,
               status_word(), rope, rd, rope_pos0};
    if (!a.status) return DS_ECUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (topk == 0) {   // nothing to attend to: every output is 0 (then rotated, as a separate pass would)
        if (cudaMemsetAsync(o, 0, (size_t)b * m * h * d * sizeof(uint16_t), st) != cudaSuccess) return DS_ECUDA;
        if (!rope) return DS_OK;
        (void)table_rows;
        return launch_apply_rotary(o, (int64_t)b * m * h, d, rd, h, m, rope_pos0, rope, true, st);
    }
    return launch_sparse_attn_tc(a, st);
}

}  // namespace dsattn

using namespace dsattn;

extern "C" {

int ds_window_topk_idxs(int32_t *idx, int64_t ld, int b, int s, int64_t start_pos, int window, int *cols_out,
                        ds_stream_t stream) {
    const Range range("ds_window_topk_idxs");
    if (!idx || b < 0 || s < 1 || window < 1 || start_pos < 0) return DS_EINVAL;
    if (start_pos > 0 && s != 1) return DS_EUNSUPPORTED;
    const int cols = start_pos == 0 ? (s < window ? s : window) : window;
    const int rows = start_pos == 0 ? s : 1;
    if (ld < cols) return DS_EINVAL;
    if (cols_out) *cols_out = cols;
    return launch_window_idx(idx, ld, b, rows, cols, start_pos, window, reinterpret_cast<cudaStream_t>(stream));
}

int ds_kv_quant_ring_write(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride, int b, int s,
                           int d, int64_t start_pos, int window, ds_stream_t stream) {
    const Range range("ds_kv_quant_ring_write");
    if (!kv || b < 0 || s < 0 || d <= 0 || d % 32 != 0 || window < 1 || start_pos < 0) return DS_EINVAL;
    if (kv_bstride < (int64_t)s * d || kv_bstride % 8 != 0 || !aligned16(kv)) return DS_EINVAL;
    if (ring && (ring_bstride < (int64_t)window * d || ring_bstride % 8 != 0 || !aligned16(ring))) return DS_EINVAL;
    return launch_kv_quant_ring(kv, kv_bstride, ring, ring_bstride, b, s, d, start_pos, window,
                                reinterpret_cast<cudaStream_t>(stream));
}

size_t ds_sparse_attn_workspace_bytes(int b, int m, int h, int d, int topk) {
    if (b < 0 || m < 0 || h < 1 || h > 128 || topk < 0 || !supported_head_dim(d)) return 0;
    return sparse_attn_tc_workspace_bytes(b, m, h, d, topk);
}

int ds_sparse_attn(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink, const int32_t *idx,
                   int topk, float scale, uint16_t *o, int b, int m, int h, int d, void *workspace,
                   size_t workspace_bytes, ds_stream_t stream) {
    const Range range("ds_sparse_attn");
    return sparse_attn_bf16(q, kv, n, sink, idx, topk, scale, o, b, m, h, d, workspace, workspace_bytes, nullptr, 0,
                            0, 0, stream);
}

int ds_sparse_attn_rope(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink, const int32_t *idx,
                        int topk, float scale, uint16_t *o, int b, int m, int h, int d, void *workspace,
                        size_t workspace_bytes, int rd, const float *table, int64_t table_rows, int64_t start_pos,
                        ds_stream_t stream) {
    const Range range("ds_sparse_attn_rope");
    if (rd <= 0 || rd % 8 != 0 || rd > d || start_pos < 0 || table_rows < 0) return DS_EINVAL;
    if (!table || (reinterpret_cast<uintptr_t>(table) & 7u) != 0) return DS_EINVAL;
    if (m > 0 && start_pos + m - 1 >= table_rows) return DS_EINVAL;   // a position outside the table
    return sparse_attn_bf16(q, kv, n, sink, idx, topk, scale, o, b, m, h, d, workspace, workspace_bytes, table, rd,
                            start_pos, table_rows, stream);
}

// ---- prefill: two neighbouring queries per gather ------------------------------------------------

namespace {
constexpr int kPrefillMaxTopk = 8192;          // index rows the union kernel sorts in shared memory
constexpr int64_t kPrefillMaxRows = (int64_t)1 << 29;   // rows addressable beside the listing bits

size_t prefill_union_bytes(int b, int m, int topk) {
    const size_t bytes = (size_t)b * ((m + 1) / 2) * (size_t)(2 * topk) * sizeof(int32_t);
    return (bytes + 255) & ~(size_t)255;
}
}  // namespace

size_t ds_sparse_attn_prefill_workspace_bytes(int b, int m, int h, int d, int topk) {
    if (b < 0 || m < 0 || h < 1 || h > 64 || topk < 1 || topk > kPrefillMaxTopk || (d != 64 && d != 512)) return 0;
    if ((int64_t)b * m == 0) return 0;
    return prefill_union_bytes(b, m, topk) + sparse_attn_tc_workspace_bytes(b, m, h, d, topk, true);
}

int ds_sparse_attn_prefill(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink, const int32_t *idx,
                           int topk, float scale, uint16_t *o, int b, int m, int h, int d, void *workspace,
                           size_t workspace_bytes, ds_stream_t stream) {
    const Range range("ds_sparse_attn_prefill");
    if (b < 0 || m < 0 || n < 0 || topk < 0 || h < 1) return DS_EINVAL;
    if ((d != 64 && d != 512) || h > 64 || topk > kPrefillMaxTopk || n > kPrefillMaxRows) return DS_EUNSUPPORTED;
    if ((int64_t)b * m == 0) return DS_OK;
    if (!q || !o || !sink || (topk > 0 && (!idx || !kv))) return DS_EINVAL;
    if (!aligned16(q) || !aligned16(o) || (kv && !aligned16(kv))) return DS_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (topk == 0)
        return cudaMemsetAsync(o, 0, (size_t)b * m * h * d * sizeof(uint16_t), st) == cudaSuccess ? DS_OK : DS_ECUDA;
    const size_t need = ds_sparse_attn_prefill_workspace_bytes(b, m, h, d, topk);
    if (workspace_bytes < need || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return DS_EWORKSPACE;
    unsigned int *status = status_word();
    if (!status) return DS_ECUDA;
    int32_t *uidx = static_cast<int32_t *>(workspace);
    const size_t ub = prefill_union_bytes(b, m, topk);
    int rc = launch_pair_union(idx, b, m, topk, n, uidx, status, st);
    if (rc != DS_OK) return rc;
    AttnArgs a{q, kv, nullptr, nullptr, n, sink, uidx, 2 * topk, scale, o, b, m, h, d,
               static_cast<char *>(workspace) + ub, workspace_bytes - ub, status, nullptr, 0, 0, true};
    return launch_sparse_attn_tc(a, st);
}

int ds_apply_rotary(uint16_t *x, int64_t rows, int row_len, int rd, int64_t rows_per_pos, int64_t positions_per_seq,
                    int64_t start_pos, const float *table, int64_t table_rows, int inverse, ds_stream_t stream) {
    const Range range("ds_apply_rotary");
    if (rows < 0 || rd <= 0 || rd % 8 != 0 || row_len < rd || row_len % 8 != 0 || rows_per_pos < 1 ||
        positions_per_seq < 1 || start_pos < 0)
        return DS_EINVAL;
    if (rows == 0) return DS_OK;
    if (!x || !table || !aligned16(x) || (reinterpret_cast<uintptr_t>(table) & 7u) != 0) return DS_EINVAL;
    const int64_t groups = (rows - 1) / rows_per_pos + 1;     // rows sharing a position, counted
    const int64_t span = groups < positions_per_seq ? groups : positions_per_seq;
    if (start_pos + span - 1 >= table_rows) return DS_EINVAL;   // a position outside the table
    return launch_apply_rotary(x, rows, row_len, rd, rows_per_pos, positions_per_seq, start_pos, table, inverse != 0,
                               reinterpret_cast<cudaStream_t>(stream));
}

int ds_kv_rope_quant_ring_write(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride, int b, int s,
                                int d, int64_t start_pos, int window, int rd, const float *table, int64_t table_rows,
                                ds_stream_t stream) {
    const Range range("ds_kv_rope_quant_ring_write");
    if (!kv || !table || b < 0 || s < 0 || d <= 0 || d % 32 != 0 || window < 1 || start_pos < 0) return DS_EINVAL;
    if (rd <= 0 || rd % 32 != 0 || rd > d || (reinterpret_cast<uintptr_t>(table) & 7u) != 0) return DS_EINVAL;
    if (s > 0 && start_pos + s - 1 >= table_rows) return DS_EINVAL;
    if (kv_bstride < (int64_t)s * d || kv_bstride % 8 != 0 || !aligned16(kv)) return DS_EINVAL;
    if (ring && (ring_bstride < (int64_t)window * d || ring_bstride % 8 != 0 || !aligned16(ring))) return DS_EINVAL;
    return launch_kv_rope_quant_ring(kv, kv_bstride, ring, ring_bstride, b, s, d, start_pos, window, rd, table,
                                     reinterpret_cast<cudaStream_t>(stream));
}

int ds_kv_quantize_fp8(const uint16_t *x, int64_t rows, int d, uint8_t *codes, int8_t *exps, ds_stream_t stream) {
    const Range range("ds_kv_quantize_fp8");
    if (rows < 0 || d <= 0 || d % 32 != 0) return DS_EINVAL;
    if (rows == 0) return DS_OK;
    if (!x || !codes || !exps || !aligned16(x) || !aligned16(codes)) return DS_EINVAL;
    return launch_kv_quantize_fp8(x, rows, d, codes, exps, reinterpret_cast<cudaStream_t>(stream));
}

int ds_kv_quant_ring_write_fp8(uint16_t *kv, int64_t kv_bstride, uint8_t *ring_codes, int8_t *ring_exps,
                               int64_t ring_bstride, int b, int s, int d, int64_t start_pos, int window,
                               ds_stream_t stream) {
    const Range range("ds_kv_quant_ring_write_fp8");
    if (!kv || !ring_codes || !ring_exps || b < 0 || s < 0 || d <= 0 || d % 32 != 0 || window < 1 || start_pos < 0)
        return DS_EINVAL;
    if (kv_bstride < (int64_t)s * d || kv_bstride % 8 != 0 || !aligned16(kv)) return DS_EINVAL;
    if (ring_bstride < window || !aligned16(ring_codes)) return DS_EINVAL;
    return launch_kv_quant_ring_fp8(kv, kv_bstride, ring_codes, ring_exps, ring_bstride, b, s, d, start_pos, window,
                                    reinterpret_cast<cudaStream_t>(stream));
}

int ds_sparse_attn_fp8kv(const uint16_t *q, const uint8_t *kv_codes, const int8_t *kv_exps, int64_t n,
                         const float *sink, const int32_t *idx, int topk, float scale, uint16_t *o, int b, int m,
                         int h, int d, void *workspace, size_t workspace_bytes, ds_stream_t stream) {
    const Range range("ds_sparse_attn_fp8kv");
    if (b < 0 || m < 0 || n < 0 || topk < 0 || h < 1) return DS_EINVAL;
    if (d != 512 || h > 128) return DS_EUNSUPPORTED;
    if ((int64_t)b * m == 0) return DS_OK;
    if (!q || !o || !sink || (topk > 0 && (!idx || !kv_codes || !kv_exps))) return DS_EINVAL;
    if (!aligned16(q) || !aligned16(o) || (kv_codes && !aligned16(kv_codes))) return DS_EINVAL;
    const size_t need = ds_sparse_attn_workspace_bytes(b, m, h, d, topk);
    if (workspace_bytes < need || (need > 0 && !workspace)) return DS_EWORKSPACE;
    AttnArgs a{q, nullptr, kv_codes, kv_exps, n, sink, idx, topk, scale, o, b, m, h, d, workspace,
               workspace_bytes, status_word()};
    if (!a.status) return DS_ECUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (topk == 0) {   // nothing to attend to: every output is 0
        return cudaMemsetAsync(o, 0, (size_t)b * m * h * d * sizeof(uint16_t), st) == cudaSuccess ? DS_OK : DS_ECUDA;
    }
    return launch_sparse_attn_tc(a, st);
}

// ---- the Indexer --------------------------------------------------------------------------------

namespace {
int64_t indexer_visible(int s, int64_t start_pos, int ratio) { return (start_pos + s) / ratio; }

int indexer_check(const uint16_t *q, const uint16_t *k, const float *w, int b, int s, int H, int D, int64_t T,
                  int64_t start_pos, int ratio) {
    if (b < 0 || s < 1 || H < 1 || T < 0 || start_pos < 0 || ratio < 1) return DS_EINVAL;
    if ((D != 64 && D != 128) || H % 16 != 0 || H > 256) return DS_EUNSUPPORTED;
    if (T < indexer_visible(s, start_pos, ratio)) return DS_EINVAL;          // keys the queries can see
    if (b == 0 || indexer_visible(s, start_pos, ratio) == 0) return DS_OK;   // nothing to score
    if (!q || !k || !w || !aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(w) & 3u) != 0)
        return DS_EINVAL;
    return DS_OK;
}
}  // namespace

size_t ds_indexer_workspace_bytes(int b, int s, int64_t start_pos, int ratio) {
    if (b < 0 || s < 1 || start_pos < 0 || ratio < 1) return 0;
    const int64_t Tv = indexer_visible(s, start_pos, ratio);
    return (size_t)b * s * (size_t)((Tv + 3) / 4 * 4) * sizeof(float);
}

int ds_indexer_scores(const uint16_t *q, const uint16_t *k, const float *w, int b, int s, int H, int D, int64_t T,
                      int64_t start_pos, int ratio, float *scores, int64_t ld, ds_stream_t stream) {
    const Range range("ds_indexer_scores");
    int st = indexer_check(q, k, w, b, s, H, D, T, start_pos, ratio);
    const int64_t Tv = indexer_visible(s, start_pos, ratio);
    if (st != DS_OK || b == 0 || Tv == 0) return st;
    if (!scores || ld < Tv || (reinterpret_cast<uintptr_t>(scores) & 3u) != 0) return DS_EINVAL;
    IndexerArgs a{q, k, w, b, s, H, D, T, start_pos, ratio, 0, 0, status_word()};
    if (!a.status) return DS_ECUDA;
    return launch_indexer_scores(a, scores, ld, reinterpret_cast<cudaStream_t>(stream));
}

int ds_indexer_select(const float *scores, int64_t ld, int b, int s, int64_t start_pos, int ratio, int topk,
                      int64_t offset, int32_t *idx, ds_stream_t stream) {
    const Range range("ds_indexer_select");
    if (b < 0 || s < 1 || start_pos < 0 || ratio < 1 || topk < 0) return DS_EINVAL;
    const int64_t Tv = indexer_visible(s, start_pos, ratio);
    const int64_t kk = topk < Tv ? topk : Tv;
    if (b == 0 || kk == 0) return DS_OK;
    if (!scores || !idx || ld < Tv || (reinterpret_cast<uintptr_t>(scores) & 3u) != 0) return DS_EINVAL;
    if (offset + Tv > INT32_MAX || offset < INT32_MIN) return DS_EINVAL;      // shifted positions fit int32
    IndexerArgs a{nullptr, nullptr, nullptr, b, s, 0, 0, 0, start_pos, ratio, topk, offset, nullptr};
    return launch_indexer_select(scores, ld, a, idx, reinterpret_cast<cudaStream_t>(stream));
}

int ds_indexer_topk(const uint16_t *q, const uint16_t *k, const float *w, int b, int s, int H, int D, int64_t T,
                    int64_t start_pos, int ratio, int topk, int64_t offset, int32_t *idx, void *workspace,
                    size_t workspace_bytes, ds_stream_t stream) {
    const Range range("ds_indexer_topk");
    if (topk < 0) return DS_EINVAL;
    int st = indexer_check(q, k, w, b, s, H, D, T, start_pos, ratio);
    const int64_t Tv = indexer_visible(s, start_pos, ratio);
    const int64_t kk = topk < Tv ? topk : Tv;
    if (st != DS_OK || b == 0 || kk == 0) return st;
    if (!idx) return DS_EINVAL;
    if (offset + Tv > INT32_MAX || offset < INT32_MIN) return DS_EINVAL;
    const size_t need = ds_indexer_workspace_bytes(b, s, start_pos, ratio);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return DS_EWORKSPACE;
    const int64_t ld = (Tv + 3) / 4 * 4;
    IndexerArgs a{q, k, w, b, s, H, D, T, start_pos, ratio, topk, offset, status_word()};
    if (!a.status) return DS_ECUDA;
    cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    float *scores = static_cast<float *>(workspace);
    st = launch_indexer_scores(a, scores, ld, strm);
    if (st != DS_OK) return st;
    return launch_indexer_select(scores, ld, a, idx, strm);
}

void ds_test_set_stall(int on) { set_test_stall(on != 0); }

int ds_sparse_attn_launches(int b, int m, int h, int d, int topk, int *kernel, size_t *workspace_bytes) {
    if (b < 0 || m < 0 || h < 1 || h > 128 || topk < 0 || !supported_head_dim(d)) return DS_EINVAL;
    return sparse_attn_plan(b, m, h, d, topk, kernel, workspace_bytes);
}

int ds_test_set_kernel(int which) {
    if (which < 0 || which > 2) return DS_EINVAL;
    set_test_kernel(which);
    return DS_OK;
}

int ds_device_status(ds_stream_t stream, unsigned int *bits_out) {
    unsigned int *p = status_word();
    if (!p) return DS_ECUDA;
    unsigned int bits = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return DS_ECUDA;
    if (cudaMemcpy(&bits, p, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess) return DS_ECUDA;
    if (bits) {
        const unsigned int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return DS_ECUDA;
    }
    if (bits_out) *bits_out = bits;
    return bits ? DS_EDEVICE : DS_OK;
}

const char *ds_status_string(int status) {
    switch (status) {
        case DS_OK: return "ok";
        case DS_EINVAL: return "invalid argument";
        case DS_EUNSUPPORTED: return "unsupported shape";
        case DS_EWORKSPACE: return "workspace too small";
        case DS_ECUDA: return "CUDA error";
        case DS_EDEVICE: return "a kernel flagged a device-side problem";
        default: return "unknown status";
    }
}

}  // extern "C"
