/*
 * dsattn.h -- C ABI of libdsattn, the GB300 (sm_103a) hot path of DeepSeek-V4.1 sparse latent
 * attention: the sliding-window index rows, the fp8 round trip of new KV rows into the ring,
 * and sparse_attn itself (gathered-row latent attention with an attention sink); beside them the
 * RoPE rotation (fused into the ring write, or on its own for the output's inverse rotation) and
 * an fp8 row store that keeps KV rows as their e4m3 codes.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers, owned by the caller.  The library allocates no
 *     device memory and keeps no state between calls (apart from one device status word per
 *     device, see ds_device_status).
 *   - bf16 tensors are passed as uint16_t bit patterns; all tensors are dense, row-major.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *     and never synchronises.  A returned DS_OK means the work was enqueued.
 *   - Errors are returned as negative codes (below); nothing is enqueued on an argument error.
 *
 * Sources are cited by page title and section:
 *   "DeepSeek V4.1", attention/attend        get_window_topk_idxs, sparse_attn_kernel, sparse_attn
 *   "DeepSeek V4.1", attention/query-latent  Attention.__init__ (window_kv_cache ring),
 *                                            Attention.forward (window + compressed concatenation)
 *   "Module attn" (deepseek_v41_ref)         Precision paragraph, ring-cache paragraph, FP8_BLOCK,
 *                                            act_quant_inplace, pow2_ceil, sparse_attn,
 *                                            window_topk_idxs, WindowCache, attention,
 *                                            apply_rotary, freqs_cis
 */
#ifndef DSATTN_H
#define DSATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st *ds_stream_t;

/* Status codes. */
#define DS_OK 0
#define DS_EINVAL (-1)        /* null pointer, negative size, misaligned pointer or stride    */
#define DS_EUNSUPPORTED (-2)  /* a shape outside the compiled set (see each call)              */
#define DS_EWORKSPACE (-3)    /* workspace smaller than ds_sparse_attn_workspace_bytes()      */
#define DS_ECUDA (-4)         /* a CUDA runtime call or kernel launch failed                  */
#define DS_EDEVICE (-5)       /* ds_device_status: a kernel flagged a problem (see bits below) */

/* Bits of the device status word (ds_device_status). */
#define DS_DEV_TIMEOUT 1u     /* a bounded wait inside a kernel gave up; that launch's output is invalid */
/* Every wait inside ds_sparse_attn's kernel gives up after 2 s, sets DS_DEV_TIMEOUT, drains the
 * launch's own copies and MMAs and returns, so the context stays usable (ds_test_set_stall
 * exercises that path). */
#define DS_DEV_BAD_INDEX 2u   /* an index >= n was seen; the entry was skipped                       */

/*
 * ds_window_topk_idxs -- sliding-window ring-slot index rows.
 * Source: "DeepSeek V4.1", attention/attend, get_window_topk_idxs; "Module attn", window_topk_idxs.
 *
 *   start_pos == 0 (prefill, s queries): cols = min(s, window).  Row q, column j holds
 *       v = max(0, q - window + 1) + j, or -1 when v > q (the causal window of query q into the
 *       chunk itself).  Rows are written for q = 0..s-1.
 *   start_pos  > 0 (decode, s must be 1): cols = window.  The single row lists the whole ring
 *       oldest first: column j holds v = (start_pos % window + 1 + j) mod window, or -1 when
 *       v > start_pos (ring still filling).
 *
 * idx        device int32, row (bi, q) starts at idx + (bi * rows + q) * ld, rows = s (prefill)
 *            or 1 (decode); only columns [0, cols) are written, so compressed indices can sit in
 *            columns [cols, ld) of the same rows (the concatenation of Attention.forward).
 * ld         row stride in int32 elements, >= cols.
 * b          sequences; the rows are the same for every sequence.
 * cols_out   optional HOST pointer that receives cols.
 * Errors: DS_EINVAL (null idx, b < 0, s < 1, window < 1, start_pos < 0, ld < cols);
 *         DS_EUNSUPPORTED for a chunked prefill (start_pos > 0 and s > 1), which the pages do not
 *         define.
 */
int ds_window_topk_idxs(int32_t *idx, int64_t ld, int b, int s, int64_t start_pos, int window,
                        int *cols_out, ds_stream_t stream);

/*
 * ds_kv_quant_ring_write -- fp8 round trip of new KV rows, in place, and their ring store.
 * Sources: "Module attn", FP8_BLOCK, pow2_ceil, act_quant_inplace, the Precision paragraph (the
 * round trip is bf16-exact) and the ring-cache paragraph; "DeepSeek V4.1", attention/query-latent,
 * Attention.__init__ (window_kv_cache [max_batch][window][head_dim]).
 *
 * Every block of 32 consecutive values of each row: amax = max |x| floored at 1e-4;
 * scale = 2^ceil(log2(amax / 448)) (f32 division, IEEE fields); x / scale clamped to +-448 and
 * rounded to e4m3 (round to nearest even); the result times scale, which is exact in bf16,
 * replaces x.  Then the token at position start_pos + t is stored to ring slot
 * (start_pos + t) % window when t >= s - window (the last `window` rows of the chunk).
 *
 * kv         device bf16 [b][s][d] rows, row stride d, batch stride kv_bstride (elements); in/out.
 * ring       device bf16, slot (bi, k) at ring + bi * ring_bstride + k * d; may be NULL when no
 *            ring store is wanted.  The ring may live inside a larger kv tensor (ring_bstride =
 *            that tensor's batch stride) so sparse_attn reads it without a copy.
 * d          multiple of 32; pointers 16-byte aligned; strides multiples of 8 elements.
 * Bit-exact with the definition above.  The ring slots written must not overlap the rows read.
 * Errors: DS_EINVAL (null kv, d % 32 != 0, misalignment, negative sizes, window < 1).
 */
int ds_kv_quant_ring_write(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride,
                           int b, int s, int d, int64_t start_pos, int window, ds_stream_t stream);

/*
 * ds_sparse_attn_workspace_bytes -- bytes of device workspace ds_sparse_attn needs for this
 * shape on the current device (0 when none).  Pure host function; the result depends on the
 * current device's SM count.  Returns 0 for shapes ds_sparse_attn rejects.
 */
size_t ds_sparse_attn_workspace_bytes(int b, int m, int h, int d, int topk);

/*
 * ds_sparse_attn -- gathered-row latent attention with an attention sink.
 * Sources: "Module attn", sparse_attn and the Precision paragraph; "DeepSeek V4.1",
 * attention/attend, sparse_attn_kernel and its sparse_attn wrapper; attention/query-latent,
 * Attention.forward (kv = window rows then compressed rows, indices concatenated likewise).
 *
 * For each sequence bi, query t and head hh, over the entries j of idx[bi][t] with idx >= 0:
 *     s_j = scale * dot(q[bi][t][hh], kv[bi][idx_j])
 *     o[bi][t][hh] = sum_j exp(s_j) * kv[bi][idx_j] / (sum_j exp(s_j) + exp(sink[hh]))
 * The sink counts in the denominator only; the gathered rows are both keys and values; entries
 * < 0 are skipped; a query with no entry gives o = 0.  Scores, softmax and accumulation are f32;
 * the probabilities are rounded to bf16 before the value product (as the pages' kernel does);
 * o is bf16.  Agreement with an f32 evaluation: |diff| <= 1e-2 + 1.6e-2 * |ref| elementwise.
 * Duplicate indices count as often as they are listed.
 *
 * q          device bf16 [b][m][h][d]
 * kv         device bf16 [b][n][d]
 * n          rows per sequence in kv (indices must be < n; larger ones are skipped and flagged
 *            with DS_DEV_BAD_INDEX)
 * sink       device f32 [h]
 * idx        device int32 [b][m][topk]
 * scale      softmax scale (head_dim^-0.5 in the model)
 * o          device bf16 [b][m][h][d], written
 * workspace  device scratch of at least ds_sparse_attn_workspace_bytes(b, m, h, d, topk) bytes,
 *            256-byte aligned (may be NULL when that size is 0); contents need no initialisation
 *            and are not meaningful after the call.  That size covers either attention kernel;
 *            the call checks the need of the kernel it runs (DS_EWORKSPACE when it is larger
 *            than workspace_bytes, before anything is enqueued).
 * Supported: d in {64, 128, 256, 512}; 1 <= h <= 128; topk >= 0; pointers 16-byte aligned.
 * Errors: DS_EINVAL, DS_EUNSUPPORTED, DS_EWORKSPACE, DS_ECUDA.
 */
int ds_sparse_attn(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink,
                   const int32_t *idx, int topk, float scale, uint16_t *o, int b, int m, int h, int d,
                   void *workspace, size_t workspace_bytes, ds_stream_t stream);

/*
 * ds_sparse_attn_rope -- ds_sparse_attn with the inverse RoPE of its output fused in.
 * Sources: "DeepSeek V4.1", attention/query-latent, Attention.forward (the attention output is
 * rotated back, apply_rotary_emb(o, inverse=True), before the output projection); "Module attn",
 * apply_rotary and freqs_cis.
 *
 * The result is bit-identical to ds_sparse_attn followed by
 *     ds_apply_rotary(o, b * m * h, d, rd, h, m, start_pos, table, table_rows, 1)
 * i.e. the last rd values of o[bi][t][hh] are rotated back by the angle of position start_pos + t
 * (the stored bf16 pair, f32 products, bf16 result), in the attention kernel's epilogue and in the
 * combine of tokens split across CTAs, without a second pass over o.
 * Arguments before rd are those of ds_sparse_attn (same workspace); rd, table and table_rows are
 * those of ds_apply_rotary: rd a multiple of 8 and <= d, table f32 [table_rows][rd / 2][2] of
 * (cos, sin), 8-byte aligned, start_pos + m - 1 < table_rows.
 * Errors: those of ds_sparse_attn, and DS_EINVAL for rd, table or start_pos outside the above.
 */
int ds_sparse_attn_rope(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink,
                        const int32_t *idx, int topk, float scale, uint16_t *o, int b, int m, int h, int d,
                        void *workspace, size_t workspace_bytes, int rd, const float *table,
                        int64_t table_rows, int64_t start_pos, ds_stream_t stream);

/*
 * ds_sparse_attn_prefill -- ds_sparse_attn for a prefill chunk, two neighbouring queries per
 * gather.  Sources: "DeepSeek V4.1", attention/attend, get_window_topk_idxs (prefill branch:
 * query q's causal window max(0, q - W + 1) .. q) and attention/query-latent (the Indexer's
 * compressed positions, re-sorted ascending); the operation is that of ds_sparse_attn.
 *
 * Queries 2j and 2j + 1 of every sequence are processed together: the sorted union of the valid
 * entries of their two index rows is gathered once and multiplied against the heads of both
 * queries (2 h rows of the tensor-core tile), each query's softmax keeping only the rows its own
 * index row lists.  Neighbouring prefill queries share all but one of their window rows and many
 * compressed rows, so the gathers and the MMA work per query shrink.
 * The result equals ds_sparse_attn's (same tolerance to an f32 evaluation) when the valid
 * entries of each index row are distinct, as window rows and the Indexer's positions are; a row
 * listed twice by one query counts once here, and DS_DEV_BAD_INDEX is raised for it.
 * Arguments and layouts are those of ds_sparse_attn; the workspace is
 * ds_sparse_attn_prefill_workspace_bytes(b, m, h, d, topk) bytes, 256-byte aligned (the union
 * rows, then the partials of pairs split across CTAs).
 * Supported: d in {64, 512}; 1 <= h <= 64; topk <= 8192; n <= 2^29 (DS_EUNSUPPORTED otherwise).
 * Errors: DS_EINVAL, DS_EUNSUPPORTED, DS_EWORKSPACE, DS_ECUDA.
 */
size_t ds_sparse_attn_prefill_workspace_bytes(int b, int m, int h, int d, int topk);
int ds_sparse_attn_prefill(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink,
                           const int32_t *idx, int topk, float scale, uint16_t *o, int b, int m, int h, int d,
                           void *workspace, size_t workspace_bytes, ds_stream_t stream);

/*
 * ds_apply_rotary -- RoPE (or its inverse) on the last rd values of rows of bf16 values, in place.
 * Sources: "Module attn", apply_rotary, freqs_cis and the Precision paragraph; "DeepSeek V4.1",
 * attention/query-latent, precompute_freqs_cis, apply_rotary_emb and Attention.forward (RoPE on
 * the last rope_dim of q and of the kv row; the inverse rotation on the attention output).
 *
 * Row r is at position pos = start_pos + (r / rows_per_pos) % positions_per_seq.  For each pair
 * j < rd / 2 of its last rd values, (a, b) = (x[2j], x[2j+1]) and (c, s) = table[pos][j]
 * (s negated when inverse != 0):  a' = a c - b s,  b' = a s + b c,  each product and sum rounded
 * to f32 separately (no fused multiply-add), then to bf16 (nearest even).  Bit-exact with that.
 *
 * x          device bf16 [rows][row_len], 16-byte aligned; in/out.  For q or o [b][m][h][d]:
 *            rows = b m h, row_len = d, rows_per_pos = h, positions_per_seq = m.
 * table      device f32 [table_rows][rd / 2][2] of (cos, sin), 8-byte aligned: the RoPE table of
 *            the layer (the ratio-0 layers: freq_j = 1 / base^(2j / rd), angle = pos freq_j)
 * rd         multiple of 8, <= row_len; row_len multiple of 8.
 * Errors: DS_EINVAL (null pointer, sizes, alignment, a position >= table_rows).
 */
int ds_apply_rotary(uint16_t *x, int64_t rows, int row_len, int rd, int64_t rows_per_pos, int64_t positions_per_seq,
                    int64_t start_pos, const float *table, int64_t table_rows, int inverse, ds_stream_t stream);

/*
 * ds_kv_rope_quant_ring_write -- ds_kv_quant_ring_write for a ratio-0 layer's new kv rows with
 * their RoPE fused in front: the last rd values of row t are first rotated to position
 * start_pos + t exactly as ds_apply_rotary does (bf16 result), then the block round trip and the
 * ring store follow ("Module attn": RoPE on the last rope_dim, then the kv row rounded through
 * fp8 in place, then the ring).  rd is a multiple of 32 (whole blocks), <= d; table as for
 * ds_apply_rotary, with start_pos + s - 1 < table_rows.  Other arguments and errors are those of
 * ds_kv_quant_ring_write.
 */
int ds_kv_rope_quant_ring_write(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride, int b, int s,
                                int d, int64_t start_pos, int window, int rd, const float *table, int64_t table_rows,
                                ds_stream_t stream);

/*
 * fp8 row store -- KV rows kept as their quantised values instead of the bf16 round trip.
 * Sources: "Module attn", act_quant_inplace and the Precision paragraph (the quantised value is
 * an e4m3 code times a power-of-two scale per block of 32, exact in bf16); "DeepSeek V4.1",
 * attention/query-latent (the compressed cache holds quantised values).  The pages define the
 * quantisation; storing its codes, rather than the bf16 values they decode to, is this
 * library's layout:
 *     codes  uint8 [rows][d]        e4m3fn bit pattern of x / scale (clamped, nearest even)
 *     exps   int8  [rows][d / 32]   k with scale = 2^k for the block (k in [-22, 120] for finite x)
 * A row decodes to exactly the bf16 row that ds_kv_quant_ring_write leaves behind, at 1 + 1/32
 * bytes per value instead of 2.
 */

/*
 * ds_kv_quantize_fp8 -- rows of bf16 values into the fp8 row store (x is not modified).
 * x          device bf16 [rows][d], contiguous, 16-byte aligned
 * codes      device uint8 [rows][d], 16-byte aligned, written
 * exps       device int8 [rows][d / 32], written
 * d          multiple of 32.  Bit-exact with the definition of ds_kv_quant_ring_write's scale and
 *            rounding.  Errors: DS_EINVAL (null pointer, rows < 0, d % 32 != 0, misalignment).
 */
int ds_kv_quantize_fp8(const uint16_t *x, int64_t rows, int d, uint8_t *codes, int8_t *exps,
                       ds_stream_t stream);

/*
 * ds_kv_quant_ring_write_fp8 -- ds_kv_quant_ring_write with an fp8 row store as the ring.
 * kv rows are rounded in place exactly as ds_kv_quant_ring_write does; the token at position
 * start_pos + t with t >= s - window stores its codes and exponents (from the same single
 * quantisation pass) in ring row (bi, (start_pos + t) % window), i.e. codes at
 * ring_codes + (bi * ring_bstride + slot) * d and exps at ring_exps + (bi * ring_bstride + slot)
 * * (d / 32).  ring_bstride is in rows (>= window), so the ring may be the first rows of an fp8
 * row store of [b][n][d] that ds_sparse_attn_fp8kv reads.
 * Errors: DS_EINVAL (null pointer, d % 32 != 0, misalignment, negative sizes, window < 1,
 *         ring_bstride < window).
 */
int ds_kv_quant_ring_write_fp8(uint16_t *kv, int64_t kv_bstride, uint8_t *ring_codes, int8_t *ring_exps,
                               int64_t ring_bstride, int b, int s, int d, int64_t start_pos, int window,
                               ds_stream_t stream);

/*
 * ds_sparse_attn_fp8kv -- ds_sparse_attn reading its rows from an fp8 row store.
 * The gathered rows are decoded on chip to the same bf16 values, so the result is bit-identical
 * to ds_sparse_attn on the decoded rows (same shape, same device), at half the gathered bytes.
 * kv_codes   device uint8 [b][n][d], 16-byte aligned
 * kv_exps    device int8 [b][n][d / 32]; every exponent must lie in [-126, 127]
 * Other arguments, the workspace (ds_sparse_attn_workspace_bytes) and the errors are those of
 * ds_sparse_attn.  Supported: d = 512, 1 <= h <= 128 (DS_EUNSUPPORTED otherwise).
 */
int ds_sparse_attn_fp8kv(const uint16_t *q, const uint8_t *kv_codes, const int8_t *kv_exps, int64_t n,
                         const float *sink, const int32_t *idx, int topk, float scale, uint16_t *o, int b,
                         int m, int h, int d, void *workspace, size_t workspace_bytes, ds_stream_t stream);

/*
 * ds_sparse_attn_static_scratch -- ds_sparse_attn for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for integration.  Some callers cannot
 * call cudaMalloc where they run attention (a runtime or memory manager that owns every device
 * allocation, a plugin handed only its input and output buffers, a hot path where allocation is
 * forbidden).  This call takes no workspace: the scratch that ds_sparse_attn would take from the
 * caller lives in a fixed device array of ds_sparse_attn_static_scratch_capacity() bytes
 * (32 MiB) compiled into the library, which every device that loads the library keeps reserved
 * until the process exits.  Nothing is allocated by the call.
 *
 * Arguments, layouts, results and errors are those of ds_sparse_attn, except that a shape whose
 * scratch need (that of the attention kernel the call runs) exceeds the capacity is refused with
 * DS_EWORKSPACE before anything is launched.
 * The first call on each device looks up that device's copy of the array (cudaGetSymbolAddress)
 * and so should happen before any stream capture on that device.  Every call on a device shares
 * the one array, and it keeps whatever the last call left there (no call needs it cleared):
 * calls whose work overlaps on the GPU (different streams, no ordering) race on it.
 */
int ds_sparse_attn_static_scratch(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink,
                                  const int32_t *idx, int topk, float scale, uint16_t *o, int b, int m, int h,
                                  int d, ds_stream_t stream);

/* Bytes of the fixed scratch array behind ds_sparse_attn_static_scratch (pure host function). */
size_t ds_sparse_attn_static_scratch_capacity(void);

/*
 * The Indexer: scores of compressed positions and the top-k kept per query.
 * Source: "DeepSeek V4.1", attention/query-latent, Indexer.forward (index_score = einsum of the
 * query's index heads with the shared index keys, relu, times weights_proj's per-head weights,
 * summed over heads; the causal compress_lens mask; topk = min(index_topk, end_pos // ratio); the
 * positions re-sorted ascending; -1 where a kept position is not visible, the others + offset).
 *
 * For query i (0 <= i < s) of sequence bi, at position start_pos + i, with
 *     lens_i = (start_pos + i + 1) / ratio      (compressed positions the query can see)
 *     Tv     = (start_pos + s) / ratio          (positions scored; end_pos // ratio)
 * the score of position t < Tv is
 *     score[t] = sum_h relu(dot(q[bi][i][h], k[bi][t])) * w[bi][i][h]    for t < lens_i
 *     score[t] = -inf                                                      for t >= lens_i
 * computed in f32 (dot products of bf16 values accumulated in f32, the head sum in f32).
 * The kk = min(topk, Tv) positions with the largest scores are kept (equal scores at the cut: the
 * smaller position first), written in ascending position order, t + offset, or -1 for t >= lens_i.
 * Layouts: q bf16 [b][s][H][D]; k bf16 [b][T][D] (T >= Tv rows per sequence); w f32 [b][s][H];
 * idx int32 [b][s][kk]; all contiguous, q and k 16-byte aligned, w 4-byte aligned.
 * Supported: D in {64, 128}; H a multiple of 16, <= 256 (DS_EUNSUPPORTED otherwise).
 * The q and k values are used as given (the pages' fp4 rounding of both is outside this call).
 */

/* ds_indexer_workspace_bytes -- scratch that ds_indexer_topk needs: the f32 scores of every query,
 * b * s * round_up(Tv, 4) * 4 bytes (pure host function; 0 for invalid arguments). */
size_t ds_indexer_workspace_bytes(int b, int s, int64_t start_pos, int ratio);

/* ds_indexer_scores -- the scores alone: scores[(bi * s + i) * ld + t] for t < Tv (f32, -inf where
 * t >= lens_i); ld >= Tv, scores 4-byte aligned.  Errors: DS_EINVAL, DS_EUNSUPPORTED, DS_ECUDA. */
int ds_indexer_scores(const uint16_t *q, const uint16_t *k, const float *w, int b, int s, int H, int D, int64_t T,
                      int64_t start_pos, int ratio, float *scores, int64_t ld, ds_stream_t stream);

/* ds_indexer_select -- the selection alone, from scores laid out as ds_indexer_scores writes them
 * (only t < lens_i of each row is read; the rest counts as -inf).  Exact: for the same scores the
 * kept positions and their order are fully determined.  offset + Tv must fit in int32.
 * Errors: DS_EINVAL, DS_ECUDA. */
int ds_indexer_select(const float *scores, int64_t ld, int b, int s, int64_t start_pos, int ratio, int topk,
                      int64_t offset, int32_t *idx, ds_stream_t stream);

/* ds_indexer_topk -- scores then selection, the scores kept in the caller's workspace
 * (>= ds_indexer_workspace_bytes, 16-byte aligned; DS_EWORKSPACE otherwise).
 * Errors: DS_EINVAL, DS_EUNSUPPORTED, DS_EWORKSPACE, DS_ECUDA. */
int ds_indexer_topk(const uint16_t *q, const uint16_t *k, const float *w, int b, int s, int H, int D, int64_t T,
                    int64_t start_pos, int ratio, int topk, int64_t offset, int32_t *idx, void *workspace,
                    size_t workspace_bytes, ds_stream_t stream);

/*
 * ds_device_status -- synchronise `stream`, then read and clear the current device's status word
 * (DS_DEV_* bits set by kernels since the last read).  Returns DS_OK when the word was 0,
 * DS_EDEVICE when a bit was set (the bits are stored to *bits_out when it is not NULL), or
 * DS_ECUDA.  This is the only call that synchronises.
 */
int ds_device_status(ds_stream_t stream, unsigned int *bits_out);

/*
 * ds_test_set_stall -- test hook for the bounded waits (no counterpart on the pages).  While `on`
 * is nonzero (process-wide, every device), each ds_sparse_attn / ds_sparse_attn_fp8kv launch has
 * its gather warps withhold the first tile's arrivals: the launch's waits run out after about
 * 2 s, it drains its own copies and MMAs, raises DS_DEV_TIMEOUT and returns with its output
 * invalid; no GPU fault is involved.  Default off; nothing in the library turns it on.
 */
void ds_test_set_stall(int on);

/*
 * ds_sparse_attn_launches -- the kernels a ds_sparse_attn call of this shape enqueues on the
 * current device (no counterpart on the pages; for accounting and tests).  Returns how many (0 for
 * an empty batch; 1 for topk = 0, the zero fill); stores to *kernel which attention kernel runs
 * (1 the 2-CTA cluster kernel, 2 the one-CTA kernel; see ds_test_set_kernel) and to
 * *workspace_bytes the workspace that kernel needs (at most ds_sparse_attn_workspace_bytes).
 * Either pointer may be NULL.  Pure host function.  Returns DS_EINVAL for a shape ds_sparse_attn
 * rejects.
 */
int ds_sparse_attn_launches(int b, int m, int h, int d, int topk, int *kernel, size_t *workspace_bytes);

/*
 * ds_test_set_kernel -- test hook for the choice of attention kernel (no counterpart on the
 * pages).  ds_sparse_attn runs one of two kernels with the same operation and tolerance: the
 * 2-CTA cluster kernel (any supported shape) or, for d = 512 and h <= 64, the one-CTA kernel
 * with a transposed accumulator (ds_sparse_attn_rope likewise; ds_sparse_attn_fp8kv always runs
 * the cluster kernel).  which = 0: that automatic choice (default); 1: always the cluster kernel;
 * 2: the one-CTA kernel wherever it is built for the shape (the same as 0 today).
 * Process-wide; nothing in the library sets it.  The workspace of
 * ds_sparse_attn_workspace_bytes suffices for either choice.
 * Returns DS_OK, or DS_EINVAL for another value of which.
 */
int ds_test_set_kernel(int which);

/* ds_status_string -- static text for a status code. */
const char *ds_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* DSATTN_H */
