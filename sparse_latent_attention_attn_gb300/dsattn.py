"""Python binding of libdsattn (include/dsattn.h): argument marshalling only.

Every function here takes torch tensors that already live on the current CUDA device, checks
dtypes and shapes, and passes raw pointers, sizes and the current stream to the C ABI of the
same name.  All computation happens in the library's CUDA kernels; there is no fallback of any
kind: importing this module fails when ``libdsattn.so`` is missing.

Sources, by page title and section: "DeepSeek V4.1", attention/attend (get_window_topk_idxs,
sparse_attn_kernel, sparse_attn wrapper); attention/query-latent (Attention.__init__ ring buffer,
Attention.forward concatenation); "Module attn" (act_quant_inplace, pow2_ceil, FP8_BLOCK,
sparse_attn, window_topk_idxs, the ring-cache and Precision paragraphs).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m sparse_latent_attention_attn_gb300.build`"
                      " (or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

DS_OK = 0
DS_EINVAL = -1
DS_EUNSUPPORTED = -2
DS_EWORKSPACE = -3
DS_ECUDA = -4
DS_EDEVICE = -5
DS_DEV_TIMEOUT = 1
DS_DEV_BAD_INDEX = 2

_P = ctypes.c_void_p
_i32, _i64, _f32, _sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

_lib.ds_window_topk_idxs.argtypes = [_P, _i64, _i32, _i32, _i64, _i32, ctypes.POINTER(_i32), _P]
_lib.ds_window_topk_idxs.restype = _i32
_lib.ds_kv_quant_ring_write.argtypes = [_P, _i64, _P, _i64, _i32, _i32, _i32, _i64, _i32, _P]
_lib.ds_kv_quant_ring_write.restype = _i32
_lib.ds_sparse_attn_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.ds_sparse_attn_workspace_bytes.restype = _sz
_lib.ds_sparse_attn.argtypes = [_P, _P, _i64, _P, _P, _i32, _f32, _P, _i32, _i32, _i32, _i32, _P, _sz, _P]
_lib.ds_sparse_attn.restype = _i32
_lib.ds_sparse_attn_prefill_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.ds_sparse_attn_prefill_workspace_bytes.restype = _sz
_lib.ds_sparse_attn_prefill.argtypes = [_P, _P, _i64, _P, _P, _i32, _f32, _P, _i32, _i32, _i32, _i32, _P, _sz, _P]
_lib.ds_sparse_attn_prefill.restype = _i32
_lib.ds_sparse_attn_rope.argtypes = [_P, _P, _i64, _P, _P, _i32, _f32, _P, _i32, _i32, _i32, _i32, _P, _sz, _i32, _P,
                                    _i64, _i64, _P]
_lib.ds_sparse_attn_rope.restype = _i32
_lib.ds_apply_rotary.argtypes = [_P, _i64, _i32, _i32, _i64, _i64, _i64, _P, _i64, _i32, _P]
_lib.ds_apply_rotary.restype = _i32
_lib.ds_kv_rope_quant_ring_write.argtypes = [_P, _i64, _P, _i64, _i32, _i32, _i32, _i64, _i32, _i32, _P, _i64, _P]
_lib.ds_kv_rope_quant_ring_write.restype = _i32
_lib.ds_kv_quantize_fp8.argtypes = [_P, _i64, _i32, _P, _P, _P]
_lib.ds_kv_quantize_fp8.restype = _i32
_lib.ds_kv_quant_ring_write_fp8.argtypes = [_P, _i64, _P, _P, _i64, _i32, _i32, _i32, _i64, _i32, _P]
_lib.ds_kv_quant_ring_write_fp8.restype = _i32
_lib.ds_sparse_attn_fp8kv.argtypes = [_P, _P, _P, _i64, _P, _P, _i32, _f32, _P, _i32, _i32, _i32, _i32, _P, _sz, _P]
_lib.ds_sparse_attn_fp8kv.restype = _i32
_lib.ds_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_uint)]
_lib.ds_device_status.restype = _i32
_lib.ds_indexer_workspace_bytes.argtypes = [_i32, _i32, _i64, _i32]
_lib.ds_indexer_workspace_bytes.restype = _sz
_lib.ds_indexer_scores.argtypes = [_P, _P, _P, _i32, _i32, _i32, _i32, _i64, _i64, _i32, _P, _i64, _P]
_lib.ds_indexer_scores.restype = _i32
_lib.ds_indexer_select.argtypes = [_P, _i64, _i32, _i32, _i64, _i32, _i32, _i64, _P, _P]
_lib.ds_indexer_select.restype = _i32
_lib.ds_indexer_topk.argtypes = [_P, _P, _P, _i32, _i32, _i32, _i32, _i64, _i64, _i32, _i32, _i64, _P, _P, _sz, _P]
_lib.ds_indexer_topk.restype = _i32
_lib.ds_test_set_stall.argtypes = [_i32]
_lib.ds_test_set_stall.restype = None
_lib.ds_test_set_kernel.argtypes = [_i32]
_lib.ds_test_set_kernel.restype = _i32
_lib.ds_sparse_attn_launches.argtypes = [_i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32),
                                         ctypes.POINTER(ctypes.c_size_t)]
_lib.ds_sparse_attn_launches.restype = _i32
_lib.ds_status_string.argtypes = [_i32]
_lib.ds_status_string.restype = ctypes.c_char_p


class DsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_lib.ds_status_string(status).decode()} ({status})")
        self.status = status


def _check(fn: str, status: int) -> None:
    if status != DS_OK:
        raise DsError(fn, status)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


def window_topk_idxs(idx: torch.Tensor, b: int, s: int, start_pos: int, window: int, stream=None) -> int:
    """Write window index rows into ``idx`` (int32, last dim = row stride ``ld``); returns cols.

    ``idx`` is viewed as rows of length ``idx.shape[-1]``: row (bi, q) is ``idx.view(-1, ld)[bi*rows+q]``.
    """
    _need(idx, torch.int32, "idx")
    ld = idx.shape[-1]
    if idx.stride(-1) != 1 or not idx.is_contiguous():
        raise ValueError("idx must be contiguous")
    cols = _i32(0)
    _check("ds_window_topk_idxs",
           _lib.ds_window_topk_idxs(_ptr(idx), ld, b, s, start_pos, window, ctypes.byref(cols), _stream(stream)))
    return cols.value


def kv_quant_ring_write(kv: torch.Tensor, ring: torch.Tensor | None, start_pos: int, window: int,
                        stream=None) -> None:
    """fp8 round trip of ``kv`` [b][s][d] (bf16, rows contiguous) in place, then the ring store.

    ``ring`` is a bf16 view [b][>=window][d] whose rows are contiguous (it may be the leading
    ``window`` rows of a larger per-sequence kv tensor).
    """
    _need(kv, torch.bfloat16, "kv")
    b, s, d = kv.shape
    if kv.stride(2) != 1 or kv.stride(1) != d:
        raise ValueError("kv rows must be contiguous")
    ring_bstride = 0
    if ring is not None:
        _need(ring, torch.bfloat16, "ring")
        if ring.shape[0] != b or ring.shape[2] != d or ring.shape[1] < window or ring.stride(2) != 1 \
                or ring.stride(1) != d:
            raise ValueError("ring must be [b][>=window][d] with contiguous rows")
        ring_bstride = ring.stride(0)
    _check("ds_kv_quant_ring_write",
           _lib.ds_kv_quant_ring_write(_ptr(kv), kv.stride(0), _ptr(ring), ring_bstride, b, s, d, start_pos, window,
                                       _stream(stream)))


def sparse_attn_workspace_bytes(b: int, m: int, h: int, d: int, topk: int) -> int:
    return int(_lib.ds_sparse_attn_workspace_bytes(b, m, h, d, topk))


def sparse_attn(q: torch.Tensor, kv: torch.Tensor, sink: torch.Tensor, idx: torch.Tensor, scale: float,
                o: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """o[b][m][h][d] = sparse_attn(q[b][m][h][d], kv[b][n][d], sink[h], idx[b][m][topk], scale)."""
    _need(q, torch.bfloat16, "q")
    _need(kv, torch.bfloat16, "kv")
    _need(sink, torch.float32, "sink")
    _need(idx, torch.int32, "idx")
    b, m, h, d = q.shape
    n = kv.shape[1]
    topk = idx.shape[2]
    if kv.shape != (b, n, d) or idx.shape[:2] != (b, m) or sink.shape != (h,):
        raise ValueError("shape mismatch")
    for t, name in ((q, "q"), (kv, "kv"), (idx, "idx"), (sink, "sink")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if o is None:
        o = torch.empty_like(q)
    elif o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("o must be a contiguous bf16 tensor shaped like q")
    need = sparse_attn_workspace_bytes(b, m, h, d, topk)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("ds_sparse_attn",
           _lib.ds_sparse_attn(_ptr(q), _ptr(kv), n, _ptr(sink), _ptr(idx), topk, float(scale), _ptr(o), b, m, h, d,
                               _ptr(workspace), ws_bytes, _stream(stream)))
    return o


def sparse_attn_prefill_workspace_bytes(b: int, m: int, h: int, d: int, topk: int) -> int:
    return int(_lib.ds_sparse_attn_prefill_workspace_bytes(b, m, h, d, topk))


def sparse_attn_prefill(q: torch.Tensor, kv: torch.Tensor, sink: torch.Tensor, idx: torch.Tensor, scale: float,
                        o: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """``sparse_attn`` for a prefill chunk, queries 2j and 2j + 1 sharing one gather of the union
    of their index rows (valid entries of a row must be distinct)."""
    _need(q, torch.bfloat16, "q")
    _need(kv, torch.bfloat16, "kv")
    _need(sink, torch.float32, "sink")
    _need(idx, torch.int32, "idx")
    b, m, h, d = q.shape
    n = kv.shape[1]
    topk = idx.shape[2]
    if kv.shape != (b, n, d) or idx.shape[:2] != (b, m) or sink.shape != (h,):
        raise ValueError("shape mismatch")
    for t, name in ((q, "q"), (kv, "kv"), (idx, "idx"), (sink, "sink")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if o is None:
        o = torch.empty_like(q)
    elif o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("o must be a contiguous bf16 tensor shaped like q")
    need = sparse_attn_prefill_workspace_bytes(b, m, h, d, topk)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("ds_sparse_attn_prefill",
           _lib.ds_sparse_attn_prefill(_ptr(q), _ptr(kv), n, _ptr(sink), _ptr(idx), topk, float(scale), _ptr(o), b, m,
                                       h, d, _ptr(workspace), ws_bytes, _stream(stream)))
    return o


def sparse_attn_rope(q: torch.Tensor, kv: torch.Tensor, sink: torch.Tensor, idx: torch.Tensor, scale: float, rd: int,
                     table: torch.Tensor, start_pos: int, o: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """``sparse_attn`` with the inverse RoPE of the output's last ``rd`` values fused in: token t of
    every sequence is rotated back by the angle of position ``start_pos + t`` (``table`` as for
    ``apply_rotary``).  Bit-identical to ``sparse_attn`` then ``apply_rotary(o, ..., inverse=True)``."""
    _need(q, torch.bfloat16, "q")
    _need(kv, torch.bfloat16, "kv")
    _need(sink, torch.float32, "sink")
    _need(idx, torch.int32, "idx")
    _check_table(table, rd)
    b, m, h, d = q.shape
    n = kv.shape[1]
    topk = idx.shape[2]
    if kv.shape != (b, n, d) or idx.shape[:2] != (b, m) or sink.shape != (h,):
        raise ValueError("shape mismatch")
    for t, name in ((q, "q"), (kv, "kv"), (idx, "idx"), (sink, "sink")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if o is None:
        o = torch.empty_like(q)
    elif o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("o must be a contiguous bf16 tensor shaped like q")
    need = sparse_attn_workspace_bytes(b, m, h, d, topk)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("ds_sparse_attn_rope",
           _lib.ds_sparse_attn_rope(_ptr(q), _ptr(kv), n, _ptr(sink), _ptr(idx), topk, float(scale), _ptr(o), b, m,
                                    h, d, _ptr(workspace), ws_bytes, rd, _ptr(table), table.shape[0], start_pos,
                                    _stream(stream)))
    return o


def _check_table(table: torch.Tensor, rd: int) -> None:
    _need(table, torch.float32, "table")
    if table.dim() != 3 or table.shape[1] * 2 != rd or table.shape[2] != 2 or not table.is_contiguous():
        raise ValueError("table must be a contiguous f32 [positions][rd/2][2] of (cos, sin)")


def apply_rotary(x: torch.Tensor, rd: int, table: torch.Tensor, start_pos: int, rows_per_pos: int,
                 positions_per_seq: int, inverse: bool = False, stream=None) -> torch.Tensor:
    """Rotate the last ``rd`` values of every row of ``x [..., row_len]`` (bf16, contiguous) in place;
    row r is at position start_pos + (r // rows_per_pos) % positions_per_seq.  For q or o
    ``[b][m][h][d]``: rows_per_pos = h, positions_per_seq = m."""
    _need(x, torch.bfloat16, "x")
    _check_table(table, rd)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    row_len = x.shape[-1]
    _check("ds_apply_rotary",
           _lib.ds_apply_rotary(_ptr(x), x.numel() // row_len if row_len else 0, row_len, rd, rows_per_pos,
                                positions_per_seq, start_pos, _ptr(table), table.shape[0], 1 if inverse else 0,
                                _stream(stream)))
    return x


def kv_rope_quant_ring_write(kv: torch.Tensor, ring: torch.Tensor | None, start_pos: int, window: int, rd: int,
                             table: torch.Tensor, stream=None) -> None:
    """RoPE on the last ``rd`` values of ``kv`` [b][s][d] (row t at start_pos + t), then the fp8
    round trip in place and the ring store (see ``kv_quant_ring_write``)."""
    _need(kv, torch.bfloat16, "kv")
    _check_table(table, rd)
    b, s, d = kv.shape
    if kv.stride(2) != 1 or kv.stride(1) != d:
        raise ValueError("kv rows must be contiguous")
    ring_bstride = 0
    if ring is not None:
        _need(ring, torch.bfloat16, "ring")
        if ring.shape[0] != b or ring.shape[2] != d or ring.shape[1] < window or ring.stride(2) != 1 \
                or ring.stride(1) != d:
            raise ValueError("ring must be [b][>=window][d] with contiguous rows")
        ring_bstride = ring.stride(0)
    _check("ds_kv_rope_quant_ring_write",
           _lib.ds_kv_rope_quant_ring_write(_ptr(kv), kv.stride(0), _ptr(ring), ring_bstride, b, s, d, start_pos,
                                            window, rd, _ptr(table), table.shape[0], _stream(stream)))


def kv_quantize_fp8(x: torch.Tensor, codes: torch.Tensor | None = None, exps: torch.Tensor | None = None,
                    stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """fp8 row store of bf16 rows ``x [..., d]`` (contiguous): e4m3fn codes ``[..., d]`` uint8 and
    per-32 scale exponents ``[..., d / 32]`` int8 (scale = 2^k)."""
    _need(x, torch.bfloat16, "x")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    d = x.shape[-1]
    if d % 32:
        raise ValueError("the last dimension must be a multiple of 32")
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if exps is None:
        exps = torch.empty(x.shape[:-1] + (d // 32,), dtype=torch.int8, device=x.device)
    _need(codes, torch.uint8, "codes")
    _need(exps, torch.int8, "exps")
    if codes.shape != x.shape or exps.shape != x.shape[:-1] + (d // 32,) or not codes.is_contiguous() \
            or not exps.is_contiguous():
        raise ValueError("codes must be shaped like x and exps like x with d / 32 columns, both contiguous")
    _check("ds_kv_quantize_fp8",
           _lib.ds_kv_quantize_fp8(_ptr(x), x.numel() // d if d else 0, d, _ptr(codes), _ptr(exps), _stream(stream)))
    return codes, exps


def kv_quant_ring_write_fp8(kv: torch.Tensor, ring_codes: torch.Tensor, ring_exps: torch.Tensor, start_pos: int,
                            window: int, stream=None) -> None:
    """fp8 round trip of ``kv`` [b][s][d] in place; the ring is an fp8 row store ``ring_codes``
    [b][R][d] uint8, ``ring_exps`` [b][R][d/32] int8 (R >= window; it may be the leading rows of
    the store ``sparse_attn_fp8kv`` reads)."""
    _need(kv, torch.bfloat16, "kv")
    _need(ring_codes, torch.uint8, "ring_codes")
    _need(ring_exps, torch.int8, "ring_exps")
    b, s, d = kv.shape
    if kv.stride(2) != 1 or kv.stride(1) != d:
        raise ValueError("kv rows must be contiguous")
    R = ring_codes.shape[1]
    if ring_codes.shape != (b, R, d) or ring_exps.shape != (b, R, d // 32) or not ring_codes.is_contiguous() \
            or not ring_exps.is_contiguous() or R < window:
        raise ValueError("the ring must be contiguous [b][>=window][d] codes and [b][>=window][d/32] exps")
    _check("ds_kv_quant_ring_write_fp8",
           _lib.ds_kv_quant_ring_write_fp8(_ptr(kv), kv.stride(0), _ptr(ring_codes), _ptr(ring_exps), R, b, s, d,
                                           start_pos, window, _stream(stream)))


def sparse_attn_fp8kv(q: torch.Tensor, kv_codes: torch.Tensor, kv_exps: torch.Tensor, sink: torch.Tensor,
                      idx: torch.Tensor, scale: float, o: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """``sparse_attn`` with the rows read from an fp8 row store: kv_codes [b][n][d] uint8,
    kv_exps [b][n][d/32] int8.  Bit-identical to ``sparse_attn`` on the decoded rows."""
    _need(q, torch.bfloat16, "q")
    _need(kv_codes, torch.uint8, "kv_codes")
    _need(kv_exps, torch.int8, "kv_exps")
    _need(sink, torch.float32, "sink")
    _need(idx, torch.int32, "idx")
    b, m, h, d = q.shape
    n = kv_codes.shape[1]
    topk = idx.shape[2]
    if kv_codes.shape != (b, n, d) or kv_exps.shape != (b, n, d // 32) or idx.shape[:2] != (b, m) \
            or sink.shape != (h,):
        raise ValueError("shape mismatch")
    for t, name in ((q, "q"), (kv_codes, "kv_codes"), (kv_exps, "kv_exps"), (idx, "idx"), (sink, "sink")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if o is None:
        o = torch.empty_like(q)
    elif o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("o must be a contiguous bf16 tensor shaped like q")
    need = sparse_attn_workspace_bytes(b, m, h, d, topk)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("ds_sparse_attn_fp8kv",
           _lib.ds_sparse_attn_fp8kv(_ptr(q), _ptr(kv_codes), _ptr(kv_exps), n, _ptr(sink), _ptr(idx), topk,
                                     float(scale), _ptr(o), b, m, h, d, _ptr(workspace), ws_bytes,
                                     _stream(stream)))
    return o


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status bits (0 = clean)."""
    bits = ctypes.c_uint(0)
    st = _lib.ds_device_status(_stream(stream), ctypes.byref(bits))
    if st not in (DS_OK, DS_EDEVICE):
        raise DsError("ds_device_status", st)
    return bits.value


def _indexer_inputs(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor):
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(w, torch.float32, "w")
    b, s, H, D = q.shape
    T = k.shape[1]
    if k.shape != (b, T, D) or w.shape != (b, s, H):
        raise ValueError("shape mismatch: q [b][s][H][D], k [b][T][D], w [b][s][H]")
    for t, name in ((q, "q"), (k, "k"), (w, "w")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    return b, s, H, D, T


def indexer_visible(s: int, start_pos: int, ratio: int) -> int:
    """Compressed positions scored for a step of s queries at start_pos: (start_pos + s) // ratio."""
    return (start_pos + s) // ratio


def indexer_scores(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, start_pos: int, ratio: int,
                   scores: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """f32 scores [b][s][Tv] of the Indexer (-inf where a position is not visible yet)."""
    b, s, H, D, T = _indexer_inputs(q, k, w)
    Tv = indexer_visible(s, start_pos, ratio)
    if scores is None:
        scores = torch.empty((b, s, Tv), dtype=torch.float32, device=q.device)
    _need(scores, torch.float32, "scores")
    if scores.shape[:2] != (b, s) or scores.shape[2] < Tv or scores.stride(2) != 1 or scores.stride(1) != scores.shape[2] \
            or scores.stride(0) != s * scores.shape[2]:
        raise ValueError("scores must be a contiguous f32 [b][s][>= Tv]")
    _check("ds_indexer_scores",
           _lib.ds_indexer_scores(_ptr(q), _ptr(k), _ptr(w), b, s, H, D, T, start_pos, ratio, _ptr(scores),
                                  scores.shape[2], _stream(stream)))
    return scores


def indexer_select(scores: torch.Tensor, start_pos: int, ratio: int, topk: int, offset: int = 0,
                   idx: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Top-k positions per query from scores [b][s][>= Tv] (contiguous f32): int32 [b][s][kk]."""
    _need(scores, torch.float32, "scores")
    if not scores.is_contiguous():
        raise ValueError("scores must be contiguous")
    b, s, ld = scores.shape
    kk = min(topk, indexer_visible(s, start_pos, ratio))
    if idx is None:
        idx = torch.empty((b, s, kk), dtype=torch.int32, device=scores.device)
    _need(idx, torch.int32, "idx")
    if idx.shape != (b, s, kk) or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous int32 [b][s][kk]")
    _check("ds_indexer_select",
           _lib.ds_indexer_select(_ptr(scores), ld, b, s, start_pos, ratio, topk, offset, _ptr(idx), _stream(stream)))
    return idx


def indexer_workspace_bytes(b: int, s: int, start_pos: int, ratio: int) -> int:
    return int(_lib.ds_indexer_workspace_bytes(b, s, start_pos, ratio))


def indexer_topk(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, start_pos: int, ratio: int, topk: int,
                 offset: int = 0, idx: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """The Indexer's kept positions: int32 [b][s][min(topk, Tv)], ascending, + offset, -1 if unseen."""
    b, s, H, D, T = _indexer_inputs(q, k, w)
    kk = min(topk, indexer_visible(s, start_pos, ratio))
    if idx is None:
        idx = torch.empty((b, s, kk), dtype=torch.int32, device=q.device)
    _need(idx, torch.int32, "idx")
    if idx.shape != (b, s, kk) or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous int32 [b][s][kk]")
    need = indexer_workspace_bytes(b, s, start_pos, ratio)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check("ds_indexer_topk",
           _lib.ds_indexer_topk(_ptr(q), _ptr(k), _ptr(w), b, s, H, D, T, start_pos, ratio, topk, offset, _ptr(idx),
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return idx


def test_set_stall(on: bool) -> None:
    """Test hook: while on, every sparse_attn launch has a bounded wait run out (DS_DEV_TIMEOUT)."""
    _lib.ds_test_set_stall(1 if on else 0)


KERNEL_AUTO, KERNEL_CLUSTER, KERNEL_ONE_CTA = 0, 1, 2


def sparse_attn_launches(b: int, m: int, h: int, d: int, topk: int) -> tuple[int, int]:
    """(kernels a sparse_attn call of this shape launches, the attention kernel it runs:
    KERNEL_CLUSTER or KERNEL_ONE_CTA)."""
    n, which, _ = sparse_attn_plan(b, m, h, d, topk)
    return n, which


def sparse_attn_plan(b: int, m: int, h: int, d: int, topk: int) -> tuple[int, int, int]:
    """(kernels launched, attention kernel, workspace bytes that kernel needs) for a sparse_attn
    call of this shape."""
    which = ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    n = _lib.ds_sparse_attn_launches(b, m, h, d, topk, ctypes.byref(which), ctypes.byref(ws))
    if n < 0:
        raise DsError("ds_sparse_attn_launches", n)
    return n, which.value, ws.value


def test_set_kernel(which: int) -> None:
    """Test hook: the attention kernel ds_sparse_attn runs (KERNEL_AUTO, KERNEL_CLUSTER or
    KERNEL_ONE_CTA, the latter wherever it is built for the shape)."""
    _check("ds_test_set_kernel", _lib.ds_test_set_kernel(int(which)))


def status_string(status: int) -> str:
    return _lib.ds_status_string(status).decode()
