"""CPU oracle for the sparse latent attention hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  The CUDA library never imports, links or calls it, and this package never touches
the CUDA library: the two share nothing but the seeded input generators.

The arithmetic lives in ``oracle.c`` (plain C11 loops, f32 where the pages fix f32, with a
float64 variant of ``sparse_attn``); this module only marshals numpy arrays through ctypes.
bf16 tensors travel as their raw ``uint16`` bit patterns.

Sources, by page title and section:
  * "DeepSeek V4.1", attention/attend: ``get_window_topk_idxs``, ``sparse_attn_kernel``.
  * "DeepSeek V4.1", attention/query-latent: ``Attention.__init__`` (ring buffer),
    ``Attention.forward`` (window and compressed rows concatenated before ``sparse_attn``).
  * "Module attn" (deepseek_v41_ref API page): Precision paragraph, ring-cache paragraph,
    ``FP8_BLOCK``, ``act_quant_inplace``, ``pow2_ceil``, ``sparse_attn``, ``window_topk_idxs``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

FP8_BLOCK = 32


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (plain gcc, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC,
             "-lm", "-lpthread"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.oracle_window_topk_idxs.argtypes = [P, i32, i64, i32]
        lib.oracle_window_topk_idxs.restype = i32
        lib.oracle_pow2_ceil.argtypes = [f32]
        lib.oracle_pow2_ceil.restype = f32
        lib.oracle_e4m3_round.argtypes = [f32]
        lib.oracle_e4m3_round.restype = f32
        lib.oracle_act_quant_inplace.argtypes = [P, i64]
        lib.oracle_act_quant_inplace.restype = i32
        lib.oracle_kv_quant_ring_write.argtypes = [P, i64, P, i64, i32, i32, i32, i64, i32]
        lib.oracle_kv_quant_ring_write.restype = i32
        lib.oracle_kv_quantize_fp8.argtypes = [P, i64, i32, P, P]
        lib.oracle_kv_quantize_fp8.restype = i32
        lib.oracle_kv_dequantize_fp8.argtypes = [P, P, i64, i32, P]
        lib.oracle_kv_dequantize_fp8.restype = i32
        lib.oracle_kv_quant_ring_write_fp8.argtypes = [P, i64, P, P, i64, i32, i32, i32, i64, i32]
        lib.oracle_kv_quant_ring_write_fp8.restype = i32
        lib.oracle_rope_table.argtypes = [P, i64, i32, ctypes.c_double]
        lib.oracle_rope_table.restype = i32
        lib.oracle_apply_rotary.argtypes = [P, i64, i32, i32, i64, i64, i64, P, i64, i32]
        lib.oracle_apply_rotary.restype = i32
        lib.oracle_kv_rope_quant_ring_write.argtypes = [P, i64, P, i64, i32, i32, i32, i64, i32, i32, P, i64]
        lib.oracle_kv_rope_quant_ring_write.restype = i32
        lib.oracle_indexer_topk.argtypes = [P, P, P, i32, i32, i32, i32, i64, i64, i32, i32, i64, P, P]
        lib.oracle_indexer_topk.restype = i32
        lib.oracle_indexer_select.argtypes = [P, i64, i32, i32, i64, i32, i32, i64, P]
        lib.oracle_indexer_select.restype = i32
        attn_args = [P, P, i64, P, P, i32, f32, P, i32, i32, i32, i32, P, i64, i32]
        lib.oracle_sparse_attn.argtypes = attn_args
        lib.oracle_sparse_attn.restype = i32
        lib.oracle_sparse_attn_f64.argtypes = attn_args
        lib.oracle_sparse_attn_f64.restype = i32
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def window_topk_idxs(s: int, start_pos: int, window: int) -> np.ndarray:
    """Index rows ``[queries][cols]`` int32 for one sequence (replicate over the batch yourself)."""
    lib = _load()
    rows = s if start_pos == 0 else 1
    out = np.empty((rows, max(min(s, window) if start_pos == 0 else window, 0)), dtype=np.int32)
    cols = lib.oracle_window_topk_idxs(_ptr(out), s, start_pos, window)
    if cols < 0:
        raise ValueError(f"window_topk_idxs undefined for s={s}, start_pos={start_pos}, window={window}")
    return out


def pow2_ceil(v: float) -> float:
    return float(_load().oracle_pow2_ceil(v))


def e4m3_round(y: float) -> float:
    return float(_load().oracle_e4m3_round(y))


def act_quant_inplace(x_bits: np.ndarray) -> np.ndarray:
    """fp8 round trip of bf16 bit patterns (uint16, size a multiple of 32), in place."""
    assert x_bits.dtype == np.uint16
    if _load().oracle_act_quant_inplace(_ptr(x_bits), x_bits.size) != 0:
        raise ValueError("act_quant_inplace needs a multiple of 32 values")
    return x_bits


def kv_quant_ring_write(kv_bits: np.ndarray, ring_bits: np.ndarray, start_pos: int, window: int) -> None:
    """kv_bits ``[b][s][d]`` (rounded in place) and ring_bits ``[b][window][d]`` (updated)."""
    assert kv_bits.dtype == np.uint16 and ring_bits.dtype == np.uint16
    b, s, d = kv_bits.shape
    assert ring_bits.shape == (b, window, d)
    rc = _load().oracle_kv_quant_ring_write(_ptr(kv_bits), s * d, _ptr(ring_bits), window * d, b, s, d,
                                            start_pos, window)
    if rc != 0:
        raise ValueError("kv_quant_ring_write: bad arguments")


def kv_quantize_fp8(x_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp8 row store of bf16 bit patterns ``[..., d]``: (e4m3fn codes ``[..., d]`` uint8,
    per-32 scale exponents ``[..., d / 32]`` int8, scale = 2^k)."""
    assert x_bits.dtype == np.uint16 and x_bits.shape[-1] % FP8_BLOCK == 0
    x = np.ascontiguousarray(x_bits)
    d = x.shape[-1]
    rows = x.size // d
    codes = np.empty(x.shape, dtype=np.uint8)
    exps = np.empty(x.shape[:-1] + (d // FP8_BLOCK,), dtype=np.int8)
    if _load().oracle_kv_quantize_fp8(_ptr(x), rows, d, _ptr(codes), _ptr(exps)) != 0:
        raise ValueError("kv_quantize_fp8: bad arguments")
    return codes, exps


def kv_dequantize_fp8(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of an fp8 row store (inverse of ``kv_quantize_fp8`` up to the round trip)."""
    assert codes.dtype == np.uint8 and exps.dtype == np.int8
    d = codes.shape[-1]
    assert exps.shape == codes.shape[:-1] + (d // FP8_BLOCK,)
    c, e = np.ascontiguousarray(codes), np.ascontiguousarray(exps)
    out = np.empty(codes.shape, dtype=np.uint16)
    if _load().oracle_kv_dequantize_fp8(_ptr(c), _ptr(e), c.size // d, d, _ptr(out)) != 0:
        raise ValueError("kv_dequantize_fp8: bad arguments")
    return out


def kv_quant_ring_write_fp8(kv_bits: np.ndarray, codes: np.ndarray, exps: np.ndarray, start_pos: int,
                            window: int) -> None:
    """kv_bits ``[b][s][d]`` (rounded in place); the fp8 ring ``codes [b][R][d]``, ``exps
    [b][R][d/32]`` (R >= window rows per sequence, slots 0..window-1 updated)."""
    assert kv_bits.dtype == np.uint16 and codes.dtype == np.uint8 and exps.dtype == np.int8
    b, s, d = kv_bits.shape
    R = codes.shape[1]
    assert codes.shape == (b, R, d) and exps.shape == (b, R, d // FP8_BLOCK) and R >= window
    rc = _load().oracle_kv_quant_ring_write_fp8(_ptr(kv_bits), s * d, _ptr(codes), _ptr(exps), R, b, s, d,
                                                start_pos, window)
    if rc != 0:
        raise ValueError("kv_quant_ring_write_fp8: bad arguments")


def rope_table(npos: int, dim: int, base: float) -> np.ndarray:
    """The ratio-0 RoPE table ``[npos][dim/2][2]`` f32 of (cos, sin), no YaRN."""
    out = np.empty((npos, dim // 2, 2), dtype=np.float32)
    if _load().oracle_rope_table(_ptr(out), npos, dim, float(base)) != 0:
        raise ValueError("rope_table: bad arguments")
    return out


def apply_rotary(x_bits: np.ndarray, rd: int, table: np.ndarray, start_pos: int, rows_per_pos: int,
                 positions_per_seq: int, inverse: bool = False) -> np.ndarray:
    """Rotate the last ``rd`` values of every row of ``x_bits [..., row_len]`` (bf16 bits, in place);
    row r is at position start_pos + (r // rows_per_pos) % positions_per_seq."""
    assert x_bits.dtype == np.uint16 and x_bits.flags["C_CONTIGUOUS"] and table.dtype == np.float32
    row_len = x_bits.shape[-1]
    assert table.shape[1] * 2 == rd
    rc = _load().oracle_apply_rotary(_ptr(x_bits), x_bits.size // row_len, row_len, rd, rows_per_pos,
                                     positions_per_seq, start_pos, _ptr(np.ascontiguousarray(table)),
                                     table.shape[0], 1 if inverse else 0)
    if rc != 0:
        raise ValueError("apply_rotary: bad arguments or a position outside the table")
    return x_bits


def kv_rope_quant_ring_write(kv_bits: np.ndarray, ring_bits: np.ndarray, start_pos: int, window: int, rd: int,
                             table: np.ndarray) -> None:
    """RoPE on the last rd values of kv_bits ``[b][s][d]`` (row t at start_pos + t), then the fp8
    round trip in place and the ring store into ring_bits ``[b][window][d]``."""
    assert kv_bits.dtype == np.uint16 and ring_bits.dtype == np.uint16 and table.dtype == np.float32
    b, s, d = kv_bits.shape
    assert ring_bits.shape == (b, window, d) and table.shape[1] * 2 == rd
    rc = _load().oracle_kv_rope_quant_ring_write(_ptr(kv_bits), s * d, _ptr(ring_bits), window * d, b, s, d,
                                                 start_pos, window, rd, _ptr(np.ascontiguousarray(table)),
                                                 table.shape[0])
    if rc != 0:
        raise ValueError("kv_rope_quant_ring_write: bad arguments")


def indexer_topk(q_bits: np.ndarray, k_bits: np.ndarray, w: np.ndarray, start_pos: int, ratio: int, topk: int,
                 offset: int = 0, return_scores: bool = False):
    """Indexer scores and top-k: q_bits ``[b][s][H][D]``, k_bits ``[b][T][D]`` (bf16 bits), w
    ``[b][s][H]`` f32.  Returns idx ``[b][s][kk]`` int32 (and scores ``[b][s][T]`` f32)."""
    assert q_bits.dtype == np.uint16 and k_bits.dtype == np.uint16 and w.dtype == np.float32
    b, s, H, D = q_bits.shape
    T = k_bits.shape[1]
    assert k_bits.shape == (b, T, D) and w.shape == (b, s, H)
    kk = min(topk, (start_pos + s) // ratio)
    idx = np.empty((b, s, max(kk, 0)), dtype=np.int32)
    scores = np.empty((b, s, T), dtype=np.float32) if return_scores else None
    got = _load().oracle_indexer_topk(_ptr(np.ascontiguousarray(q_bits)), _ptr(np.ascontiguousarray(k_bits)),
                                      _ptr(np.ascontiguousarray(w)), b, s, H, D, T, start_pos, ratio, topk, offset,
                                      None if scores is None else _ptr(scores), _ptr(idx))
    if got != kk:
        raise ValueError("indexer_topk: bad arguments (fewer compressed keys than the top-k needs?)")
    return (idx, scores) if return_scores else idx


def indexer_select(scores: np.ndarray, start_pos: int, ratio: int, topk: int, offset: int = 0) -> np.ndarray:
    """The Indexer's selection from given f32 scores ``[b][s][>= Tv]``: idx ``[b][s][kk]`` int32."""
    assert scores.dtype == np.float32 and scores.ndim == 3
    b, s, ld = scores.shape
    kk = min(topk, (start_pos + s) // ratio)
    idx = np.empty((b, s, max(kk, 0)), dtype=np.int32)
    got = _load().oracle_indexer_select(_ptr(np.ascontiguousarray(scores)), ld, b, s, start_pos, ratio, topk, offset,
                                        _ptr(idx))
    if got != kk:
        raise ValueError("indexer_select: bad arguments")
    return idx


def sparse_attn(q_bits: np.ndarray, kv_bits: np.ndarray, sink: np.ndarray, idx: np.ndarray, scale: float,
                tokens: np.ndarray | None = None, nthreads: int | None = None, f64: bool = False) -> np.ndarray:
    """Oracle sparse_attn.

    q_bits ``[b][m][h][d]`` uint16 (bf16 bits); kv_bits ``[b][n][d]`` uint16; sink ``[h]`` f32;
    idx ``[b][m][topk]`` int32.  ``tokens``: optional flattened token numbers ``bi*m + t`` to
    compute.  Returns bf16 bits ``[ntok][h][d]`` (uint16) from the f32 oracle, or float64 values
    from the f64 variant.  Without ``tokens`` the result is shaped ``[b][m][h][d]``.
    """
    lib = _load()
    b, m, h, d = q_bits.shape
    n = kv_bits.shape[1]
    topk = idx.shape[2]
    assert kv_bits.shape == (b, n, d) and idx.shape[:2] == (b, m)
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kv_bits = np.ascontiguousarray(kv_bits, dtype=np.uint16)
    sink = np.ascontiguousarray(sink, dtype=np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    if tokens is not None:
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        ntok = tokens.size
    else:
        ntok = b * m
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    if f64:
        out = np.zeros((ntok, h, d), dtype=np.float64)
        fn = lib.oracle_sparse_attn_f64
    else:
        out = np.zeros((ntok, h, d), dtype=np.uint16)
        fn = lib.oracle_sparse_attn
    rc = fn(_ptr(q_bits), _ptr(kv_bits), n, _ptr(sink), _ptr(idx), topk, float(scale), _ptr(out), b, m, h, d,
            _ptr(tokens) if tokens is not None else None, ntok, int(nthreads))
    if rc != 0:
        raise ValueError("oracle sparse_attn: bad arguments or index out of range")
    if tokens is None:
        out = out.reshape(b, m, h, d)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
