"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the pages or the mathematics fix: the ring-cache
worked example printed in "Module attn" (golden files), an independent enumeration of the window
(brute force), PyTorch's own float8_e4m3fn conversion and softmax / scaled_dot_product_attention
(library routines), closed forms, and invariances stated in "DeepSeek V4.1", attention/attend.
A plausible slip in the oracle (a dropped sink, a wrong scale, a transposed operand, an off-by-one
in the ring, a wrong rounding tie) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------------------
# helpers (bf16 <-> numbers through torch, independent of the oracle's C conversions)
# ----------------------------------------------------------------------------------------------

def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return from_bits(b).to(torch.float64).numpy()


def read_golden_ring():
    rows = {}
    with open(os.path.join(GOLDEN, "ring_cache_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            if line[0] == "decode":
                step = int(line[1])
                slot = int(line[3])
                ring = [int(x) for x in line[5:13]]
                row = [int(x) for x in line[14:22]]
                rows.setdefault("decode", []).append((step, slot, ring, row))
            else:
                rows[line[0]] = [int(x) for x in line[1:]]
    return rows


# ----------------------------------------------------------------------------------------------
# window_topk_idxs
# ----------------------------------------------------------------------------------------------

def test_window_rows_prefill_golden(oracle_mod):
    rows = oracle_mod.window_topk_idxs(12, 0, 8)
    assert rows.shape == (12, 8)
    with open(os.path.join(GOLDEN, "window_rows_prefill.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            q = int(line[0][1:])
            assert rows[q].tolist() == [int(x) for x in line[1:]], q


def test_window_rows_decode_golden(oracle_mod):
    g = read_golden_ring()
    for step, _slot, _ring, row in g["decode"]:
        got = oracle_mod.window_topk_idxs(1, step, g["window"][0])
        assert got.shape == (1, 8)
        assert got[0].tolist() == row


def _brute_decode_row(p, W):
    # the W most recent tokens p-W+1 .. p, oldest first; token t sits in slot t mod W; a token
    # before the sequence start leaves its slot empty
    return [(t % W) if t >= 0 else -1 for t in range(p - W + 1, p + 1)]


def _brute_prefill_rows(s, W):
    cols = min(s, W)
    out = []
    for q in range(s):
        seen = list(range(max(0, q - W + 1), q + 1))
        out.append(seen + [-1] * (cols - len(seen)))
    return out


@pytest.mark.parametrize("W", [1, 2, 3, 8, 128])
def test_window_rows_decode_bruteforce(oracle_mod, W):
    for p in list(range(1, 3 * W + 2)) + [10000, 16384, 131072]:
        got = oracle_mod.window_topk_idxs(1, p, W)[0].tolist()
        assert got == _brute_decode_row(p, W), (p, W)


@pytest.mark.parametrize("s,W", [(1, 8), (5, 8), (8, 8), (12, 8), (37, 16), (300, 128)])
def test_window_rows_prefill_bruteforce(oracle_mod, s, W):
    got = oracle_mod.window_topk_idxs(s, 0, W)
    assert got.tolist() == _brute_prefill_rows(s, W)


def test_window_rows_ring_filling_case(oracle_mod):
    # position 3 in an 8-slot ring: only slots 0..3 hold tokens yet
    assert oracle_mod.window_topk_idxs(1, 3, 8)[0].tolist() == [-1, -1, -1, -1, 0, 1, 2, 3]


def test_window_rows_chunked_prefill_undefined(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.window_topk_idxs(4, 5, 8)


# ----------------------------------------------------------------------------------------------
# fp8 round trip
# ----------------------------------------------------------------------------------------------

def _pow2_ceil_math(v: float) -> float:
    m, e = math.frexp(v)       # v = m * 2**e, 0.5 <= m < 1
    return v if m == 0.5 else math.ldexp(1.0, e)


def test_pow2_ceil_matches_math(oracle_mod):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        (2.0 ** rng.integers(-120, 120, 500)).astype(np.float32),
        rng.uniform(1e-30, 1e30, 2000).astype(np.float32),
        (rng.standard_normal(2000).astype(np.float32) ** 2 + np.float32(1e-20)),
        np.array([1.0, 0.75, 1.5, 2.0 ** -126, 3.0e38], dtype=np.float32),
    ])
    for v in vals:
        v = float(v)
        # 2**128 is not an f32: the power above the largest binade overflows to inf
        with np.errstate(over="ignore"):
            want = float(np.float32(_pow2_ceil_math(v)))
        assert oracle_mod.pow2_ceil(v) == want, v


def _torch_e4m3(y: torch.Tensor) -> torch.Tensor:
    return y.to(torch.float8_e4m3fn).to(torch.float32)


def test_e4m3_round_matches_torch_cast(oracle_mod):
    # every e4m3 value, every midpoint between neighbours (ties), and random points, both signs
    codes = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    mids = (codes[:-1] + codes[1:]) / 2
    rng = np.random.default_rng(2)
    rand = torch.from_numpy(rng.uniform(0, 448, 3000))
    ys = torch.cat([codes, mids, rand, codes[1:] * (1 + 2 ** -12), codes[1:] * (1 - 2 ** -12)])
    ys = torch.cat([ys, -ys]).to(torch.float32).clamp(-448, 448)
    want = _torch_e4m3(ys)
    got = torch.tensor([oracle_mod.e4m3_round(float(y)) for y in ys], dtype=torch.float32)
    assert torch.equal(got, want)


def _quant_reference_torch(x_bf16: torch.Tensor) -> torch.Tensor:
    """The round trip with library primitives: f32 amax/448, frexp pow2 ceiling, torch fp8 cast."""
    x = x_bf16.to(torch.float32).view(-1, 32)
    amax = x.abs().amax(dim=1).clamp(min=torch.tensor(1e-4, dtype=torch.float32))
    r = amax / torch.tensor(448.0, dtype=torch.float32)
    m, e = torch.frexp(r)
    scale = torch.where(m == 0.5, r, torch.ldexp(torch.ones_like(r), e))
    y = (x / scale[:, None]).clamp(-448, 448)
    return (_torch_e4m3(y) * scale[:, None]).to(torch.bfloat16).view(x_bf16.shape)


def test_quant_exhaustive_bf16_patterns_consecutive_blocks(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = from_bits(pats).to(torch.float32)
    finite = torch.isfinite(vals).numpy()
    pats = np.where(finite, pats, np.uint16(0))
    x = from_bits(pats).clone()
    want = to_bits(_quant_reference_torch(x))
    got = oracle_mod.act_quant_inplace(pats.copy())
    assert np.array_equal(got, want)


@pytest.mark.parametrize("anchor_exp", [-20, -9, -6, -1, 0, 3, 7, 12, 40])
def test_quant_every_bf16_value_at_fixed_scale(oracle_mod, anchor_exp):
    # each finite bf16 value of magnitude <= anchor goes through a block whose amax is the anchor,
    # so the whole e4m3 range (subnormals and ties included) is exercised at one scale
    anchor = 448.0 * 2.0 ** anchor_exp
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = from_bits(pats).to(torch.float64)
    keep = torch.isfinite(vals) & (vals.abs() <= anchor)
    vals = vals[keep].to(torch.bfloat16)
    nb = (vals.numel() + 30) // 31
    blocks = torch.zeros((nb, 32), dtype=torch.bfloat16)
    flat = torch.zeros(nb * 31, dtype=torch.bfloat16)
    flat[: vals.numel()] = vals
    blocks[:, :31] = flat.view(nb, 31)
    blocks[:, 31] = anchor
    want = to_bits(_quant_reference_torch(blocks))
    got = oracle_mod.act_quant_inplace(to_bits(blocks).reshape(-1))
    assert np.array_equal(got, want.reshape(-1))


def test_quant_random_blocks_match_library(oracle_mod):
    g = torch.Generator().manual_seed(3)
    x = torch.randn((4096, 32), generator=g) * torch.exp(torch.randn((4096, 1), generator=g) * 6)
    x = x.to(torch.bfloat16)
    want = to_bits(_quant_reference_torch(x))
    got = oracle_mod.act_quant_inplace(to_bits(x).reshape(-1))
    assert np.array_equal(got, want.reshape(-1))


def test_quant_properties(oracle_mod):
    g = torch.Generator().manual_seed(4)
    x = to_bits(torch.randn((512, 32), generator=g)).reshape(-1)
    once = oracle_mod.act_quant_inplace(x.copy())
    twice = oracle_mod.act_quant_inplace(once.copy())
    assert np.array_equal(once, twice)                       # idempotent
    zero = np.zeros(64, dtype=np.uint16)
    assert np.array_equal(oracle_mod.act_quant_inplace(zero.copy()), zero)   # amax floor, no NaN
    # values already on the e4m3 grid times a block-wide power of two are unchanged
    codes = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
    rng = np.random.default_rng(5)
    for k in (-12, -3, 0, 5, 20):
        blk = codes[rng.integers(0, 127, 32)] * (2.0 ** k)
        blk[0] = 448.0 * 2.0 ** k
        blk = blk * torch.from_numpy(rng.choice([-1.0, 1.0], 32)).to(torch.float32)
        b = to_bits(blk)
        assert np.array_equal(oracle_mod.act_quant_inplace(b.copy()), b)
    # every output is e4m3 * 2^k for the block's scale: dividing by the scale lands on the grid
    vals = bits_to_f64(once).reshape(-1, 32)
    src = bits_to_f64(x).reshape(-1, 32)
    for r in range(0, 512, 37):
        amax = max(np.abs(src[r]).max(), 1e-4)
        scale = _pow2_ceil_math(float(np.float32(np.float32(amax) / np.float32(448.0))))
        y = torch.from_numpy(vals[r] / scale).to(torch.float32)
        assert torch.equal(_torch_e4m3(y), y)


# ----------------------------------------------------------------------------------------------
# ring write: the worked example
# ----------------------------------------------------------------------------------------------

def _token_rows(tokens, d):
    # row of token t holds the value t+1 everywhere: small integers sit on the fp8 grid, so the
    # round trip leaves them unchanged and the ring contents name their tokens
    return to_bits(torch.tensor([[float(t + 1)] * d for t in tokens], dtype=torch.float32))


def test_ring_worked_example(oracle_mod):
    g = read_golden_ring()
    W, S = g["window"][0], g["prefill_tokens"][0]
    d = 64
    ring = np.zeros((1, W, d), dtype=np.uint16)
    chunk = _token_rows(range(S), d).reshape(1, S, d)
    oracle_mod.kv_quant_ring_write(chunk, ring, 0, W)
    slot_tokens = bits_to_f64(ring)[0, :, 0].astype(int) - 1
    assert slot_tokens.tolist() == g["ring_after_prefill"]
    for step, slot, ring_after, _row in g["decode"]:
        new = _token_rows([step], d).reshape(1, 1, d)
        before = ring.copy()
        oracle_mod.kv_quant_ring_write(new, ring, step, W)
        changed = np.nonzero((ring != before).any(axis=2)[0])[0].tolist()
        assert changed == [slot]
        assert (bits_to_f64(ring)[0, :, 0].astype(int) - 1).tolist() == ring_after


def test_ring_write_rounds_in_place_and_keeps_last_window(oracle_mod):
    g = torch.Generator().manual_seed(6)
    b, s, d, W, p0 = 3, 20, 64, 8, 37
    raw = to_bits(torch.randn((b, s, d), generator=g))
    kv = raw.copy()
    ring = np.full((b, W, d), 0x7f7f, dtype=np.uint16)
    oracle_mod.kv_quant_ring_write(kv, ring, p0, W)
    want = oracle_mod.act_quant_inplace(raw.copy().reshape(-1)).reshape(b, s, d)
    assert np.array_equal(kv, want)
    for t in range(s - W, s):
        assert np.array_equal(ring[:, (p0 + t) % W], want[:, t])


# ----------------------------------------------------------------------------------------------
# fp8 row store (codes + per-32 power-of-two exponents)
# ----------------------------------------------------------------------------------------------

def _fp8_store_reference_torch(x_bf16: torch.Tensor):
    """Codes and exponents with library primitives: f32 amax/448, frexp pow2 ceiling, torch's
    float8_e4m3fn cast read back as its bit pattern."""
    x = x_bf16.to(torch.float32).reshape(-1, 32)
    amax = x.abs().amax(dim=1).clamp(min=torch.tensor(1e-4, dtype=torch.float32))
    r = amax / torch.tensor(448.0, dtype=torch.float32)
    m, e = torch.frexp(r)
    scale = torch.where(m == 0.5, r, torch.ldexp(torch.ones_like(r), e))
    k = torch.frexp(scale)[1] - 1
    y = (x / scale[:, None]).clamp(-448, 448)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy().reshape(-1), k.to(torch.int8).numpy()


def _fp8_decode_torch(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    c = torch.from_numpy(codes.reshape(-1, 32).copy()).view(torch.float8_e4m3fn).to(torch.float32)
    v = torch.ldexp(c, torch.from_numpy(exps.reshape(-1, 1).astype(np.int32)))
    return to_bits(v.reshape(-1))


def test_fp8_store_exhaustive_bf16_patterns_match_library(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = torch.isfinite(from_bits(pats).to(torch.float32)).numpy()
    pats = np.where(finite, pats, np.uint16(0))
    want_c, want_k = _fp8_store_reference_torch(from_bits(pats).clone())
    codes, exps = oracle_mod.kv_quantize_fp8(pats.reshape(-1, 64))
    assert np.array_equal(codes.reshape(-1), want_c)
    assert np.array_equal(exps.reshape(-1), want_k)


@pytest.mark.parametrize("anchor_exp", [-20, -9, -1, 0, 7, 40])
def test_fp8_store_every_bf16_value_at_fixed_scale(oracle_mod, anchor_exp):
    anchor = 448.0 * 2.0 ** anchor_exp
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = from_bits(pats).to(torch.float64)
    vals = vals[torch.isfinite(vals) & (vals.abs() <= anchor)].to(torch.bfloat16)
    nb = (vals.numel() + 30) // 31
    blocks = torch.zeros((nb, 32), dtype=torch.bfloat16)
    flat = torch.zeros(nb * 31, dtype=torch.bfloat16)
    flat[: vals.numel()] = vals
    blocks[:, :31] = flat.view(nb, 31)
    blocks[:, 31] = anchor
    want_c, want_k = _fp8_store_reference_torch(blocks)
    codes, exps = oracle_mod.kv_quantize_fp8(to_bits(blocks))
    assert np.array_equal(codes.reshape(-1), want_c)
    assert np.array_equal(exps.reshape(-1), want_k)


def test_fp8_store_decodes_to_the_round_trip(oracle_mod):
    g = torch.Generator().manual_seed(8)
    x = torch.randn((2048, 64), generator=g) * torch.exp(torch.randn((2048, 1), generator=g) * 6)
    x = to_bits(x)
    codes, exps = oracle_mod.kv_quantize_fp8(x)
    dec = oracle_mod.kv_dequantize_fp8(codes, exps)
    assert np.array_equal(dec, to_bits(_quant_reference_torch(from_bits(x).clone())))
    assert np.array_equal(dec.reshape(-1), _fp8_decode_torch(codes, exps))
    # the decoded rows are a fixed point of the round trip
    assert np.array_equal(oracle_mod.act_quant_inplace(dec.copy().reshape(-1)), dec.reshape(-1))
    # zero blocks: every code +0 at the floor exponent of 1e-4 / 448 (2^-22)
    zc, ze = oracle_mod.kv_quantize_fp8(np.zeros((1, 32), dtype=np.uint16))
    assert (zc == 0).all() and (ze == -22).all()


def test_fp8_ring_write_matches_round_trip_and_store(oracle_mod):
    g = torch.Generator().manual_seed(9)
    b, s, d, W, p0, R = 3, 20, 64, 8, 37, 11
    raw = to_bits(torch.randn((b, s, d), generator=g) * 3)
    kv = raw.copy()
    codes = np.full((b, R, d), 0x55, dtype=np.uint8)
    exps = np.full((b, R, d // 32), 99, dtype=np.int8)
    oracle_mod.kv_quant_ring_write_fp8(kv, codes, exps, p0, W)
    assert np.array_equal(kv, oracle_mod.act_quant_inplace(raw.copy().reshape(-1)).reshape(b, s, d))
    want_c, want_k = oracle_mod.kv_quantize_fp8(raw)
    slots = set()
    for t in range(s - W, s):
        sl = (p0 + t) % W
        slots.add(sl)
        assert np.array_equal(codes[:, sl], want_c[:, t]) and np.array_equal(exps[:, sl], want_k[:, t])
    assert (codes[:, W:] == 0x55).all() and (exps[:, W:] == 99).all()   # rows past the window untouched
    assert slots == set(range(W))


# ----------------------------------------------------------------------------------------------
# RoPE (ratio-0 table, rotation of the last rope_dim values, inverse rotation)
# ----------------------------------------------------------------------------------------------

def _torch_rope_table(npos, dim, base):
    """The table as the pages build it: f32 frequencies, outer product with the positions, polar."""
    freqs = 1.0 / (base ** (torch.arange(0, dim, 2, dtype=torch.float32) / dim))
    ang = torch.outer(torch.arange(npos).float(), freqs)
    return torch.view_as_real(torch.polar(torch.ones_like(ang), ang)).numpy()


def test_rope_table_matches_library(oracle_mod):
    t = oracle_mod.rope_table(140000, 64, 10000.0)
    ref = _torch_rope_table(140000, 64, 10000.0)
    assert np.abs(t - ref).max() <= 1.2e-7          # cos / sin rounded to f32 either way
    assert (t[0, :, 0] == 1).all() and (t[0, :, 1] == 0).all()
    t2 = oracle_mod.rope_table(50, 32, 500.0)
    assert np.abs(t2 - _torch_rope_table(50, 32, 500.0)).max() <= 1.2e-7


def _torch_rotary(x: torch.Tensor, table: np.ndarray, pos: np.ndarray, rd: int, inverse: bool) -> torch.Tensor:
    """The pages' apply_rotary_emb with library complex arithmetic; x [rows][d], pos [rows]."""
    fc = torch.view_as_complex(torch.from_numpy(table[pos].copy()))
    if inverse:
        fc = fc.conj()
    y = x.clone()
    xc = torch.view_as_complex(y[:, -rd:].float().unflatten(-1, (-1, 2)))
    y[:, -rd:] = torch.view_as_real(xc * fc).flatten(-2).to(torch.bfloat16)
    return y


@pytest.mark.parametrize("inverse", [False, True])
def test_apply_rotary_matches_library(oracle_mod, inverse):
    g = torch.Generator().manual_seed(12)
    b, m, h, d, rd, p0 = 2, 5, 3, 128, 64, 1000
    x = (torch.randn((b, m, h, d), generator=g) * 5).to(torch.bfloat16)
    table = oracle_mod.rope_table(1100, rd, 10000.0)
    got = oracle_mod.apply_rotary(to_bits(x), rd, table, p0, h, m, inverse)
    pos = p0 + (np.arange(b * m * h) // h) % m
    want = to_bits(_torch_rotary(x.view(-1, d), table, pos, rd, inverse))
    assert np.array_equal(got.reshape(-1), want.reshape(-1))
    assert np.array_equal(got.reshape(-1, d)[:, : d - rd], to_bits(x).reshape(-1, d)[:, : d - rd])


def test_apply_rotary_properties(oracle_mod):
    g = torch.Generator().manual_seed(13)
    x = torch.randn((64, 512), generator=g).to(torch.bfloat16)
    table = oracle_mod.rope_table(5000, 64, 10000.0)
    xb = to_bits(x)
    # position 0 is the identity, exactly
    assert np.array_equal(oracle_mod.apply_rotary(xb.copy(), 64, table, 0, 64, 1), xb)
    # the inverse undoes the rotation up to the two bf16 roundings; norms of pairs are kept
    fwd = oracle_mod.apply_rotary(xb.copy(), 64, table, 4321, 1, 1)
    back = oracle_mod.apply_rotary(fwd.copy(), 64, table, 4321, 1, 1, inverse=True)
    x64, f64, b64 = bits_to_f64(xb)[:, -64:], bits_to_f64(fwd)[:, -64:], bits_to_f64(back)[:, -64:]
    assert np.abs(b64 - x64).max() <= 2 * 2.0 ** -8 * np.abs(x64).max()
    n0 = x64[:, 0::2] ** 2 + x64[:, 1::2] ** 2
    n1 = f64[:, 0::2] ** 2 + f64[:, 1::2] ** 2
    assert np.allclose(n1, n0, rtol=2 ** -6, atol=1e-6)
    assert not np.array_equal(fwd, xb)


def test_rope_ring_write_is_rotation_then_round_trip(oracle_mod):
    g = torch.Generator().manual_seed(14)
    b, s, d, W, p0, rd = 2, 12, 64, 8, 0, 32
    raw = to_bits(torch.randn((b, s, d), generator=g) * 3)
    table = oracle_mod.rope_table(64, rd, 10000.0)
    kv = raw.copy()
    ring = np.zeros((b, W, d), dtype=np.uint16)
    oracle_mod.kv_rope_quant_ring_write(kv, ring, p0, W, rd, table)
    want = raw.copy()
    for bi in range(b):
        oracle_mod.apply_rotary(want[bi], rd, table, p0, 1, s)
    want_ring = np.zeros_like(ring)
    oracle_mod.kv_quant_ring_write(want, want_ring, p0, W)
    assert np.array_equal(kv, want) and np.array_equal(ring, want_ring)
    # and the rotation is by each row's own position: row t of sequence 0, done by the library
    lib_rot = to_bits(_torch_rotary(from_bits(raw[0]).clone(), table, p0 + np.arange(s), rd, False))
    assert np.array_equal(oracle_mod.act_quant_inplace(lib_rot.reshape(-1)).reshape(s, d), kv[0])


# ----------------------------------------------------------------------------------------------
# Indexer scoring and top-k
# ----------------------------------------------------------------------------------------------

def _indexer_case(seed, b=2, s=24, H=4, D=32, ratio=4, start_pos=0):
    g = torch.Generator().manual_seed(seed)
    T = (start_pos + s) // ratio
    q = torch.randn((b, s, H, D), generator=g).to(torch.bfloat16)
    k = torch.randn((b, T, D), generator=g).to(torch.bfloat16)
    w = torch.rand((b, s, H), generator=g) * 0.2
    return q, k, w


def test_indexer_scores_match_library(oracle_mod):
    q, k, w = _indexer_case(30)
    idx, sc = oracle_mod.indexer_topk(to_bits(q), to_bits(k), w.numpy(), 0, 4, 3, return_scores=True)
    dots = torch.einsum("bshd,btd->bsht", q.double(), k.double()).relu()
    ref = (dots * w.double().unsqueeze(-1)).sum(dim=2)
    lens = (torch.arange(1, 25) // 4).view(1, -1, 1)
    ref = ref.masked_fill(torch.arange(6).view(1, 1, -1) >= lens, -math.inf)
    fin = np.isfinite(sc)
    assert np.array_equal(fin, np.isfinite(ref.numpy()))
    assert np.allclose(sc[fin], ref.numpy()[fin], rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("start_pos,s,topk,offset", [(0, 24, 3, 0), (0, 40, 64, 128), (37, 1, 5, 128), (400, 1, 50, 7)])
def test_indexer_topk_matches_library_selection(oracle_mod, start_pos, s, topk, offset):
    q, k, w = _indexer_case(31 + start_pos, s=s, start_pos=start_pos)
    idx, sc = oracle_mod.indexer_topk(to_bits(q), to_bits(k), w.numpy(), start_pos, 4, topk, offset,
                                      return_scores=True)
    kk = min(topk, (start_pos + s) // 4)
    assert idx.shape == (2, s, kk)
    sct = torch.from_numpy(sc)
    for bi in range(2):
        for i in range(s):
            lens = (start_pos + i + 1) // 4
            want_valid = sorted(t for t in torch.topk(sct[bi, i], kk).indices.tolist() if t < lens)
            row = idx[bi, i]
            assert [int(v) - offset for v in row if v >= 0] == want_valid       # ascending, shifted
            assert (row == -1).sum() == kk - len(want_valid)                     # the rest is -1
            assert list(row[: len(want_valid)]) == [v + offset for v in want_valid]


def test_indexer_properties(oracle_mod):
    q, k, w = _indexer_case(32, s=32, H=6)
    base = oracle_mod.indexer_topk(to_bits(q), to_bits(k), w.numpy(), 0, 4, 4)
    perm = torch.randperm(6, generator=torch.Generator().manual_seed(1))
    assert np.array_equal(oracle_mod.indexer_topk(to_bits(q[:, :, perm]), to_bits(k), w[:, :, perm].numpy().copy(),
                                                  0, 4, 4), base)
    assert np.array_equal(oracle_mod.indexer_topk(to_bits(q), to_bits(k), (w * 4).numpy(), 0, 4, 4), base)
    # a head with weight 0 does not matter; a key that dominates every head is always selected
    w0 = w.clone()
    w0[:, :, 2] = 0
    q2 = q.clone()
    q2[:, :, 2] = torch.randn_like(q2[:, :, 2].float()).to(torch.bfloat16)
    assert np.array_equal(oracle_mod.indexer_topk(to_bits(q2), to_bits(k), w0.numpy(), 0, 4, 4),
                          oracle_mod.indexer_topk(to_bits(q), to_bits(k), w0.numpy(), 0, 4, 4))
    k2 = k.clone()
    k2[:, 1] = q.float().mean(dim=(1, 2)).mul(50).to(torch.bfloat16)
    got = oracle_mod.indexer_topk(to_bits(q), to_bits(k2), w.numpy(), 0, 4, 4)
    for i in range(4, 32):          # visible from query 7 on (compress_lens = (i + 1) // 4 > 1)
        if (i + 1) // 4 > 1:
            assert 1 in got[:, i].tolist()[0] and 1 in got[:, i].tolist()[1]


def _brute_select(scores, start_pos, ratio, topk, offset):
    """Textbook selection: order positions by (score descending, position ascending), keep the
    first kk, list them ascending, -1 for an unseen position."""
    b, s, _ = scores.shape
    Tv = (start_pos + s) // ratio
    kk = min(topk, Tv)
    out = np.empty((b, s, kk), dtype=np.int32)
    for bi in range(b):
        for i in range(s):
            lens = (start_pos + i + 1) // ratio
            vals = [(-(float(scores[bi, i, t]) if t < lens else -math.inf), t) for t in range(Tv)]
            keep = sorted(t for _, t in sorted(vals)[:kk])
            out[bi, i] = [t + offset if t < lens else -1 for t in keep]
    return out


@pytest.mark.parametrize("start_pos,s,topk,offset", [(0, 40, 6, 0), (0, 40, 64, 128), (99, 1, 7, 3), (400, 2, 30, 0)])
def test_indexer_select_is_the_ordered_cut(oracle_mod, start_pos, s, topk, offset):
    """The selection from given scores, with many exact ties (scores on a coarse grid, and +0 next
    to -0), against a brute-force ordering by (score, position)."""
    g = torch.Generator().manual_seed(34 + s)
    Tv = (start_pos + s) // 4
    sc = (torch.randint(-4, 5, (2, s, Tv + 3), generator=g).float() * 0.5).numpy()
    sc[0, :, ::7] = -0.0
    got = oracle_mod.indexer_select(sc, start_pos, 4, topk, offset)
    assert np.array_equal(got, _brute_select(sc, start_pos, 4, topk, offset))


def test_indexer_select_agrees_with_topk_on_its_own_scores(oracle_mod):
    q, k, w = _indexer_case(35, s=40)
    idx, sc = oracle_mod.indexer_topk(to_bits(q), to_bits(k), w.numpy(), 0, 4, 5, 7, return_scores=True)
    assert np.array_equal(oracle_mod.indexer_select(sc, 0, 4, 5, 7), idx)


def test_indexer_prefill_row_equals_decode_step(oracle_mod):
    q, k, w = _indexer_case(33, b=1, s=40, H=3)
    pre = oracle_mod.indexer_topk(to_bits(q), to_bits(k), w.numpy(), 0, 4, 6)
    for i in (3, 7, 20, 39):
        T = (i + 1) // 4
        dec = oracle_mod.indexer_topk(to_bits(q[:, i:i + 1]).copy(), to_bits(k[:, :T]).copy(),
                                      w[:, i:i + 1].numpy().copy(), i, 4, 6)
        assert [v for v in pre[0, i] if v >= 0] == [v for v in dec[0, 0] if v >= 0]


# ----------------------------------------------------------------------------------------------
# sparse_attn
# ----------------------------------------------------------------------------------------------

def _rand_case(seed, b=2, m=3, h=5, d=32, n=40, topk=24, neg=0.2, dup=False):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((b, m, h, d), generator=g).to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g).to(torch.bfloat16)
    sink = torch.randn((h,), generator=g)
    if dup:
        idx = torch.randint(0, n, (b, m, topk), generator=g)
    else:
        idx = torch.stack([torch.randperm(n, generator=g)[:topk] for _ in range(b * m)]).view(b, m, topk)
    mask = torch.rand((b, m, topk), generator=g) < neg
    idx = torch.where(mask, -1, idx).to(torch.int32)
    return q, kv, sink, idx


def _dense_masked_reference(q, kv, sink, idx, scale):
    """Textbook dense attention over all n rows with a -inf mask for rows not in the index set,
    plus one sink column appended to the scores and dropped after the softmax.  Requires distinct
    indices per row (a set, like the mask it builds)."""
    q64, kv64 = q.to(torch.float64), kv.to(torch.float64)
    b, m, h, d = q.shape
    n = kv.shape[1]
    out = torch.zeros((b, m, h, d), dtype=torch.float64)
    for bi in range(b):
        scores = torch.einsum("mhd,nd->mhn", q64[bi], kv64[bi]) * scale
        mask = torch.full((m, n), float("-inf"), dtype=torch.float64)
        for t in range(m):
            sel = idx[bi, t][idx[bi, t] >= 0].long()
            mask[t, sel] = 0.0
        scores = scores + mask[:, None, :]
        scores = torch.cat([scores, sink.to(torch.float64)[None, :, None].expand(m, h, 1)], dim=-1)
        p = torch.softmax(scores, dim=-1)[..., :n]
        out[bi] = torch.einsum("mhn,nd->mhd", p, kv64[bi])
    return out


def _gathered_reference(q, kv, sink, idx, scale):
    """Softmax over the gathered list (duplicates count as often as listed) plus the sink."""
    q64, kv64 = q.to(torch.float64), kv.to(torch.float64)
    b, m, h, d = q.shape
    out = torch.zeros((b, m, h, d), dtype=torch.float64)
    for bi in range(b):
        for t in range(m):
            sel = idx[bi, t][idx[bi, t] >= 0].long()
            rows = kv64[bi, sel]                                   # [k, d]
            sc = (q64[bi, t] @ rows.T) * scale                     # [h, k]
            sc = torch.cat([sc, sink.to(torch.float64)[:, None]], dim=1)
            p = torch.softmax(sc, dim=1)[:, :-1]
            out[bi, t] = p @ rows
    return out


def f32(x: float) -> float:
    """The softmax scale crosses every interface as an f32."""
    return float(np.float32(x))


def _run_oracle(oracle_mod, q, kv, sink, idx, scale, f64=True, tokens=None):
    return oracle_mod.sparse_attn(to_bits(q), to_bits(kv), sink.numpy(), idx.numpy(), scale,
                                  tokens=tokens, f64=f64, nthreads=2)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_attn_matches_dense_masked_softmax(oracle_mod, seed):
    q, kv, sink, idx = _rand_case(seed)
    scale = f32(32 ** -0.5)
    want = _dense_masked_reference(q, kv, sink, idx, scale).numpy()
    got64 = _run_oracle(oracle_mod, q, kv, sink, idx, scale)
    np.testing.assert_allclose(got64, want, rtol=1e-12, atol=1e-13)
    got32 = bits_to_f64(_run_oracle(oracle_mod, q, kv, sink, idx, scale, f64=False))
    # f32 arithmetic then one bf16 rounding: within half a bf16 ulp plus f32 noise
    np.testing.assert_allclose(got32, want, rtol=2 ** -8 + 1e-5, atol=1e-6)


def test_attn_duplicates_count_as_listed(oracle_mod):
    q, kv, sink, idx = _rand_case(7, dup=True, n=10, topk=24)
    scale = f32(0.3)
    want = _gathered_reference(q, kv, sink, idx, scale).numpy()
    got = _run_oracle(oracle_mod, q, kv, sink, idx, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_attn_sink_to_minus_infinity_is_sdpa(oracle_mod):
    q, kv, sink, idx = _rand_case(8, neg=0.0)
    scale = f32(32 ** -0.5)
    sink_off = torch.full_like(sink, -1e30)
    got = _run_oracle(oracle_mod, q, kv, sink_off, idx, scale)
    b, m, h, d = q.shape
    for bi in range(b):
        for t in range(m):
            rows = kv[bi, idx[bi, t].long()].to(torch.float64)
            want = torch.nn.functional.scaled_dot_product_attention(
                q[bi, t].to(torch.float64)[None], rows[None], rows[None], scale=scale)[0]
            np.testing.assert_allclose(got[bi * m + t] if got.ndim == 3 else got[bi, t], want.numpy(),
                                       rtol=1e-12, atol=1e-13)


def test_attn_probability_mass_below_one_and_tends_to_one(oracle_mod):
    # with every gathered row equal to v, o = v * sum_j p_j, so the mass is read off o / v
    g = torch.Generator().manual_seed(9)
    d, h, k = 16, 3, 6
    v = torch.randn((d,), generator=g).to(torch.bfloat16)
    kv = v[None, None, :].expand(1, k, d).contiguous()
    q = torch.randn((1, 1, h, d), generator=g).to(torch.bfloat16)
    idx = torch.arange(k, dtype=torch.int32).view(1, 1, k)
    scale = f32(0.25)
    s = (q[0, 0].to(torch.float64) @ v.to(torch.float64)) * scale               # [h]
    v64 = v.to(torch.float64).numpy()
    masses = []
    for sink_val in (3.0, 0.0, -5.0, -40.0, -1e30):
        sink = torch.full((h,), sink_val)
        got = _run_oracle(oracle_mod, q, kv, sink, idx, scale)[0, 0]
        mass_closed = 1.0 / (1.0 + torch.exp(torch.tensor(sink_val, dtype=torch.float64) - s - math.log(k)))
        np.testing.assert_allclose(got, (mass_closed[:, None] * v.to(torch.float64)[None]).numpy(),
                                   rtol=1e-12, atol=1e-14)
        masses.append(got @ v64 / (v64 @ v64))               # the mass each head put on the rows
    masses = np.array(masses)
    assert (masses[:3] < 1).all()                           # the sink takes a share
    assert (np.diff(masses, axis=0) >= 0).all()             # and gives it back as it falls
    np.testing.assert_allclose(masses[-1], 1.0, rtol=1e-14)


def test_attn_single_valid_row_closed_form(oracle_mod):
    q, kv, sink, idx = _rand_case(10, topk=9, neg=0.0)
    idx[:] = -1
    idx[:, :, 4] = 7
    scale = f32(0.2)
    got = _run_oracle(oracle_mod, q, kv, sink, idx, scale)
    b, m, h, d = q.shape
    for bi in range(b):
        row = kv[bi, 7].to(torch.float64)
        for t in range(m):
            s = (q[bi, t].to(torch.float64) @ row) * scale
            w = torch.sigmoid(s - sink.to(torch.float64))
            np.testing.assert_allclose(got[bi, t], (w[:, None] * row[None]).numpy(), rtol=1e-12, atol=1e-14)


def test_attn_all_invalid_row_is_zero(oracle_mod):
    q, kv, sink, idx = _rand_case(11)
    idx[1, 2] = -1
    got32 = _run_oracle(oracle_mod, q, kv, sink, idx, 0.5, f64=False)
    got64 = _run_oracle(oracle_mod, q, kv, sink, idx, 0.5)
    assert (got32[1, 2] == 0).all() and (got64[1, 2] == 0).all()
    assert (got64[0, 0] != 0).any()


def test_attn_order_and_padding_invariance(oracle_mod):
    q, kv, sink, idx = _rand_case(12, neg=0.3)
    scale = f32(0.17)
    base = _run_oracle(oracle_mod, q, kv, sink, idx, scale)
    g = torch.Generator().manual_seed(13)
    perm = torch.randperm(idx.shape[-1], generator=g)
    np.testing.assert_allclose(_run_oracle(oracle_mod, q, kv, sink, idx[..., perm].contiguous(), scale), base,
                               rtol=1e-12, atol=1e-14)
    padded = torch.cat([torch.full_like(idx[..., :5], -1), idx, torch.full_like(idx[..., :3], -1)], dim=-1)
    np.testing.assert_allclose(_run_oracle(oracle_mod, q, kv, sink, padded.contiguous(), scale), base,
                               rtol=1e-12, atol=1e-14)


def test_attn_token_subset_matches_full(oracle_mod):
    q, kv, sink, idx = _rand_case(14, b=3, m=4)
    full = _run_oracle(oracle_mod, q, kv, sink, idx, 0.3, f64=False)
    toks = np.array([11, 0, 5], dtype=np.int64)
    sub = _run_oracle(oracle_mod, q, kv, sink, idx, 0.3, f64=False, tokens=toks)
    for k, tok in enumerate(toks):
        assert np.array_equal(sub[k], full.reshape(-1, *full.shape[2:])[tok])


def test_attn_rejects_out_of_range_index(oracle_mod):
    q, kv, sink, idx = _rand_case(15)
    idx[0, 0, 0] = kv.shape[1]
    with pytest.raises(ValueError):
        _run_oracle(oracle_mod, q, kv, sink, idx, 0.3)
