"""GPU-vs-oracle parity through the C ABI.

Index rows and the fp8 round trip / ring contents must match the oracle bit for bit; attention
outputs must satisfy |gpu - oracle| <= 1e-2 + 1.6e-2 * |oracle| elementwise ("Module attn",
Precision paragraph: f32 arithmetic, bf16 result, compared at bf16 tolerance, window indices
exactly).
"""
from contextlib import contextmanager

import numpy as np
import pytest
import torch

import oracle
from pathcheck import GpuStep, OracleStep, assert_close_bf16, bits
from sparse_latent_attention_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ds():
    from sparse_latent_attention_attn_gb300 import dsattn
    dsattn.device_status()      # clear anything left over
    return dsattn


@contextmanager
def _kernel(ds, which):
    """Run ds_sparse_attn on one attention kernel (ds_test_set_kernel) inside the block."""
    ds.test_set_kernel(which)
    try:
        yield
    finally:
        ds.test_set_kernel(ds.KERNEL_AUTO)


def _bf16_from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


# ----------------------------------------------------------------------------------------------
# window_topk_idxs
# ----------------------------------------------------------------------------------------------

WINDOW_CASES = [(s, 0, W) for s, W in [(1, 8), (5, 8), (12, 8), (37, 16), (300, 128), (4096, 128), (7, 1)]] + \
               [(1, p, W) for p, W in [(1, 8), (3, 8), (7, 8), (8, 8), (12, 8), (13, 8), (127, 128), (128, 128),
                                        (10000, 128), (16384, 128), (131072, 128), (5, 1), (9, 3)]]


@pytest.mark.parametrize("s,start_pos,W", WINDOW_CASES)
def test_window_idx_exact(ds, s, start_pos, W):
    b, pad = 3, 5
    rows = s if start_pos == 0 else 1
    ref = oracle.window_topk_idxs(s, start_pos, W)
    cols = ref.shape[1]
    idx = torch.full((b, rows, cols + pad), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    got_cols = ds.window_topk_idxs(idx, b, s, start_pos, W)
    assert got_cols == cols
    got = idx.cpu().numpy()
    for bi in range(b):
        assert np.array_equal(got[bi, :, :cols], ref)
    assert (got[:, :, cols:] == 0x5A5A5A5A).all()          # columns past cols untouched


def test_window_idx_rejects_chunked_prefill(ds):
    idx = torch.zeros((1, 4, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(ds.DsError) as e:
        ds.window_topk_idxs(idx, 1, 4, 5, 8)
    assert e.value.status == ds.DS_EUNSUPPORTED


# ----------------------------------------------------------------------------------------------
# fp8 round trip and ring
# ----------------------------------------------------------------------------------------------

def _all_finite_bf16_patterns() -> np.ndarray:
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (pats >> 7) & 0xFF
    return np.where(exp == 0xFF, np.uint16(0), pats)


@pytest.mark.parametrize("d", [512, 64])
def test_quant_exhaustive_bit_exact(ds, d):
    pats = _all_finite_bf16_patterns()
    rng = np.random.default_rng(d)
    for order in ("sorted", "shuffled"):
        x = pats.copy() if order == "sorted" else rng.permutation(pats)
        kv = _bf16_from_bits(x).view(1, -1, d).cuda()
        ds.kv_quant_ring_write(kv, None, 0, 1)
        want = oracle.act_quant_inplace(x.copy())
        assert np.array_equal(bits(kv).reshape(-1), want), order


@pytest.mark.parametrize("anchor_exp", [-20, -9, -6, 0, 7, 40])
def test_quant_every_value_at_fixed_scale(ds, anchor_exp):
    anchor = 448.0 * 2.0 ** anchor_exp
    pats = _all_finite_bf16_patterns()
    vals = _bf16_from_bits(pats).to(torch.float64)
    vals = vals[vals.abs() <= anchor].to(torch.bfloat16)
    nb = (vals.numel() + 30) // 31
    nb += (-nb) % 16                                  # whole rows of d = 512
    flat = torch.zeros(nb * 31, dtype=torch.bfloat16)
    flat[: vals.numel()] = vals
    blocks = torch.empty((nb, 32), dtype=torch.bfloat16)
    blocks[:, :31] = flat.view(nb, 31)
    blocks[:, 31] = anchor
    x = bits(blocks).reshape(-1)
    kv = blocks.view(1, -1, 512).cuda()
    ds.kv_quant_ring_write(kv, None, 0, 1)
    assert np.array_equal(bits(kv).reshape(-1), oracle.act_quant_inplace(x.copy()))


@pytest.mark.parametrize("b,s,d,W,p0", [(1, 12, 64, 8, 0), (3, 20, 64, 8, 37), (2, 5, 512, 8, 0),
                                        (4, 1, 512, 128, 10000), (2, 300, 512, 128, 0), (1, 7, 256, 16, 3)])
def test_ring_write_bit_exact(ds, b, s, d, W, p0):
    g = torch.Generator().manual_seed(b * 1000 + s)
    raw = (torch.randn((b, s, d), generator=g) * torch.exp(torch.randn((b, s, 1), generator=g) * 3)).to(
        torch.bfloat16)
    extra = 9                                         # the ring sits inside a wider kv tensor
    canary = 0x7F7F
    big = torch.full((b, W + extra, d), canary, dtype=torch.int16).view(torch.bfloat16).cuda()
    kv = raw.cuda()
    ds.kv_quant_ring_write(kv, big[:, :W], p0, W)
    want_kv = bits(raw).copy()
    want_ring = np.full((b, W, d), canary, dtype=np.uint16)
    oracle.kv_quant_ring_write(want_kv, want_ring, p0, W)
    assert np.array_equal(bits(kv), want_kv)
    got_big = bits(big)
    assert np.array_equal(got_big[:, :W], want_ring)
    assert (got_big[:, W:] == canary).all()


def test_ring_worked_example_gpu(ds):
    # "Module attn", ring-cache paragraph: rows valued t+1 are on the fp8 grid and name their token
    W, d = 8, 64
    ring = torch.zeros((1, W, d), dtype=torch.bfloat16, device="cuda")
    chunk = torch.tensor([[float(t + 1)] * d for t in range(12)]).to(torch.bfloat16).view(1, 12, d).cuda()
    ds.kv_quant_ring_write(chunk, ring, 0, W)
    assert (ring[0, :, 0].float().cpu().numpy().astype(int) - 1).tolist() == [8, 9, 10, 11, 4, 5, 6, 7]
    for step, ring_after in ((12, [8, 9, 10, 11, 12, 5, 6, 7]), (13, [8, 9, 10, 11, 12, 13, 6, 7])):
        new = torch.full((1, 1, d), float(step + 1)).to(torch.bfloat16).cuda()
        ds.kv_quant_ring_write(new, ring, step, W)
        assert (ring[0, :, 0].float().cpu().numpy().astype(int) - 1).tolist() == ring_after


# ----------------------------------------------------------------------------------------------
# the ratio-0 fixture: prefill 12 tokens, then decode 12 and 13 through one cache
# ----------------------------------------------------------------------------------------------

def test_fixture_sequence(ds):
    fx = wl.fixture_inputs(device="cuda")
    w = fx["w"]
    W, d, h = w.window, w.d, w.h
    sink = fx["sink"]
    # --- GPU ---------------------------------------------------------------------------------
    from sparse_latent_attention_attn_gb300 import path
    ring = torch.zeros((w.b, W, d), dtype=torch.bfloat16, device="cuda")
    kv = fx["prefill_kv"].clone()
    idx = torch.empty((w.b, w.s, min(w.s, W)), dtype=torch.int32, device="cuda")
    o_pre = path.prefill_step(fx["prefill_q"], kv, ring, sink, idx, W, w.scale)
    # --- oracle --------------------------------------------------------------------------------
    ring_o = np.zeros((w.b, W, d), dtype=np.uint16)
    chunk_o = bits(fx["prefill_kv"])
    oracle.kv_quant_ring_write(chunk_o, ring_o, 0, W)
    win = oracle.window_topk_idxs(w.s, 0, W)
    idx_o = np.ascontiguousarray(win[None])
    o_pre_o = oracle.sparse_attn(bits(fx["prefill_q"]), chunk_o, sink.cpu().numpy(), idx_o, w.scale)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    assert np.array_equal(bits(kv), chunk_o)
    assert np.array_equal(bits(ring), ring_o)
    assert_close_bf16(bits(o_pre), o_pre_o, "prefill o")
    for step in fx["decode"]:
        p = step["start_pos"]
        new = step["new_kv"].clone()
        idx_d = torch.empty((w.b, 1, W), dtype=torch.int32, device="cuda")
        o_d = path.decode_step(step["q"], ring, new, sink, idx_d, p, W, w.scale)
        oracle.kv_quant_ring_write(bits(step["new_kv"]), ring_o, p, W)
        win_d = oracle.window_topk_idxs(1, p, W)
        o_d_o = oracle.sparse_attn(bits(step["q"]), ring_o, sink.cpu().numpy(), np.ascontiguousarray(win_d[None]),
                                   w.scale)
        assert np.array_equal(idx_d.cpu().numpy()[0], win_d)
        assert np.array_equal(bits(ring), ring_o), f"ring after decode {p}"
        assert_close_bf16(bits(o_d), o_d_o, f"decode {p} o")
    assert ds.device_status() == 0


# ----------------------------------------------------------------------------------------------
# the four model-scale workloads, at full size, sampled where the oracle would be slow
# ----------------------------------------------------------------------------------------------

SAMPLE_SEQS = {1: [0, 17, 63], 2: [0], 3: [0, 5, 31], 4: [0, 101, 255]}
SAMPLE_TOKENS_PREFILL = [0, 1, 2, 3, 7, 127, 128, 129, 511, 1000, 2047, 2048, 2049, 3333, 4094, 4095]


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_workload_parity(ds, cfg):
    w = wl.WORKLOADS[cfg]
    gs = GpuStep(w)
    gs.run()
    torch.cuda.synchronize()
    orc = OracleStep(gs, seqs=SAMPLE_SEQS[cfg])
    sel = torch.tensor(orc.seqs, device="cuda")
    # index rows and ring: exact
    assert np.array_equal(gs.idx.index_select(0, sel).cpu().numpy(), orc.idx)
    ring_gpu = bits(gs.ring.index_select(0, sel))
    assert np.array_equal(ring_gpu, orc.ring)
    if not w.decode:
        assert np.array_equal(bits(gs.kv.index_select(0, sel)[:, : w.s]), orc.chunk)
    # attention: tolerance, on sampled tokens
    if w.decode:
        got = bits(gs.o.index_select(0, sel)).reshape(len(orc.seqs), w.h, w.d)
        ref = orc.attend()
        assert_close_bf16(got, ref.reshape(len(orc.seqs), w.h, w.d), f"cfg{cfg} o")
    else:
        toks = np.array(SAMPLE_TOKENS_PREFILL, dtype=np.int64)
        got = bits(gs.o[0, torch.from_numpy(toks).cuda()])
        ref = orc.attend(tokens=toks)
        assert_close_bf16(got, ref, f"cfg{cfg} o")
    # every output is finite, and the step is repeatable bit for bit
    assert torch.isfinite(gs.o.float()).all()
    first = gs.o.clone()
    gs.reset()
    gs.run()
    assert torch.equal(first, gs.o)
    assert ds.device_status() == 0


# ----------------------------------------------------------------------------------------------
# sparse_attn edge cases on small shapes (every output element checked)
# ----------------------------------------------------------------------------------------------

def _case(seed, b, m, h, d, n, topk, neg=0.1, dup=False, sink_val=None, tail_pad=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((b, m, h, d), generator=g).to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g).to(torch.bfloat16)
    sink = torch.randn((h,), generator=g) if sink_val is None else torch.full((h,), float(sink_val))
    if dup or topk > n:
        idx = torch.randint(0, n, (b, m, topk), generator=g)
    else:
        idx = torch.stack([torch.randperm(n, generator=g)[:topk] for _ in range(b * m)]).view(b, m, topk) \
            if topk else torch.zeros((b, m, 0), dtype=torch.long)
    idx = torch.where(torch.rand((b, m, topk), generator=g) < neg, -1, idx).to(torch.int32)
    if tail_pad:
        idx[..., -tail_pad:] = -1
    return q, kv, sink, idx


def _check_case(ds, q, kv, sink, idx, scale):
    o = ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), scale)
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), idx.numpy(), scale)
    assert_close_bf16(bits(o), ref)
    return o, ref


EDGE = [
    # seed, b, m, h, d, n, topk, neg, dup
    (1, 2, 3, 4, 64, 40, 24, 0.1, False),
    (2, 1, 5, 1, 64, 10, 8, 0.0, False),
    (3, 3, 2, 16, 128, 300, 200, 0.2, False),
    (4, 2, 2, 64, 512, 700, 640, 0.05, False),
    (5, 1, 3, 128, 512, 2000, 1000, 0.02, False),
    (6, 2, 2, 100, 256, 500, 65, 0.0, False),
    (7, 2, 2, 128, 512, 300, 63, 0.0, False),
    (8, 2, 2, 128, 512, 300, 64, 0.0, False),
    (9, 2, 2, 33, 512, 300, 129, 0.3, False),
    (10, 2, 2, 8, 64, 20, 50, 0.1, True),        # duplicates count as listed
    (11, 1, 1, 128, 512, 100, 1, 0.0, False),
    (12, 1, 4, 64, 512, 5000, 2176, 0.02, False),
    # index rows longer than any tile ring: one or two tokens split over 32 clusters each
    (13, 1, 2, 32, 256, 9000, 5000, 0.05, False),
    (14, 1, 1, 64, 512, 12000, 8192, 0.02, False),
]


@pytest.mark.parametrize("case", EDGE, ids=[f"e{c[0]}" for c in EDGE])
def test_attn_edge_shapes(ds, case):
    seed, b, m, h, d, n, topk, neg, dup = case
    q, kv, sink, idx = _case(seed, b, m, h, d, n, topk, neg, dup)
    _check_case(ds, q, kv, sink, idx, d ** -0.5)
    assert ds.device_status() == 0


@pytest.mark.parametrize("qscale", [8.0, 32.0])
def test_attn_peaked_scores_on_the_split_path(ds, qscale):
    """Large logits on the d = 512 path, where each CTA of the cluster adds the peer's partial
    scores (f32) to its own.  q is scaled so the partial logits reach tens to hundreds of log2
    units: attention that is nearly one-hot, where a score error shows up directly in the
    weights.  Also a workload where the two halves' partials cancel: q's second half is minus its
    first half and kv's halves are equal, so every full score is 0 and the output is the plain
    mean of the rows (with the sink)."""
    q, kv, sink, idx = _case(30, 2, 2, 128, 512, 1500, 700, 0.02)
    q = (q.float() * qscale).to(torch.bfloat16)
    _check_case(ds, q, kv, sink, idx, 512 ** -0.5)
    assert ds.device_status() == 0
    qc = q.clone()
    qc[..., 256:] = -qc[..., :256]
    kvc = kv.clone()
    kvc[..., 256:] = kvc[..., :256]
    _check_case(ds, qc, kvc, sink, idx, 512 ** -0.5)
    assert ds.device_status() == 0


@pytest.mark.parametrize("d,h,ntok,topk", [(512, 16, 200, 300), (512, 8, 160, 129), (64, 8, 400, 200)])
def test_attn_stream_k_every_token(ds, d, h, ntok, topk):
    """More tokens than co-resident clusters: each cluster runs a range of the (token, entry)
    space that starts and ends inside tokens, weighted by a fixed cost per token, and the combine
    kernel merges every cut token.  Every token is checked, cut or whole."""
    q, kv, sink, idx = _case(50 + topk, ntok // 2, 2, h, d, 3 * topk, topk, 0.05)
    _check_case(ds, q, kv, sink, idx, d ** -0.5)
    assert ds.device_status() == 0


def _out_of_tolerance(got: np.ndarray, ref64: np.ndarray) -> int:
    """Elements of got (f32 values) outside |got - ref| <= 1e-2 + 1.6e-2 |ref| of the f64 result."""
    return int((np.abs(got.astype(np.float64) - ref64) > 1e-2 + 1.6e-2 * np.abs(ref64)).sum())


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("d,h,b,m,topk", [(512, 64, 100, 2, 300), (512, 128, 2, 2, 1500), (256, 32, 3, 2, 500)])
def test_attn_wide_range_rows_as_accurate_as_f32(ds, fp8, d, h, b, m, topk):
    """Rows whose 32-blocks span 2^-20 .. 2^20 (a range the fp8 round trip keeps): logits reach
    about 10^6, where an f32 evaluation itself is no longer within the bf16 tolerance everywhere
    (its rounding of a logit near 7e5 is 0.06, which moves a near-tie's weights by percent).
    Scores, softmax and accumulation are f32 ("Module attn", Precision paragraph), so measured
    against the f64 evaluation the kernel may miss the tolerance only where f32 arithmetic does:
    it must have no more elements out of tolerance than the f32 oracle on the same input (a
    score carried with fewer bits than f32 across the d split shows up here as many more)."""
    if fp8 and d != 512:
        pytest.skip("the fp8 row store is read by the d = 512 kernel")
    q, _, sink, idx = _case(300 + d + b, b, m, h, d, 2 * topk, topk, 0.05)
    kv = _spread_rows(300 + b, b * 2 * topk, d).view(b, 2 * topk, d)
    kv_rt = _bf16_from_bits(oracle.act_quant_inplace(bits(kv).copy().reshape(-1)).reshape(kv.shape))
    if fp8:
        codes, exps = ds.kv_quantize_fp8(kv.cuda())
        o = ds.sparse_attn_fp8kv(q.cuda(), codes, exps, sink.cuda(), idx.cuda(), d ** -0.5)
    else:
        o = ds.sparse_attn(q.cuda(), kv_rt.cuda(), sink.cuda(), idx.cuda(), d ** -0.5)
    ref64 = oracle.sparse_attn(bits(q), bits(kv_rt), sink.numpy(), idx.numpy(), d ** -0.5, f64=True)
    ref32 = oracle.bf16_bits_to_f32(oracle.sparse_attn(bits(q), bits(kv_rt), sink.numpy(), idx.numpy(), d ** -0.5))
    got = oracle.bf16_bits_to_f32(bits(o))
    assert np.isfinite(got).all()
    n_gpu, n_f32 = _out_of_tolerance(got, ref64), _out_of_tolerance(ref32, ref64)
    print(f"\nwide-range rows d={d} h={h} fp8={fp8}: out of tolerance against f64: kernel {n_gpu}, "
          f"f32 oracle {n_f32} of {got.size}")
    assert n_gpu <= n_f32
    assert ds.device_status() == 0


@pytest.mark.parametrize("d,h,b,m,topk", [(512, 128, 3, 2, 700), (256, 32, 2, 3, 300), (64, 8, 2, 2, 100)])
def test_attn_q_and_o_aligned_to_16_bytes_only(ds, d, h, b, m, topk):
    """q and o 16 bytes past a 32-byte boundary (the interface asks for 16): the kernel moves
    their rows in 16-byte accesses instead of 32-byte ones, and the output is bit-identical to the
    one written from 32-byte aligned buffers."""
    q, kv, sink, idx = _case(40 + d, b, m, h, d, 2 * topk, topk, 0.05)
    o_aligned, _ = _check_case(ds, q, kv, sink, idx, d ** -0.5)
    qbuf = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    obuf = torch.zeros(q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    q16, o16 = qbuf[8:].view(q.shape), obuf[8:].view(q.shape)
    assert q16.data_ptr() % 32 == 16 and o16.data_ptr() % 32 == 16
    q16.copy_(q.cuda())
    ds.sparse_attn(q16, kv.cuda(), sink.cuda(), idx.cuda(), d ** -0.5, o=o16)
    assert torch.equal(o16, o_aligned)
    assert ds.device_status() == 0


def test_attn_all_invalid_rows_give_zero(ds):
    q, kv, sink, idx = _case(20, 2, 3, 64, 512, 300, 130)
    idx[1, 2] = -1
    idx[0, 0] = -1
    o, _ = _check_case(ds, q, kv, sink, idx, 512 ** -0.5)
    assert (o[1, 2].float() == 0).all() and (o[0, 0].float() == 0).all()


@pytest.mark.parametrize("d,h,b", [(64, 8, 400), (256, 32, 300), (512, 128, 200)])
def test_attn_tokens_without_rows_inside_ranges(ds, d, h, b):
    """More tokens than clusters, so each work range holds several tokens, some listing no valid
    row (scattered, three in a row, the last): zeros out for those, and the right q for the
    tokens after them in the same range (cluster kernel at every head_dim it takes; d < 512
    loads each q in the softmax warps, d = 512 after a segment without rows only)."""
    q, kv, sink, idx = _case(90 + d, b, 1, h, d, 300, 150, 0.05)
    empty = [3, 4, 150, 151, 152, b - 1]
    for t in empty:
        idx[t] = -1
    o, _ = _check_case(ds, q, kv, sink, idx, d ** -0.5)
    for t in empty:
        assert (o[t].float() == 0).all()
    assert ds.device_status() == 0


def test_attn_empty_topk(ds):
    q, kv, sink, idx = _case(21, 2, 2, 16, 64, 10, 0)
    o, _ = _check_case(ds, q, kv, sink, idx, 0.125)
    assert (o.float() == 0).all()


@pytest.mark.parametrize("sink_val", [-1e30, -30.0, 30.0, 1e30])
def test_attn_extreme_sinks(ds, sink_val):
    q, kv, sink, idx = _case(22, 2, 2, 32, 512, 400, 256, sink_val=sink_val)
    _check_case(ds, q, kv, sink, idx, 512 ** -0.5)


def test_attn_tail_padding_and_permutation(ds):
    q, kv, sink, idx = _case(23, 2, 2, 64, 512, 1000, 300, neg=0.0, tail_pad=37)
    o1, _ = _check_case(ds, q, kv, sink, idx, 512 ** -0.5)
    perm = torch.randperm(idx.shape[-1], generator=torch.Generator().manual_seed(1))
    o2, _ = _check_case(ds, q, kv, sink, idx[..., perm].contiguous(), 512 ** -0.5)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2


def test_attn_out_of_range_index_is_skipped_and_flagged(ds):
    q, kv, sink, idx = _case(24, 1, 2, 16, 64, 50, 20, neg=0.0)
    bad = idx.clone()
    bad[0, 1, 3] = 50          # == n: out of range
    o = ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), bad.cuda(), 0.125)
    assert ds.device_status() & ds.DS_DEV_BAD_INDEX
    skipped = bad.clone()
    skipped[0, 1, 3] = -1
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), skipped.numpy(), 0.125)
    assert_close_bf16(bits(o), ref)
    assert ds.device_status() == 0


def test_repeated_calls_finish_without_timeouts(ds):
    """Many back-to-back calls on a stream-K split with many segments per cluster (prefill: 4096
    tokens over the clusters, every boundary cutting a token) and on decode_large: every call
    finishes with the same output and no bounded wait inside the kernel gives up."""
    for cfg, reps in ((2, 20), (4, 5)):
        w = wl.WORKLOADS[cfg]
        gs = GpuStep(w)
        gs.run()
        torch.cuda.synchronize()
        first = gs.o.clone()
        for _ in range(reps):
            gs.attend_only()
        torch.cuda.synchronize()
        assert ds.device_status() == 0, f"cfg{cfg}: a kernel wait timed out"
        assert torch.equal(first, gs.o), f"cfg{cfg}: repeated calls differ"


@pytest.mark.parametrize("d,h,b,topk", [(512, 64, 4, 700), (512, 128, 4, 700), (64, 8, 2, 300)])
def test_timed_out_wait_is_reported_and_context_stays_usable(ds, d, h, b, topk):
    """The kernel's bounded waits, made to run out without any GPU fault: with the test hook
    ds_test_set_stall on, the gather warps withhold the first tile's arrivals, so the MMA thread's
    wait gives up after its time limit.  The call must end (no hang), raise DS_DEV_TIMEOUT, and
    leave the context usable: the next call without the switch is clean and agrees with the
    oracle.  Covers the 2-CTA cluster kernel (d = 512, forced for 64 heads, where a decode batch
    would otherwise take the one-CTA kernel) and its single-CTA form (d = 64)."""
    q, kv, sink, idx = _case(40 + d + h, b, 1, h, d, 2048, topk)
    scale = d ** -0.5
    assert ds.device_status() == 0
    ds.test_set_kernel(ds.KERNEL_CLUSTER)
    try:
        ds.test_set_stall(True)
        try:
            ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), scale)
            bits_after = ds.device_status()
        finally:
            ds.test_set_stall(False)
        assert bits_after & ds.DS_DEV_TIMEOUT, f"expected a timeout, status bits {bits_after}"
        _check_case(ds, q, kv, sink, idx, scale)
    finally:
        ds.test_set_kernel(ds.KERNEL_AUTO)
    assert ds.device_status() == 0


def test_attn_argument_errors(ds):
    q, kv, sink, idx = _case(25, 1, 1, 4, 64, 10, 8)
    q, kv, sink, idx = q.cuda(), kv.cuda(), sink.cuda(), idx.cuda()
    with pytest.raises(ds.DsError) as e:
        ds.sparse_attn(q.view(1, 1, 4, 64)[..., :48].contiguous().view(1, 1, 4, 48),
                       kv[..., :48].contiguous(), sink, idx, 0.1)
    assert e.value.status == ds.DS_EUNSUPPORTED
    big_h = torch.zeros((1, 1, 129, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ds.DsError) as e:
        ds.sparse_attn(big_h, kv, torch.zeros(129, device="cuda"), idx, 0.1)
    assert e.value.status == ds.DS_EUNSUPPORTED


# ----------------------------------------------------------------------------------------------
# fp8 row store (codes + per-32 exponents) and sparse_attn reading it
# ----------------------------------------------------------------------------------------------

def _spread_rows(seed, rows, d):
    """bf16 rows whose 32-blocks span magnitudes from 2^-20 to 2^20 (subnormal e4m3 codes, ties)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, d), generator=g) * torch.exp2(torch.randint(-20, 21, (rows, d // 32), generator=g)
                                                          .float().repeat_interleave(32, dim=1))
    return x.to(torch.bfloat16)


def test_fp8_quantize_bit_exact(ds):
    x = _spread_rows(60, 1500, 512)
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    pats = np.where(np.isfinite(bits_to_f32(pats)), pats, np.uint16(0)).reshape(-1, 64)
    for xb in (bits(x), pats):
        codes, exps = ds.kv_quantize_fp8(_bf16_from_bits(xb).cuda())
        want_c, want_k = oracle.kv_quantize_fp8(xb)
        assert np.array_equal(codes.cpu().numpy(), want_c)
        assert np.array_equal(exps.cpu().numpy(), want_k)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("b,s,d,W,p0", [(3, 20, 64, 8, 37), (2, 1, 512, 128, 10000), (1, 300, 512, 128, 0)])
def test_fp8_ring_write_bit_exact(ds, b, s, d, W, p0):
    g = torch.Generator().manual_seed(61 + s)
    kv = (torch.randn((b, s, d), generator=g) * 4).to(torch.bfloat16)
    R = W + 5
    codes = torch.full((b, R, d), 0x55, dtype=torch.uint8)
    exps = torch.full((b, R, d // 32), 99, dtype=torch.int8)
    kv_o, codes_o, exps_o = bits(kv).copy(), codes.numpy().copy(), exps.numpy().copy()   # bits() of a CPU tensor is a view
    oracle.kv_quant_ring_write_fp8(kv_o, codes_o, exps_o, p0, W)
    kv_g, codes_g, exps_g = kv.cuda(), codes.cuda(), exps.cuda()
    ds.kv_quant_ring_write_fp8(kv_g, codes_g, exps_g, p0, W)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kv_g), kv_o)
    assert np.array_equal(codes_g.cpu().numpy(), codes_o)
    assert np.array_equal(exps_g.cpu().numpy(), exps_o)


FP8_ATTN = [
    # seed, b, m, h, n, topk, neg
    (70, 2, 2, 64, 700, 640, 0.05),
    (71, 1, 3, 128, 2000, 1000, 0.02),
    (72, 2, 2, 128, 300, 63, 0.0),
    (73, 2, 2, 33, 300, 129, 0.3),
    (74, 1, 4, 64, 5000, 2176, 0.02),
    (75, 100, 2, 16, 900, 300, 0.05),     # more tokens than clusters: cut tokens and the combine
    (76, 1, 1, 64, 12000, 8192, 0.02),    # one token split over many clusters
]


@pytest.mark.parametrize("case", FP8_ATTN, ids=[f"f{c[0]}" for c in FP8_ATTN])
def test_attn_fp8kv_is_bit_identical_to_bf16_on_decoded_rows(ds, case):
    """The fp8 gather decodes each row on chip to the bf16 values of the round trip, so the MMA
    sees identical operands: the output must equal ds_sparse_attn on the decoded rows bit for bit
    (the same cluster kernel, which the fp8 row store always runs), and match the oracle on those
    rows."""
    seed, b, m, h, n, topk, neg = case
    q, _, sink, idx = _case(seed, b, m, h, 512, n, topk, neg)
    kv = _spread_rows(seed, b * n, 512).view(b, n, 512)
    codes, exps = ds.kv_quantize_fp8(kv.cuda())
    dec = oracle.kv_dequantize_fp8(codes.cpu().numpy(), exps.cpu().numpy())
    assert np.array_equal(dec, oracle.act_quant_inplace(bits(kv).copy().reshape(-1)).reshape(dec.shape))
    kv_dec = _bf16_from_bits(dec)
    with _kernel(ds, ds.KERNEL_CLUSTER):
        o_bf16, _ = _check_case(ds, q, kv_dec, sink, idx, 512 ** -0.5)
    o_f8 = ds.sparse_attn_fp8kv(q.cuda(), codes, exps, sink.cuda(), idx.cuda(), 512 ** -0.5)
    assert torch.equal(o_f8, o_bf16)
    assert ds.device_status() == 0


def test_attn_fp8kv_tokens_without_rows_inside_ranges(ds):
    """The fp8 row store's gather with tokens listing no valid row inside multi-token ranges:
    bit-identical to ds_sparse_attn on the decoded rows, zeros for those tokens."""
    b, h, n, topk = 200, 128, 600, 200
    q, _, sink, idx = _case(95, b, 1, h, 512, n, topk, 0.05)
    empty = [0, 7, 8, 9, 120, b - 1]
    for t in empty:
        idx[t] = -1
    kv = torch.randn((b, n, 512), generator=torch.Generator().manual_seed(96)).to(torch.bfloat16)
    codes, exps = ds.kv_quantize_fp8(kv.cuda())
    kv_dec = _bf16_from_bits(oracle.kv_dequantize_fp8(codes.cpu().numpy(), exps.cpu().numpy()))
    o_bf16, _ = _check_case(ds, q, kv_dec, sink, idx, 512 ** -0.5)
    o_f8 = ds.sparse_attn_fp8kv(q.cuda(), codes, exps, sink.cuda(), idx.cuda(), 512 ** -0.5)
    assert torch.equal(o_f8, o_bf16)
    for t in empty:
        assert (o_f8[t].float() == 0).all()
    assert ds.device_status() == 0


def test_attn_fp8kv_decode_large_full_size(ds):
    """The fp8 row store on decode_large at full size, in the launch configuration
    `bench.py --kv fp8` times (256 sequences, 128 heads, 2176 entries over 32896 rows each): the
    whole output bit-identical to ds_sparse_attn on the round-tripped rows, and three sampled
    sequences against the oracle on those rows."""
    w = wl.WORKLOADS[4]
    gs = GpuStep(w)
    gs.run()
    torch.cuda.synchronize()
    codes, exps = ds.kv_quantize_fp8(gs.kv)
    kv_rt = gs.kv.clone()
    ds.kv_quant_ring_write(kv_rt, None, 0, 1)          # every row through the round trip, in place
    q, sink = gs.inp.q, gs.inp.sink
    o_bf16 = ds.sparse_attn(q, kv_rt, sink, gs.idx, w.scale)
    o_f8 = ds.sparse_attn_fp8kv(q, codes, exps, sink, gs.idx, w.scale)
    assert torch.equal(o_f8, o_bf16)
    for bi in (0, 101, 255):
        ref = oracle.sparse_attn(bits(q[bi:bi + 1]), bits(kv_rt[bi:bi + 1]), sink.cpu().numpy(),
                                 gs.idx[bi:bi + 1].cpu().numpy(), w.scale)
        assert_close_bf16(bits(o_f8[bi:bi + 1]), ref, f"fp8 decode_large sequence {bi}")
    assert ds.device_status() == 0


def test_attn_fp8kv_ring_then_attend(ds):
    """The fp8 ring write into the leading rows of an fp8 row store, then attention over window
    and compressed rows: equal to the bf16 pipeline (round-tripped ring inside a bf16 kv)."""
    b, W, ncomp, h, d, p0 = 4, 128, 1500, 64, 512, 5000
    n = W + ncomp
    g = torch.Generator().manual_seed(80)
    kv = _spread_rows(81, b * n, d).view(b, n, d)
    new = (torch.randn((b, 1, d), generator=g) * 2).to(torch.bfloat16)
    codes, exps = ds.kv_quantize_fp8(kv.cuda())
    kv_bf = _bf16_from_bits(oracle.kv_dequantize_fp8(codes.cpu().numpy(), exps.cpu().numpy())).cuda()
    new_a, new_b = new.cuda(), new.cuda()
    ds.kv_quant_ring_write_fp8(new_a, codes, exps, p0, W)
    ds.kv_quant_ring_write(new_b, kv_bf, p0, W)
    q, _, sink, idx = _case(82, b, 1, h, d, n, 700, 0.02)
    o_f8 = ds.sparse_attn_fp8kv(q.cuda(), codes, exps, sink.cuda(), idx.cuda(), d ** -0.5)
    with _kernel(ds, ds.KERNEL_CLUSTER):
        o_bf = ds.sparse_attn(q.cuda(), kv_bf, sink.cuda(), idx.cuda(), d ** -0.5)
    assert torch.equal(new_a, new_b)
    assert torch.equal(o_f8, o_bf)
    ref = oracle.sparse_attn(bits(q), bits(kv_bf), sink.numpy(), idx.numpy(), d ** -0.5)
    assert_close_bf16(bits(o_f8), ref)
    assert ds.device_status() == 0


def test_attn_fp8kv_timed_out_wait_is_reported(ds):
    """The bounded-wait abort on the fp8 gather path (see the bf16 test above)."""
    q, _, sink, idx = _case(90, 4, 1, 64, 512, 2048, 700)
    kv = _spread_rows(90, 4 * 2048, 512).view(4, 2048, 512)
    codes, exps = ds.kv_quantize_fp8(kv.cuda())
    assert ds.device_status() == 0
    ds.test_set_stall(True)
    try:
        ds.sparse_attn_fp8kv(q.cuda(), codes, exps, sink.cuda(), idx.cuda(), 512 ** -0.5)
        bits_after = ds.device_status()
    finally:
        ds.test_set_stall(False)
    assert bits_after & ds.DS_DEV_TIMEOUT, f"expected a timeout, status bits {bits_after}"
    o = ds.sparse_attn_fp8kv(q.cuda(), codes, exps, sink.cuda(), idx.cuda(), 512 ** -0.5)
    dec = oracle.kv_dequantize_fp8(codes.cpu().numpy(), exps.cpu().numpy())
    ref = oracle.sparse_attn(bits(q), dec, sink.numpy(), idx.numpy(), 512 ** -0.5)
    assert_close_bf16(bits(o), ref)
    assert ds.device_status() == 0


# ----------------------------------------------------------------------------------------------
# RoPE: the rotation (and its inverse) and the RoPE-then-round-trip ring write
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("b,m,h,d,rd,p0,inverse", [(2, 3, 4, 128, 64, 100, False), (2, 3, 4, 128, 64, 100, True),
                                                   (4, 1, 128, 512, 64, 131072, True), (1, 40, 8, 64, 32, 0, False),
                                                   (3, 1, 5, 512, 512, 9, False)])
def test_apply_rotary_bit_exact(ds, b, m, h, d, rd, p0, inverse):
    g = torch.Generator().manual_seed(100 + d + m)
    x = (torch.randn((b, m, h, d), generator=g) * 4).to(torch.bfloat16)
    table = oracle.rope_table(p0 + m, rd, 10000.0)
    want = oracle.apply_rotary(bits(x).copy(), rd, table, p0, h, m, inverse)
    xg = x.cuda()
    ds.apply_rotary(xg, rd, torch.from_numpy(table).cuda(), p0, h, m, inverse)
    assert np.array_equal(bits(xg), want)


@pytest.mark.parametrize("b,s,d,W,p0,rd", [(1, 12, 64, 8, 0, 32), (3, 20, 64, 8, 37, 64), (4, 1, 512, 128, 10000, 64),
                                           (2, 300, 512, 128, 0, 64)])
def test_kv_rope_ring_write_bit_exact(ds, b, s, d, W, p0, rd):
    g = torch.Generator().manual_seed(200 + s)
    raw = (torch.randn((b, s, d), generator=g) * torch.exp(torch.randn((b, s, 1), generator=g) * 2)).to(torch.bfloat16)
    table = oracle.rope_table(p0 + s, rd, 10000.0)
    kv_o = bits(raw).copy()
    ring_o = np.zeros((b, W, d), dtype=np.uint16)
    oracle.kv_rope_quant_ring_write(kv_o, ring_o, p0, W, rd, table)
    kv = raw.cuda()
    ring = torch.zeros((b, W, d), dtype=torch.bfloat16, device="cuda")
    ds.kv_rope_quant_ring_write(kv, ring, p0, W, rd, torch.from_numpy(table).cuda())
    assert np.array_equal(bits(kv), kv_o)
    assert np.array_equal(bits(ring), ring_o)


@pytest.mark.parametrize("kernel", ["cluster", "one_cta"])
@pytest.mark.parametrize("d,h,b,m,topk,rd,p0", [(512, 64, 100, 2, 300, 64, 4000),    # cut tokens: the combine
                                                 (512, 128, 3, 1, 2176, 64, 131072),  # whole tokens, decode
                                                 (512, 16, 1, 5, 200, 512, 0),        # every column rotated
                                                 (512, 64, 32, 1, 640, 64, 16384),    # 4-CTA clusters merge
                                                 (512, 40, 6, 1, 300, 24, 77),        # 2 parts; rd not a multiple of 32
                                                 (64, 4, 1, 12, 8, 16, 0),            # the ratio-0 fixture's shape
                                                 (256, 32, 60, 3, 129, 32, 77)])
def test_sparse_attn_rope_equals_attention_then_inverse_rotation(ds, kernel, d, h, b, m, topk, rd, p0):
    """The inverse RoPE of the output fused into the attention epilogue, the in-cluster merge and
    the combine ("DeepSeek V4.1", attention/query-latent, Attention.forward rotates o back by its
    position): bit-identical to ds_sparse_attn followed by ds_apply_rotary(inverse) on the same
    kernel (each kernel where it is built for the shape), and to the oracle's rotation of that
    attention output; the attention itself matches the oracle within the tolerance."""
    if kernel == "one_cta" and (d != 512 or h > 64):
        pytest.skip("the one-CTA kernel is built for head_dim 512 and at most 64 heads")
    q, kv, sink, idx = _case(700 + d + m, b, m, h, d, 2 * topk, topk, 0.05)
    table = oracle.rope_table(p0 + m, rd, 10000.0)
    tg = torch.from_numpy(table).cuda()
    qg, kvg, sg, ig = q.cuda(), kv.cuda(), sink.cuda(), idx.cuda()
    with _kernel(ds, ds.KERNEL_CLUSTER if kernel == "cluster" else ds.KERNEL_ONE_CTA):
        fused = ds.sparse_attn_rope(qg, kvg, sg, ig, d ** -0.5, rd, tg, p0)
        plain = ds.sparse_attn(qg, kvg, sg, ig, d ** -0.5)
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), idx.numpy(), d ** -0.5)
    assert_close_bf16(bits(plain), ref)
    want = oracle.apply_rotary(bits(plain).copy(), rd, table, p0, h, m, True)
    assert np.array_equal(bits(fused), want)
    ds.apply_rotary(plain, rd, tg, p0, h, m, True)
    assert torch.equal(fused, plain)
    assert ds.device_status() == 0


def test_sparse_attn_rope_empty_topk_rotates_zeros(ds):
    """No index entries: o is zero, then rotated like any other output (the sign of a rotated
    zero follows the table, exactly as the separate rotation pass gives it)."""
    q, kv, sink, idx = _case(710, 2, 3, 8, 64, 10, 0)
    table = oracle.rope_table(40, 16, 10000.0)
    fused = ds.sparse_attn_rope(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), 0.125, 16, torch.from_numpy(table).cuda(),
                                30)
    want = oracle.apply_rotary(np.zeros((2, 3, 8, 64), dtype=np.uint16), 16, table, 30, 8, 3, True)
    assert np.array_equal(bits(fused), want)


def test_apply_rotary_rate(ds):
    """The inverse rotation of decode_large's output (256 tokens x 128 heads x 512, last 64 values
    rotated) as a memory-bound kernel: CUDA events over repeated launches, printed as GB/s of the
    bytes it must move (the rotated 128 bytes of each row read and written, the table row read)."""
    b, h, d, rd, p0 = 256, 128, 512, 64, 131072
    o = torch.randn((b, 1, h, d), device="cuda").to(torch.bfloat16)
    table = torch.from_numpy(oracle.rope_table(p0 + 1, rd, 10000.0)).cuda()
    for _ in range(3):
        ds.apply_rotary(o, rd, table, p0, h, 1, True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 50
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n):
        ds.apply_rotary(o, rd, table, p0, h, 1, True)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    moved = b * h * rd * 2 * 2 + rd * 4
    print(f"\napply_rotary on decode_large's o: {us:.2f} us per launch, {moved / us / 1e3:.0f} GB/s of {moved} bytes")
    assert us > 0


# ----------------------------------------------------------------------------------------------
# output canaries: every write of a call stays inside its output and workspace
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("d,h,b,m,topk", [(512, 64, 100, 2, 300), (512, 128, 1, 1, 5000), (64, 8, 300, 1, 200)])
def test_writes_stay_inside_o_and_workspace(ds, fp8, d, h, b, m, topk):
    """o sits between two 128-byte canary bands inside a larger buffer, the workspace has a 4 KB
    canary band after the size the library asks for; after the call every canary byte is as it
    was and o matches the oracle (shapes with cut tokens, so the workspace is used)."""
    if fp8 and d != 512:
        pytest.skip("the fp8 row store is read by the d = 512 kernel")
    q, kv, sink, idx = _case(300 + d + b, b, m, h, d, 2 * topk, topk, 0.05)
    pad, canary = 64, 0x5A5A
    big = torch.full((q.numel() + 2 * pad,), canary, dtype=torch.int16, device="cuda")
    o = big[pad:pad + q.numel()].view(torch.bfloat16).view(q.shape)
    need = ds.sparse_attn_workspace_bytes(b, m, h, d, topk)
    ws_big = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = ws_big[:need] if need else None
    if fp8:
        # the same N(0,1) rows, kept as the fp8 row store (this test is about where writes land;
        # wide-range rows are the subject of test_attn_wide_range_rows_as_accurate_as_f32)
        codes, exps = ds.kv_quantize_fp8(kv.cuda())
        ds.sparse_attn_fp8kv(q.cuda(), codes, exps, sink.cuda(), idx.cuda(), d ** -0.5, o=o, workspace=ws)
        kv_ref = oracle.kv_dequantize_fp8(codes.cpu().numpy(), exps.cpu().numpy())
    else:
        ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), d ** -0.5, o=o, workspace=ws)
        kv_ref = bits(kv)
    torch.cuda.synchronize()
    bb = big.cpu()
    assert (bb[:pad] == canary).all() and (bb[pad + q.numel():] == canary).all()
    assert (ws_big[need:].cpu() == 0xA5).all()
    ref = oracle.sparse_attn(bits(q), kv_ref, sink.numpy(), idx.numpy(), d ** -0.5)
    assert_close_bf16(bits(o), ref)
    assert ds.device_status() == 0


# ----------------------------------------------------------------------------------------------
# prefill in pairs: queries 2j and 2j + 1 share one gather of the union of their rows
# ----------------------------------------------------------------------------------------------

def _prefill_rows(seed, b, m, n, window, K, ncomp, neg_tail=True):
    """Index rows shaped like a prefill chunk's: query q's causal window rows (chunk positions
    max(0, q - window + 1) .. q, -1 before the chunk start) then K compressed positions drawn
    without replacement from the first q // 4 of ncomp (shifted past the chunk), ascending,
    -1 padded at the tail."""
    g = torch.Generator().manual_seed(seed)
    W = min(m, window)
    idx = torch.full((b, m, W + K), -1, dtype=torch.int32)
    for qi in range(m):
        lo = max(0, qi - window + 1)
        win = torch.arange(lo, lo + W)
        idx[:, qi, :W] = torch.where(win <= qi, win, -1).to(torch.int32)
        avail = min(qi // 4, ncomp)
        for bi in range(b):
            if avail:
                sel = torch.sort(torch.randperm(avail, generator=g)[:min(K, avail)]).values
                idx[bi, qi, W:W + len(sel)] = (sel + m).to(torch.int32)
    return idx


PAIR_CASES = [
    # seed, b, m, h, d, window, K, ncomp
    (1, 1, 12, 4, 64, 8, 0, 0),            # the ratio-0 fixture's prefill shape
    (2, 2, 37, 8, 64, 16, 24, 40),         # odd query count: the last pair has one query
    (3, 1, 300, 64, 512, 128, 64, 200),    # more pairs than clusters: pairs cut across CTAs
    (4, 3, 21, 64, 512, 128, 512, 1024),   # wide rows, few queries
    (5, 1, 130, 32, 512, 128, 40, 60),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=[f"p{c[0]}" for c in PAIR_CASES])
def test_prefill_pairs_match_oracle(ds, case):
    seed, b, m, h, d, window, K, ncomp = case
    n = m + ncomp
    g = torch.Generator().manual_seed(600 + seed)
    q = torch.randn((b, m, h, d), generator=g).to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g).to(torch.bfloat16)
    sink = torch.randn((h,), generator=g)
    idx = _prefill_rows(seed, b, m, n, window, K, ncomp)
    o = ds.sparse_attn_prefill(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), d ** -0.5)
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), idx.numpy(), d ** -0.5)
    assert_close_bf16(bits(o), ref)
    assert ds.device_status() == 0
    # the same rows in any order (the union is sorted on the GPU), and repeatable bit for bit
    perm = torch.randperm(idx.shape[-1], generator=torch.Generator().manual_seed(seed))
    o2 = ds.sparse_attn_prefill(q.cuda(), kv.cuda(), sink.cuda(), idx[..., perm].contiguous().cuda(), d ** -0.5)
    assert torch.equal(o, o2)


def test_prefill_pairs_empty_and_shared_rows(ds):
    """Pairs whose rows are all -1 (zeros out), pairs where only one query lists anything, and
    pairs listing exactly the same rows."""
    b, m, h, d, n = 2, 8, 16, 512, 200
    g = torch.Generator().manual_seed(620)
    q = torch.randn((b, m, h, d), generator=g).to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g).to(torch.bfloat16)
    sink = torch.randn((h,), generator=g)
    idx = torch.stack([torch.randperm(n, generator=g)[:90] for _ in range(b * m)]).view(b, m, 90).to(torch.int32)
    idx[0, 0:2] = -1                  # pair 0 of sequence 0: nothing at all
    idx[0, 3] = -1                    # pair 1: only its first query lists rows
    idx[1, 5] = idx[1, 4]             # pair 2 of sequence 1: the same rows twice
    o = ds.sparse_attn_prefill(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), d ** -0.5)
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), idx.numpy(), d ** -0.5)
    assert_close_bf16(bits(o), ref)
    assert (o[0, 0:2].float() == 0).all() and (o[0, 3].float() == 0).all()
    assert ds.device_status() == 0


def test_prefill_pairs_without_rows_inside_ranges(ds):
    """More query pairs than clusters (several pairs per work range), some pairs listing no
    row at all, one pair where only the second query lists rows."""
    b, m, h, d, n = 1, 700, 16, 512, 400
    g = torch.Generator().manual_seed(640)
    q = torch.randn((b, m, h, d), generator=g).to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g).to(torch.bfloat16)
    sink = torch.randn((h,), generator=g)
    idx = torch.stack([torch.randperm(n, generator=g)[:100] for _ in range(b * m)]).view(b, m, 100).to(torch.int32)
    for j in (10, 11, 200, 201, 202, 349):     # pairs (2j, 2j + 1) with nothing
        idx[0, 2 * j:2 * j + 2] = -1
    idx[0, 2 * 50] = -1                        # pair 50: only its second query
    o = ds.sparse_attn_prefill(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), d ** -0.5)
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), idx.numpy(), d ** -0.5)
    assert_close_bf16(bits(o), ref)
    for j in (10, 11, 200, 201, 202, 349):
        assert (o[0, 2 * j:2 * j + 2].float() == 0).all()
    assert ds.device_status() == 0


def test_prefill_pairs_flag_a_row_listed_twice(ds):
    """This path counts a row once per query: a row listed twice by one query raises
    DS_DEV_BAD_INDEX, and the output is that of the row listed once."""
    b, m, h, d, n = 1, 4, 8, 64, 50
    g = torch.Generator().manual_seed(630)
    q = torch.randn((b, m, h, d), generator=g).to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g).to(torch.bfloat16)
    sink = torch.randn((h,), generator=g)
    idx = torch.stack([torch.randperm(n, generator=g)[:20] for _ in range(m)]).view(b, m, 20).to(torch.int32)
    dup = idx.clone()
    dup[0, 2, 5] = dup[0, 2, 4]
    o = ds.sparse_attn_prefill(q.cuda(), kv.cuda(), sink.cuda(), dup.cuda(), 0.125)
    assert ds.device_status() & ds.DS_DEV_BAD_INDEX
    once = dup.clone()
    once[0, 2, 5] = -1
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), once.numpy(), 0.125)
    assert_close_bf16(bits(o), ref)
    assert ds.device_status() == 0


def test_prefill_workload_in_pairs(ds):
    """The prefill workload at full size (4096 queries, 64 heads, 512 wide, 128 window + 512
    compressed rows) through the pair path, sampled tokens against the oracle, repeatable."""
    w = wl.WORKLOADS[2]
    gs = GpuStep(w)
    need = ds.sparse_attn_prefill_workspace_bytes(w.b, w.m, w.h, w.d, w.topk)
    gs.workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    from sparse_latent_attention_attn_gb300 import path
    inp = gs.inp
    path.prefill_step(inp.q, gs.kv, gs.ring, inp.sink, gs.idx, w.window, w.scale, o=gs.o, workspace=gs.workspace,
                      pairs=True)
    torch.cuda.synchronize()
    orc = OracleStep(gs, seqs=[0])
    toks = np.array(SAMPLE_TOKENS_PREFILL, dtype=np.int64)
    assert_close_bf16(bits(gs.o[0, torch.from_numpy(toks).cuda()]), orc.attend(tokens=toks), "prefill pairs o")
    first = gs.o.clone()
    ds.sparse_attn_prefill(inp.q, gs.kv, inp.sink, gs.idx, w.scale, o=gs.o, workspace=gs.workspace)
    torch.cuda.synchronize()
    diff = (first.float() - gs.o.float()).abs()
    where = (diff > 0).any(dim=3).any(dim=2)[0].nonzero().flatten().tolist()
    assert not where, (f"repeated call differs at {int((diff > 0).sum())} outputs (max {diff.max().item()}) "
                       f"of tokens {where[:16]} ({len(where)} tokens)")
    assert ds.device_status() == 0
