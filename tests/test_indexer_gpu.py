"""The Indexer on the GPU through the C ABI, against the oracle ("DeepSeek V4.1",
attention/query-latent, Indexer.forward).

* Scores: f32 on both sides, so they agree within the rounding of an f32 evaluation: the dot
  products (D terms) and the head sum (H terms) each add at most a few units of 2^-24 relative to
  the sum of the absolute values of their terms.  The bound used is 4 (D + H) 2^-24 times
  sum_h |w_h| sum_d |q_hd k_td|, computed in float64 from the inputs; unseen positions must be
  -inf on both sides.
* Selection alone (ds_indexer_select on the oracle's own scores, ties included): bit-exact with
  the oracle's selection, since both take the larger score first and, at equal scores, the
  smaller position.
* Scores and selection together: the two sides' scores differ by rounding, so a position whose
  score sits within that bound of the cut may be kept by one side and not the other.  The GPU
  row must be a valid selection (kk entries, ascending, distinct, the right -1 count), keep
  every position the oracle scores clearly above the cut, and keep none clearly below it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_latent_attention_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

EPS32 = 2.0 ** -24


@pytest.fixture(scope="module")
def ds():
    from sparse_latent_attention_attn_gb300 import dsattn
    dsattn.device_status()
    return dsattn


def _bits(t: torch.Tensor) -> np.ndarray:
    return wl.bits(t)


def _case(seed, b, s, H, D, start_pos, ratio=4, extra_rows=0):
    g = torch.Generator().manual_seed(seed)
    Tv = (start_pos + s) // ratio
    q = torch.randn((b, s, H, D), generator=g).to(torch.bfloat16)
    k = torch.randn((b, Tv + extra_rows, D), generator=g).to(torch.bfloat16)
    w = torch.randn((b, s, H), generator=g).to(torch.bfloat16).float() * (D ** -0.5 * H ** -0.5)
    return q, k, w


def _score_bound(q, k, w, start_pos, ratio):
    """Per (bi, i, t) rounding bound of an f32 evaluation of the score (float64)."""
    b, s, H, D = q.shape
    Tv = (start_pos + s) // ratio
    mag = torch.einsum("bshd,btd->bsht", q.double().abs(), k[:, :Tv].double().abs())
    return 4 * (D + H) * EPS32 * (mag * w.double().abs().unsqueeze(-1)).sum(dim=2)


def _check_scores(got, ref, bound):
    """got, ref [b][s][Tv] f32; -inf at the same places, finite ones within bound."""
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "unseen positions differ"
    assert (got[~fin] == -np.inf).all() and (ref[~fin] == -np.inf).all()
    err = np.abs(got[fin].astype(np.float64) - ref[fin].astype(np.float64))
    bad = err > bound[fin]
    assert not bad.any(), f"{int(bad.sum())} scores outside the f32 bound; worst excess {float((err - bound[fin]).max())}"


def _check_selection(got_row, ref_scores_row, lens, kk, offset, tol):
    """got_row: the GPU's kk entries for one query; ref_scores_row: oracle scores [Tv]."""
    got = np.asarray(got_row, dtype=np.int64)
    assert got.shape == (kk,)
    nvis = min(lens, kk)
    valid = got[got >= 0]
    assert (got[:len(valid)] >= 0).all(), "-1 entries must follow the kept positions"
    assert len(valid) == nvis and (got[nvis:] == -1).all(), f"{len(valid)} kept of {nvis}"
    pos = valid - offset
    assert (np.diff(pos) > 0).all(), "kept positions must be ascending and distinct"
    assert (pos >= 0).all() and (pos < lens).all()
    if lens <= kk:
        assert np.array_equal(pos, np.arange(lens))
        return
    sc = ref_scores_row[:lens].astype(np.float64)
    cut = np.sort(sc)[::-1][kk - 1]
    assert (sc[pos] >= cut - tol).all(), "a kept position scores clearly below the cut"
    must = np.nonzero(sc > cut + tol)[0]
    assert np.isin(must, pos).all(), "a position clearly above the cut was not kept"


SCORE_CASES = [
    # seed, b, s, H, D, start_pos, extra key rows
    (1, 2, 1, 64, 128, 4000, 0),       # decode, 1001 positions (ragged last tile)
    (2, 1, 37, 64, 128, 0, 0),         # prefill, causal, a ragged query block
    (3, 3, 1, 16, 64, 130, 5),         # narrow heads, small width, key rows beyond the visible ones
    (4, 1, 300, 32, 128, 0, 0),        # prefill, 8 queries per block
    (5, 2, 2, 48, 128, 9000, 0),       # two queries per sequence at once
    (6, 1, 1, 256, 64, 700, 0),        # 256 heads: one query fills N
    # more query blocks than SMs (several waves of CTAs), ragged blocks and chunks
    (7, 1, 700, 64, 128, 0, 0),        # 350 blocks of 2 queries, 2 key tiles each
    (8, 2, 400, 16, 64, 2000, 3),      # 8 queries per block, 3 key chunks per block, start_pos > 0
    (9, 1, 600, 256, 64, 0, 0),        # 256 heads: one query per block, N = 256
]


@pytest.mark.parametrize("case", SCORE_CASES, ids=[f"i{c[0]}" for c in SCORE_CASES])
def test_indexer_scores_match_oracle(ds, case):
    seed, b, s, H, D, p0, extra = case
    q, k, w = _case(seed, b, s, H, D, p0, extra_rows=extra)
    _, ref = oracle.indexer_topk(_bits(q), _bits(k), w.numpy(), p0, 4, 1, return_scores=True)
    Tv = (p0 + s) // 4
    got = ds.indexer_scores(q.cuda(), k.cuda(), w.cuda(), p0, 4).cpu().numpy()
    _check_scores(got, ref[..., :Tv], _score_bound(q, k, w, p0, 4).numpy())
    assert ds.device_status() == 0


@pytest.mark.parametrize("start_pos,s,topk,offset,grid", [(0, 64, 5, 0, 0.5), (0, 300, 20, 4096, 0.25),
                                                          (4000, 1, 512, 128, 0.125), (131071, 1, 2048, 128, 1.0),
                                                          (400, 3, 20, 7, 0.0), (240000, 1, 3000, 0, 0.5)])
def test_indexer_select_is_exact_on_given_scores(ds, start_pos, s, topk, offset, grid):
    """ds_indexer_select on scores with many exact ties (values on a coarse grid; grid 0 makes
    every score equal), including -0 next to +0: the same entries as the oracle, in order.  Rows
    of up to 4096 positions, up to 49152 (order keys kept in shared memory) and longer (read from
    L2 in every pass) take different kernel variants."""
    g = torch.Generator().manual_seed(11 + s)
    Tv = (start_pos + s) // 4
    b = 3 if Tv <= 40000 else 1
    sc = torch.randn((b, s, Tv + 5), generator=g)
    sc = (sc / grid).round() * grid if grid > 0 else torch.zeros_like(sc)
    sc[:, :, 1::9] = -0.0
    sc = sc.contiguous()
    want = oracle.indexer_select(sc.numpy(), start_pos, 4, topk, offset)
    got = ds.indexer_select(sc.cuda(), start_pos, 4, topk, offset).cpu().numpy()
    assert np.array_equal(got, want)


@pytest.mark.parametrize("case", SCORE_CASES, ids=[f"i{c[0]}" for c in SCORE_CASES])
def test_indexer_topk_small(ds, case):
    seed, b, s, H, D, p0, extra = case
    q, k, w = _case(seed, b, s, H, D, p0, extra_rows=extra)
    topk, offset = 40, 100
    idx_o, ref = oracle.indexer_topk(_bits(q), _bits(k), w.numpy(), p0, 4, topk, offset, return_scores=True)
    got = ds.indexer_topk(q.cuda(), k.cuda(), w.cuda(), p0, 4, topk, offset).cpu().numpy()
    kk = min(topk, (p0 + s) // 4)
    assert got.shape == idx_o.shape == (b, s, kk)
    bound = _score_bound(q, k, w, p0, 4).numpy()
    for bi in range(b):
        for i in range(s):
            lens = (p0 + i + 1) // 4
            _check_selection(got[bi, i], ref[bi, i], lens, kk, offset, 2 * float(bound[bi, i].max()))
    assert ds.device_status() == 0


SAMPLE = {2: [0, 3, 4, 511, 2047, 2048, 3000, 4095], 3: [0, 17, 31], 4: [0, 101, 255]}


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_indexer_workload_parity(ds, cfg):
    """The three Indexer workloads at full size in the bench's launch configuration; sampled
    queries (decode: sequences, prefill: query tokens) are scored and selected by the oracle one
    by one, each as the decode step at that position."""
    iw = wl.INDEXER_WORKLOADS[cfg]
    q, k, w = wl.indexer_inputs(iw, device="cuda")
    idx = ds.indexer_topk(q, k, w, iw.start_pos, iw.ratio, iw.topk, iw.offset)
    scores = ds.indexer_scores(q, k, w, iw.start_pos, iw.ratio)
    torch.cuda.synchronize()
    kk = min(iw.topk, iw.Tv)
    for j in SAMPLE[cfg]:
        bi, i = (j, 0) if iw.s == 1 else (0, j)
        pos = iw.start_pos + i
        lens = (pos + 1) // iw.ratio
        if lens == 0:                 # sees no compressed position yet: every entry is -1
            assert (idx[bi, i] == -1).all()
            assert (scores[bi, i] == -math.inf).all()
            continue
        qs = _bits(q[bi:bi + 1, i:i + 1])
        ks = _bits(k[bi:bi + 1, :lens])
        ws = w[bi:bi + 1, i:i + 1].cpu().numpy()
        idx_o, ref = oracle.indexer_topk(qs, ks, ws, pos, iw.ratio, iw.topk, iw.offset, return_scores=True)
        qc, kc, wc = q[bi:bi + 1, i:i + 1].cpu(), k[bi:bi + 1, :lens].cpu(), w[bi:bi + 1, i:i + 1].cpu()
        bound = _score_bound(qc, kc, wc, pos, iw.ratio).numpy()[0, 0]
        got_sc = scores[bi, i, :lens].cpu().numpy()
        _check_scores(got_sc[None, None], ref[:, :, :lens], bound[None, None, :lens])
        _check_selection(idx[bi, i].cpu().numpy(), ref[0, 0], lens, kk, iw.offset, 2 * float(bound.max()))
    again = ds.indexer_topk(q, k, w, iw.start_pos, iw.ratio, iw.topk, iw.offset)
    assert torch.equal(idx, again), "repeated calls differ"
    assert ds.device_status() == 0


def test_indexer_all_kept_and_empty(ds):
    """kk equal to every visible position (the row is 0 .. lens - 1 then -1), and a step that
    sees no compressed position yet (nothing to write)."""
    q, k, w = _case(20, 2, 8, 16, 64, 0)
    got = ds.indexer_topk(q.cuda(), k.cuda(), w.cuda(), 0, 4, 99, 5).cpu().numpy()   # kk = Tv = 2
    want = oracle.indexer_topk(_bits(q), _bits(k), w.numpy(), 0, 4, 99, 5)
    assert np.array_equal(got, want)
    q1, k1, w1 = _case(21, 2, 2, 16, 64, 0)       # Tv = 0
    out = ds.indexer_topk(q1.cuda(), k1.cuda(), w1.cuda(), 0, 4, 10)
    assert out.shape == (2, 2, 0)


def test_indexer_argument_errors(ds):
    q, k, w = _case(22, 1, 1, 16, 64, 100)
    with pytest.raises(ds.DsError) as e:
        ds.indexer_topk(q[..., :48].contiguous().cuda(), k[..., :48].contiguous().cuda(), w.cuda(), 100, 4, 8)
    assert e.value.status == ds.DS_EUNSUPPORTED
    with pytest.raises(ds.DsError) as e:              # fewer key rows than positions visible
        ds.indexer_topk(q.cuda(), k[:, :10].contiguous().cuda(), w.cuda(), 100, 4, 8)
    assert e.value.status == ds.DS_EINVAL
    q2, k2, w2 = _case(23, 1, 1, 24, 64, 100)       # 24 heads: not a multiple of 16
    with pytest.raises(ds.DsError) as e:
        ds.indexer_topk(q2.cuda(), k2.cuda(), w2.cuda(), 100, 4, 8)
    assert e.value.status == ds.DS_EUNSUPPORTED
