"""The one-CTA sparse_attn kernel (head_dim 512, at most 64 heads, transposed accumulator) against
the oracle, through the C ABI.

ds_sparse_attn picks this kernel by itself wherever it is built for the shape; the test switch
ds_test_set_kernel forces either kernel, so every case here runs on both and each result is held
to the attention tolerance against the oracle ("Module attn", sparse_attn and the
Precision paragraph: |gpu - ref| <= 1e-2 + 1.6e-2 |ref|).  Cases cover whole and cut tokens
(parts merged inside a cluster of 2, 3 or 4 CTAs, or by the combine kernel), ragged last tiles, odd head counts, entries that are
-1, duplicated or out of range, rows with no valid entry, many parts per token, more tokens than
SMs (several segments per CTA), and scores that grow along the index row so the running
max moves and the accumulator is rescaled.
"""
import numpy as np
import pytest
import torch

import oracle
from pathcheck import assert_close_bf16, bits

pytestmark = pytest.mark.gpu

KERNELS = {"cluster": 1, "one_cta": 2}


@pytest.fixture(scope="module")
def ds():
    from sparse_latent_attention_attn_gb300 import dsattn
    dsattn.device_status()
    return dsattn


@pytest.fixture(params=list(KERNELS), ids=list(KERNELS))
def kernel(ds, request):
    ds.test_set_kernel(KERNELS[request.param])
    yield request.param
    ds.test_set_kernel(ds.KERNEL_AUTO)


def _case(seed, b, m, h, n, topk, neg=0.05, dup=False, grow=0.0, qscale=1.0, d=512):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn((b, m, h, d), generator=g) * qscale).to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g)
    if grow:
        # row r scaled by 1 + grow * r / n: with ascending indices the later tiles score higher
        kv = kv * (1.0 + grow * torch.arange(n, dtype=torch.float32) / n).view(1, n, 1)
    kv = kv.to(torch.bfloat16)
    sink = torch.randn((h,), generator=g)
    if dup or topk > n:
        idx = torch.randint(0, n, (b, m, topk), generator=g)
    else:
        idx = torch.stack([torch.randperm(n, generator=g)[:topk] for _ in range(b * m)]).view(b, m, topk)
    if grow:
        idx = idx.sort(dim=-1).values
    idx = torch.where(torch.rand((b, m, topk), generator=g) < neg, -1, idx).to(torch.int32)
    return q, kv, sink, idx


def _check(ds, q, kv, sink, idx, what):
    d = q.shape[-1]
    scale = d ** -0.5
    o = ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), scale)
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), idx.numpy(), scale)
    assert_close_bf16(bits(o), ref, what)
    return o


CASES = [
    # seed, b, m, h, n, topk, neg
    (1, 2, 2, 64, 700, 640, 0.05),       # 4 tokens, each cut over several CTAs
    (2, 1, 1, 64, 300, 1, 0.0),          # a single entry
    (3, 3, 1, 33, 500, 129, 0.3),        # odd head count, ragged last tile, many -1
    (4, 4, 1, 16, 900, 300, 0.1),
    (5, 40, 2, 64, 1000, 200, 0.05),     # 80 tokens
    (6, 32, 1, 64, 4224, 640, 0.05),     # decode_comp's shape
    (7, 1, 4, 64, 5000, 2176, 0.02),     # decode_large's index width, 64 heads
    (8, 1, 1, 64, 12000, 8192, 0.02),    # one token over 32 CTAs
    (9, 64, 1, 64, 128, 128, 0.0),       # decode_window's shape: whole tokens, no combine
    (10, 2, 1, 8, 200, 70, 0.0),         # 8 heads, a 6-entry last tile
    (11, 8, 2, 40, 900, 300, 0.05),      # two queries per sequence, 40 heads, 2-CTA merges
    (12, 45, 1, 48, 1000, 400, 0.05),    # 45 tokens in 3 parts each: 3-CTA merges
    (13, 15, 3, 64, 900, 384, 0.05),     # the same with three queries per sequence
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{c[0]}" for c in CASES])
def test_attn_matches_oracle_on_both_kernels(ds, kernel, case):
    seed, b, m, h, n, topk, neg = case
    q, kv, sink, idx = _case(seed, b, m, h, n, topk, neg)
    _check(ds, q, kv, sink, idx, f"{kernel} c{seed}")
    assert ds.device_status() == 0


@pytest.mark.parametrize("ntok,h,topk", [(200, 8, 257), (300, 64, 640), (1000, 32, 130)])
def test_more_tokens_than_sms(ds, kernel, ntok, h, topk):
    """Several segments per CTA (stream-K ranges cut inside tokens): every token is checked."""
    q, kv, sink, idx = _case(60 + h, ntok, 1, h, 3 * topk, topk, 0.05)
    _check(ds, q, kv, sink, idx, f"{kernel} stream-k")
    assert ds.device_status() == 0


@pytest.mark.parametrize("grow,qscale", [(3.0, 4.0), (8.0, 8.0)])
def test_running_max_moves_along_the_row(ds, kernel, grow, qscale):
    """Index rows ascending over rows whose norms grow along kv: each tile's scores exceed the
    running max of the earlier ones by many log2 units, so the lazy rescale of the accumulator
    runs, on whole tokens and on cut ones."""
    q, kv, sink, idx = _case(70, 3, 1, 64, 6000, 1500, 0.02, grow=grow, qscale=qscale)
    _check(ds, q, kv, sink, idx, f"{kernel} rescale")
    assert ds.device_status() == 0


def test_invalid_duplicate_and_out_of_range_entries(ds, kernel):
    """-1 everywhere in one token (its output is 0), duplicates counted as listed, and entries
    >= n skipped and flagged with DS_DEV_BAD_INDEX."""
    q, kv, sink, idx = _case(80, 4, 1, 64, 300, 400, 0.1, dup=True)
    idx[1] = -1
    o = _check(ds, q, kv, sink, idx, f"{kernel} dup")
    assert (o[1].float() == 0).all()
    assert ds.device_status() == 0
    bad = idx.clone()
    bad[2, 0, 5] = 300
    bad[3, 0, 399] = 1 << 30
    ref_idx = bad.clone()
    ref_idx[ref_idx >= 300] = -1
    scale = 512 ** -0.5
    got = ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), bad.cuda(), scale)
    ref = oracle.sparse_attn(bits(q), bits(kv), sink.numpy(), ref_idx.numpy(), scale)
    assert_close_bf16(bits(got), ref, f"{kernel} out of range")
    assert ds.device_status() & ds.DS_DEV_BAD_INDEX
    assert ds.device_status() == 0


def test_tokens_without_rows_inside_ranges(ds, kernel):
    """More tokens than CTAs or clusters, so each work range holds several tokens, some of
    them listing no valid row at all (scattered, three in a row, and the last): such a token's
    output is 0, and the tokens after it in the same range get their own q (the cluster kernel
    loads it in the softmax warps after a segment without rows, in its exchange warps after any
    other segment)."""
    q, kv, sink, idx = _case(85, 300, 1, 64, 500, 200, 0.05)
    empty = [5, 6, 100, 151, 152, 153, 299]
    for t in empty:
        idx[t] = -1
    o = _check(ds, q, kv, sink, idx, f"{kernel} empty tokens")
    for t in empty:
        assert (o[t].float() == 0).all()
    assert ds.device_status() == 0


def test_twenty_thousand_tokens_sampled(ds, kernel):
    """20000 tokens of 16 entries, far more than CTAs: every work range walks over a hundred
    tokens (segment changes, q loads and index arithmetic over long ranges).  Sampled tokens,
    the first and last ones and those at range-like boundaries among them, against the oracle."""
    b, h, d, n, topk = 20000, 64, 512, 16, 16
    g = torch.Generator(device="cuda").manual_seed(97)
    q = torch.randn((b, 1, h, d), generator=g, device="cuda").to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g, device="cuda").to(torch.bfloat16)
    sink = torch.randn((h,), generator=g, device="cuda")
    idx = torch.argsort(torch.rand((b, 1, n), generator=g, device="cuda"), dim=-1)[..., :topk].to(torch.int32)
    idx[torch.rand((b, 1, topk), generator=g, device="cuda") < 0.05] = -1
    scale = d ** -0.5
    o = ds.sparse_attn(q, kv, sink, idx, scale)
    torch.cuda.synchronize()
    pick = [0, 1, 2, 131, 132, 151, 152, 153, 9999, 10000, 19997, 19998, 19999]
    pick += torch.randint(0, b, (24,), generator=torch.Generator().manual_seed(98)).tolist()
    sk = sink.cpu().numpy()
    for t in pick:
        ref = oracle.sparse_attn(bits(q[t:t + 1]), bits(kv[t:t + 1]), sk, idx[t:t + 1].cpu().numpy(), scale)
        assert_close_bf16(bits(o[t:t + 1]), ref, f"{kernel} token {t}")
    assert ds.device_status() == 0


def test_plan_query_names_the_kernel(ds):
    """ds_sparse_attn_launches reports the kernel ds_sparse_attn picks and how many kernels it
    enqueues (the combine kernel only where tokens are cut and not merged inside a cluster)."""
    assert ds.sparse_attn_launches(32, 1, 64, 512, 640) == (1, ds.KERNEL_ONE_CTA)   # 4-CTA clusters merge
    assert ds.sparse_attn_launches(64, 1, 64, 512, 128) == (1, ds.KERNEL_ONE_CTA)   # whole tokens
    assert ds.sparse_attn_launches(4, 1, 64, 512, 700) == (2, ds.KERNEL_ONE_CTA)    # 5 parts: the combine
    assert ds.sparse_attn_launches(256, 1, 128, 512, 2176)[1] == ds.KERNEL_CLUSTER  # 128 heads
    assert ds.sparse_attn_launches(4, 1, 8, 64, 700)[1] == ds.KERNEL_CLUSTER        # head_dim 64
    assert ds.sparse_attn_launches(4, 1, 64, 512, 0) == (1, ds.KERNEL_ONE_CTA)      # the zero fill
    try:
        ds.test_set_kernel(ds.KERNEL_CLUSTER)
        assert ds.sparse_attn_launches(32, 1, 64, 512, 640)[1] == ds.KERNEL_CLUSTER
    finally:
        ds.test_set_kernel(ds.KERNEL_AUTO)


def test_both_kernels_agree_and_repeat_exactly(ds):
    """On decode_comp's shape the two kernels give results within the attention tolerance of each
    other, and each repeats bit for bit."""
    q, kv, sink, idx = _case(90, 32, 1, 64, 4224, 640, 0.05)
    scale = 512 ** -0.5
    outs = {}
    try:
        for name, which in KERNELS.items():
            ds.test_set_kernel(which)
            a = ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), scale)
            b = ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), scale)
            assert torch.equal(a, b), f"{name}: repeated calls differ"
            outs[name] = bits(a)
    finally:
        ds.test_set_kernel(ds.KERNEL_AUTO)
    assert_close_bf16(outs["one_cta"], outs["cluster"], "one_cta against cluster")
    assert ds.device_status() == 0


@pytest.mark.parametrize("b,topk", [(4, 700), (32, 640)])
def test_timed_out_wait_is_reported(ds, b, topk):
    """The one-CTA kernel's bounded waits, made to run out with the stall hook (the gather warps
    withhold the first tile's arrivals): the call ends, raises DS_DEV_TIMEOUT, and the next call
    is clean and correct.  With 32 tokens of 640 entries the CTAs of a token form a cluster that
    merges in the kernel; with 4 tokens of 700 a combine kernel merges the parts."""
    q, kv, sink, idx = _case(95, b, 1, 64, 2048, topk)
    scale = 512 ** -0.5
    assert ds.device_status() == 0
    ds.test_set_kernel(KERNELS["one_cta"])
    try:
        ds.test_set_stall(True)
        try:
            ds.sparse_attn(q.cuda(), kv.cuda(), sink.cuda(), idx.cuda(), scale)
            status_bits = ds.device_status()
        finally:
            ds.test_set_stall(False)
        assert status_bits & ds.DS_DEV_TIMEOUT, f"expected a timeout, status bits {status_bits}"
        _check(ds, q, kv, sink, idx, "after a timeout")
    finally:
        ds.test_set_kernel(ds.KERNEL_AUTO)
    assert ds.device_status() == 0
