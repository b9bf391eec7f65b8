"""Seeded synthetic workloads for the sparse latent attention hot path.

This module holds only shapes and seeded random inputs.  It contains none of the method's
arithmetic (no quantisation, no index rows, no attention), so that both the CUDA path and the
CPU oracle can be fed from it without sharing any of the computation.

The five workloads follow the decode and prefill regimes of "DeepSeek V4.1", attention/attend and
attention/query-latent (a sliding-window ring of raw KV plus ``index_topk`` compressed positions
concatenated behind it), and the ratio-0 fixture of "Module attn" (ring-cache paragraph):

* ``fixture``        bsz 1, 4 heads, head_dim 64, 8-slot ring; prefill 12 tokens, decode 12, 13.
* ``decode_window``  bsz 64, 64 heads, head_dim 512, 128-slot ring full (start_pos 10000).
* ``prefill``        bsz 1, 4096 queries at start_pos 0, 64 heads, head_dim 512, 128-token causal
                     window plus 512 compressed indices per query drawn without replacement from
                     the first floor(q/4) of 1024 compressed rows (tail padded with -1).
* ``decode_comp``    bsz 32, 64 heads, 128-slot ring full plus 512 compressed indices per query from
                     4096 compressed rows, exactly round(0.05*512) entries set to -1.
* ``decode_large``   bsz 256, 128 heads, 128-slot ring plus 2048 compressed indices per query from
                     32768 compressed rows, exactly round(0.02*2048) entries set to -1.

Values: q, kv ~ N(0,1) rounded to bf16; sink ~ N(0,1) in f32; softmax scale head_dim**-0.5
(Attention.__init__).  Window rows are raw here: the step itself rounds each new row through
fp8 on its way into the ring, and a decode workload's older ring slots are handed over raw
(``hist``) so that each side rounds them with its own quantiser.  Compressed rows stay plain bf16.
Compressed indices are sorted ascending per row (the Indexer re-sorts its top-k into position
order) and already shifted past the window rows, as ``Attention.forward`` concatenates them.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    b: int          # sequences
    h: int          # heads
    d: int          # head_dim (latent row width)
    window: int     # ring slots
    start_pos: int  # position of the first query of the step
    s: int          # queries per sequence in the step (1 for decode)
    n_comp: int     # compressed rows per sequence (0: pure sliding window)
    topk_comp: int  # compressed indices per query
    neg_frac: float  # fraction of compressed entries that are -1 (exact count per row)
    comp_mode: str  # "none" | "uniform" | "prefill_causal"
    rope_dim: int

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    @property
    def decode(self) -> bool:
        return self.start_pos > 0

    @property
    def m(self) -> int:
        return self.s

    @property
    def win_cols(self) -> int:
        return self.window if self.decode else min(self.s, self.window)

    @property
    def topk(self) -> int:
        return self.win_cols + self.topk_comp

    @property
    def win_rows(self) -> int:
        """Rows of kv in front of the compressed rows: the ring (decode) or the chunk (prefill)."""
        return self.window if self.decode else self.s

    @property
    def n(self) -> int:
        return self.win_rows + self.n_comp

    @property
    def seed(self) -> int:
        return 1000 + self.index


WORKLOADS = {
    0: Workload(0, "fixture", b=1, h=4, d=64, window=8, start_pos=0, s=12, n_comp=0, topk_comp=0,
                neg_frac=0.0, comp_mode="none", rope_dim=16),
    1: Workload(1, "decode_window", b=64, h=64, d=512, window=128, start_pos=10000, s=1, n_comp=0,
                topk_comp=0, neg_frac=0.0, comp_mode="none", rope_dim=64),
    2: Workload(2, "prefill", b=1, h=64, d=512, window=128, start_pos=0, s=4096, n_comp=1024,
                topk_comp=512, neg_frac=0.0, comp_mode="prefill_causal", rope_dim=64),
    3: Workload(3, "decode_comp", b=32, h=64, d=512, window=128, start_pos=16384, s=1, n_comp=4096,
                topk_comp=512, neg_frac=0.05, comp_mode="uniform", rope_dim=64),
    4: Workload(4, "decode_large", b=256, h=128, d=512, window=128, start_pos=131072, s=1, n_comp=32768,
                topk_comp=2048, neg_frac=0.02, comp_mode="uniform", rope_dim=64),
}

# decode steps the fixture runs after its 12-token prefill, through the same ring
FIXTURE_DECODE_STEPS = (12, 13)


@dataclass(frozen=True)
class IndexerWorkload:
    """The Indexer step that produces a workload's compressed indices ("DeepSeek V4.1",
    attention/query-latent, Indexer.forward): H index heads of width D per query, one shared key
    per compressed position, compress ratio 4, index_topk kept, shifted past the window rows."""
    index: int
    name: str
    b: int
    s: int
    H: int
    D: int
    start_pos: int
    ratio: int
    topk: int
    offset: int

    @property
    def Tv(self) -> int:
        return (self.start_pos + self.s) // self.ratio

    @property
    def seed(self) -> int:
        return 2000 + self.index


# The pages name the Indexer's head count and width (index_n_heads, index_head_dim) without
# values; these workloads take 64 heads of 128.  The compressed positions, top-k and window offset
# are those of the attention workload with the same number.
INDEXER_WORKLOADS = {
    2: IndexerWorkload(2, "indexer_prefill", b=1, s=4096, H=64, D=128, start_pos=0, ratio=4, topk=512, offset=4096),
    3: IndexerWorkload(3, "indexer_decode_comp", b=32, s=1, H=64, D=128, start_pos=16384, ratio=4, topk=512,
                       offset=128),
    4: IndexerWorkload(4, "indexer_decode_large", b=256, s=1, H=64, D=128, start_pos=131072, ratio=4, topk=2048,
                       offset=128),
}


def indexer_inputs(w: IndexerWorkload, device="cpu", seed: int | None = None):
    """q [b][s][H][D] and k [b][Tv][D] ~ N(0,1) bf16; w [b][s][H] f32 ~ N(0,1) * D^-0.5 * H^-0.5
    (weights_proj's output times the softmax scale and n_heads^-0.5, rounded to bf16 first)."""
    g = _gen(device, w.seed if seed is None else seed)
    q = torch.empty((w.b, w.s, w.H, w.D), dtype=torch.bfloat16, device=device)
    _fill_rows_bf16(q, g)
    k = torch.empty((w.b, w.Tv, w.D), dtype=torch.bfloat16, device=device)
    _fill_rows_bf16(k, g)
    wt = torch.randn((w.b, w.s, w.H), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16).float()
    wt = wt * (w.D ** -0.5 * w.H ** -0.5)
    return q, k, wt


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def _fill_rows_bf16(t: torch.Tensor, g: torch.Generator, chunk_rows: int = 1 << 20) -> None:
    """Fill a [..., d] bf16 tensor with N(0,1) in bounded chunks (keeps the f32 staging small)."""
    flat = t.view(-1, t.shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, t.shape[-1]), generator=g, device=t.device,
                                  dtype=torch.float32).to(torch.bfloat16)


def compressed_indices(w: Workload, g: torch.Generator, device) -> torch.Tensor:
    """int32 [b][m][topk_comp]: compressed indices shifted by ``w.win_rows``; -1 for nothing."""
    b, m, K, C = w.b, w.m, w.topk_comp, w.n_comp
    if K == 0:
        return torch.empty((b, m, 0), dtype=torch.int32, device=device)
    if w.comp_mode == "uniform":
        # K distinct draws per query, uniform without replacement, sorted ascending
        keys = torch.rand((b * m, C), generator=g, device=device)
        sel = keys.topk(K, dim=-1).indices.sort(dim=-1).values
        out = (sel + w.win_rows).to(torch.int32)
        nneg = int(round(w.neg_frac * K))
        if nneg:
            pos = torch.rand((b * m, K), generator=g, device=device).topk(nneg, dim=-1).indices
            out.scatter_(1, pos, -1)
        return out.view(b, m, K)
    if w.comp_mode == "prefill_causal":
        # query q may draw from the first floor(q/4) compressed rows; tail padded with -1
        assert w.b == 1
        qpos = torch.arange(w.start_pos, w.start_pos + m, device=device)
        avail = (qpos // 4).clamp(max=C)
        keys = torch.rand((m, C), generator=g, device=device)
        keys = torch.where(torch.arange(C, device=device)[None, :] < avail[:, None], keys, -1.0)
        vals, sel = keys.topk(K, dim=-1)
        sel = torch.where(vals >= 0, sel, C + 1)       # unreachable draws sort to the tail
        sel = sel.sort(dim=-1).values
        out = torch.where(sel <= C, sel + w.win_rows, -1).to(torch.int32)
        return out.view(1, m, K)
    raise ValueError(w.comp_mode)


@dataclass
class StepInputs:
    """One step's inputs (all tensors on one device; bf16 tensors hold raw, unquantised rows).

    kv      [b][n][d]  rows [0, win_rows): the chunk (prefill, raw) or the ring (decode, raw history
                       rounded by whichever side consumes it); rows [win_rows, n): compressed, plain.
    hist    decode only: [b][window][d] raw rows of tokens start_pos-window .. start_pos-1 that the
            ring held before the step (the ring is seeded from them: row i goes to slot
            (start_pos - window + i) % window).
    new_kv  decode only: [b][1][d] raw row of the step's own token.
    q       [b][m][h][d]; sink [h] f32; cidx [b][m][topk_comp] int32 (already shifted).
    """
    w: Workload
    q: torch.Tensor
    kv: torch.Tensor
    hist: torch.Tensor | None
    new_kv: torch.Tensor | None
    sink: torch.Tensor
    cidx: torch.Tensor


def make_step_inputs(w: Workload, device="cpu", seed: int | None = None) -> StepInputs:
    seed = w.seed if seed is None else seed
    g = _gen(device, seed)
    q = torch.empty((w.b, w.m, w.h, w.d), dtype=torch.bfloat16, device=device)
    _fill_rows_bf16(q, g)
    sink = torch.randn((w.h,), generator=g, device=device, dtype=torch.float32)
    kv = torch.empty((w.b, w.n, w.d), dtype=torch.bfloat16, device=device)
    _fill_rows_bf16(kv, g)
    hist = new_kv = None
    if w.decode:
        hist = kv[:, : w.window].clone()
        new_kv = torch.empty((w.b, 1, w.d), dtype=torch.bfloat16, device=device)
        _fill_rows_bf16(new_kv, g)
    cidx = compressed_indices(w, g, device)
    return StepInputs(w, q, kv, hist, new_kv, sink, cidx)


def fixture_inputs(device="cpu", seed: int | None = None) -> dict:
    """The ratio-0 fixture: a 12-token prefill chunk and the rows/queries of decode steps 12, 13."""
    w = WORKLOADS[0]
    g = _gen(device, w.seed if seed is None else seed)
    out = {
        "w": w,
        "prefill_kv": randn_bf16((w.b, w.s, w.d), g, device),
        "prefill_q": randn_bf16((w.b, w.s, w.h, w.d), g, device),
        "sink": torch.randn((w.h,), generator=g, device=device, dtype=torch.float32),
        "decode": [],
    }
    for p in FIXTURE_DECODE_STEPS:
        out["decode"].append({
            "start_pos": p,
            "new_kv": randn_bf16((w.b, 1, w.d), g, device),
            "q": randn_bf16((w.b, 1, w.h, w.d), g, device),
        })
    return out


def bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a tensor as a numpy uint16 array (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
