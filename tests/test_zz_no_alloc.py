"""ds_sparse_attn_static_scratch: sparse_attn without a caller-provided workspace.

Some callers cannot allocate device memory where they run attention (an owning runtime or memory
manager, a plugin handed only its buffers), so this entry point keeps its scratch in a fixed
device array inside the library.  The test calls it through the C ABI on a shape that needs
scratch (tokens split across CTAs), twice in a row.  Both entry points run the same
deterministic kernels on the same inputs, so every output must equal ds_sparse_attn's (with an
allocated workspace) bit for bit, and match the oracle within the attention tolerance.  It lives
in its own file, collected last.
"""
import ctypes

import pytest
import torch

import oracle
from pathcheck import assert_close_bf16, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from sparse_latent_attention_attn_gb300 import dsattn
    L = dsattn._lib
    P = ctypes.c_void_p
    L.ds_sparse_attn_static_scratch.argtypes = [P, P, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_float, P,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    L.ds_sparse_attn_static_scratch.restype = ctypes.c_int
    L.ds_sparse_attn_static_scratch_capacity.argtypes = []
    L.ds_sparse_attn_static_scratch_capacity.restype = ctypes.c_size_t
    return L


def _inputs(b, m, h, d, n, topk, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = torch.randn((b, m, h, d), generator=g, device="cuda").to(torch.bfloat16)
    kv = torch.randn((b, n, d), generator=g, device="cuda").to(torch.bfloat16)
    sink = torch.randn((h,), generator=g, device="cuda")
    idx = torch.rand((b * m, n), generator=g, device="cuda").topk(topk, dim=-1).indices.to(torch.int32)
    idx = idx.view(b, m, topk).contiguous()
    idx[..., -13:] = -1
    return q, kv, sink, idx


def _call_static(lib, q, kv, sink, idx, scale, o):
    b, m, h, d = q.shape
    return lib.ds_sparse_attn_static_scratch(q.data_ptr(), kv.data_ptr(), kv.shape[1], sink.data_ptr(),
                                             idx.data_ptr(), idx.shape[2], scale, o.data_ptr(), b, m, h, d,
                                             torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("b,m,h,d,n,topk", [(4, 1, 64, 512, 900, 700),       # parts merged by a combine kernel
                                            (32, 1, 64, 512, 4224, 640)])   # decode_comp's shape: 4-CTA merges
def test_static_scratch_matches_workspace_path(lib, b, m, h, d, n, topk):
    from sparse_latent_attention_attn_gb300 import dsattn
    scale = d ** -0.5
    need = dsattn.sparse_attn_plan(b, m, h, d, topk)[2]                   # the running kernel's need
    assert need > 0                                                        # the shape really uses scratch
    assert need <= lib.ds_sparse_attn_static_scratch_capacity()
    for call, seed in enumerate((11, 12)):                                 # two calls in a row
        q, kv, sink, idx = _inputs(b, m, h, d, n, topk, seed)
        ref = dsattn.sparse_attn(q, kv, sink, idx, scale)
        o = torch.full_like(q, float("nan"))
        assert _call_static(lib, q, kv, sink, idx, scale, o) == 0
        torch.cuda.synchronize()
        assert torch.equal(o, ref), f"call {call}: differs from ds_sparse_attn with a workspace"
        want = oracle.sparse_attn(bits(q), bits(kv), sink.cpu().numpy(), idx.cpu().numpy(), scale)
        assert_close_bf16(bits(o), want, f"call {call}: o against the oracle")
    assert dsattn.device_status() == 0


def test_static_scratch_refuses_shapes_beyond_capacity(lib):
    """128 heads run the cluster kernel; with more tokens than clusters every range boundary cuts
    a token, and two f32 partial slots of 128 heads x 512 per cluster exceed the 32 MiB array."""
    from sparse_latent_attention_attn_gb300 import dsattn
    b, m, h, d, n, topk = 128, 1, 128, 512, 300, 256
    need = dsattn.sparse_attn_workspace_bytes(b, m, h, d, topk)
    if need <= lib.ds_sparse_attn_static_scratch_capacity():
        pytest.skip("on this device the shape fits the static scratch")
    q, kv, sink, idx = _inputs(b, m, h, d, n, topk, 13)
    o = torch.zeros_like(q)
    assert _call_static(lib, q, kv, sink, idx, d ** -0.5, o) == dsattn.DS_EWORKSPACE
    torch.cuda.synchronize()
    assert (o.float() == 0).all()                                          # nothing was launched
