"""nc_attention_bwd_noalloc: the attention backward for callers that cannot
give the library device memory where they run it -- e.g. an operator inside
another framework's runtime that owns all device memory and hands this op no
scratch, or a hot loop that must not call cudaMalloc.  Its one scratch
buffer is a fixed device array inside the library.

The test checks, through the C ABI, that two calls in a row (different
inputs each time, so the second call runs on the first call's leftover
scratch) give the same results as nc_attention_bwd with a caller workspace,
and that an oversized shape is refused before anything is launched.  It
lives in its own file, collected last, and needs no state from other tests.
"""
import numpy as np
import pytest
import torch

from pretraining_step_pretrain_b300 import build, nc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    nc.lib()


def _case(dtype, B, T, H, h, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    r = lambda *s: torch.randn(*s, generator=g, device="cuda").to(dt)  # noqa: E731
    q, k, v, do = r(B, T, H, h), r(B, T, h), r(B, T, h), r(B, T, H, h)
    code = nc.NC_BF16 if dtype == "bf16" else nc.NC_F32
    o = torch.empty_like(q)
    lse = torch.empty(B, T, H, device="cuda")
    nc.attention_fwd(code, B, T, H, h, q, k, v, o, lse)
    return code, q, k, v, o, lse, do


def _grads(fn, code, B, T, H, h, q, k, v, o, lse, do):
    W = (H + 2) * h
    dqkv = torch.full((B * T, W), 3.0, dtype=q.dtype, device="cuda")
    fn(code, B, T, H, h, q, k, v, o, lse, do, dqkv[:, :H * h], W, dqkv[:, H * h:H * h + h], W,
       dqkv[:, H * h + h:], W)
    torch.cuda.synchronize()
    return dqkv.float()


@pytest.mark.parametrize("dtype,B,T,H,h", [("bf16", 2, 300, 10, 128), ("f32", 3, 77, 2, 64)])
def test_noalloc_matches_workspace_version_two_calls(dtype, B, T, H, h):
    for seed in (1, 2):                       # two calls in a row on the shared scratch
        args = _case(dtype, B, T, H, h, seed)
        ref = _grads(nc.attention_bwd, *args[:1], B, T, H, h, *args[1:])
        got = _grads(nc.attention_bwd_noalloc, *args[:1], B, T, H, h, *args[1:])
        rel = float((got - ref).norm() / ref.norm())
        assert rel <= (1e-5 if dtype == "f32" else 1e-3), (seed, rel)
        assert np.isfinite(got.cpu().numpy()).all()


def test_noalloc_refuses_more_rows_than_its_scratch():
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(16, device="cuda")
    B, T, H, h = 64, 8192, 10, 128            # 5.2M query rows > 2^21
    with pytest.raises(nc.NcError) as e:
        nc.attention_bwd_noalloc(nc.NC_BF16, B, T, H, h, q, q, q, q, lse, q, q, H * h, q, h, q, h)
    assert e.value.status == 2 and "scratch" in str(e.value)
