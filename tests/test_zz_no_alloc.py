"""nc_attention_bwd_noalloc: the attention backward for callers that cannot
give the library device memory where they run it -- e.g. an operator inside
another framework's runtime that owns all device memory and hands this op no
scratch, or a hot loop that must not call cudaMalloc.  Its one scratch
buffer is a fixed device array inside the library, and so is its device
error word (read with nc_attention_bwd_noalloc_status).

The tests check, through the C ABI, that two calls in a row (different
inputs each time, so the second call runs on the first call's leftover
scratch) give bit for bit the results of nc_attention_bwd with a caller
workspace -- the same kernels on the same inputs, so any read of stale
scratch would show -- with a clean status after each call; that a bounded
wait which runs out is reported through that status word; and that an
oversized shape is refused before anything is launched.  The file is
collected last and needs no state from other tests.
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
    return dqkv


@pytest.mark.parametrize("dtype,B,T,H,h", [("bf16", 2, 300, 10, 128), ("f32", 3, 77, 2, 64)])
def test_noalloc_matches_workspace_version_two_calls(dtype, B, T, H, h):
    assert nc.attention_bwd_noalloc_status() == 0
    for seed in (1, 2):                       # two calls in a row on the shared scratch
        args = _case(dtype, B, T, H, h, seed)
        ref = _grads(nc.attention_bwd, *args[:1], B, T, H, h, *args[1:])
        got = _grads(nc.attention_bwd_noalloc, *args[:1], B, T, H, h, *args[1:])
        assert nc.attention_bwd_noalloc_status() == 0
        assert torch.equal(got, ref), seed
        assert np.isfinite(got.float().cpu().numpy()).all()


def test_noalloc_status_reports_a_wait_that_ran_out():
    """A CTA waits on an mbarrier nothing completes for 2 ms and records the
    timeout in the no-alloc calls' error word; the status call reports it
    once and clears it, and the next backward runs normally."""
    assert nc.attention_bwd_noalloc_status() == 0
    nc.selftest_wait_timeout(2000, None)
    assert nc.attention_bwd_noalloc_status() == 5          # NC_ERR_TIMEOUT
    assert nc.attention_bwd_noalloc_status() == 0          # read once, then clear
    args = _case("bf16", 1, 64, 2, 128, 3)
    ref = _grads(nc.attention_bwd, *args[:1], 1, 64, 2, 128, *args[1:])
    got = _grads(nc.attention_bwd_noalloc, *args[:1], 1, 64, 2, 128, *args[1:])
    assert nc.attention_bwd_noalloc_status() == 0
    assert torch.equal(got, ref)


def test_noalloc_refuses_more_rows_than_its_scratch():
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(16, device="cuda")
    B, T, H, h = 64, 8192, 10, 128            # 5.2M query rows > 2^21
    with pytest.raises(nc.NcError) as e:
        nc.attention_bwd_noalloc(nc.NC_BF16, B, T, H, h, q, q, q, q, lse, q, q, H * h, q, h, q, h)
    assert e.value.status == 2 and "scratch" in str(e.value)
