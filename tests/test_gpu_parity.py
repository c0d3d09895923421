"""Parity of the whole CUDA step (nc_step and the per-call C ABI) with the
fp64 oracle on the same seeded inputs.  Tolerances in tests/helpers.py."""
import math

import numpy as np
import pytest
import torch

import nc_synth
import oracle
from pretraining_step_pretrain_b300 import build, nc
from tests.helpers import assert_parity, inputs, run_cuda_step, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    nc.lib()


RAGGED = nc_synth.ModelShape(depth=2, d_model=256, n_head=2, head_dim=128, d_mlp=512, vocab=4160)
# Many heads: the QK-norm + RoPE backward's per-warp staging slots no longer
# fit in shared memory (fp32 from 16 heads, bf16 from 33), so these take its
# register path.
WIDE_F32 = nc_synth.ModelShape(depth=1, d_model=128, n_head=20, head_dim=128, d_mlp=128, vocab=256)
WIDE_BF16 = nc_synth.ModelShape(depth=1, d_model=128, n_head=36, head_dim=128, d_mlp=128, vocab=256)


@pytest.mark.parametrize("case", [
    # name, shape, B, T, dtype, ids, zero
    ("tiny_f32", nc_synth.TINY.shape, 2, 64, "f32", "uniform", ()),
    ("tiny_f32_zero_heads", nc_synth.TINY.shape, 2, 64, "f32", "uniform", ("w_lm", "w_o", "w_proj")),
    ("tiny_f32_zero_out_proj", nc_synth.TINY.shape, 2, 64, "f32", "uniform", ("w_o", "w_proj")),
    ("tiny_f32_ragged", nc_synth.TINY.shape, 3, 37, "f32", "zipf", ()),
    ("small_bf16", nc_synth.SMALL.shape, 8, 256, "bf16", "zipf", ()),
    ("ragged_bf16", RAGGED, 3, 100, "bf16", "zipf", ()),
    ("tiny_len1_bf16", RAGGED, 2, 1, "bf16", "zipf", ()),
    ("wide_heads_f32", WIDE_F32, 2, 24, "f32", "uniform", ()),
    ("wide_heads_bf16", WIDE_BF16, 2, 40, "bf16", "zipf", ()),
], ids=lambda c: c[0])
def test_step_matches_oracle(case):
    name, shape, B, T, dtype, dist, zero = case
    ids, tg, w = inputs(shape, B, T, dtype, ids_dist=dist, zero=zero)
    ref_loss, ref_grads = run_oracle(shape, ids, tg, w)
    loss, grads, status = run_cuda_step(shape, dtype, ids, tg, w)
    assert status == 0
    assert_parity(dtype, ref_loss, ref_grads, loss, grads)
    if "zero_heads" in name:
        assert loss == pytest.approx(math.log(shape.vocab), rel=1e-6)
        for k, g in grads.items():
            if k != "w_lm":
                assert np.all(g == 0.0), k


def test_accumulate_adds_into_gradients():
    shape = nc_synth.SMALL.shape
    ids, tg, w = inputs(shape, 4, 128, "bf16")
    ref_loss, ref_grads = run_oracle(shape, ids, tg, w)
    loss, grads, status = run_cuda_step(shape, "bf16", ids, tg, w, accumulate_runs=2)
    assert status == 0
    assert_parity("bf16", ref_loss, {k: 2 * v for k, v in ref_grads.items()}, loss, grads)


def test_ignored_targets():
    shape = nc_synth.SMALL.shape
    ids, tg, w = inputs(shape, 2, 64, "bf16")
    tg[0, :10] = -1
    tg[1, 5] = -1
    ref_loss, ref_grads = run_oracle(shape, ids, tg, w)
    loss, grads, status = run_cuda_step(shape, "bf16", ids, tg, w)
    assert status == 0
    assert_parity("bf16", ref_loss, ref_grads, loss, grads)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_per_call_abi_composes_to_nc_step(dtype):
    """nc_embed_norm -> nc_block_fwd* -> nc_lmhead_softcap_ce_fwd_bwd ->
    nc_block_bwd* -> nc_embed_norm_bwd gives nc_step's results bit for bit."""
    shape = nc_synth.TINY.shape if dtype == "f32" else nc_synth.SMALL.shape
    B, T = (2, 64) if dtype == "f32" else (4, 128)
    ids, tg, w = inputs(shape, B, T, dtype)
    st = nc.Step(shape, dtype, B, T, w)
    ids_d, tg_d = torch.from_numpy(ids).cuda(), torch.from_numpy(tg).cuda()
    st.run(ids_d, tg_d)
    ref = {k: v.clone() for k, v in st.g.items()}
    ref_loss = st.loss.clone()
    M, d = B * T, shape.d_model
    x = torch.zeros(M, d, device="cuda")
    dx = torch.zeros(M, d, device="cuda")
    g = {k: torch.full_like(v, 3.0) for k, v in st.g.items()}
    loss = torch.zeros(1, device="cuda")
    cfg, ws = st.cfg, st.ws
    nc.embed_norm(cfg, B, T, ids_d, st.w["wte"], x, ws)
    for l in range(shape.depth):
        nc.block_fwd(cfg, l, B, T, st.layers[l], x, ws)
    nc.lmhead_softcap_ce_fwd_bwd(cfg, B, T, x, st.w["w_lm"], tg_d, loss, dx, g["w_lm"], 0, ws)
    for l in reversed(range(shape.depth)):
        gl = nc.NcLayerG(g[f"w_qkv.{l}"].data_ptr(), g[f"w_o.{l}"].data_ptr(),
                         g[f"w_fc.{l}"].data_ptr(), g[f"w_proj.{l}"].data_ptr())
        nc.block_bwd(cfg, l, B, T, st.layers[l], dx, gl, 0, ws)
    nc.embed_norm_bwd(cfg, B, T, ids_d, st.w["wte"], dx, g["wte"], 0, ws)
    torch.cuda.synchronize()
    assert nc.get_device_status(ws) == 0
    assert torch.equal(loss, ref_loss)
    for k in ref:
        assert torch.equal(g[k], ref[k]), k


def test_step_is_deterministic():
    shape = nc_synth.SMALL.shape
    ids, tg, w = inputs(shape, 8, 256, "bf16")
    a = run_cuda_step(shape, "bf16", ids, tg, w)
    b = run_cuda_step(shape, "bf16", ids, tg, w)
    assert a[0] == b[0]
    for k in a[1]:
        assert np.array_equal(a[1][k], b[1][k]), k


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_eval_matches_oracle(dtype):
    """nc_eval (forward only): mean loss and bits per byte against the oracle,
    with a byte table that has zero-length (special) tokens; its loss equals
    the training step's."""
    shape = nc_synth.TINY.shape if dtype == "f32" else nc_synth.SMALL.shape
    B, T = (2, 64) if dtype == "f32" else (4, 128)
    ids, tg, w = inputs(shape, B, T, dtype)
    tg[0, :4] = -1
    rng = np.random.default_rng(9)
    nbytes = rng.integers(1, 9, size=shape.vocab).astype(np.int32)
    nbytes[:3] = 0
    P = {k: v.astype(np.float64) for k, v in w.items()}
    ref_loss, ref_bpb = oracle.evaluate(shape, P, ids, tg, nbytes)
    st = nc.Step(shape, dtype, B, T, w)
    ids_d, tg_d = torch.from_numpy(ids).cuda(), torch.from_numpy(tg).cuda()
    out = st.evaluate(ids_d, tg_d, torch.from_numpy(nbytes).cuda()).cpu().numpy()
    no_bytes = st.evaluate(ids_d, tg_d).cpu().numpy()
    step_loss = float(st.run(ids_d, tg_d).item())
    torch.cuda.synchronize()
    assert st.status() == 0
    tol = 1e-5 if dtype == "f32" else 2e-3
    assert abs(out[0] - ref_loss) <= tol * ref_loss, (out[0], ref_loss)
    assert abs(out[1] - ref_bpb) <= tol * ref_bpb, (out[1], ref_bpb)
    assert np.isnan(no_bytes[1]) and no_bytes[0] == out[0]
    assert out[0] == pytest.approx(step_loss, rel=1e-6)
