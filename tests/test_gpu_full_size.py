"""Checks at the depth-20 shape in the launch configuration the bench times
(B = 32 rows x T = 2048 tokens, V = 65536): outputs the oracle can compute
for sampled sequences, and properties that hold at any size."""
import math

import numpy as np
import pytest
import torch

import nc_synth
import oracle
from pretraining_step_pretrain_b300 import build, nc
from tests.helpers import assert_parity, grad_metrics, inputs, run_cuda_step, run_oracle

pytestmark = pytest.mark.gpu

D20 = nc_synth.D20


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    nc.lib()


def test_d20_widths_short_sequence_match_oracle():
    """Full d20 widths (d 1280, 10 heads, f 5120, V 65536), one row of 128 tokens."""
    shape = D20.shape
    ids, tg, w = inputs(shape, 1, 128, "bf16")
    ref_loss, ref_grads = run_oracle(shape, ids, tg, w)
    loss, grads, status = run_cuda_step(shape, "bf16", ids, tg, w)
    assert status == 0
    assert_parity("bf16", ref_loss, ref_grads, loss, grads)


@pytest.fixture(scope="module")
def d20_full():
    shape = D20.shape
    B, T = D20.batch, D20.seq
    ids, tg, w = inputs(shape, B, T, "bf16")
    return shape, B, T, ids, tg, w


def test_d20_full_size_first_block_sampled_rows(d20_full):
    """nc_embed_norm + nc_block_fwd(0) over all 32 x 2048 tokens; the oracle
    recomputes layer 0 for two sampled sequences."""
    shape, B, T, ids, tg, w = d20_full
    st = nc.Step(shape, "bf16", B, T, w)
    ids_d = torch.from_numpy(ids).cuda()
    x = torch.zeros(B * T, shape.d_model, device="cuda")
    nc.embed_norm(st.cfg, B, T, ids_d, st.w["wte"], x, st.ws)
    nc.block_fwd(st.cfg, 0, B, T, st.layers[0], x, st.ws)
    torch.cuda.synchronize()
    assert nc.get_device_status(st.ws) == 0
    got = x.view(B, T, -1).double().cpu().numpy()
    one = nc_synth.ModelShape(1, shape.d_model, shape.n_head, shape.head_dim, shape.d_mlp,
                              shape.vocab)
    P = {k: w[k].astype(np.float64) for k in ("wte", "w_qkv.0", "w_o.0", "w_fc.0", "w_proj.0",
                                               "w_lm")}
    for b in (0, B - 1):
        cache = oracle.forward(one, P, ids[b:b + 1])
        ref = cache["x_out"][0]
        cos, rel = grad_metrics(ref, got[b])
        assert cos > 0.9999 and rel < 1e-2, (b, cos, rel)
    del st
    torch.cuda.empty_cache()


def test_d20_full_size_zero_heads_closed_form(d20_full):
    """LM head, attention output and MLP output projections at zero: the
    residual stream stays norm(embedding), the loss is ln V exactly, dW_lm has
    the closed form (1/N) sum_t (1/V - [y_t = v]) xf_t with
    xf_t = norm(norm(wte[id_t])), and every other gradient is exactly zero --
    all of which hold at any size."""
    shape, B, T, ids, tg, w = d20_full
    w = dict(w)
    for name in list(w):
        if name.split(".")[0] in ("w_lm", "w_o", "w_proj"):
            w[name] = np.zeros_like(w[name])
    loss, grads, status = run_cuda_step(shape, "bf16", ids, tg, w)
    assert status == 0
    assert abs(loss - math.log(shape.vocab)) / math.log(shape.vocab) < 2e-3
    for k, g in grads.items():
        if k != "w_lm":
            assert np.all(g == 0.0), k
    emb = w["wte"].astype(np.float64)[ids.reshape(-1)]
    xf = oracle.rmsnorm(oracle.rmsnorm(emb, shape.eps)[0], shape.eps)[0]
    y = tg.reshape(-1)
    rows = np.array([0, 1, 2, 17, 1000, 40000, shape.vocab - 1])
    ref = np.stack([(xf.sum(0) / shape.vocab - xf[y == v].sum(0)) / y.size for v in rows])
    cos, rel = grad_metrics(ref, grads["w_lm"][rows])
    assert cos > 0.999 and rel < 3e-2, (cos, rel)


def test_d20_full_size_step_finite_deterministic(d20_full):
    shape, B, T, ids, tg, w = d20_full
    a = run_cuda_step(shape, "bf16", ids, tg, w)
    b = run_cuda_step(shape, "bf16", ids, tg, w)
    assert a[2] == 0 and b[2] == 0
    lnv = math.log(shape.vocab)
    assert lnv - 1.0 < a[0] < lnv + 2.0
    assert a[0] == b[0]
    for k in a[1]:
        assert np.all(np.isfinite(a[1][k])), k
        assert np.array_equal(a[1][k], b[1][k]), k


D30 = nc_synth.D30


def test_d30_widths_short_sequence_match_oracle():
    """The next rung of the depth ladder (depth 30: 1920 channels, 15 heads,
    f 7680, V 65536), one row of 128 tokens, every gradient against the oracle."""
    shape = D30.shape
    ids, tg, w = inputs(shape, 1, 128, "bf16")
    ref_loss, ref_grads = run_oracle(shape, ids, tg, w)
    loss, grads, status = run_cuda_step(shape, "bf16", ids, tg, w)
    assert status == 0
    assert_parity("bf16", ref_loss, ref_grads, loss, grads)


def test_d30_gradient_accumulation_over_micro_batches():
    """Two micro-batches accumulated into the same gradient buffers
    (accumulate = 1 on the second) equal the oracle's sum of both batches'
    gradients at the d30 widths."""
    shape = D30.shape
    ids, tg, w = inputs(shape, 2, 64, "bf16")
    ref_a = run_oracle(shape, ids[:1], tg[:1], w)
    ref_b = run_oracle(shape, ids[1:], tg[1:], w)
    st = nc.Step(shape, "bf16", 1, 64, w)
    st.run(torch.from_numpy(ids[:1].copy()).cuda(), torch.from_numpy(tg[:1].copy()).cuda())
    st.run(torch.from_numpy(ids[1:].copy()).cuda(), torch.from_numpy(tg[1:].copy()).cuda(),
           accumulate=True)
    torch.cuda.synchronize()
    assert st.status() == 0
    for k in ref_a[1]:
        ref = ref_a[1][k] + ref_b[1][k]
        cos, rel = grad_metrics(ref, st.g[k].double().cpu().numpy())
        assert cos > 0.999 and rel < 3e-2, (k, cos, rel)
