"""Parity at full sequence length, on the paths the timed configurations take.

The pages' pretraining step runs rows of 2048 tokens (walkthrough, section
"预训练": 32 rows x 2048 tokens per GPU forward/backward); the long-context
configuration uses rows of 8192.  Here the CUDA path is compared with the
fp64 oracle on whole 2048- and 8192-token rows: the full step at the depth-20
widths, and the attention kernels with more than eight sequences (the
backward launches its key tiles in groups of eight sequences) and with many
query tiles per key tile.  Tolerances are those of tests/helpers.py (bf16:
cosine >= 0.999 and ||delta|| / ||ref|| <= 3e-2 per gradient tensor; the
attention outputs of a single kernel are held to <= 2e-2)."""
import numpy as np
import pytest
import torch

import nc_synth
import oracle
from pretraining_step_pretrain_b300 import build, nc
from tests.helpers import assert_parity, grad_metrics, inputs, run_cuda_step, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    nc.lib()


def test_d20_full_sequence_step_matches_oracle():
    """nc_step at the depth-20 shape (20 blocks, d 1280, 10 heads x 128,
    f 5120, V 65536) on one whole row of 2048 tokens: the loss and every
    weight gradient against the oracle."""
    shape = nc_synth.D20.shape
    ids, tg, w = inputs(shape, 1, nc_synth.D20.seq, "bf16")
    loss, grads, status = run_cuda_step(shape, "bf16", ids, tg, w)
    torch.cuda.empty_cache()
    assert status == 0
    ref_loss, ref_grads = run_oracle(shape, ids, tg, w)
    assert_parity("bf16", ref_loss, ref_grads, loss, grads)


def _bf16_normal(rng, shape):
    a = rng.standard_normal(shape, dtype=np.float32)
    return torch.from_numpy(a).to(torch.bfloat16)


def _attention_gpu(q, k, v, do):
    """Forward and backward of the bf16 attention kernels through the C ABI;
    the gradients land inside one (B*T, (H+2)h) buffer as in the step."""
    B, T, H, h = q.shape
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty(B, T, H, device="cuda")
    nc.attention_fwd(nc.NC_BF16, B, T, H, h, qd, kd, vd, o, lse)
    W = (H + 2) * h
    dqkv = torch.full((B * T, W), 7.0, dtype=torch.bfloat16, device="cuda")
    nc.attention_bwd(nc.NC_BF16, B, T, H, h, qd, kd, vd, o, lse, dod, dqkv[:, :H * h], W,
                     dqkv[:, H * h:H * h + h], W, dqkv[:, H * h + h:], W)
    torch.cuda.synchronize()
    dqkv = dqkv.view(B, T, W)
    return {"o": o.cpu(), "lse": lse.cpu(), "dq": dqkv[..., :H * h].reshape(B, T, H, h).cpu(),
            "dk": dqkv[..., H * h:H * h + h].cpu(), "dv": dqkv[..., H * h + h:].cpu()}


def _lse_oracle(q, k):
    """Natural-log sum of exp of the oracle's scaled causal scores, (T, H) for
    one sequence, from the oracle's own score function."""
    from oracle import nanochat_step as ns
    s = ns._causal_scores(q, k)[0]                                   # (H, T, T)
    m = s.max(-1, keepdims=True)
    return (m + np.log(np.exp(s - m).sum(-1, keepdims=True)))[..., 0].T


@pytest.mark.parametrize("B,T,H,check", [
    (9, 2048, 10, (0, 7, 8)),      # the bench's rows and heads; nine sequences cross a group of eight
    (2, 8192, 2, (1,)),            # 8192-token rows: 64 key tiles, 128 query tiles per sequence
], ids=["T2048_H10_B9", "T8192_H2_B2"])
def test_attention_full_sequences_match_oracle(B, T, H, check):
    h = 128
    rng = np.random.default_rng(T + H)
    q, do = _bf16_normal(rng, (B, T, H, h)), _bf16_normal(rng, (B, T, H, h))
    k, v = _bf16_normal(rng, (B, T, h)), _bf16_normal(rng, (B, T, h))
    got = _attention_gpu(q, k, v, do)
    for b in check:
        qb, kb, vb, dob = (t[b:b + 1].double().numpy() for t in (q, k, v, do))
        ref = {"o": oracle.attention(qb, kb, vb)}
        ref["dq"], ref["dk"], ref["dv"] = oracle.attention_bwd(dob, qb, kb, vb)
        for name, r in ref.items():
            cos, rel = grad_metrics(r, got[name][b:b + 1].double().numpy())
            assert cos > 0.999 and rel < 2e-2, (b, name, cos, rel)
        np.testing.assert_allclose(got["lse"][b].double().numpy(), _lse_oracle(qb, kb), atol=2e-2)


def test_attention_long_context_heads_match_oracle():
    """The long-context configuration's attention (4 rows x 8192 tokens, 10
    heads) on the GPU; the oracle checks two heads of the last row in full.
    Heads are independent given the shared K/V head, so one head's output,
    log-sum-exp and query gradient are the oracle's with that head alone."""
    B, T, H, h = 4, 8192, 10, 128
    rng = np.random.default_rng(8192)
    q, do = _bf16_normal(rng, (B, T, H, h)), _bf16_normal(rng, (B, T, H, h))
    k, v = _bf16_normal(rng, (B, T, h)), _bf16_normal(rng, (B, T, h))
    got = _attention_gpu(q, k, v, do)
    b = B - 1
    kb, vb = k[b:b + 1].double().numpy(), v[b:b + 1].double().numpy()
    for hd in (0, H - 1):
        qh = q[b:b + 1, :, hd:hd + 1].double().numpy()
        doh = do[b:b + 1, :, hd:hd + 1].double().numpy()
        o_ref = oracle.attention(qh, kb, vb)
        dq_ref, _, _ = oracle.attention_bwd(doh, qh, kb, vb)
        for name, r, g in (("o", o_ref, got["o"][b:b + 1, :, hd:hd + 1]),
                           ("dq", dq_ref, got["dq"][b:b + 1, :, hd:hd + 1])):
            cos, rel = grad_metrics(r, g.double().numpy())
            assert cos > 0.999 and rel < 2e-2, (hd, name, cos, rel)
        np.testing.assert_allclose(got["lse"][b, :, hd].double().numpy(),
                                   _lse_oracle(qh, kb)[:, 0], atol=2e-2)


def test_fp32_tiny_step_elementwise():
    """The fp32 debug mode element by element: every loss and gradient entry
    within 1e-5 of its own magnitude, with an absolute floor of 1e-6 of the
    tensor's largest entry (entries that cancel to near zero carry the
    rounding of the large terms they cancel)."""
    shape = nc_synth.TINY.shape
    ids, tg, w = inputs(shape, 2, 64, "f32", ids_dist="uniform")
    ref_loss, ref_grads = run_oracle(shape, ids, tg, w)
    loss, grads, status = run_cuda_step(shape, "f32", ids, tg, w)
    assert status == 0
    assert abs(loss - ref_loss) <= 1e-5 * abs(ref_loss)
    for k, r in ref_grads.items():
        g = grads[k]
        bound = 1e-5 * np.abs(r) + 1e-6 * np.abs(r).max()
        worst = float(np.max(np.abs(g - r) - bound))
        assert worst <= 0.0, (k, worst, float(np.abs(g - r).max()), float(np.abs(r).max()))


def test_attention_backward_exact_zeros_and_repeatable_at_bench_shape():
    """At the bench's attention shape (32 rows x 2048 tokens, 10 heads): with
    dO = 0 every gradient is exactly zero (dP = 0 and delta = 0, so dS = 0,
    and dV = P^T dO = 0) on each of many repeats, and a repeated backward on
    random dO is bit-identical.  A product that read a shared-memory tile
    before its load landed, or a tensor-memory buffer before it was written,
    shows up here even when it stays inside the tolerance of a parity test."""
    B, T, H, h = 32, 2048, 10, 128
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn(B, T, H, h, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, T, h, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, T, h, generator=g, device="cuda").to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(B, T, H, device="cuda")
    ws = nc.attention_fwd(nc.NC_BF16, B, T, H, h, q, k, v, o, lse)
    W = (H + 2) * h

    def bwd(do):
        dqkv = torch.full((B * T, W), 5.0, dtype=torch.bfloat16, device="cuda")
        nc.attention_bwd(nc.NC_BF16, B, T, H, h, q, k, v, o, lse, do, dqkv[:, :H * h], W,
                         dqkv[:, H * h:H * h + h], W, dqkv[:, H * h + h:], W, ws=ws)
        return dqkv

    zero = torch.zeros_like(q)
    for it in range(12):
        got = bwd(zero)
        torch.cuda.synchronize()
        assert not bool(got.any()), (it, int((got.float().abs().amax(1) > 0).sum()))
    do = torch.randn(B, T, H, h, generator=g, device="cuda").to(torch.bfloat16)
    ref = bwd(do)
    for it in range(4):
        assert torch.equal(bwd(do), ref), it
