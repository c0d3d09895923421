"""Parity of the optimizer step (nc_optimizer_step: Muon for the block
matrices, AdamW for the embedding and the LM head) with the fp64 oracle in
oracle/optimizer.py, and of the batched GEMM it is built on with a plain
PyTorch fp32 contraction."""
import math

import numpy as np
import pytest
import torch

import nc_synth
from oracle import optimizer as opt
from pretraining_step_pretrain_b300 import build, nc
from tests.helpers import grad_metrics

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    nc.lib()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("layout", ["NT", "NN"])
@pytest.mark.parametrize("epi", ["store", "axpby"])
def test_batched_gemm_matches_torch(dtype, layout, epi):
    """Six independent products in one launch (the Newton-Schulz shapes:
    square Gram matrices and wide iterates), ragged M against the tiles."""
    batch, M, N, K = 6, 320, 576 if layout == "NN" else 320, 320 if layout == "NN" else 576
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device="cuda").manual_seed(7)
    A = torch.randn(batch, M, K, generator=g, device="cuda").to(dt)
    if layout == "NT":
        B = (torch.randn(batch, N, K, generator=g, device="cuda") / K ** 0.5).to(dt)
        ref = A.float() @ B.float().transpose(1, 2)
        lay, ldb = nc.GEMM_NT, K
    else:
        B = (torch.randn(batch, K, N, generator=g, device="cuda") / K ** 0.5).to(dt)
        ref = A.float() @ B.float()
        lay, ldb = nc.GEMM_NN, N
    aux = torch.randn(batch, M, N, generator=g, device="cuda").to(dt)
    C = torch.zeros(batch, M, N, dtype=dt, device="cuda")
    if epi == "axpby":
        alpha, beta = -0.75, 1.5
        expect = alpha * aux.float() + beta * ref
        nc.gemm_batched(nc.NC_BF16 if dtype == "bf16" else nc.NC_F32, lay, nc.EPI_AXPBY, batch,
                        M, N, K, A, K, M * K, B, ldb, B[0].numel(), C, N, M * N, aux=aux,
                        alpha=alpha, beta=beta)
    else:
        expect = ref
        nc.gemm_batched(nc.NC_BF16 if dtype == "bf16" else nc.NC_F32, lay, nc.EPI_STORE, batch,
                        M, N, K, A, K, M * K, B, ldb, B[0].numel(), C, N, M * N)
    torch.cuda.synchronize()
    for z in range(batch):
        err = float((C[z].float() - expect[z]).norm() / expect[z].norm())
        assert err < (8e-3 if dtype == "bf16" else 2e-5), (z, err)


def _setup(shape, dtype, seed):
    """Random master weights (fp32, N(0, 1/fan_in)), random gradients."""
    rng = np.random.default_rng(seed)
    w = nc_synth.make_weights(shape, seed=seed, bf16=False)
    grads = {k: (rng.standard_normal(v.shape) * 0.01).astype(np.float32) for k, v in w.items()}
    st = nc.Step(shape, dtype, 1, 8, w)
    for k, gv in grads.items():
        st.g[k].copy_(torch.from_numpy(gv))
    return st, w, grads


HP = dict(lr_muon=0.02, momentum=0.95, lr_embed=0.3, lr_lm=0.004, betas=(0.8, 0.95), eps=1e-10,
          weight_decay=0.01)


def _run(shape, dtype, steps, seed=3):
    st, w, grads = _setup(shape, dtype, seed)
    o = nc.Optimizer(st, lr_muon=HP["lr_muon"], momentum=HP["momentum"], lr_embed=HP["lr_embed"],
                     lr_lm=HP["lr_lm"], betas=HP["betas"], eps=HP["eps"],
                     weight_decay=HP["weight_decay"], masters=w)
    P = {k: v.astype(np.float64) for k, v in w.items()}
    S = {}
    for t in range(1, steps + 1):
        lrm = 1.0 if t == 1 else 0.5
        o.step(t, lrm)
        P, S = opt.optimizer_step(P, {k: v.astype(np.float64) for k, v in grads.items()}, S, t,
                                  shape.d_model, lrm, HP["lr_muon"], HP["momentum"],
                                  HP["lr_embed"], HP["lr_lm"], HP["betas"], HP["eps"],
                                  HP["weight_decay"])
    torch.cuda.synchronize()
    got = {k: v.double().cpu().numpy() for k, v in o.p.items()}
    return st, o, w, got, P


def test_optimizer_f32_matches_oracle_two_steps():
    """fp32 debug mode: two steps (state carried over, lrm 1 then 0.5) agree
    with the fp64 oracle to 1e-5 relative on every parameter's update."""
    shape = nc_synth.TINY.shape
    st, o, w, got, ref = _run(shape, "f32", 2)
    for k in ref:
        upd_ref = ref[k] - w[k].astype(np.float64)
        upd_got = got[k] - w[k].astype(np.float64)
        rel = np.linalg.norm(upd_got - upd_ref) / np.linalg.norm(upd_ref)
        assert rel < 1e-5, (k, rel)
    # the compute copies hold the updated masters
    for k in got:
        assert np.array_equal(st.w[k].double().cpu().numpy(), got[k]), k


def test_optimizer_bf16_matches_oracle():
    """bf16 mode: the Newton-Schulz iterates are bf16 (tensor cores); every
    update agrees with the fp64 oracle to cosine >= 0.999 and relative error
    <= 3e-2, AdamW parameters (fp32 element-wise) to 1e-5."""
    shape = nc_synth.SMALL.shape
    st, o, w, got, ref = _run(shape, "bf16", 2)
    for k in ref:
        upd_ref = ref[k] - w[k].astype(np.float64)
        upd_got = got[k] - w[k].astype(np.float64)
        if k in ("wte", "w_lm"):
            rel = np.linalg.norm(upd_got - upd_ref) / np.linalg.norm(upd_ref)
            assert rel < 1e-5, (k, rel)
        else:
            cos, rel = grad_metrics(upd_ref, upd_got)
            assert cos > 0.999 and rel < 3e-2, (k, cos, rel)
    bf = {k: v.to(torch.bfloat16).float().double().cpu().numpy() for k, v in o.p.items()}
    for k in bf:
        assert np.array_equal(st.w[k].double().cpu().numpy(), bf[k]), k


def test_optimizer_is_deterministic():
    shape = nc_synth.SMALL.shape
    a = _run(shape, "bf16", 1, seed=11)[3]
    b = _run(shape, "bf16", 1, seed=11)[3]
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_optimizer_muon_update_is_orthogonal_like():
    """The Muon update of a well-conditioned matrix has every singular value
    of update / (lr sqrt(max(1, r/c))) inside the quintic's band around 1.
    The random gradients of the rectangular matrices (aspect 2 to 4) have
    their smallest singular value well away from 0; a square random matrix
    (w_o) does not, and five steps cannot lift a near-zero one into the band."""
    shape = nc_synth.SMALL.shape
    st, o, w, got, ref = _run(shape, "bf16", 1, seed=5)
    for k in ("w_qkv.0", "w_fc.1", "w_proj.2", "w_fc.3"):
        r, c = w[k].shape
        u = (w[k].astype(np.float64) - got[k]) / (HP["lr_muon"] * math.sqrt(max(1.0, r / c)))
        s = np.linalg.svd(u, compute_uv=False)
        assert s.min() > 0.45 and s.max() < 1.35, (k, s.min(), s.max())
