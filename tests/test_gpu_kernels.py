"""GPU tests of single kernels through the C ABI: every GEMM layout and
epilogue (tcgen05 bf16 and fp32 SIMT) against a plain PyTorch fp32 matmul,
and the MQA attention forward/backward against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from pretraining_step_pretrain_b300 import build, nc
from tests.helpers import grad_metrics

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    nc.lib()


def _operands(layout, M, N, K, dt, gen):
    """A ~ N(0, 1), B ~ N(0, 1/K) so that outputs are O(1)."""
    def a(*s):
        return torch.randn(*s, generator=gen, device="cuda").to(dt)

    def b(*s):
        return (torch.randn(*s, generator=gen, device="cuda") / np.sqrt(K)).to(dt)
    if layout == nc.GEMM_NT:
        A, B = a(M, K), b(N, K)
        ref = A.float() @ B.float().T
        lda, ldb = K, K
    elif layout == nc.GEMM_NN:
        A, B = a(M, K), b(K, N)
        ref = A.float() @ B.float()
        lda, ldb = K, N
    else:
        A, B = a(K, M), b(K, N)
        ref = A.float().T @ B.float()
        lda, ldb = M, N
    return A, lda, B, ldb, ref


SHAPES = [(300, 320, 200), (128, 256, 64), (1000, 512, 1024), (64, 32, 8)]
EPIS = [nc.EPI_STORE, nc.EPI_STORE_F32, nc.EPI_ADD_F32, nc.EPI_RELU2, nc.EPI_RELU2_BWD]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("layout", [nc.GEMM_NT, nc.GEMM_NN, nc.GEMM_TN], ids=["NT", "NN", "TN"])
@pytest.mark.parametrize("epi", EPIS, ids=["store", "store_f32", "add_f32", "relu2", "relu2_bwd"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_matches_torch(dtype, layout, epi, shape):
    M, N, K = shape
    if layout == nc.GEMM_TN:
        # A is stored (K, M): its row stride M must be a multiple of 8; the
        # reduction length K (tokens) stays ragged.
        M, K = -(-M // 8) * 8, K + 13
    gen = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K + layout * 11 + epi)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    A, lda, B, ldb, ref = _operands(layout, M, N, K, dt, gen)
    code = nc.NC_BF16 if dtype == "bf16" else nc.NC_F32
    aux = None
    if epi in (nc.EPI_STORE_F32, nc.EPI_ADD_F32):
        C = torch.randn(M, N, generator=gen, device="cuda")
        C0 = C.clone()
        acc = 1
        expect = ref + C0
    elif epi == nc.EPI_RELU2_BWD:
        C = torch.zeros(M, N, dtype=dt, device="cuda")
        aux = torch.relu(torch.randn(M, N, generator=gen, device="cuda")).square().to(dt)
        acc = 0
        expect = ref * 2 * aux.float().sqrt()
    else:
        C = torch.zeros(M, N, dtype=dt, device="cuda")
        acc = 0
        expect = torch.relu(ref).square() if epi == nc.EPI_RELU2 else ref
    nc.gemm(code, layout, epi, M, N, K, A, lda, B, ldb, C, N, aux=aux, accumulate=acc)
    torch.cuda.synchronize()
    err = (C.float() - expect).norm() / expect.norm()
    fp32_out = epi in (nc.EPI_STORE_F32, nc.EPI_ADD_F32) or dtype == "f32"
    assert err < (2e-5 if fp32_out and dtype == "f32" else 1e-4 if fp32_out else 8e-3), float(err)


@pytest.mark.parametrize("layout", [nc.GEMM_NT, nc.GEMM_NN, nc.GEMM_TN], ids=["NT", "NN", "TN"])
@pytest.mark.parametrize("epi", [nc.EPI_STORE, nc.EPI_ADD_F32, nc.EPI_RELU2_BWD],
                         ids=["store", "add_f32", "relu2_bwd"])
def test_gemm_many_tiles_per_cta_pair(layout, epi):
    """More output tiles than CTA pairs (33 x 10 tiles of 256 x 256), so every
    pair walks several tiles: both accumulators and every ring stage are
    reused many times; ragged M and N edges."""
    M, N, K = 8296, 2528, 320  # the API needs N % 32 == 0 and 16-byte row strides
    gen = torch.Generator(device="cuda").manual_seed(layout * 5 + epi)
    A, lda, B, ldb, ref = _operands(layout, M, N, K, torch.bfloat16, gen)
    aux = None
    if epi == nc.EPI_ADD_F32:
        C = torch.randn(M, N, generator=gen, device="cuda")
        expect = ref + C
    elif epi == nc.EPI_RELU2_BWD:
        C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
        aux = torch.relu(torch.randn(M, N, generator=gen, device="cuda")).square().to(torch.bfloat16)
        expect = ref * 2 * aux.float().sqrt()
    else:
        C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
        expect = ref
    nc.gemm(nc.NC_BF16, layout, epi, M, N, K, A, lda, B, ldb, C, N, aux=aux)
    torch.cuda.synchronize()
    err = float((C.float() - expect).norm() / expect.norm())
    assert err < (1e-4 if epi == nc.EPI_ADD_F32 else 8e-3), err
    # every tile was written (no tile skipped by the persistent walk)
    assert bool(torch.isfinite(C.float()).all())
    rows = (C.float() - expect).abs().amax(dim=1)
    assert float(rows.max()) < 0.1 * float(expect.abs().max()), float(rows.max())


@pytest.mark.parametrize("K", [8192, 65536])
def test_gemm_split_k_weight_gradient(K):
    # dW-shaped: few output tiles, long reduction -> split-K with a fixed-order slab sum
    M, N = 256, 384
    gen = torch.Generator(device="cuda").manual_seed(K)
    A = torch.randn(K, M, generator=gen, device="cuda").to(torch.bfloat16)
    B = torch.randn(K, N, generator=gen, device="cuda").to(torch.bfloat16)
    ref = A.float().T @ B.float()
    C = torch.full((M, N), 0.5, device="cuda")
    ws = nc.gemm(nc.NC_BF16, nc.GEMM_TN, nc.EPI_STORE_F32, M, N, K, A, M, B, N, C, N, accumulate=1)
    torch.cuda.synchronize()
    assert ws.numel() > 1024                      # the split-K slabs were requested
    err = (C - 0.5 - ref).norm() / ref.norm()
    assert err < 5e-5, float(err)
    C2 = torch.zeros(M, N, device="cuda")
    C3 = torch.zeros(M, N, device="cuda")
    nc.gemm(nc.NC_BF16, nc.GEMM_TN, nc.EPI_STORE_F32, M, N, K, A, M, B, N, C2, N, ws=ws)
    nc.gemm(nc.NC_BF16, nc.GEMM_TN, nc.EPI_STORE_F32, M, N, K, A, M, B, N, C3, N, ws=ws)
    torch.cuda.synchronize()
    assert float((C2 - ref).norm() / ref.norm()) < 5e-5
    assert torch.equal(C2, C3)                     # fixed-order reduction: run-to-run identical


# ---------------------------------------------------------------- attention
def _attn_case(B, T, H, h, dtype, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, h))
    k = rng.standard_normal((B, T, h))
    v = rng.standard_normal((B, T, h))
    do = rng.standard_normal((B, T, H, h))
    if dtype == "bf16":
        rt = lambda a: torch.from_numpy(a).to(torch.bfloat16).double().numpy()  # noqa: E731
        q, k, v, do = rt(q), rt(k), rt(v), rt(do)
    return q, k, v, do


@pytest.mark.parametrize("dtype,h", [("bf16", 128), ("f32", 128), ("f32", 64)])
@pytest.mark.parametrize("B,T,H", [(2, 100, 3), (1, 1, 2), (1, 129, 10), (3, 64, 1)])
def test_attention_fwd_bwd_matches_oracle(dtype, h, B, T, H):
    q, k, v, do = _attn_case(B, T, H, h, dtype, seed=T * 31 + H)
    o_ref = oracle.attention(q, k, v)
    dq_ref, dk_ref, dv_ref = oracle.attention_bwd(do, q, k, v)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    code = nc.NC_BF16 if dtype == "bf16" else nc.NC_F32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda()  # noqa: E731
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    o = torch.zeros_like(qd)
    lse = torch.zeros(B, T, H, device="cuda")
    nc.attention_fwd(code, B, T, H, h, qd, kd, vd, o, lse)
    # gradients land inside one (B*T, (H+2)h) buffer, as in the step
    W = (H + 2) * h
    dqkv = torch.full((B * T, W), 7.0, dtype=dt, device="cuda")
    nc.attention_bwd(code, B, T, H, h, qd, kd, vd, o, lse, dod, dqkv[:, :H * h], W,
                     dqkv[:, H * h:H * h + h], W, dqkv[:, H * h + h:], W)
    torch.cuda.synchronize()
    got = {"o": o.double().cpu().numpy(),
           "dq": dqkv[:, :H * h].double().cpu().numpy().reshape(B, T, H, h),
           "dk": dqkv[:, H * h:H * h + h].double().cpu().numpy().reshape(B, T, h),
           "dv": dqkv[:, H * h + h:].double().cpu().numpy().reshape(B, T, h)}
    ref = {"o": o_ref, "dq": dq_ref, "dk": dk_ref, "dv": dv_ref}
    s = np.einsum("bthd,bjd->bhtj", q, k) / np.sqrt(h)
    s = np.where(np.triu(np.ones((T, T), bool), 1)[None, None], -np.inf, s)
    m = s.max(-1, keepdims=True)
    lse_ref = (m + np.log(np.exp(s - m).sum(-1, keepdims=True)))[..., 0].transpose(0, 2, 1)
    np.testing.assert_allclose(lse.double().cpu().numpy(), lse_ref,
                               atol=2e-2 if dtype == "bf16" else 1e-5)
    for name in ref:
        if not np.any(ref[name]):
            # One visible key (T = 1): P = 1 and dP = delta, so dS and dq are
            # exactly zero; the GPU's two fp32 reductions (the dP MMA and the
            # delta row sum) leave only rounding-level residue.
            assert np.abs(got[name]).max() < 1e-3, (name, np.abs(got[name]).max())
            continue
        cos, rel = grad_metrics(ref[name], got[name])
        if dtype == "bf16":
            assert cos > 0.999 and rel < 2e-2, (name, cos, rel)
        else:
            assert rel < 2e-5, (name, rel)


def test_attention_running_maximum_grows_every_key_tile():
    """Scores that rise along the keys (k_t = c (t / T) u + noise, q = 16 u +
    noise for a unit vector u): from one 128-key tile to the next a row's
    maximum grows by ~40 nats (~58 in log2 units), far past the 2^8 margin
    within which the online softmax keeps its running maximum, so the
    forward rescales its output accumulator on every key tile.  Output,
    log-sum-exp, dK and dV against the oracle.  dQ is left out: with P nearly
    one-hot, dP - delta is a difference of nearly equal terms, weighted by
    keys of norm ~141, and the bf16 rounding of the stored output that enters
    delta = rowsum(O * dO) moves dQ by ~5 % on its own (an fp64 replay of the
    method with only that rounding gives cos 0.9989): a conditioning property
    of this input, not of the running maximum tested here."""
    B, T, H, h = 2, 640, 3, 128
    rng = np.random.default_rng(640)
    u = rng.standard_normal(h)
    u /= np.linalg.norm(u)
    c = 200.0 * np.sqrt(h) / 16.0                 # last key's score ~200 nats
    q = 16.0 * u + 0.3 * rng.standard_normal((B, T, H, h))
    k = c * (np.arange(T) / T)[None, :, None] * u + 0.3 * rng.standard_normal((B, T, h))
    v = rng.standard_normal((B, T, h))
    do = rng.standard_normal((B, T, H, h))
    rt = lambda a: torch.from_numpy(a).to(torch.bfloat16).double().numpy()  # noqa: E731
    q, k, v, do = rt(q), rt(k), rt(v), rt(do)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).cuda()  # noqa: E731
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    o = torch.zeros_like(qd)
    lse = torch.zeros(B, T, H, device="cuda")
    nc.attention_fwd(nc.NC_BF16, B, T, H, h, qd, kd, vd, o, lse)
    W = (H + 2) * h
    dqkv = torch.full((B * T, W), 7.0, dtype=torch.bfloat16, device="cuda")
    nc.attention_bwd(nc.NC_BF16, B, T, H, h, qd, kd, vd, o, lse, dod, dqkv[:, :H * h], W,
                     dqkv[:, H * h:H * h + h], W, dqkv[:, H * h + h:], W)
    torch.cuda.synchronize()
    s = np.einsum("bthd,bjd->bhtj", q, k) / np.sqrt(h)
    s = np.where(np.triu(np.ones((T, T), bool), 1)[None, None], -np.inf, s)
    m = s.max(-1, keepdims=True)
    assert float(m[..., -1, 0].min()) > 150.0      # the construction did what it says
    lse_ref = (m + np.log(np.exp(s - m).sum(-1, keepdims=True)))[..., 0].transpose(0, 2, 1)
    np.testing.assert_allclose(lse.double().cpu().numpy(), lse_ref, rtol=1e-4, atol=2e-2)
    _, dk_ref, dv_ref = oracle.attention_bwd(do, q, k, v)
    got = {"o": o.double().cpu().numpy(),
           "dk": dqkv[:, H * h:H * h + h].double().cpu().numpy().reshape(B, T, h),
           "dv": dqkv[:, H * h + h:].double().cpu().numpy().reshape(B, T, h)}
    ref = {"o": oracle.attention(q, k, v), "dk": dk_ref, "dv": dv_ref}
    for name in ref:
        cos, rel = grad_metrics(ref[name], got[name])
        assert cos > 0.999 and rel < 2e-2, (name, cos, rel)
