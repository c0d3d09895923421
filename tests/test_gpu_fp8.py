"""Parity of the 8-bit floating-point contraction (nc_gemm_fp8: E4M3
operands on the tcgen05 kernel) with the fp64 oracle in oracle/fp8.py.

Tolerance from the arithmetic: every product of two E4M3 values is exact in
fp32, so the only error is the fp32 summation, bounded element-wise by
K u S with u = 2^-24 and S = |scale| sum_k |a_ik b_jk|, plus the output
rounding (|C| 2^-24 for fp32, |C| 2^-8 for bf16)."""
import numpy as np
import pytest
import torch

import nc_synth
from oracle import fp8
from pretraining_step_pretrain_b300 import build, nc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    nc.lib()


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 288, 512), (1000, 1024, 1040),
                                   (2304, 1536, 2048), (1, 32, 16)])
def test_fp8_gemm_matches_oracle(out, M, N, K):
    a = nc_synth.make_e4m3_codes(M, K, seed=M + K)
    b = nc_synth.make_e4m3_codes(N, K, seed=N + 7 * K)
    scale = 0.3
    ref = fp8.gemm_e4m3(a, b, scale)
    bound = K * 2.0 ** -24 * (abs(scale) * (np.abs(fp8.e4m3_decode(a)) @ np.abs(fp8.e4m3_decode(b)).T))
    bound += np.abs(ref) * (2.0 ** -24 if out == "f32" else 2.0 ** -8)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    C = torch.full((M, N), 7.0, dtype=dt, device="cuda")
    nc.gemm_fp8(M, N, K, torch.from_numpy(a).cuda(), K, torch.from_numpy(b).cuda(), K, C, N, scale)
    torch.cuda.synchronize()
    got = C.double().cpu().numpy()
    err = np.abs(got - ref)
    assert np.all(err <= bound * 1.0001 + 1e-30), (float(err.max()), float((err / (bound + 1e-30)).max()))


def test_fp8_gemm_strided_operands_and_output():
    """Leading dimensions wider than the rows: only the first K (N) columns count."""
    M, N, K, lda, ldb, ldc = 200, 64, 96, 144, 128, 72
    a = nc_synth.make_e4m3_codes(M, lda, seed=1)
    b = nc_synth.make_e4m3_codes(N, ldb, seed=2)
    ref = fp8.gemm_e4m3(a[:, :K], b[:, :K], 1.0)
    C = torch.full((M, ldc), -3.0, dtype=torch.float32, device="cuda")
    nc.gemm_fp8(M, N, K, torch.from_numpy(a).cuda(), lda, torch.from_numpy(b).cuda(), ldb, C, ldc)
    torch.cuda.synchronize()
    got = C.double().cpu().numpy()
    assert np.allclose(got[:, :N], ref, rtol=1e-6, atol=1e-6)
    assert np.all(got[:, N:] == -3.0)   # columns past N untouched


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fp8_gemm_full_code_range(out):
    """Operands drawn from every non-NaN code, with whole rows of zeros (both
    signs), of subnormals only, and of +-448 (the largest finite magnitude),
    and columns of the same kinds in B; the element-wise bound as above."""
    M, N, K = 520, 288, 640
    a = nc_synth.make_e4m3_codes_full(M, K, seed=11)
    b = nc_synth.make_e4m3_codes_full(N, K, seed=12)
    rng = np.random.default_rng(13)
    sign = lambda *s: (rng.integers(0, 2, size=s, dtype=np.uint8) << 7)  # noqa: E731
    a[0] = sign(K)                                           # +-0
    a[1] = sign(K) | rng.integers(1, 8, size=K, dtype=np.uint8)   # subnormals s.0000.mmm
    a[2] = sign(K) | 0x7E                                    # +-448
    a[3, ::2] = 0x7E                                         # mixed extremes and zeros
    a[3, 1::2] = 0x80
    b[0] = sign(K) | 0x7E
    b[5] = sign(K) | rng.integers(1, 8, size=K, dtype=np.uint8)
    b[7] = sign(K)
    assert not np.isnan(fp8.e4m3_decode(a)).any() and not np.isnan(fp8.e4m3_decode(b)).any()
    scale = 1.0 / 448.0
    ref = fp8.gemm_e4m3(a, b, scale)
    bound = K * 2.0 ** -24 * (abs(scale) * (np.abs(fp8.e4m3_decode(a)) @ np.abs(fp8.e4m3_decode(b)).T))
    bound += np.abs(ref) * (2.0 ** -24 if out == "f32" else 2.0 ** -8)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    C = torch.full((M, N), 7.0, dtype=dt, device="cuda")
    nc.gemm_fp8(M, N, K, torch.from_numpy(a).cuda(), K, torch.from_numpy(b).cuda(), K, C, N, scale)
    torch.cuda.synchronize()
    got = C.double().cpu().numpy()
    err = np.abs(got - ref)
    assert np.all(err <= bound * 1.0001 + 1e-30), (float(err.max()), float((err / (bound + 1e-30)).max()))
    assert np.all(got[0] == 0.0) and np.all(got[:, 7] == 0.0)
