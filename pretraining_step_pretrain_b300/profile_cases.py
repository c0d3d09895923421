"""Run one kernel of the step on synthetic inputs, for profiler captures
(ncu) and quick timing.  Every case goes through the C ABI.

    python -m pretraining_step_pretrain_b300.profile_cases gemm --layout NT --epi relu2 \
        --M 16384 --N 5120 --K 1280 --iters 3
    python -m pretraining_step_pretrain_b300.profile_cases attn --B 4 --T 2048 --H 10 --bwd
    python -m pretraining_step_pretrain_b300.profile_cases step --workload small_bf16
    python -m pretraining_step_pretrain_b300.profile_cases step --workload d20_bf16 --depth 1 \
        --vocab 4096 --iters 2
    python -m pretraining_step_pretrain_b300.profile_cases gemm_fp8 --M 65536 --N 5120 --K 1280

The gemm and gemm_fp8 cases also print the mean time and FLOP rate of their
launches after the first (CUDA events on the launching stream).
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from pretraining_step_pretrain_b300 import nc  # noqa: E402

LAYOUTS = {"NT": nc.GEMM_NT, "NN": nc.GEMM_NN, "TN": nc.GEMM_TN}
EPIS = {"store": nc.EPI_STORE, "store_f32": nc.EPI_STORE_F32, "add_f32": nc.EPI_ADD_F32,
        "relu2": nc.EPI_RELU2, "relu2_bwd": nc.EPI_RELU2_BWD}


def gemm(a):
    L, E = LAYOUTS[a.layout], EPIS[a.epi]
    M, N, K = a.M, a.N, a.K
    g = torch.Generator(device="cuda").manual_seed(0)
    bf = torch.bfloat16
    A = torch.randn(*((M, K) if L != nc.GEMM_TN else (K, M)), generator=g, device="cuda").to(bf)
    B = (torch.randn(*((N, K) if L == nc.GEMM_NT else (K, N)), generator=g, device="cuda")
         / K ** 0.5).to(bf)
    lda = K if L != nc.GEMM_TN else M
    ldb = K if L == nc.GEMM_NT else N
    f32_out = E in (nc.EPI_STORE_F32, nc.EPI_ADD_F32)
    C = torch.zeros(M, N, device="cuda", dtype=torch.float32 if f32_out else bf)
    aux = torch.rand(M, N, generator=g, device="cuda").to(bf) if E == nc.EPI_RELU2_BWD else None
    ws = nc.gemm(nc.NC_BF16, L, E, M, N, K, A, lda, B, ldb, C, N, aux=aux)
    ms = _timed(lambda: nc.gemm(nc.NC_BF16, L, E, M, N, K, A, lda, B, ldb, C, N, aux=aux, ws=ws),
                a.iters - 1)
    print(f"gemm {a.layout} {a.epi} M={M} N={N} K={K}: ok" + _rate(ms, 2.0 * M * N * K))


def _timed(fn, n):
    """Mean ms of n calls of fn, CUDA events on the current stream (None if n < 1)."""
    if n < 1:
        torch.cuda.synchronize()
        return None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def _rate(ms, flop):
    return "" if ms is None else f", {ms:.3f} ms per launch, {flop / ms * 1e-9:.0f} TFLOP/s"


def gemm_fp8(a):
    """C (bf16) = A . B^T with E4M3 operands (random codes, exponents 3..10)."""
    import nc_synth
    M, N, K = a.M, a.N, a.K
    A = torch.from_numpy(nc_synth.make_e4m3_codes(M, K, seed=1)).cuda()
    B = torch.from_numpy(nc_synth.make_e4m3_codes(N, K, seed=2)).cuda()
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = nc.gemm_fp8(M, N, K, A, K, B, K, C, N, 1.0 / 64)
    ms = _timed(lambda: nc.gemm_fp8(M, N, K, A, K, B, K, C, N, 1.0 / 64, ws=ws), a.iters - 1)
    print(f"gemm_fp8 NT M={M} N={N} K={K}: ok" + _rate(ms, 2.0 * M * N * K))


def attn(a):
    B, T, H, h = a.B, a.T, a.H, 128
    g = torch.Generator(device="cuda").manual_seed(0)
    bf = torch.bfloat16
    q = torch.randn(B, T, H, h, generator=g, device="cuda").to(bf)
    k = torch.randn(B, T, h, generator=g, device="cuda").to(bf)
    v = torch.randn(B, T, h, generator=g, device="cuda").to(bf)
    o = torch.empty_like(q)
    lse = torch.empty(B, T, H, device="cuda")
    ws = nc.attention_fwd(nc.NC_BF16, B, T, H, h, q, k, v, o, lse)
    causal = B * H * T * T * h            # one causal-half matmul
    ms = _timed(lambda: nc.attention_fwd(nc.NC_BF16, B, T, H, h, q, k, v, o, lse, ws=ws),
                a.iters - 1)
    print(f"attention fwd B={B} T={T} H={H}: ok" + _rate(ms, 2.0 * causal))
    if a.bwd:
        do = torch.randn_like(q, dtype=torch.float32).to(bf)
        W = (H + 2) * h
        dqkv = torch.empty(B * T, W, dtype=bf, device="cuda")

        def bwd():
            nc.attention_bwd(nc.NC_BF16, B, T, H, h, q, k, v, o, lse, do, dqkv[:, :H * h], W,
                             dqkv[:, H * h:H * h + h], W, dqkv[:, H * h + h:], W, ws=ws)
        bwd()
        ms = _timed(bwd, a.iters - 1)
        print(f"attention bwd B={B} T={T} H={H}: ok" + _rate(ms, 5.0 * causal))


def step(a):
    """nc_step on a named workload; --depth / --vocab / --batch / --seq override its
    shape (e.g. one block at the depth-20 widths, for captures of every kernel
    of a step on inputs larger than L2 but a few GB on the device)."""
    import dataclasses

    import nc_synth
    w = nc_synth.WORKLOADS[a.workload]
    shape = w.shape
    if a.depth:
        shape = dataclasses.replace(shape, depth=a.depth)
    if a.vocab:
        shape = dataclasses.replace(shape, vocab=a.vocab)
    B, T = a.batch or w.batch, a.seq or w.seq
    ids, tg = nc_synth.make_tokens(shape.vocab, B, T, seed=0, dist=w.ids)
    st = nc.Step(shape, w.dtype, B, T, nc_synth.make_weights(shape, seed=1, bf16=(w.dtype == "bf16")))
    st.ids.copy_(torch.from_numpy(ids))
    st.targets.copy_(torch.from_numpy(tg))
    for _ in range(a.iters):
        st.run()
    torch.cuda.synchronize()
    assert st.status() == 0
    print(f"step {a.workload} depth={shape.depth} V={shape.vocab} B={B} T={T}: "
          f"loss {float(st.loss.item()):.5f}, {nc.launch_count() // max(a.iters, 1)} launches per step")


def main():
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="case", required=True)
    p = sub.add_parser("gemm")
    p.add_argument("--layout", default="NT", choices=sorted(LAYOUTS))
    p.add_argument("--epi", default="store", choices=sorted(EPIS))
    p.add_argument("--M", type=int, default=16384)
    p.add_argument("--N", type=int, default=5120)
    p.add_argument("--K", type=int, default=1280)
    p.add_argument("--iters", type=int, default=3)
    p = sub.add_parser("gemm_fp8")
    p.add_argument("--M", type=int, default=16384)
    p.add_argument("--N", type=int, default=5120)
    p.add_argument("--K", type=int, default=1280)
    p.add_argument("--iters", type=int, default=3)
    p = sub.add_parser("attn")
    p.add_argument("--B", type=int, default=4)
    p.add_argument("--T", type=int, default=2048)
    p.add_argument("--H", type=int, default=10)
    p.add_argument("--bwd", action="store_true")
    p.add_argument("--iters", type=int, default=3)
    p = sub.add_parser("step")
    p.add_argument("--workload", default="small_bf16")
    p.add_argument("--iters", type=int, default=2)
    p.add_argument("--depth", type=int, default=0)
    p.add_argument("--vocab", type=int, default=0)
    p.add_argument("--batch", type=int, default=0)
    p.add_argument("--seq", type=int, default=0)
    a = ap.parse_args()
    {"gemm": gemm, "gemm_fp8": gemm_fp8, "attn": attn, "step": step}[a.case](a)


if __name__ == "__main__":
    main()
