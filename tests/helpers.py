"""Shared test helpers: run the CUDA step on seeded inputs, run the oracle on
the same inputs, and compare with the parity tolerances.

Tolerances (CUDA path vs fp64 oracle):
  bf16 mode: relative loss error <= 2e-3; for every gradient tensor cosine
             similarity >= 0.999 and ||delta|| / ||ref|| <= 3e-2;
  fp32 mode: every output within 1e-5 relative (loss; gradients in norm).
"""
from __future__ import annotations

import numpy as np

import nc_synth

LOSS_RTOL_BF16 = 2e-3
COS_MIN_BF16 = 0.999
REL_MAX_BF16 = 3e-2
RTOL_F32 = 1e-5


def inputs(shape, B, T, dtype, ids_dist="zipf", seed_ids=0, seed_w=1, zero=()):
    ids, tg = nc_synth.make_tokens(shape.vocab, B, T, seed=seed_ids, dist=ids_dist)
    w = nc_synth.make_weights(shape, seed=seed_w, bf16=(dtype == "bf16"), zero=zero)
    return ids, tg, w


def run_cuda_step(shape, dtype, ids, tg, weights, accumulate_runs=1):
    import torch

    from pretraining_step_pretrain_b300 import nc
    B, T = ids.shape
    st = nc.Step(shape, dtype, B, T, weights)
    ids_d = torch.from_numpy(ids).cuda()
    tg_d = torch.from_numpy(tg).cuda()
    for i in range(accumulate_runs):
        st.run(ids_d, tg_d, accumulate=i > 0)
    torch.cuda.synchronize()
    status = st.status()
    loss = float(st.loss.item())
    grads = {k: v.double().cpu().numpy() for k, v in st.g.items()}
    return loss, grads, status


def run_oracle(shape, ids, tg, weights):
    import oracle
    return oracle.step(shape, {k: v.astype(np.float64) for k, v in weights.items()}, ids, tg)


def grad_metrics(ref: np.ndarray, got: np.ndarray) -> tuple[float, float]:
    r, g = ref.ravel(), got.ravel()
    nr, ng = np.linalg.norm(r), np.linalg.norm(g)
    if nr == 0.0:
        return (1.0 if ng == 0.0 else 0.0), (0.0 if ng == 0.0 else np.inf)
    cos = float(r @ g / (nr * ng)) if ng > 0 else 0.0
    return cos, float(np.linalg.norm(r - g) / nr)


def assert_parity(dtype, ref_loss, ref_grads, loss, grads):
    report = []
    if dtype == "bf16":
        assert abs(loss - ref_loss) / abs(ref_loss) <= LOSS_RTOL_BF16, (loss, ref_loss)
        for k in sorted(ref_grads):
            cos, rel = grad_metrics(ref_grads[k], grads[k])
            report.append((k, cos, rel))
            assert cos >= COS_MIN_BF16 and rel <= REL_MAX_BF16, (k, cos, rel)
    else:
        assert abs(loss - ref_loss) / abs(ref_loss) <= RTOL_F32, (loss, ref_loss)
        for k in sorted(ref_grads):
            cos, rel = grad_metrics(ref_grads[k], grads[k])
            report.append((k, cos, rel))
            assert rel <= RTOL_F32, (k, rel)
    return report
