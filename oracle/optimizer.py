"""fp64 CPU oracle of the optimizer step that follows the pretraining step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA path.

What the pages fix (launch article's Q&A, vpshk.cn, section
"卡帕西亲自揭秘背后技术", architecture list; imeisheng.com walkthrough
"100美元成本、8000行代码纯手搓克隆ChatGPT", section "预训练"):

  * the optimizer is Muon + AdamW, after modded-nanoGPT;
  * Muon updates the matrices (here: every weight inside the blocks), AdamW
    the embedding and the unembedding -- there are no other parameters;
  * learning rates scale as 1/sqrt(dim);
  * ``lrm``, the learning-rate multiplier, falls linearly to 0 near the end
    of training.

Everything else is a reading, stated where it is used:

  * AdamW is the decoupled-weight-decay Adam of Loshchilov & Hutter with bias
    correction; betas, eps and the weight decay are caller inputs.
  * Muon is the published method (K. Jordan et al., 2024, "Muon: an optimizer
    for hidden layers"): momentum buffer b <- mu b + g, Nesterov look-ahead
    u = g + mu b, orthogonalisation of u by an odd-polynomial Newton-Schulz
    iteration on X = u / ||u||_F, update W <- W - lr * sqrt(max(1, r/c)) * X
    for an r x c matrix.  The iteration's coefficients (a, b, c) and step
    count are caller inputs; the defaults are the quintic published with Muon.
  * 1/sqrt(dim) scaling: the AdamW learning rates are multiplied by
    d_model^(-1/2) (an orthogonalised Muon update has unit spectral norm at
    any width, so Muon's rate is left unscaled).
  * ``lrm`` schedule: 1 until the last ``warmdown`` fraction of the steps,
    then linear to 0 at the final step.

Random numbers are never drawn here; callers pass the arrays.
"""
from __future__ import annotations

import math

import numpy as np

# Odd quintic published with Muon: p(x) = a x + b x^3 + c x^5, five steps.
MUON_NS_COEFFS = (3.4445, -4.7750, 2.0315)
MUON_NS_STEPS = 5
# Classical cubic Newton-Schulz step for the polar factor (Higham, "Functions
# of Matrices", section 8.3): X <- 1.5 X - 0.5 X X^T X.
CUBIC_NS_COEFFS = (1.5, -0.5, 0.0)


def lr_multiplier(step: int, total_steps: int, warmdown: float) -> float:
    """lrm at `step` (0-based) of `total_steps`: 1, then linear to 0 over the
    final `warmdown` fraction (walkthrough: lrm falls linearly to 0 near the end)."""
    n_down = int(round(warmdown * total_steps))
    start = total_steps - n_down
    if n_down <= 0 or step < start:
        return 1.0
    return max(0.0, (total_steps - 1 - step) / n_down) if n_down > 0 else 1.0


def adamw(p, g, m, v, t: int, lr: float, beta1: float, beta2: float, eps: float, wd: float):
    """One AdamW update (t = 1 on the first step).  Returns new (p, m, v)."""
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    p = p - lr * wd * p - lr * mhat / (np.sqrt(vhat) + eps)
    return p, m, v


def newton_schulz(G: np.ndarray, coeffs=MUON_NS_COEFFS, steps: int = MUON_NS_STEPS,
                  norm_eps: float = 1e-7) -> np.ndarray:
    """Odd-polynomial Newton-Schulz iteration towards the polar factor of G.

    X0 = G / (||G||_F + norm_eps), taken as the wide orientation (rows <= cols,
    so that X X^T is the smaller Gram matrix); each step
    X <- a X + (b A + c A A) X with A = X X^T.
    """
    a, b, c = coeffs
    X = np.asarray(G, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = X / (np.linalg.norm(X) + norm_eps)
    for _ in range(steps):
        A = X @ X.T
        Bm = b * A + c * (A @ A)
        X = a * X + Bm @ X
    return X.T if tall else X


def muon(p, g, buf, lr: float, momentum: float, nesterov: bool = True, coeffs=MUON_NS_COEFFS,
         steps: int = MUON_NS_STEPS):
    """One Muon update of an r x c matrix.  Returns new (p, buf)."""
    buf = momentum * buf + g
    u = g + momentum * buf if nesterov else buf
    o = newton_schulz(u, coeffs, steps)
    r, c = p.shape
    p = p - lr * math.sqrt(max(1.0, r / c)) * o
    return p, buf


def is_muon_param(name: str) -> bool:
    """Matrices inside the blocks go to Muon; the embedding and the LM head to AdamW."""
    return name.split(".")[0] in ("w_qkv", "w_o", "w_fc", "w_proj")


def optimizer_step(params: dict, grads: dict, state: dict, t: int, d_model: int, lrm: float,
                   lr_muon: float, momentum: float, lr_embed: float, lr_lm: float,
                   betas=(0.9, 0.999), eps: float = 1e-8, wd: float = 0.0,
                   ns_coeffs=MUON_NS_COEFFS, ns_steps: int = MUON_NS_STEPS):
    """Update every parameter once (fp64 master weights).  `state` maps a name
    to {"buf"} (Muon) or {"m", "v"} (AdamW); missing entries start at zero.
    `t` counts optimizer steps from 1.  Returns (params, state) as new dicts."""
    scale = 1.0 / math.sqrt(d_model)
    new_p, new_s = {}, {}
    for name, p in params.items():
        g = grads[name]
        st = state.get(name, {})
        if is_muon_param(name):
            buf = st.get("buf", np.zeros_like(p))
            new_p[name], b = muon(p, g, buf, lr_muon * lrm, momentum, True, ns_coeffs, ns_steps)
            new_s[name] = {"buf": b}
        else:
            lr = (lr_embed if name == "wte" else lr_lm) * lrm * scale
            m = st.get("m", np.zeros_like(p))
            v = st.get("v", np.zeros_like(p))
            new_p[name], m, v = adamw(p, g, m, v, t, lr, betas[0], betas[1], eps, wd)
            new_s[name] = {"m": m, "v": v}
    return new_p, new_s
