"""Pins of the fp64 optimizer oracle (oracle/optimizer.py) against closed
forms, invariants and library special cases -- never against a retyping of
its own formulas."""
import math

import numpy as np
import pytest

from oracle import optimizer as opt


def test_lrm_is_one_then_linear_to_zero():
    """Walkthrough, section "预训练": lrm falls linearly to 0 near the end."""
    N, wd = 100, 0.2
    lr = [opt.lr_multiplier(s, N, wd) for s in range(N)]
    assert lr[:80] == [1.0] * 80
    assert lr[-1] == 0.0
    steps = np.diff(lr[79:])
    assert np.allclose(steps, -1.0 / 20)          # one straight line down to 0
    assert opt.lr_multiplier(5, 10, 0.0) == 1.0    # no warmdown: constant


def test_adamw_first_step_is_sign_like():
    """With zero moments, bias correction makes the first update
    lr * g / (|g| + eps) exactly (mhat = g, vhat = g^2)."""
    rng = np.random.default_rng(0)
    p = rng.standard_normal(50)
    g = rng.standard_normal(50)
    lr, eps, wd = 0.01, 1e-8, 0.1
    new, m, v = opt.adamw(p, g, np.zeros(50), np.zeros(50), 1, lr, 0.8, 0.95, eps, wd)
    assert np.allclose(new, p * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=0, atol=1e-15)
    assert np.allclose(m, 0.2 * g) and np.allclose(v, 0.05 * g * g)


@pytest.mark.parametrize("t_steps", [2, 7])
def test_adamw_constant_gradient_has_unbiased_moments(t_steps):
    """A constant gradient keeps mhat = g and vhat = g^2 at every step, so
    every update is the same lr * g / (|g| + eps) (no weight decay)."""
    g = np.array([0.3, -2.0, 1e-3])
    p = np.zeros(3)
    m = np.zeros(3)
    v = np.zeros(3)
    lr, eps = 0.05, 1e-10
    for t in range(1, t_steps + 1):
        p_old = p
        p, m, v = opt.adamw(p, g, m, v, t, lr, 0.9, 0.999, eps, 0.0)
        assert np.allclose(p_old - p, lr * g / (np.abs(g) + eps), rtol=1e-12)


def _scalar_ns(x, coeffs, steps):
    a, b, c = coeffs
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


@pytest.mark.parametrize("shape", [(12, 20), (20, 12), (16, 16)])
@pytest.mark.parametrize("coeffs", [opt.MUON_NS_COEFFS, opt.CUBIC_NS_COEFFS])
def test_newton_schulz_acts_on_singular_values(shape, coeffs):
    """An odd polynomial iteration on X = G/||G||_F keeps the singular vectors
    and maps every singular value s by the scalar iteration of p(x) = a x +
    b x^3 + c x^5: NS(G) = U diag(p^k(s/||G||_F)) V^T (SVD from LAPACK)."""
    rng = np.random.default_rng(shape[0] * 31 + shape[1])
    G = rng.standard_normal(shape)
    U, s, Vt = np.linalg.svd(G, full_matrices=False)
    expect = (U * _scalar_ns(s / (np.linalg.norm(G) + 1e-7), coeffs, 5)) @ Vt
    got = opt.newton_schulz(G, coeffs, 5)
    assert got.shape == G.shape
    assert np.allclose(got, expect, atol=1e-12)


def test_cubic_newton_schulz_converges_to_polar_factor():
    """Enough classical cubic steps give the orthogonal polar factor U V^T."""
    rng = np.random.default_rng(3)
    G = rng.standard_normal((16, 24))
    U, _, Vt = np.linalg.svd(G, full_matrices=False)
    X = opt.newton_schulz(G, opt.CUBIC_NS_COEFFS, 40)
    assert np.allclose(X, U @ Vt, atol=1e-10)
    assert np.allclose(X @ X.T, np.eye(16), atol=1e-10)


def test_muon_quintic_squashes_spectrum_into_band():
    """The published quintic does not converge to 1; after 5 steps every
    singular value of a full-rank matrix lies in a band around 1."""
    rng = np.random.default_rng(4)
    G = rng.standard_normal((64, 96))
    s = np.linalg.svd(opt.newton_schulz(G), compute_uv=False)
    assert s.min() > 0.5 and s.max() < 1.3, (s.min(), s.max())


def test_muon_first_step_and_shape_scale():
    """Zero momentum buffer, Nesterov: u = (1 + mu) g and NS is scale-free, so
    the first update is lr sqrt(max(1, r/c)) NS(g); the buffer becomes g."""
    rng = np.random.default_rng(5)
    for r, c in ((30, 10), (10, 30)):
        p = rng.standard_normal((r, c))
        g = rng.standard_normal((r, c))
        new, buf = opt.muon(p, g, np.zeros((r, c)), 0.02, 0.95)
        scale = math.sqrt(max(1.0, r / c))
        assert np.allclose(buf, g)
        assert np.allclose(p - new, 0.02 * scale * opt.newton_schulz(g), atol=1e-9)


def test_optimizer_routes_matrices_to_muon_and_embeddings_to_adamw():
    """Architecture list: Muon for the matrices, AdamW for the embedding and
    unembedding; AdamW rates carry lrm and the 1/sqrt(d_model) factor."""
    rng = np.random.default_rng(6)
    d = 16
    params = {"wte": rng.standard_normal((32, d)), "w_qkv.0": rng.standard_normal((24, d)),
              "w_lm": rng.standard_normal((32, d))}
    grads = {k: rng.standard_normal(v.shape) for k, v in params.items()}
    new, state = opt.optimizer_step(params, grads, {}, 1, d, 0.5, lr_muon=0.02, momentum=0.95,
                                    lr_embed=0.3, lr_lm=0.004, betas=(0.8, 0.95), eps=1e-10)
    assert set(state["w_qkv.0"]) == {"buf"} and set(state["wte"]) == {"m", "v"}
    step_embed = params["wte"] - new["wte"]
    assert np.allclose(step_embed, 0.3 * 0.5 / 4.0 * grads["wte"] / (np.abs(grads["wte"]) + 1e-10))
    step_lm = params["w_lm"] - new["w_lm"]
    assert np.allclose(step_lm, 0.004 * 0.5 / 4.0 * grads["w_lm"] / (np.abs(grads["w_lm"]) + 1e-10))
    step_m = params["w_qkv.0"] - new["w_qkv.0"]
    assert np.allclose(step_m, 0.02 * 0.5 * math.sqrt(24 / 16) * opt.newton_schulz(grads["w_qkv.0"]),
                       atol=1e-9)
