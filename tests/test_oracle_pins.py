"""Pins of the fp64 oracle against things fixed outside it: closed forms,
invariants, special cases that reduce to library routines (torch SDPA, scipy
log_softmax), brute force on tiny inputs, and central differences.

Each test names the part of the method it pins; a plausible mistake (dropped
term, wrong sign or index, transposed operand) in that part fails it.
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import nc_synth
import oracle
from oracle import nanochat_step as ns

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _tiny_params(shape, seed=1, zero=()):
    return {k: v.astype(np.float64) for k, v in
            nc_synth.make_weights(shape, seed=seed, bf16=False, zero=zero).items()}


# ------------------------------------------------------------------ RMSNorm
def test_rmsnorm_rms_closed_form():
    x = RNG.standard_normal((7, 33)) * 3.0
    eps = 1e-6
    y, r = oracle.rmsnorm(x, eps)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), np.sqrt(ms / (ms + eps)),
                               rtol=1e-14)
    y0, _ = oracle.rmsnorm(x, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y0 * y0, axis=-1)), 1.0, rtol=1e-14)


def test_rmsnorm_eps_placement():
    # eps sits inside the square root: a constant row of value a maps to a/sqrt(a^2+eps)
    a, eps = 1e-3, 1e-6
    y, _ = oracle.rmsnorm(np.full((1, 8), a), eps)
    np.testing.assert_allclose(y, a / math.sqrt(a * a + eps), rtol=1e-14)


def test_rmsnorm_scale_invariant_without_eps():
    x = RNG.standard_normal((5, 16))
    y1, _ = oracle.rmsnorm(x, 0.0)
    y2, _ = oracle.rmsnorm(17.0 * x, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-13)


def test_rmsnorm_bwd_central_difference():
    x = RNG.standard_normal((3, 12))
    dy = RNG.standard_normal((3, 12))
    eps = 1e-3
    _, r = oracle.rmsnorm(x, eps)
    dx = oracle.rmsnorm_bwd(dy, x, r)
    num = np.zeros_like(x)
    hstep = 1e-6
    for idx in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += hstep
        xm[idx] -= hstep
        num[idx] = (np.sum(oracle.rmsnorm(xp, eps)[0] * dy) -
                    np.sum(oracle.rmsnorm(xm, eps)[0] * dy)) / (2 * hstep)
    np.testing.assert_allclose(dx, num, rtol=1e-7, atol=1e-9)


# ------------------------------------------------------------------ RoPE
def test_rope_closed_form_golden():
    g = json.load(open(os.path.join(GOLDEN, "rope_closed_form.json")))
    h, base = g["head_dim"], g["base"]
    for case in g["cases"]:
        T = case["t"] + 1
        cos, sin = oracle.rope_tables(T, h, base)
        e = np.zeros(h)
        e[case["unit_index"]] = 1.0
        out = oracle.rope(e, cos[case["t"]], sin[case["t"]])
        expect = np.zeros(h)
        for i, val in case["expect_index_pairs"]:
            expect[i] = val
        np.testing.assert_allclose(out, expect, atol=1e-12)


def test_rope_identity_at_position_zero_and_norm_preserving():
    T, h = 50, 16
    cos, sin = oracle.rope_tables(T, h, 10000.0)
    x = RNG.standard_normal((T, h))
    y = oracle.rope(x, cos, sin)
    np.testing.assert_array_equal(y[0], x[0])
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_dot_depends_on_relative_position_only():
    T, h = 64, 16
    cos, sin = oracle.rope_tables(T, h, 10000.0)
    q, k = RNG.standard_normal(h), RNG.standard_normal(h)
    for m, n in [(5, 2), (40, 3), (10, 10)]:
        ref = oracle.rope(q, cos[m], sin[m]) @ oracle.rope(k, cos[n], sin[n])
        for delta in (1, 7, 13):
            got = oracle.rope(q, cos[m + delta], sin[m + delta]) @ oracle.rope(k, cos[n + delta], sin[n + delta])
            assert abs(got - ref) < 1e-12


def test_rope_bwd_is_transpose():
    T, h = 9, 8
    cos, sin = oracle.rope_tables(T, h, 10000.0)
    x, dy = RNG.standard_normal((T, h)), RNG.standard_normal((T, h))
    assert abs(np.sum(oracle.rope(x, cos, sin) * dy) - np.sum(x * oracle.rope_bwd(dy, cos, sin))) < 1e-12


def test_norm_and_rope_commute():
    # RoPE is orthogonal, so normalising before or after rotating is the same map.
    T, h = 20, 16
    cos, sin = oracle.rope_tables(T, h, 10000.0)
    x = RNG.standard_normal((T, h)) * 2.0
    a = oracle.rope(oracle.rmsnorm(x, 1e-6)[0], cos, sin)
    b = oracle.rmsnorm(oracle.rope(x, cos, sin), 1e-6)[0]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ softcap
def test_softcap_bounded_and_identity_near_zero():
    c = 15.0
    z = np.array([-1e30, -1e4, -40.0, 40.0, 1e4, 1e30])
    s = oracle.softcap(z, c)
    assert np.all(np.abs(s) <= c)
    assert s[0] == -c and s[-1] == c
    zs = np.array([-1e-3, 2e-4, 5e-3])
    np.testing.assert_allclose(oracle.softcap(zs, c), zs - zs ** 3 / (3 * c * c), rtol=1e-10)


def test_softcap_bwd_derivative():
    c, z = 15.0, np.linspace(-40, 40, 81)
    s = oracle.softcap(z, c)
    np.testing.assert_allclose(oracle.softcap_bwd(np.ones_like(z), s, c),
                               1.0 / np.cosh(z / c) ** 2, rtol=1e-12)


# ------------------------------------------------------------------ attention
def _torch_mqa_reference(q, k, v):
    """MQA as textbook MHA (torch SDPA, causal) with the one K/V head repeated."""
    B, T, H, h = q.shape
    qt = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_(True)
    kt = torch.tensor(k)[:, None].expand(B, H, T, h).clone().requires_grad_(True)
    vt = torch.tensor(v)[:, None].expand(B, H, T, h).clone().requires_grad_(True)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    return qt, kt, vt, o


def test_attention_matches_torch_sdpa_fwd_and_bwd():
    B, T, H, h = 2, 11, 3, 8
    q, k, v = (RNG.standard_normal(s) for s in ((B, T, H, h), (B, T, h), (B, T, h)))
    do = RNG.standard_normal((B, T, H, h))
    o = oracle.attention(q, k, v)
    qt, kt, vt, ot = _torch_mqa_reference(q, k, v)
    np.testing.assert_allclose(o, ot.permute(0, 2, 1, 3).detach().numpy(), rtol=1e-12, atol=1e-13)
    ot.backward(torch.tensor(do).permute(0, 2, 1, 3))
    dq, dk, dv = oracle.attention_bwd(do, q, k, v)
    np.testing.assert_allclose(dq, qt.grad.permute(0, 2, 1, 3).numpy(), rtol=1e-11, atol=1e-12)
    # one shared K/V head: its gradient is the sum over query heads of MHA's
    np.testing.assert_allclose(dk, kt.grad.sum(1).numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.sum(1).numpy(), rtol=1e-11, atol=1e-12)


def test_attention_brute_force_loops():
    B, T, H, h = 1, 6, 2, 4
    q, k, v = (RNG.standard_normal(s) for s in ((B, T, H, h), (B, T, h), (B, T, h)))
    o = oracle.attention(q, k, v)
    for hd in range(H):
        for i in range(T):
            w = [math.exp(float(q[0, i, hd] @ k[0, j]) / math.sqrt(h)) for j in range(i + 1)]
            z = sum(w)
            ref = sum(w[j] / z * v[0, j] for j in range(i + 1))
            np.testing.assert_allclose(o[0, i, hd], ref, rtol=1e-12)


def test_attention_single_position_returns_v():
    q, k, v = RNG.standard_normal((2, 1, 4, 8)), RNG.standard_normal((2, 1, 8)), RNG.standard_normal((2, 1, 8))
    o = oracle.attention(q, k, v)
    for hd in range(4):
        np.testing.assert_array_equal(o[:, 0, hd], v[:, 0])


def test_causal_mask_by_token_perturbation():
    shape = nc_synth.GRADCHECK
    P = _tiny_params(shape)
    ids, tg = nc_synth.make_tokens(shape.vocab, 1, 10, seed=3, dist="uniform")
    base = oracle.forward(shape, P, ids)["s"]
    for j in (0, 4, 9):
        ids2 = ids.copy()
        ids2[0, j] = (ids2[0, j] + 1) % shape.vocab
        s2 = oracle.forward(shape, P, ids2)["s"]
        np.testing.assert_array_equal(s2[0, :j], base[0, :j])     # bit-identical before j
        assert np.all(np.any(s2[0, j:] != base[0, j:], axis=-1))  # every later position moves


# ------------------------------------------------------------------ loss
def test_cross_entropy_matches_scipy_and_ignore_index():
    s = RNG.standard_normal((9, 13)) * 4.0
    y = RNG.integers(0, 13, size=9)
    y[3] = -1
    loss, ds = oracle.cross_entropy(s, y)
    valid = y >= 0
    ref = -np.mean(scipy.special.log_softmax(s[valid], axis=-1)[np.arange(valid.sum()), y[valid]])
    assert abs(loss - ref) < 1e-13
    np.testing.assert_allclose(ds.sum(-1), 0.0, atol=1e-15)
    assert np.all(ds[3] == 0.0)


@pytest.mark.parametrize("vocab,expect", [(512, 6.238325), (4096, 8.317766), (65536, 11.090355)])
def test_zero_lm_head_loss_is_log_vocab(vocab, expect):
    # closed form: all logits 0 -> uniform softmax -> loss = ln V
    assert abs(math.log(vocab) - expect) < 5e-7
    shape = nc_synth.ModelShape(1, 32, 2, 16, 64, vocab)
    P = _tiny_params(shape, zero=("w_lm",))
    ids, tg = nc_synth.make_tokens(vocab, 2, 5, seed=5, dist="zipf")
    loss, g = oracle.step(shape, P, ids, tg)
    assert abs(loss - math.log(vocab)) < 1e-12
    cache = oracle.forward(shape, P, ids, tg)
    xf = cache["xf"].reshape(-1, shape.d_model)
    y = tg.reshape(-1)
    onehot = np.zeros((y.size, vocab))
    onehot[np.arange(y.size), y] = 1.0
    np.testing.assert_allclose(g["w_lm"], (1.0 / vocab - onehot).T @ xf / y.size, rtol=1e-12, atol=1e-15)
    for name, val in g.items():
        if name != "w_lm":
            assert np.all(val == 0.0), name


def test_zero_output_projections_reduce_to_softmax_regression():
    shape = nc_synth.GRADCHECK
    P = _tiny_params(shape, zero=("w_o", "w_proj"))
    ids, tg = nc_synth.make_tokens(shape.vocab, 2, 7, seed=9, dist="uniform")
    loss, g = oracle.step(shape, P, ids, tg)
    emb = P["wte"][ids]
    x = emb / np.sqrt(np.mean(emb ** 2, -1, keepdims=True) + shape.eps)
    cache = oracle.forward(shape, P, ids, tg)
    np.testing.assert_allclose(cache["x_embed"], x, rtol=1e-14)
    for lc in cache["layers"]:
        np.testing.assert_array_equal(lc["x_in"], cache["x_embed"])  # residual carries norm(embedding)
    np.testing.assert_array_equal(cache["x_out"], cache["x_embed"])
    xf = x / np.sqrt(np.mean(x ** 2, -1, keepdims=True) + shape.eps)
    s = 15.0 * np.tanh((xf @ P["w_lm"].T) / 15.0)
    ref = np.mean(scipy.special.logsumexp(s, axis=-1) - np.take_along_axis(s, tg[..., None], -1)[..., 0])
    assert abs(loss - ref) < 1e-12
    for l in range(shape.depth):
        assert np.all(g[f"w_qkv.{l}"] == 0.0) and np.all(g[f"w_fc.{l}"] == 0.0)
        assert np.abs(g[f"w_o.{l}"]).max() > 1e-6 and np.abs(g[f"w_proj.{l}"]).max() > 1e-6


# ------------------------------------------------------------------ where RoPE acts in forward()
def _one_layer_cache(ids):
    shape = dataclasses.replace(nc_synth.GRADCHECK, depth=1)
    return shape, oracle.forward(shape, _tiny_params(shape, seed=21), ids)


def _rotate_closed_form(x, h, base):
    """Rotate x (B, T, [heads,] h) by position t = 0..T-1 of its own row, written
    out from the rotary definition (pairs (i, i + h/2), angle t base^(-2i/h)),
    without the oracle's tables."""
    T = x.shape[1]
    ang = np.array([[t * base ** (-2.0 * i / h) for i in range(h // 2)] for t in range(T)])
    c, s = np.cos(ang), np.sin(ang)
    if x.ndim == 4:
        c, s = c[:, None, :], s[:, None, :]
    x1, x2 = x[..., : h // 2], x[..., h // 2:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def test_forward_rotates_queries_and_keys_at_each_rows_own_positions():
    """Architecture list: rotary embeddings act on the (QK-normed) queries and
    key at each token's position within its row, and nothing else is rotated.
    Fails if q or k is left unrotated, v is rotated, or positions run on
    across rows instead of restarting at 0."""
    ids, _ = nc_synth.make_tokens(32, 3, 9, seed=31, dist="uniform")
    shape, cache = _one_layer_cache(ids)
    lc = cache["layers"][0]
    H, h = shape.n_head, shape.head_dim
    np.testing.assert_allclose(lc["qr"], _rotate_closed_form(lc["qn"], h, shape.rope_base),
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lc["kr"], _rotate_closed_form(lc["kn"], h, shape.rope_base),
                               rtol=1e-12, atol=1e-14)
    assert np.abs(lc["qr"][:, 1:] - lc["qn"][:, 1:]).max() > 1e-3   # really rotated
    assert np.abs(lc["kr"][:, 1:] - lc["kn"][:, 1:]).max() > 1e-3
    # v: the raw value rows of the projection, neither normed nor rotated
    w = _tiny_params(shape, seed=21)["w_qkv.0"]
    np.testing.assert_array_equal(lc["v"], lc["xn"] @ w[(H + 1) * h:].T)
    o = oracle.attention(lc["qr"], lc["kr"], lc["v"]).reshape(lc["o"].shape)
    np.testing.assert_array_equal(lc["o"], o)


def test_forward_positions_restart_in_every_row():
    """Two rows holding the same tokens give the same outputs: a position
    counted across the batch (row b starting at b T) would rotate row 1
    differently from row 0."""
    ids, _ = nc_synth.make_tokens(32, 1, 11, seed=32, dist="uniform")
    ids2 = np.concatenate([ids, ids], axis=0)
    _, cache = _one_layer_cache(ids2)
    np.testing.assert_array_equal(cache["layers"][0]["qr"][0], cache["layers"][0]["qr"][1])
    np.testing.assert_array_equal(cache["s"][0], cache["s"][1])


def test_forward_scores_of_a_constant_row_depend_on_relative_position_only():
    """With one token repeated along a row, every position has the same normed
    q and k, so after rotation the score q_i . k_j is a function of i - j
    alone -- and not a constant, which it would be without rotation."""
    ids = np.full((1, 12), 7, dtype=np.int32)
    shape, cache = _one_layer_cache(ids)
    lc = cache["layers"][0]
    T = ids.shape[1]
    for hd in range(shape.n_head):
        s = lc["qr"][0, :, hd] @ lc["kr"][0].T                    # (T, T): query i, key j
        for delta in range(T):
            diag = np.array([s[i, i - delta] for i in range(delta, T)])
            np.testing.assert_allclose(diag, diag[0], rtol=1e-12, atol=1e-13)
        lagged = np.array([s[T - 1, T - 1 - delta] for delta in range(T)])
        assert np.ptp(lagged) > 1e-3


# ------------------------------------------------------------------ structure
def test_qk_norm_makes_loss_invariant_to_query_key_scale():
    shape = nc_synth.GRADCHECK
    P = _tiny_params(shape)
    ids, tg = nc_synth.make_tokens(shape.vocab, 2, 6, seed=2, dist="uniform")
    base = oracle.step(shape, P, ids, tg)[0]
    P2 = dict(P)
    qk = (shape.n_head + 1) * shape.head_dim
    w = P["w_qkv.0"].copy()
    w[:qk] *= 3.0
    P2["w_qkv.0"] = w
    assert abs(oracle.step(shape, P2, ids, tg)[0] - base) < 1e-5    # eps only
    w = P["w_qkv.0"].copy()
    w[qk:] *= 3.0                                                  # value rows: not normalised
    P2["w_qkv.0"] = w
    assert abs(oracle.step(shape, P2, ids, tg)[0] - base) > 1e-3


def test_relu_squared_is_degree_two_homogeneous():
    # relu(a u)^2 = a^2 relu(u)^2: scaling W_fc by a equals scaling W_proj by a^2
    shape = nc_synth.GRADCHECK
    P = _tiny_params(shape)
    ids, tg = nc_synth.make_tokens(shape.vocab, 1, 8, seed=4, dist="uniform")
    a = 1.7
    Pa, Pb = dict(P), dict(P)
    Pa["w_fc.1"] = P["w_fc.1"] * a
    Pb["w_proj.1"] = P["w_proj.1"] * a * a
    la, lb = oracle.step(shape, Pa, ids, tg)[0], oracle.step(shape, Pb, ids, tg)[0]
    assert abs(la - lb) < 1e-12
    Pc = dict(P)
    Pc["w_proj.1"] = P["w_proj.1"] * a
    assert abs(oracle.step(shape, Pc, ids, tg)[0] - la) > 1e-6


# ------------------------------------------------------------------ gradients
def test_central_difference_every_weight():
    shape = nc_synth.GRADCHECK
    P = _tiny_params(shape, seed=11)
    ids, tg = nc_synth.make_tokens(shape.vocab, 2, 8, seed=12, dist="uniform")
    tg[1, 3] = -1                                                   # exercise ignore index
    _, grads = oracle.step(shape, P, ids, tg)

    def loss_of(p):
        return oracle.forward(shape, p, ids, tg)["loss"]

    for name, w in P.items():
        num = np.zeros_like(w)
        for idx in np.ndindex(*w.shape):
            hstep = 1e-5 * max(1.0, abs(w[idx]))
            orig = w[idx]
            w[idx] = orig + hstep
            lp = loss_of(P)
            w[idx] = orig - hstep
            lm = loss_of(P)
            w[idx] = orig
            num[idx] = (lp - lm) / (2 * hstep)
        err = np.abs(num - grads[name])
        tol = np.maximum(1e-9, 1e-6 * np.abs(num))
        assert np.all(err <= tol), (name, float(err.max()))


# ------------------------------------------------------------------ pages' arithmetic
def test_pages_depth20_arithmetic():
    from pretraining_step_pretrain_b300 import flops
    g = json.load(open(os.path.join(GOLDEN, "pages_d20_run.json")))
    s = nc_synth.shape_from_depth(g["depth"])
    assert (s.d_model, s.n_head, s.head_dim) == (g["channels"], g["heads"], g["head_dim"])
    assert g["rows_per_gpu"] * g["tokens_per_row"] * g["gpus"] == g["tokens_per_step"] == 2 ** 19
    n_mha = flops.n_params(s, n_kv_head=s.n_head)
    assert abs(n_mha / g["params_approx"] - 1) < 0.01
    assert abs(20 * n_mha / g["tokens_total_approx"] - 1) < 0.01
    assert abs(g["tokens_total_approx"] / g["tokens_per_step"] / g["iterations_approx"] - 1) < 0.01
    total = flops.flops_per_token(s, g["tokens_per_row"], n_kv_head=s.n_head) * g["tokens_total_approx"]
    assert abs(total / g["flops_total_approx"] - 1) < 0.05
    assert abs(flops.n_params(s) / 502.0e6 - 1) < 0.001            # MQA, as built


# ---------------------------------------------------------------- evaluation
def test_eval_bpb_closed_form_zero_head():
    """Zero LM head: every token's loss is ln V, so bpb = n ln V / (ln 2 sum
    bytes) exactly; tokens of byte length 0 drop out of both sums."""
    shape = nc_synth.TINY.shape
    ids, tg = nc_synth.make_tokens(shape.vocab, 2, 16, seed=3, dist="uniform")
    w = nc_synth.make_weights(shape, seed=1, bf16=False, zero=("w_lm",))
    P = {k: v.astype(np.float64) for k, v in w.items()}
    rng = np.random.default_rng(0)
    nbytes = rng.integers(1, 7, size=shape.vocab)
    nbytes[:5] = 0
    loss, bpb = oracle.evaluate(shape, P, ids, tg, nbytes)
    lnv = math.log(shape.vocab)
    assert loss == pytest.approx(lnv, rel=1e-12)
    y = tg.reshape(-1)
    keep = nbytes[y] > 0
    assert bpb == pytest.approx(keep.sum() * lnv / (math.log(2) * nbytes[y].sum()), rel=1e-12)


def test_eval_loss_equals_training_loss_and_one_byte_tokens_give_bits_per_token():
    shape = nc_synth.TINY.shape
    ids, tg = nc_synth.make_tokens(shape.vocab, 2, 16, seed=4, dist="uniform")
    tg[0, :3] = -1
    w = nc_synth.make_weights(shape, seed=2, bf16=False)
    P = {k: v.astype(np.float64) for k, v in w.items()}
    loss, bpb = oracle.evaluate(shape, P, ids, tg, np.ones(shape.vocab, dtype=np.int64))
    train = oracle.forward(shape, P, ids, tg)["loss"]
    assert loss == pytest.approx(train, rel=1e-12)
    assert bpb == pytest.approx(loss / math.log(2), rel=1e-12)
    assert oracle.evaluate(shape, P, ids, tg)[1] is None
