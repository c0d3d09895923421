"""fp64 CPU oracle of the nanochat-style pretraining step (forward + backward).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA path.

The computation is the plain definition, in float64 with numpy, of the model
listed in the launch article's Q&A ("安德烈·卡帕西推出nanochat…", vpshk.cn,
section "卡帕西亲自揭秘背后技术", architecture list):

  * dense decoder, Llama-like pre-norm residual stream;
  * rotary position embeddings, no learned positions;
  * QK norm (RMSNorm of every query head and of the key head);
  * untied token embedding and unembedding;
  * a norm right after the token embedding;
  * ReLU^2 MLP;
  * RMSNorm without learnable parameters;
  * bias-free linear layers;
  * multi-query attention (one K/V head shared by all query heads);
  * logit softcap at the output.

The objective is next-token prediction (imeisheng.com walkthrough
"100美元成本、8000行代码纯手搓克隆ChatGPT", section "预训练").  Constants the
pages do not give (softcap 15, RoPE base 10000, eps 1e-6, MLP width 4d, the
RoPE pairing) are readings, each noted where it is used.

Weights use the (out, in) layout: y = x @ W.T.  Activations are (B, T, ...).
Random numbers are never drawn here; callers pass the arrays.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Parameter-free RMSNorm (architecture list: RMSNorm carries no learnable gain).
# Reading: y = x / sqrt(mean(x^2) + eps), eps = 1e-6, over the last axis.
# --------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, eps: float) -> tuple[np.ndarray, np.ndarray]:
    """Return (y, r) with y = x * r and r = 1/sqrt(mean(x^2) + eps) (keepdims)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(ms + eps)
    return x * r, r


def rmsnorm_bwd(dy: np.ndarray, x: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Gradient of y = x * r(x) w.r.t. x, written from the chain rule.

    dr/dx_j = -r^3 x_j / d, so dx_j = r dy_j - (r^3 / d) x_j sum_i dy_i x_i.
    """
    d = x.shape[-1]
    dot = np.sum(dy * x, axis=-1, keepdims=True)
    return r * dy - (r ** 3 / d) * x * dot


# --------------------------------------------------------------------------
# Rotary embeddings (architecture list: rotary, no positional embeddings).
# Reading: half-split pairs (i, i + h/2), theta_i = base^(-2i/h), angle t*theta_i
# for token position t = 0..T-1 within each row.
# --------------------------------------------------------------------------
def rope_tables(T: int, h: int, base: float) -> tuple[np.ndarray, np.ndarray]:
    i = np.arange(h // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / h)
    ang = np.arange(T, dtype=np.float64)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)            # (T, h/2) each


def rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate x (..., T, [heads,] h) given tables broadcastable to (..., T, [1,] h/2)."""
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x1 * sin + x2 * cos], axis=-1)


def rope_bwd(dy: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Transpose of the rotation: rotate dy by the negated angle."""
    half = dy.shape[-1] // 2
    d1, d2 = dy[..., :half], dy[..., half:]
    return np.concatenate([d1 * cos + d2 * sin, -d1 * sin + d2 * cos], axis=-1)


# --------------------------------------------------------------------------
# Causal multi-query attention.  q: (B, T, H, h); k, v: (B, T, h) -- one K/V
# head shared by every query head.  Reading: scale 1/sqrt(h), key j visible to
# query i iff j <= i (next-token objective), no dropout.
# --------------------------------------------------------------------------
def _causal_scores(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    h = q.shape[-1]
    T = q.shape[1]
    s = np.einsum("bthd,bjd->bhtj", q, k, optimize=True) / np.sqrt(h)
    future = np.triu(np.ones((T, T), dtype=bool), k=1)      # j > i
    return np.where(future[None, None], -np.inf, s)


def _softmax(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    p = _softmax(_causal_scores(q, k))                      # (B, H, T, T)
    return np.einsum("bhtj,bjd->bthd", p, v, optimize=True)


def attention_bwd(do: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """Gradients (dq, dk, dv); dk and dv sum over all query heads (MQA)."""
    h = q.shape[-1]
    p = _softmax(_causal_scores(q, k))
    dv = np.einsum("bhtj,bthd->bjd", p, do, optimize=True)
    dp = np.einsum("bthd,bjd->bhtj", do, v, optimize=True)
    ds = p * (dp - np.sum(dp * p, axis=-1, keepdims=True))
    dq = np.einsum("bhtj,bjd->bthd", ds, k, optimize=True) / np.sqrt(h)
    dk = np.einsum("bhtj,bthd->bjd", ds, q, optimize=True) / np.sqrt(h)
    return dq, dk, dv


# --------------------------------------------------------------------------
# Logit softcap (architecture list: softcap on the output logits).  Reading: s = c tanh(z/c),
# c = 15.
# --------------------------------------------------------------------------
def softcap(z: np.ndarray, c: float) -> np.ndarray:
    return c * np.tanh(z / c)


def softcap_bwd(ds: np.ndarray, s: np.ndarray, c: float) -> np.ndarray:
    return ds * (1.0 - (s / c) ** 2)


# --------------------------------------------------------------------------
# Next-token cross-entropy, mean over targets >= 0 (ignore index -1).
# --------------------------------------------------------------------------
def cross_entropy(s: np.ndarray, y: np.ndarray) -> tuple[float, np.ndarray]:
    """Return (loss, ds) for logits s (N, V) and targets y (N,)."""
    valid = y >= 0
    n = max(int(valid.sum()), 1)
    m = np.max(s, axis=-1, keepdims=True)
    lse = (m + np.log(np.sum(np.exp(s - m), axis=-1, keepdims=True)))[:, 0]
    rows = np.nonzero(valid)[0]
    loss = float(np.sum(lse[rows] - s[rows, y[rows]]) / n)
    p = np.exp(s - lse[:, None])
    ds = p.copy()
    ds[rows, y[rows]] -= 1.0
    ds[~valid] = 0.0
    return loss, ds / n


# --------------------------------------------------------------------------
# Whole step.
# --------------------------------------------------------------------------
def _w(params: dict, name: str) -> np.ndarray:
    return np.asarray(params[name], dtype=np.float64)


def forward(shape, params: dict, ids: np.ndarray, targets: np.ndarray | None = None):
    """Forward pass.  Returns a cache dict holding every activation and, when
    targets are given, 'loss'.  `shape` carries depth, d_model, n_head,
    head_dim, d_mlp, vocab, softcap, rope_base, eps."""
    B, T = ids.shape
    L, H, h = shape.depth, shape.n_head, shape.head_dim
    eps, c = shape.eps, shape.softcap
    cos, sin = rope_tables(T, h, shape.rope_base)
    cache = {"ids": ids, "cos": cos, "sin": sin, "layers": []}

    x0 = _w(params, "wte")[ids]                              # (B, T, d) embedding
    x, r0 = rmsnorm(x0, eps)                                 # norm after embedding
    cache.update(x0=x0, r0=r0, x_embed=x)
    for l in range(L):
        lc = {"x_in": x}
        xn, r1 = rmsnorm(x, eps)
        qkv = xn @ _w(params, f"w_qkv.{l}").T                # bias-free
        q = qkv[..., : H * h].reshape(B, T, H, h)
        k = qkv[..., H * h: H * h + h]
        v = qkv[..., H * h + h:]
        qn, rq = rmsnorm(q, eps)                             # QK norm, per head
        kn, rk = rmsnorm(k, eps)
        qr = rope(qn, cos[None, :, None, :], sin[None, :, None, :])
        kr = rope(kn, cos[None], sin[None])
        o = attention(qr, kr, v).reshape(B, T, H * h)
        x_mid = x + o @ _w(params, f"w_o.{l}").T             # residual add
        xn2, r2 = rmsnorm(x_mid, eps)
        u = xn2 @ _w(params, f"w_fc.{l}").T
        a = np.maximum(u, 0.0) ** 2                          # ReLU^2
        x = x_mid + a @ _w(params, f"w_proj.{l}").T          # residual add
        lc.update(xn=xn, r1=r1, q=q, k=k, v=v, qn=qn, rq=rq, kn=kn, rk=rk,
                  qr=qr, kr=kr, o=o, x_mid=x_mid, xn2=xn2, r2=r2, u=u, a=a)
        cache["layers"].append(lc)
    xf, rf = rmsnorm(x, eps)
    z = xf @ _w(params, "w_lm").T                            # untied unembedding
    s = softcap(z, c)
    cache.update(x_out=x, xf=xf, rf=rf, z=z, s=s)
    if targets is not None:
        loss, ds = cross_entropy(s.reshape(B * T, -1), targets.reshape(-1))
        cache.update(loss=loss, ds=ds.reshape(B, T, -1))
    return cache


def evaluate(shape, params: dict, ids: np.ndarray, targets: np.ndarray,
             token_bytes: np.ndarray | None = None) -> tuple[float, float | None]:
    """Forward-only evaluation: (mean next-token loss in nats over targets >= 0,
    bits per byte or None).

    Walkthrough, section "预训练": the run reports validation bits per byte,
    the per-token loss normalised by the bytes each token stands for so that
    it does not depend on the tokenizer.  `token_bytes[v]` is the byte length
    of token v.  Reading: tokens of byte length 0 (special tokens) are left
    out of both sums; bpb = sum(loss_t) / (ln 2 * sum(bytes(y_t))).
    """
    cache = forward(shape, params, ids)
    s = cache["s"].reshape(-1, shape.vocab)
    y = targets.reshape(-1)
    rows = np.nonzero(y >= 0)[0]
    m = np.max(s[rows], axis=-1, keepdims=True)
    lse = (m + np.log(np.sum(np.exp(s[rows] - m), axis=-1, keepdims=True)))[:, 0]
    nats = lse - s[rows, y[rows]]
    loss = float(nats.sum() / max(rows.size, 1))
    if token_bytes is None:
        return loss, None
    nb = np.asarray(token_bytes, dtype=np.int64)[y[rows]]
    keep = nb > 0
    total = int(nb[keep].sum())
    bpb = float(nats[keep].sum() / (np.log(2.0) * total)) if total > 0 else float("nan")
    return loss, bpb


def backward(shape, params: dict, cache: dict) -> dict:
    """Hand-derived backward of `forward`; returns d(loss)/d(every weight)."""
    ids = cache["ids"]
    B, T = ids.shape
    L, H, h, c = shape.depth, shape.n_head, shape.head_dim, shape.softcap
    cos, sin = cache["cos"], cache["sin"]
    grads = {}

    dz = softcap_bwd(cache["ds"], cache["s"], c)              # (B, T, V)
    xf = cache["xf"]
    grads["w_lm"] = dz.reshape(B * T, -1).T @ xf.reshape(B * T, -1)
    dxf = dz @ _w(params, "w_lm")
    dx = rmsnorm_bwd(dxf, cache["x_out"], cache["rf"])
    for l in reversed(range(L)):
        lc = cache["layers"][l]
        # x_out = x_mid + a @ Wproj.T,  a = relu(u)^2,  u = norm(x_mid) @ Wfc.T
        grads[f"w_proj.{l}"] = dx.reshape(B * T, -1).T @ lc["a"].reshape(B * T, -1)
        da = dx @ _w(params, f"w_proj.{l}")
        du = da * 2.0 * np.maximum(lc["u"], 0.0)
        grads[f"w_fc.{l}"] = du.reshape(B * T, -1).T @ lc["xn2"].reshape(B * T, -1)
        dxn2 = du @ _w(params, f"w_fc.{l}")
        dx = dx + rmsnorm_bwd(dxn2, lc["x_mid"], lc["r2"])
        # x_mid = x_in + o @ Wo.T
        grads[f"w_o.{l}"] = dx.reshape(B * T, -1).T @ lc["o"].reshape(B * T, -1)
        do = (dx @ _w(params, f"w_o.{l}")).reshape(B, T, H, h)
        dqr, dkr, dv = attention_bwd(do, lc["qr"], lc["kr"], lc["v"])
        dqn = rope_bwd(dqr, cos[None, :, None, :], sin[None, :, None, :])
        dkn = rope_bwd(dkr, cos[None], sin[None])
        dq = rmsnorm_bwd(dqn, lc["q"], lc["rq"])
        dk = rmsnorm_bwd(dkn, lc["k"], lc["rk"])
        dqkv = np.concatenate([dq.reshape(B, T, H * h), dk, dv], axis=-1)
        grads[f"w_qkv.{l}"] = dqkv.reshape(B * T, -1).T @ lc["xn"].reshape(B * T, -1)
        dxn = dqkv @ _w(params, f"w_qkv.{l}")
        dx = dx + rmsnorm_bwd(dxn, lc["x_in"], lc["r1"])
    dx0 = rmsnorm_bwd(dx, cache["x0"], cache["r0"])
    dwte = np.zeros_like(_w(params, "wte"))
    np.add.at(dwte, ids.reshape(-1), dx0.reshape(B * T, -1))
    grads["wte"] = dwte
    return grads


def step(shape, params: dict, ids: np.ndarray, targets: np.ndarray):
    """One forward + backward: returns (loss, grads)."""
    cache = forward(shape, params, ids, targets)
    return cache["loss"], backward(shape, params, cache)
