"""Parameter and FLOP accounting for the nanochat-style step.

Model FLOPs per token follow the usual 6N + attention convention: every matrix
parameter costs 6 FLOPs per token (2 forward, 4 backward) and attention adds
12 * L * H * h * T (QK^T and PV, forward and backward, with the masked half of
the causal square counted).  This is the accounting under which the imeisheng.com
walkthrough's figures for the depth-20 run come out (section "预训练": about
4e19 FLOPs for about 11.2B tokens, MFU near one half at about 0.5 s per
524,288-token step on eight H100s).  The embedding lookup costs no FLOPs; the
unembedding (LM head) is counted.
"""
from __future__ import annotations


def block_params(shape, n_kv_head: int = 1) -> int:
    d, H, h, f = shape.d_model, shape.n_head, shape.head_dim, shape.d_mlp
    return d * H * h + 2 * d * n_kv_head * h + H * h * d + 2 * d * f


def n_params(shape, n_kv_head: int = 1) -> int:
    """All trainable parameters: blocks + untied embedding + LM head."""
    return shape.depth * block_params(shape, n_kv_head) + 2 * shape.vocab * shape.d_model


def flops_per_token(shape, seq: int, causal_actual: bool = False, n_kv_head: int = 1) -> float:
    L, H, h, V, d = shape.depth, shape.n_head, shape.head_dim, shape.vocab, shape.d_model
    dense = 6 * (L * block_params(shape, n_kv_head) + V * d)
    attn = (6 if causal_actual else 12) * L * H * h * seq
    return float(dense + attn)


def optimizer_cost(shape, ns_steps: int = 5) -> tuple[float, float]:
    """(Newton-Schulz FLOPs, AdamW bytes) of one optimizer step.

    Each block matrix (r x c, wide orientation m = min, n = max) costs, per
    Newton-Schulz step, 2 m^2 n (A = X X^T) + 2 m^3 (A A) + 2 m^2 n (B X).
    AdamW reads the master, gradient and both moments (fp32) and writes the
    master, both moments and the bf16 compute copy: 30 bytes per element of
    the embedding and of the LM head."""
    d, H, h, f = shape.d_model, shape.n_head, shape.head_dim, shape.d_mlp
    mats = [((H + 2) * h, d), (d, H * h), (f, d), (d, f)]
    per_layer = 0
    for r, c in mats:
        m, n = min(r, c), max(r, c)
        per_layer += ns_steps * (4 * m * m * n + 2 * m ** 3)
    return float(shape.depth * per_layer), float(2 * shape.vocab * d * 30)
