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
