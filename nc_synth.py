"""Seeded synthetic inputs for the nanochat-style pretraining step.

This module is shared by the tests, the bench and the oracle's callers.  It
holds model *shapes* and *random draws* only -- none of the step's arithmetic
(no norm, no attention, no loss).  Both the CUDA path and the CPU oracle are
fed the exact arrays produced here.

Shapes follow the nanochat description: depth d sets the width as 64 * depth
channels with 128-wide heads (the launch article on vpshk.cn, Karpathy Q&A
"卡帕西亲自揭秘背后技术": dense Transformer, MQA; the imeisheng.com walkthrough,
section "预训练": depth 20 -> 1280 channels, 10 heads of dim 128, 32 rows x 2048
tokens per device forward/backward).  The pretraining corpus (FineWeb-EDU) is
not available here; token ids are drawn from a truncated Zipf law (s = 1.1)
as a stand-in for natural-text token frequencies.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class ModelShape:
    depth: int          # L, number of transformer blocks
    d_model: int        # d, residual width
    n_head: int         # H, query heads (one shared K/V head: MQA)
    head_dim: int       # h
    d_mlp: int          # f, MLP hidden width (ReLU^2)
    vocab: int          # V
    softcap: float = 15.0
    rope_base: float = 10000.0
    eps: float = 1e-6

    @property
    def qkv_dim(self) -> int:
        return (self.n_head + 2) * self.head_dim


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    batch: int
    seq: int
    dtype: str          # "f32" (debug/parity mode) or "bf16"
    ids: str            # "uniform" or "zipf"


def shape_from_depth(depth: int, vocab: int = 65536) -> ModelShape:
    """d_model = 64 * depth, heads of 128 (depth 20 -> 1280 / 10 x 128)."""
    d = 64 * depth
    return ModelShape(depth=depth, d_model=d, n_head=d // 128, head_dim=128,
                      d_mlp=4 * d, vocab=vocab)


TINY = Workload("tiny_f32", ModelShape(2, 128, 2, 64, 512, 512), 2, 64, "f32", "uniform")
SMALL = Workload("small_bf16", ModelShape(4, 256, 2, 128, 1024, 4096), 8, 256, "bf16", "zipf")
D20 = Workload("d20_bf16", shape_from_depth(20), 32, 2048, "bf16", "zipf")
D30 = Workload("d30_bf16", shape_from_depth(30), 16, 2048, "bf16", "zipf")
D20_LONG = Workload("d20_long_bf16", shape_from_depth(20), 4, 8192, "bf16", "zipf")
WORKLOADS = {w.name: w for w in (TINY, SMALL, D20, D30, D20_LONG)}

# Gradient-check shape (tiny enough for central differences on every entry).
GRADCHECK = ModelShape(depth=2, d_model=16, n_head=2, head_dim=8, d_mlp=64, vocab=32)


def zipf_probs(vocab: int, s: float = 1.1) -> np.ndarray:
    k = np.arange(1, vocab + 1, dtype=np.float64)
    p = k ** (-s)
    return p / p.sum()


def make_tokens(vocab: int, batch: int, seq: int, seed: int = 0,
                dist: str = "zipf") -> tuple[np.ndarray, np.ndarray]:
    """Draw a (batch, seq+1) int32 stream; inputs are [:, :seq], targets [:, 1:]."""
    rng = np.random.default_rng(seed)
    if dist == "uniform":
        stream = rng.integers(0, vocab, size=(batch, seq + 1), dtype=np.int64)
    elif dist == "zipf":
        stream = rng.choice(vocab, size=(batch, seq + 1), p=zipf_probs(vocab))
    else:
        raise ValueError(dist)
    stream = stream.astype(np.int32)
    return np.ascontiguousarray(stream[:, :seq]), np.ascontiguousarray(stream[:, 1:])


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), kept as float32."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def weight_shapes(shape: ModelShape) -> dict[str, tuple[int, int]]:
    """Row-major (out, in) shapes, y = x @ W.T.  Per-layer names carry a .{l} suffix."""
    d, H, h, f, V = shape.d_model, shape.n_head, shape.head_dim, shape.d_mlp, shape.vocab
    out = {"wte": (V, d)}
    for l in range(shape.depth):
        out[f"w_qkv.{l}"] = ((H + 2) * h, d)
        out[f"w_o.{l}"] = (d, H * h)
        out[f"w_fc.{l}"] = (f, d)
        out[f"w_proj.{l}"] = (d, f)
    out["w_lm"] = (V, d)
    return out


def make_weights(shape: ModelShape, seed: int = 1, bf16: bool = True,
                 zero: tuple[str, ...] = ()) -> dict[str, np.ndarray]:
    """N(0, 1/fan_in) for every linear map, N(0, 1) for the embedding.

    `zero` lists weight families ("w_lm", "w_o", "w_proj", ...) set to exactly 0
    (the zero-init variants).  Values are float32 arrays, already rounded to
    bfloat16 when `bf16` is set, so both sides see the same numbers.
    """
    rng = np.random.default_rng(seed)
    out = {}
    for name, (rows, cols) in weight_shapes(shape).items():
        family = name.split(".")[0]
        std = 1.0 if family == "wte" else 1.0 / math.sqrt(cols)
        w = rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(std)
        if family in zero:
            w[:] = 0.0
        out[name] = round_to_bf16(w) if bf16 else w
    return out


def make_e4m3_codes(rows: int, cols: int, seed: int, exp_lo: int = 3, exp_hi: int = 10):
    """Random 8-bit codes laid out as s.eeee.mmm (uint8, (rows, cols)): sign and
    mantissa fields uniform, exponent field uniform in [exp_lo, exp_hi], so no
    code is NaN and the magnitudes stay within a few powers of two of 1.  Bit
    fields only -- the values the codes stand for are the oracle's business."""
    rng = np.random.default_rng(seed)
    s = rng.integers(0, 2, size=(rows, cols), dtype=np.uint8)
    e = rng.integers(exp_lo, exp_hi + 1, size=(rows, cols), dtype=np.uint8)
    m = rng.integers(0, 8, size=(rows, cols), dtype=np.uint8)
    return (s << 7) | (e << 3) | m


def make_e4m3_codes_full(rows: int, cols: int, seed: int):
    """Random 8-bit codes over the whole code space except the two NaN codes
    (s.1111.111): zeros of both signs, subnormals (exponent field 0), and the
    largest magnitudes (s.1111.110) all occur.  Bit fields only."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    nan = (c & 0x7F) == 0x7F
    while nan.any():
        c[nan] = rng.integers(0, 256, size=int(nan.sum()), dtype=np.uint8)
        nan = (c & 0x7F) == 0x7F
    return c
