"""CPU-only checks of the C-ABI library: it loads, exports every function that
include/nc.h declares, and rejects bad arguments on the host before any
launch (no GPU needed: validation returns before the first CUDA call)."""
import ctypes
import os
import re

import pytest

import nc_synth
from pretraining_step_pretrain_b300 import build, nc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return nc.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "nc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nc_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(nc.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def _cfg(shape=nc_synth.SMALL.shape, dtype="bf16", **over):
    c = nc.make_config(shape, dtype)
    for k, v in over.items():
        setattr(c, k, v)
    return c


def test_workspace_bytes_positive_and_monotone(lib):
    s = nc_synth.SMALL.shape
    a = nc.workspace_bytes(_cfg(s), 8, 256)
    b = nc.workspace_bytes(_cfg(s), 16, 256)
    assert 0 < a < b
    d20 = nc.workspace_bytes(_cfg(nc_synth.D20.shape), 32, 2048)
    assert 20e9 < d20 < 80e9          # saved activations of 20 layers + logits


@pytest.mark.parametrize("field,value", [("d_model", 100), ("head_dim", 96), ("vocab", 1000),
                                         ("d_mlp", 0), ("depth", 0), ("n_head", 0)])
def test_bad_shapes_rejected(lib, field, value):
    assert nc.workspace_bytes(_cfg(**{field: value}), 8, 256) == 0
    assert b"must" in lib.nc_last_error_message()


def test_bf16_mode_requires_head_dim_128(lib):
    assert nc.workspace_bytes(_cfg(nc_synth.TINY.shape, "bf16"), 2, 64) == 0
    assert nc.workspace_bytes(_cfg(nc_synth.TINY.shape, "f32"), 2, 64) > 0


def test_step_rejects_null_and_misaligned_pointers_before_launch(lib):
    cfg = _cfg()
    B, T = 8, 256
    need = nc.workspace_bytes(cfg, B, T)
    L = cfg.depth
    layers = (nc.NcLayerW * L)(*[nc.NcLayerW(4096, 4096, 4096, 4096) for _ in range(L)])
    grads = (nc.NcLayerG * L)(*[nc.NcLayerG(4096, 4096, 4096, 4096) for _ in range(L)])
    f = lib.nc_step
    # null ids
    st = f(ctypes.byref(cfg), B, T, None, 4096, 4096, layers, 4096, 4096, 4096, grads, 4096, 0,
           4096, need, None)
    assert st == 1 and b"null" in lib.nc_last_error_message()
    # misaligned weight
    st = f(ctypes.byref(cfg), B, T, 4096, 4096, 4100, layers, 4096, 4096, 4096, grads, 4096, 0,
           4096, need, None)
    assert st == 1 and b"aligned" in lib.nc_last_error_message()
    # short workspace
    st = f(ctypes.byref(cfg), B, T, 4096, 4096, 4096, layers, 4096, 4096, 4096, grads, 4096, 0,
           4096, need - 1, None)
    assert st == 3
    # bad layer pointer
    layers[1].w_fc = 0
    st = f(ctypes.byref(cfg), B, T, 4096, 4096, 4096, layers, 4096, 4096, 4096, grads, 4096, 0,
           4096, need, None)
    assert st == 1 and b"layer 1" in lib.nc_last_error_message()


def test_block_calls_reject_bad_layer_index(lib):
    cfg = _cfg()
    need = nc.workspace_bytes(cfg, 8, 256)
    w = nc.NcLayerW(4096, 4096, 4096, 4096)
    st = lib.nc_block_fwd(ctypes.byref(cfg), cfg.depth, 8, 256, ctypes.byref(w), 4096, 4096,
                          need, None)
    assert st == 1 and b"layer" in lib.nc_last_error_message()


def test_gemm_argument_checks(lib):
    f = lib.nc_gemm
    assert f(0, 0, 0, 128, 100, 64, 4096, 64, 4096, 64, 4096, 128, None, 0, 4096, 1 << 20, None) == 2
    assert f(0, 2, 0, 300, 128, 64, 4096, 300, 4096, 128, 4096, 128, None, 0, 4096, 1 << 20, None) == 2
    assert f(0, 7, 0, 128, 128, 64, 4096, 64, 4096, 64, 4096, 128, None, 0, 4096, 1 << 20, None) == 1
    assert f(0, 0, 9, 128, 128, 64, 4096, 64, 4096, 64, 4096, 128, None, 0, 4096, 1 << 20, None) == 1
    assert f(0, 0, 0, 128, 128, 64, 4096, 60, 4096, 64, 4096, 128, None, 0, 4096, 1 << 20, None) == 2
    # relu2-bwd needs its aux operand
    assert f(0, 0, 4, 128, 128, 64, 4096, 64, 4096, 64, 4096, 128, None, 0, 4096, 1 << 20, None) == 1


def test_fp8_gemm_argument_checks(lib):
    f = lib.nc_gemm_fp8
    # M N K A lda B ldb out C ldc scale ws ws_bytes stream
    assert f(128, 128, 24, 4096, 32, 4096, 32, 0, 4096, 128, 1.0, 4096, 1 << 20, None) == 2  # K % 16
    assert f(128, 100, 64, 4096, 64, 4096, 64, 0, 4096, 128, 1.0, 4096, 1 << 20, None) == 2  # N % 32
    assert f(128, 128, 64, 4096, 72, 4096, 64, 0, 4096, 128, 1.0, 4096, 1 << 20, None) == 2  # lda % 16
    assert f(128, 128, 64, 4096, 48, 4096, 64, 0, 4096, 128, 1.0, 4096, 1 << 20, None) == 2  # lda < K
    assert f(128, 128, 64, 4096, 64, 4096, 64, 5, 4096, 128, 1.0, 4096, 1 << 20, None) == 1  # out dtype
    assert f(128, 128, 64, 4096, 64, 4096, 64, 0, 4096, 128, float("inf"), 4096, 1 << 20,
             None) == 1                                                                       # scale
    assert f(128, 128, 64, 4104, 64, 4096, 64, 0, 4096, 128, 1.0, 4096, 1 << 20, None) == 1  # misaligned
    assert f(128, 128, 64, 4096, 64, 4096, 64, 0, 4096, 128, 1.0, 4096, 16, None) == 3       # tiny ws


def test_attention_argument_checks(lib):
    f = lib.nc_attention_fwd
    assert f(0, 1, 64, 2, 64, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 20, None) == 2  # bf16 h=64
    assert f(1, 0, 64, 2, 64, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 20, None) == 2  # B = 0
    assert f(1, 1, 64, 2, 64, 4096, 4096, 4096, 4096, 4096, 4096, 16, None) == 3       # tiny ws


def test_status_strings(lib):
    for k, v in nc.STATUS.items():
        assert lib.nc_status_string(k).decode() == v
