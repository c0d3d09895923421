"""Thin Python binding of libnc.so (include/nc.h).

Argument marshalling only: every function passes torch device pointers, the
current CUDA stream and plain integers straight to the C ABI.  All arithmetic
of the step runs in the library's CUDA kernels.  If libnc.so is missing or a
call fails, an exception is raised -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnc.so")

NC_BF16, NC_F32 = 0, 1
GEMM_NT, GEMM_NN, GEMM_TN = 0, 1, 2
EPI_STORE, EPI_STORE_F32, EPI_ADD_F32, EPI_RELU2, EPI_RELU2_BWD = 0, 1, 2, 3, 4
EPI_AXPBY = 6
STATUS = {0: "NC_OK", 1: "NC_ERR_INVALID_ARG", 2: "NC_ERR_UNSUPPORTED_SHAPE",
          3: "NC_ERR_WORKSPACE", 4: "NC_ERR_CUDA", 5: "NC_ERR_TIMEOUT", 6: "NC_ERR_TOKEN_RANGE"}

# Symbols declared in include/nc.h (kept in step with the header by a test).
EXPORTS = ("nc_workspace_bytes", "nc_embed_norm", "nc_block_fwd", "nc_lmhead_softcap_ce_fwd_bwd",
           "nc_block_bwd", "nc_embed_norm_bwd", "nc_step", "nc_get_device_status",
           "nc_status_string", "nc_last_error_message", "nc_gemm_workspace_bytes", "nc_gemm",
           "nc_attention_workspace_bytes", "nc_attention_fwd", "nc_attention_bwd",
           "nc_attention_bwd_noalloc", "nc_attention_bwd_noalloc_status",
           "nc_launch_count", "nc_profile_start", "nc_profile_stop", "nc_profile_record",
           "nc_selftest_wait_timeout", "nc_gemm_batched", "nc_optimizer_workspace_bytes",
           "nc_optimizer_step", "nc_eval", "nc_gemm_fp8")


class NcConfig(ctypes.Structure):
    _fields_ = [("depth", ctypes.c_int), ("d_model", ctypes.c_int), ("n_head", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("d_mlp", ctypes.c_int), ("vocab", ctypes.c_int),
                ("softcap", ctypes.c_float), ("rope_base", ctypes.c_float),
                ("eps", ctypes.c_float), ("dtype", ctypes.c_int)]


class NcLayerW(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("w_fc", ctypes.c_void_p), ("w_proj", ctypes.c_void_p)]


class NcLayerG(ctypes.Structure):
    _fields_ = [("d_qkv", ctypes.c_void_p), ("d_o", ctypes.c_void_p),
                ("d_fc", ctypes.c_void_p), ("d_proj", ctypes.c_void_p)]


class NcLayerF(ctypes.Structure):
    """float32 per-layer matrices (master weights or Muon momentum buffers)."""
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("w_fc", ctypes.c_void_p), ("w_proj", ctypes.c_void_p)]


class NcLayerWC(ctypes.Structure):
    """Per-layer compute copies the optimizer rewrites."""
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("w_fc", ctypes.c_void_p), ("w_proj", ctypes.c_void_p)]


class NcOptConfig(ctypes.Structure):
    _fields_ = [("lr_muon", ctypes.c_float), ("momentum", ctypes.c_float),
                ("lr_embed", ctypes.c_float), ("lr_lm", ctypes.c_float),
                ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("ns_a", ctypes.c_float),
                ("ns_b", ctypes.c_float), ("ns_c", ctypes.c_float), ("ns_steps", ctypes.c_int)]


class NcError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libnc.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -m pretraining_step_pretrain_b300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        C = ctypes.POINTER(NcConfig)
        sig = {
            "nc_workspace_bytes": (S, [C, I, I]),
            "nc_embed_norm": (I, [C, I, I, P, P, P, P, S, P]),
            "nc_block_fwd": (I, [C, I, I, I, ctypes.POINTER(NcLayerW), P, P, S, P]),
            "nc_lmhead_softcap_ce_fwd_bwd": (I, [C, I, I, P, P, P, P, P, P, I, P, S, P]),
            "nc_block_bwd": (I, [C, I, I, I, ctypes.POINTER(NcLayerW), P,
                                 ctypes.POINTER(NcLayerG), I, P, S, P]),
            "nc_embed_norm_bwd": (I, [C, I, I, P, P, P, P, I, P, S, P]),
            "nc_step": (I, [C, I, I, P, P, P, ctypes.POINTER(NcLayerW), P, P, P,
                            ctypes.POINTER(NcLayerG), P, I, P, S, P]),
            "nc_get_device_status": (I, [P, P]),
            "nc_status_string": (ctypes.c_char_p, [I]),
            "nc_last_error_message": (ctypes.c_char_p, []),
            "nc_gemm_workspace_bytes": (S, [I, I, I, I, I]),
            "nc_gemm": (I, [I, I, I, I, I, I, P, I, P, I, P, I, P, I, P, S, P]),
            "nc_attention_workspace_bytes": (S, [I, I, I]),
            "nc_attention_fwd": (I, [I, I, I, I, I, P, P, P, P, P, P, S, P]),
            "nc_attention_bwd": (I, [I, I, I, I, I, P, P, P, P, P, P, P, I, P, I, P, I, P, S, P]),
            "nc_attention_bwd_noalloc": (I, [I, I, I, I, I, P, P, P, P, P, P, P, I, P, I, P, I,
                                             P]),
            "nc_attention_bwd_noalloc_status": (I, [P]),
            "nc_selftest_wait_timeout": (I, [I, P, S, P]),
            "nc_launch_count": (ctypes.c_longlong, []),
            "nc_profile_start": (I, [I]),
            "nc_profile_stop": (I, []),
            "nc_profile_record": (I, [I, ctypes.POINTER(ctypes.c_char_p),
                                      ctypes.POINTER(ctypes.c_float)]),
            "nc_gemm_batched": (I, [I, I, I, I, I, I, I, P, I, ctypes.c_long, P, I, ctypes.c_long,
                                    P, I, ctypes.c_long, P, ctypes.c_float, ctypes.c_float, P, S,
                                    P]),
            "nc_optimizer_workspace_bytes": (S, [C]),
            "nc_gemm_fp8": (I, [I, I, I, P, I, P, I, I, P, I, ctypes.c_float, P, S, P]),
            "nc_eval": (I, [C, I, I, P, P, P, P, ctypes.POINTER(NcLayerW), P, P, P, S, P]),
            "nc_optimizer_step": (I, [C, ctypes.POINTER(NcOptConfig), I, ctypes.c_float, P, P,
                                      ctypes.POINTER(NcLayerF), P, P, ctypes.POINTER(NcLayerWC),
                                      P, P, ctypes.POINTER(NcLayerG), P, P, P, P,
                                      ctypes.POINTER(NcLayerF), P, S, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise NcError(status, lib().nc_last_error_message().decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device=None) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def make_config(shape, dtype: str) -> NcConfig:
    return NcConfig(shape.depth, shape.d_model, shape.n_head, shape.head_dim, shape.d_mlp,
                    shape.vocab, shape.softcap, shape.rope_base, shape.eps,
                    NC_BF16 if dtype == "bf16" else NC_F32)


def act_dtype(dtype: str) -> torch.dtype:
    return torch.bfloat16 if dtype == "bf16" else torch.float32


# ---------------------------------------------------------------- C-ABI calls
def workspace_bytes(cfg: NcConfig, B: int, T: int) -> int:
    return lib().nc_workspace_bytes(ctypes.byref(cfg), B, T)


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """Zeroed (so the device error word starts clear), 256-byte aligned."""
    return torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)


def _ws(ws: torch.Tensor) -> tuple[int, int]:
    p = ws.data_ptr()
    off = (-p) % 256
    return p + off, ws.numel() - off


def embed_norm(cfg, B, T, ids, wte, x, ws):
    p, n = _ws(ws)
    _check(lib().nc_embed_norm(ctypes.byref(cfg), B, T, _ptr(ids), _ptr(wte), _ptr(x), p, n,
                               _stream()))


def block_fwd(cfg, layer, B, T, w: NcLayerW, x, ws):
    p, n = _ws(ws)
    _check(lib().nc_block_fwd(ctypes.byref(cfg), layer, B, T, ctypes.byref(w), _ptr(x), p, n,
                              _stream()))


def lmhead_softcap_ce_fwd_bwd(cfg, B, T, x_L, w_lm, targets, loss, dx_L, dw_lm, accumulate, ws):
    p, n = _ws(ws)
    _check(lib().nc_lmhead_softcap_ce_fwd_bwd(ctypes.byref(cfg), B, T, _ptr(x_L), _ptr(w_lm),
                                              _ptr(targets), _ptr(loss), _ptr(dx_L), _ptr(dw_lm),
                                              int(accumulate), p, n, _stream()))


def block_bwd(cfg, layer, B, T, w: NcLayerW, dx, g: NcLayerG, accumulate, ws):
    p, n = _ws(ws)
    _check(lib().nc_block_bwd(ctypes.byref(cfg), layer, B, T, ctypes.byref(w), _ptr(dx),
                              ctypes.byref(g), int(accumulate), p, n, _stream()))


def embed_norm_bwd(cfg, B, T, ids, wte, dx, dwte, accumulate, ws):
    p, n = _ws(ws)
    _check(lib().nc_embed_norm_bwd(ctypes.byref(cfg), B, T, _ptr(ids), _ptr(wte), _ptr(dx),
                                   _ptr(dwte), int(accumulate), p, n, _stream()))


def step(cfg, B, T, ids, targets, wte, layers, w_lm, loss, dwte, grads, dw_lm, accumulate, ws):
    p, n = _ws(ws)
    _check(lib().nc_step(ctypes.byref(cfg), B, T, _ptr(ids), _ptr(targets), _ptr(wte), layers,
                         _ptr(w_lm), _ptr(loss), _ptr(dwte), grads, _ptr(dw_lm),
                         int(accumulate), p, n, _stream()))


def get_device_status(ws) -> int:
    p, _ = _ws(ws)
    return lib().nc_get_device_status(p, _stream())


def gemm_fp8(M, N, K, A, lda, B, ldb, C, ldc, scale=1.0, ws=None):
    """C = scale * A B^T on E4M3 operands given as uint8 tensors of codes (see
    nc_gemm_fp8); C's dtype (bfloat16 or float32) selects the output type."""
    import torch
    out = NC_F32 if C.dtype == torch.float32 else NC_BF16
    if ws is None:
        ws = alloc_workspace(256, A.device)
    p, n = _ws(ws)
    _check(lib().nc_gemm_fp8(M, N, K, _ptr(A), lda, _ptr(B), ldb, out, _ptr(C), ldc,
                             float(scale), p, n, _stream()))
    return ws


def gemm(dtype, layout, epilogue, M, N, K, A, lda, B, ldb, C, ldc, aux=None, accumulate=0,
         ws=None):
    L = lib()
    need = L.nc_gemm_workspace_bytes(dtype, layout, M, N, K)
    if ws is None:
        ws = alloc_workspace(need, A.device)
    p, n = _ws(ws)
    _check(L.nc_gemm(dtype, layout, epilogue, M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                     _ptr(aux), int(accumulate), p, n, _stream()))
    return ws


def gemm_batched(dtype, layout, epilogue, batch, M, N, K, A, lda, a_bstride, B, ldb, b_bstride,
                 C, ldc, c_bstride, aux=None, alpha=0.0, beta=1.0, ws=None):
    if ws is None:
        ws = alloc_workspace(256, A.device)
    p, n = _ws(ws)
    _check(lib().nc_gemm_batched(dtype, layout, epilogue, batch, M, N, K, _ptr(A), lda, a_bstride,
                                 _ptr(B), ldb, b_bstride, _ptr(C), ldc, c_bstride, _ptr(aux),
                                 float(alpha), float(beta), p, n, _stream()))
    return ws


def attention_fwd(dtype, B, T, H, h, q, k, v, o, lse, ws=None):
    L = lib()
    if ws is None:
        ws = alloc_workspace(L.nc_attention_workspace_bytes(B, T, H), q.device)
    p, n = _ws(ws)
    _check(L.nc_attention_fwd(dtype, B, T, H, h, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              p, n, _stream()))
    return ws


def attention_bwd(dtype, B, T, H, h, q, k, v, o, lse, dout, dq, ldq, dk, ldk, dv, ldv, ws=None):
    L = lib()
    if ws is None:
        ws = alloc_workspace(L.nc_attention_workspace_bytes(B, T, H), q.device)
    p, n = _ws(ws)
    _check(L.nc_attention_bwd(dtype, B, T, H, h, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              _ptr(dout), _ptr(dq), ldq, _ptr(dk), ldk, _ptr(dv), ldv, p, n,
                              _stream()))
    return ws


def attention_bwd_noalloc(dtype, B, T, H, h, q, k, v, o, lse, dout, dq, ldq, dk, ldk, dv, ldv):
    """nc_attention_bwd without a workspace: its scratch is a fixed device
    array inside the library (B*T*H <= 2^21; calls must not overlap)."""
    _check(lib().nc_attention_bwd_noalloc(dtype, B, T, H, h, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                          _ptr(lse), _ptr(dout), _ptr(dq), ldq, _ptr(dk), ldk,
                                          _ptr(dv), ldv, _stream()))


def attention_bwd_noalloc_status() -> int:
    """Read and clear the device error word of the allocation-free calls
    (synchronises the current stream); returns the nc_status value."""
    return lib().nc_attention_bwd_noalloc_status(_stream())


def launch_count() -> int:
    return lib().nc_launch_count()


def profile_start(max_records: int) -> None:
    _check(lib().nc_profile_start(max_records))


def profile_stop() -> list[tuple[str, float]]:
    """Stop recording; return [(launch-group name, ms)] in launch order."""
    L = lib()
    n = L.nc_profile_stop()
    out = []
    name, ms = ctypes.c_char_p(), ctypes.c_float()
    for i in range(n):
        _check(L.nc_profile_record(i, ctypes.byref(name), ctypes.byref(ms)))
        out.append((name.value.decode(), ms.value))
    return out


def selftest_wait_timeout(timeout_us: int, ws) -> None:
    """ws None: record into the allocation-free calls' error word."""
    p, n = _ws(ws) if ws is not None else (None, 0)
    _check(lib().nc_selftest_wait_timeout(timeout_us, p, n, _stream()))


# ---------------------------------------------------------------- convenience
class Step:
    """Device-resident weights, gradients and workspace for repeated nc_step
    calls on one (shape, dtype, B, T)."""

    def __init__(self, shape, dtype: str, B: int, T: int, weights: dict, device="cuda"):
        self.shape, self.dtype, self.B, self.T = shape, dtype, B, T
        self.device = torch.device(device)
        self.cfg = make_config(shape, dtype)
        adt = act_dtype(dtype)
        self.w = {k: torch.as_tensor(v).to(device=self.device, dtype=adt).contiguous()
                  for k, v in weights.items()}
        self.g = {k: torch.zeros(v.shape, dtype=torch.float32, device=self.device)
                  for k, v in self.w.items()}
        L = shape.depth
        self.layers = (NcLayerW * L)(*[NcLayerW(self.w[f"w_qkv.{l}"].data_ptr(),
                                                self.w[f"w_o.{l}"].data_ptr(),
                                                self.w[f"w_fc.{l}"].data_ptr(),
                                                self.w[f"w_proj.{l}"].data_ptr())
                                       for l in range(L)])
        self.grads = (NcLayerG * L)(*[NcLayerG(self.g[f"w_qkv.{l}"].data_ptr(),
                                               self.g[f"w_o.{l}"].data_ptr(),
                                               self.g[f"w_fc.{l}"].data_ptr(),
                                               self.g[f"w_proj.{l}"].data_ptr())
                                      for l in range(L)])
        nbytes = workspace_bytes(self.cfg, B, T)
        if nbytes == 0:
            raise NcError(2, lib().nc_last_error_message().decode())
        self.ws = alloc_workspace(nbytes, self.device)
        self.loss = torch.zeros(1, dtype=torch.float32, device=self.device)
        self.ids = torch.zeros((B, T), dtype=torch.int32, device=self.device)
        self.targets = torch.zeros((B, T), dtype=torch.int32, device=self.device)

    def run(self, ids=None, targets=None, accumulate: bool = False) -> torch.Tensor:
        """One fwd+bwd on device-resident ids/targets; returns the device loss."""
        ids = self.ids if ids is None else ids
        targets = self.targets if targets is None else targets
        step(self.cfg, self.B, self.T, ids, targets, self.w["wte"], self.layers, self.w["w_lm"],
             self.loss, self.g["wte"], self.grads, self.g["w_lm"], accumulate, self.ws)
        return self.loss

    def run_host(self, ids_host: torch.Tensor, targets_host: torch.Tensor) -> float:
        """End-to-end call from host buffers: copy ids/targets (pinned host ->
        device), run the step, read the loss back to the host."""
        self.ids.copy_(ids_host, non_blocking=True)
        self.targets.copy_(targets_host, non_blocking=True)
        self.run()
        return float(self.loss.item())

    def status(self) -> int:
        return get_device_status(self.ws)

    def evaluate(self, ids, targets, token_bytes=None) -> torch.Tensor:
        """Forward-only nc_eval on device ids/targets; returns the device
        tensor [mean loss (nats), bits per byte (NaN without token_bytes)]."""
        out = torch.zeros(2, dtype=torch.float32, device=self.device)
        p, n = _ws(self.ws)
        _check(lib().nc_eval(ctypes.byref(self.cfg), self.B, self.T, _ptr(ids), _ptr(targets),
                             _ptr(token_bytes), self.w["wte"].data_ptr(), self.layers,
                             self.w["w_lm"].data_ptr(), out.data_ptr(), p, n, _stream(self.device)))
        return out


# Muon's published defaults (momentum 0.95, the quintic Newton-Schulz
# coefficients, five steps); AdamW's betas and eps as in the AdamW paper.
MUON_NS = (3.4445, -4.7750, 2.0315)


class Optimizer:
    """float32 master weights plus Muon + AdamW state for the parameters of a
    Step.  step(t, lrm) applies nc_optimizer_step to the Step's gradients and
    rewrites the Step's compute weights (bf16 or float) from the masters."""

    def __init__(self, st: Step, lr_muon=0.02, momentum=0.95, lr_embed=0.1, lr_lm=0.01,
                 betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0, ns=MUON_NS, ns_steps=5,
                 masters: dict | None = None):
        self.st = st
        dev = st.device
        src = masters if masters is not None else st.w
        self.p = {k: torch.as_tensor(src[k]).to(device=dev, dtype=torch.float32).clone()
                  for k in st.w}
        self.state = {}
        for k, v in self.p.items():
            if k in ("wte", "w_lm"):
                self.state[k] = {"m": torch.zeros_like(v), "v": torch.zeros_like(v)}
            else:
                self.state[k] = {"buf": torch.zeros_like(v)}
        self.oc = NcOptConfig(lr_muon, momentum, lr_embed, lr_lm, betas[0], betas[1], eps,
                              weight_decay, ns[0], ns[1], ns[2], ns_steps)
        L = st.shape.depth
        self.masters = (NcLayerF * L)(*[NcLayerF(*(self.p[f"{n}.{l}"].data_ptr()
                                                   for n in ("w_qkv", "w_o", "w_fc", "w_proj")))
                                        for l in range(L)])
        self.copies = (NcLayerWC * L)(*[NcLayerWC(*(st.w[f"{n}.{l}"].data_ptr()
                                                    for n in ("w_qkv", "w_o", "w_fc", "w_proj")))
                                        for l in range(L)])
        self.mom = (NcLayerF * L)(*[NcLayerF(*(self.state[f"{n}.{l}"]["buf"].data_ptr()
                                               for n in ("w_qkv", "w_o", "w_fc", "w_proj")))
                                    for l in range(L)])
        nbytes = lib().nc_optimizer_workspace_bytes(ctypes.byref(st.cfg))
        if nbytes == 0:
            raise NcError(2, lib().nc_last_error_message().decode())
        self.ws = alloc_workspace(nbytes, dev)

    def step(self, t: int, lrm: float = 1.0) -> None:
        st, p, s = self.st, self.p, self.state
        wp, wn = _ws(self.ws)
        _check(lib().nc_optimizer_step(
            ctypes.byref(st.cfg), ctypes.byref(self.oc), int(t), float(lrm),
            p["wte"].data_ptr(), p["w_lm"].data_ptr(), self.masters,
            st.w["wte"].data_ptr(), st.w["w_lm"].data_ptr(), self.copies,
            st.g["wte"].data_ptr(), st.g["w_lm"].data_ptr(), st.grads,
            s["wte"]["m"].data_ptr(), s["wte"]["v"].data_ptr(), s["w_lm"]["m"].data_ptr(),
            s["w_lm"]["v"].data_ptr(), self.mom, wp, wn, _stream(st.device)))
