"""Thin Python binding of libmoe.so (ctypes): argument marshalling only.

Every step of the MoE path runs in the library's CUDA kernels; this module
only allocates outputs/workspaces with PyTorch, passes raw device pointers and
the current CUDA stream, and turns status codes into exceptions.  There is no
fallback: if libmoe.so is missing or fails to load, every call raises.

Names follow the C ABI (include/moe.h): route, dispatch, condense,
expert_ffn, combine, layer_forward, workspace_size, adaptive_tau,
get_device_status.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_F32, MOE_BF16 = 0, 1
GATING = {"softmax_topk": 0, "softmax_topk_renorm": 1, "sigmoid_topk": 2}
RESIDUAL = {"none": 0, "input": 1, "external": 2, "input_plus_external": 3}
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_INDEX"}

EXPORTED = ("moe_status_string", "moe_adaptive_tau", "moe_get_device_status",
            "moe_route_workspace_size", "moe_route",
            "moe_dispatch_workspace_size", "moe_dispatch", "moe_condense_workspace_size",
            "moe_condense", "moe_expert_ffn_workspace_size", "moe_expert_ffn", "moe_combine",
            "moe_workspace_size", "moe_layer_forward", "moe_layer_forward_ex",
            "moe_dispatch_static_scratch", "moe_layer_backward_workspace_size",
            "moe_layer_backward", "moe_condense_history_bytes", "moe_condense_hist")


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("H", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("H_shared", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("gating", ctypes.c_int32), ("residual", ctypes.c_int32)]


class moe_weights(ctypes.Structure):
    _fields_ = [("W_r", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("W_gu", ctypes.c_void_p), ("W_down", ctypes.c_void_p),
                ("Ws_gu", ctypes.c_void_p), ("Ws_down", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (built in-tree by routing_expert_ffn_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = load_library(LIB_PATH)
    return _lib


def load_library(path: str) -> ctypes.CDLL:
    """A build of the library at `path` with the C ABI's signatures set (lib() loads the
    product library; the timeout test loads the fault-injection build this way)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m routing_expert_ffn_gb300.build`")
    L = ctypes.CDLL(path)
    P, S, I, F = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    CFG, W = ctypes.POINTER(moe_config), ctypes.POINTER(moe_weights)
    sig = {
        "moe_status_string": (ctypes.c_char_p, [I]),
        "moe_adaptive_tau": (F, [F]),
        "moe_get_device_status": (I, [P]),
        "moe_route_workspace_size": (S, [CFG]),
        "moe_route": (I, [CFG, P, P, P, P, P, P, P, S, P]),
        "moe_dispatch_workspace_size": (S, [CFG]),
        "moe_dispatch": (I, [CFG, P, P, P, P, P, P, P, P, S, P]),
        "moe_condense_workspace_size": (S, [CFG]),
        "moe_condense": (I, [CFG, P, P, F, P, P, P, P, S, P]),
        "moe_condense_history_bytes": (S, [CFG]),
        "moe_condense_hist": (I, [CFG, P, P, P, P, F, F, F, P, P, P, P, P, P, P, S, P]),
        "moe_expert_ffn_workspace_size": (S, [CFG, I]),
        "moe_expert_ffn": (I, [CFG, W, P, P, P, P, P, P, P, S, P]),
        "moe_combine": (I, [CFG, P, P, P, P, P, P, P, P, P]),
        "moe_workspace_size": (S, [CFG, I]),
        "moe_layer_forward": (I, [CFG, W, P, P, F, P, P, P, P, S, P]),
        "moe_layer_forward_ex": (I, [CFG, W, P, P, F, P, P, P, P, P, S, P, P]),
        "moe_dispatch_static_scratch": (I, [CFG, P, P, P, P, P, P, P, P]),
        "moe_layer_backward_workspace_size": (S, [CFG, I]),
        "moe_layer_backward": (I, [CFG, W, P, P, F, P, P, P, P, P, P, P, P, P, S, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def _check(code: int, where: str) -> None:
    if code != 0:
        raise MoEError(code, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class Config:
    T: int
    d: int
    E: int
    k: int
    H: int
    n_shared: int = 0
    H_shared: int = 0
    dtype: str = "bf16"
    gating: str = "softmax_topk"
    residual: str = "input"

    @classmethod
    def from_workload(cls, w) -> "Config":
        return cls(T=w.T, d=w.d, E=w.E, k=w.k, H=w.H, n_shared=w.n_shared, H_shared=w.H_shared,
                   dtype=w.dtype, gating=w.gating, residual=w.residual)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def c(self) -> moe_config:
        return moe_config(self.T, self.d, self.E, self.k, self.H, self.n_shared, self.H_shared,
                          MOE_BF16 if self.dtype == "bf16" else MOE_F32, GATING[self.gating],
                          RESIDUAL[self.residual])


@dataclass
class Weights:
    W_r: torch.Tensor
    router_bias: torch.Tensor | None
    W_gu: torch.Tensor
    W_down: torch.Tensor
    Ws_gu: torch.Tensor | None = None
    Ws_down: torch.Tensor | None = None

    def c(self) -> moe_weights:
        return moe_weights(_ptr(self.W_r), _ptr(self.router_bias), _ptr(self.W_gu),
                           _ptr(self.W_down), _ptr(self.Ws_gu), _ptr(self.Ws_down))


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def _workspace(nbytes: int, device) -> torch.Tensor | None:
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ entry points
def status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def adaptive_tau(l_norm: float) -> float:
    return float(lib().moe_adaptive_tau(l_norm))


def get_device_status(stream=None) -> int:
    return int(lib().moe_get_device_status(_stream(stream)))


def route(cfg: Config, x, W_r, bias=None, stream=None):
    """(logits [T,E] fp32, topk_idx [T,k] int32, topk_gate [T,k] fp32)."""
    dev = x.device
    logits = _empty((cfg.T, cfg.E), torch.float32, dev)
    idx = _empty((cfg.T, cfg.k), torch.int32, dev)
    gate = _empty((cfg.T, cfg.k), torch.float32, dev)
    c = cfg.c()
    n = lib().moe_route_workspace_size(ctypes.byref(c))
    ws = _workspace(n, dev)
    _check(lib().moe_route(ctypes.byref(c), _ptr(x), _ptr(W_r), _ptr(bias), _ptr(logits),
                           _ptr(idx), _ptr(gate), _ptr(ws), n, _stream(stream)), "moe_route")
    return logits, idx, gate


def dispatch(cfg: Config, x, topk_idx, stream=None) -> dict:
    dev = x.device
    P = cfg.T * cfg.k
    c = cfg.c()
    out = dict(counts=_empty((cfg.E,), torch.int32, dev),
               offsets=_empty((cfg.E + 1,), torch.int32, dev),
               perm=_empty((max(P, 1),), torch.int32, dev),
               slot_of=_empty((cfg.T, cfg.k), torch.int32, dev),
               x_perm=_empty((max(P, 1), cfg.d), cfg.torch_dtype, dev))
    n = lib().moe_dispatch_workspace_size(ctypes.byref(c))
    ws = _workspace(n, dev)
    _check(lib().moe_dispatch(ctypes.byref(c), _ptr(x), _ptr(topk_idx), _ptr(out["counts"]),
                              _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["slot_of"]),
                              _ptr(out["x_perm"]), _ptr(ws), n, _stream(stream)), "moe_dispatch")
    return out


def dispatch_static_scratch(cfg: Config, x, topk_idx, stream=None) -> dict:
    """moe_dispatch without a workspace (scratch is a fixed array inside the library)."""
    dev = x.device
    P = cfg.T * cfg.k
    out = dict(counts=_empty((cfg.E,), torch.int32, dev),
               offsets=_empty((cfg.E + 1,), torch.int32, dev),
               perm=_empty((max(P, 1),), torch.int32, dev),
               slot_of=_empty((cfg.T, cfg.k), torch.int32, dev),
               x_perm=_empty((max(P, 1), cfg.d), cfg.torch_dtype, dev))
    _check(lib().moe_dispatch_static_scratch(
        ctypes.byref(cfg.c()), _ptr(x), _ptr(topk_idx), _ptr(out["counts"]), _ptr(out["offsets"]),
        _ptr(out["perm"]), _ptr(out["slot_of"]), _ptr(out["x_perm"]), _stream(stream)),
        "moe_dispatch_static_scratch")
    return out


def condense_history_bytes(cfg: Config) -> int:
    return int(lib().moe_condense_history_bytes(ctypes.byref(cfg.c())))


def condense_hist(cfg: Config, x_perm, offsets, perm, slot_of, tau: float, s1: float, s2: float,
                  hist_in=None, hist_out=None, stream=None):
    """Condensation with the previous call's pair classes.  hist_in / hist_out are uint8
    device tensors of condense_history_bytes(cfg) bytes (hist_out is allocated when None).
    Returns (rep_of, n_rep, n_condensed, n_cos_tiles, hist_out)."""
    dev = x_perm.device
    c = cfg.c()
    P = cfg.T * cfg.k
    rep_of = _empty((max(P, 1),), torch.int32, dev)
    n_rep = _empty((cfg.E,), torch.int32, dev)
    n_cond = _empty((1,), torch.int32, dev)
    n_cos = _empty((1,), torch.int32, dev)
    if hist_out is None:
        hist_out = torch.empty(condense_history_bytes(cfg), dtype=torch.uint8, device=dev)
    n = lib().moe_condense_workspace_size(ctypes.byref(c))
    ws = _workspace(n, dev)
    _check(lib().moe_condense_hist(ctypes.byref(c), _ptr(x_perm), _ptr(offsets), _ptr(perm),
                                   _ptr(slot_of), tau, s1, s2, _ptr(hist_in), _ptr(hist_out),
                                   _ptr(rep_of), _ptr(n_rep), _ptr(n_cond), _ptr(n_cos), _ptr(ws),
                                   n, _stream(stream)), "moe_condense_hist")
    return rep_of, n_rep, n_cond, n_cos, hist_out


def condense(cfg: Config, x_perm, offsets, tau: float, stream=None):
    """(rep_of [T*k] int32, n_rep [E] int32, n_condensed [1] int32)."""
    dev = x_perm.device
    c = cfg.c()
    P = cfg.T * cfg.k
    rep_of = _empty((max(P, 1),), torch.int32, dev)
    n_rep = _empty((cfg.E,), torch.int32, dev)
    n_cond = _empty((1,), torch.int32, dev)
    n = lib().moe_condense_workspace_size(ctypes.byref(c))
    ws = _workspace(n, dev)
    _check(lib().moe_condense(ctypes.byref(c), _ptr(x_perm), _ptr(offsets), tau, _ptr(rep_of),
                              _ptr(n_rep), _ptr(n_cond), _ptr(ws), n, _stream(stream)),
           "moe_condense")
    return rep_of, n_rep, n_cond


def expert_ffn(cfg: Config, w: Weights, x_perm, offsets, rep_of=None, x=None, stream=None):
    """(y_perm [T*k, d], shared_out [T, d] or None)."""
    dev = x_perm.device
    c = cfg.c()
    P = cfg.T * cfg.k
    y = torch.zeros((max(P, 1), cfg.d), dtype=cfg.torch_dtype, device=dev)
    so = _empty((cfg.T, cfg.d), cfg.torch_dtype, dev) if cfg.n_shared > 0 else None
    n = lib().moe_expert_ffn_workspace_size(ctypes.byref(c), int(rep_of is not None))
    ws = _workspace(n, dev)
    wc = w.c()
    _check(lib().moe_expert_ffn(ctypes.byref(c), ctypes.byref(wc), _ptr(x_perm), _ptr(offsets),
                                _ptr(rep_of), _ptr(x), _ptr(y), _ptr(so), _ptr(ws), n,
                                _stream(stream)), "moe_expert_ffn")
    return y, so


def combine(cfg: Config, y_perm, shared_out, slot_of, rep_of, topk_gate, x=None, residual=None,
            out=None, stream=None):
    dev = y_perm.device
    if out is None:
        out = _empty((cfg.T, cfg.d), cfg.torch_dtype, dev)
    _check(lib().moe_combine(ctypes.byref(cfg.c()), _ptr(y_perm), _ptr(shared_out), _ptr(slot_of),
                             _ptr(rep_of), _ptr(topk_gate), _ptr(x), _ptr(residual), _ptr(out),
                             _stream(stream)), "moe_combine")
    return out


def workspace_size(cfg: Config, condense: bool) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(cfg.c()), int(condense)))


class Layer:
    """A routed-expert MoE layer with its weights and a preallocated workspace.

    ``layer(x, residual, tau)`` is one ``moe_layer_forward`` call on the
    current stream.  tau <= 1 enables condensation; tau = nan disables it.
    With ``partial_out`` (FarSkip's partial activation r + shared) or
    ``aux_stream`` (shared experts on a second stream) it is one
    ``moe_layer_forward_ex`` call.
    """

    def __init__(self, cfg: Config, w: Weights, condense: bool = False, device=None):
        self.cfg = cfg
        self.w = w
        self.device = device or w.W_gu.device
        self._c = cfg.c()
        self._wc = w.c()
        self.condense = condense
        self.ws_bytes = workspace_size(cfg, condense)
        self.ws = _workspace(self.ws_bytes, self.device)

    def __call__(self, x, residual=None, tau: float = math.nan, out=None, topk_idx_out=None,
                 n_condensed_out=None, stream=None, partial_out=None, aux_stream=None):
        if out is None:
            out = _empty((self.cfg.T, self.cfg.d), self.cfg.torch_dtype, self.device)
        if tau <= 1.0 and not self.condense:
            raise ValueError("layer was built without condensation workspace")
        if partial_out is None and aux_stream is None:
            _check(lib().moe_layer_forward(ctypes.byref(self._c), ctypes.byref(self._wc), _ptr(x),
                                           _ptr(residual), tau, _ptr(out), _ptr(topk_idx_out),
                                           _ptr(n_condensed_out), _ptr(self.ws), self.ws_bytes,
                                           _stream(stream)), "moe_layer_forward")
        else:
            aux = aux_stream.cuda_stream if aux_stream is not None else None
            _check(lib().moe_layer_forward_ex(ctypes.byref(self._c), ctypes.byref(self._wc),
                                              _ptr(x), _ptr(residual), tau, _ptr(out),
                                              _ptr(partial_out), _ptr(topk_idx_out),
                                              _ptr(n_condensed_out), _ptr(self.ws), self.ws_bytes,
                                              _stream(stream), aux), "moe_layer_forward_ex")
        return out


def layer_forward(cfg: Config, w: Weights, x, residual=None, tau: float = math.nan, stream=None):
    return Layer(cfg, w, condense=tau <= 1.0, device=x.device)(x, residual, tau, stream=stream)


class Backward:
    """The layer's backward with a preallocated workspace and gradient buffers.

    ``bwd(x, d_out)`` is one ``moe_layer_backward`` call on the current stream and
    returns the gradient dict (the same tensors every call): d_x, d_residual (or None),
    dW_r, d_bias (or None), dW_gu, dW_down, dWs_gu, dWs_down (or None).
    """

    def __init__(self, cfg: Config, w: Weights, d_residual: bool = False, device=None,
                 condense: bool = False):
        self.cfg, self.w = cfg, w
        self.condense = condense
        dev = device or w.W_gu.device
        f32 = torch.float32
        self._c = cfg.c()
        self._wc = w.c()
        self.grads = dict(
            d_x=_empty((cfg.T, cfg.d), cfg.torch_dtype, dev),
            d_residual=_empty((cfg.T, cfg.d), cfg.torch_dtype, dev) if d_residual else None,
            dW_r=_empty((cfg.d, cfg.E), f32, dev),
            d_bias=_empty((cfg.E,), f32, dev) if w.router_bias is not None else None,
            dW_gu=_empty((cfg.E, 2 * cfg.H, cfg.d), f32, dev),
            dW_down=_empty((cfg.E, cfg.d, cfg.H), f32, dev),
            dWs_gu=_empty((cfg.n_shared, 2 * cfg.H_shared, cfg.d), f32, dev) if cfg.n_shared else None,
            dWs_down=_empty((cfg.n_shared, cfg.d, cfg.H_shared), f32, dev) if cfg.n_shared else None)
        self.ws_bytes = int(lib().moe_layer_backward_workspace_size(ctypes.byref(self._c),
                                                                    int(condense)))
        self.ws = _workspace(self.ws_bytes, dev)

    def __call__(self, x, d_out, tau: float = math.nan, stream=None) -> dict:
        if tau <= 1.0 and not self.condense:
            raise ValueError("backward was built without condensation workspace")
        g = self.grads
        _check(lib().moe_layer_backward(ctypes.byref(self._c), ctypes.byref(self._wc), _ptr(x),
                                        _ptr(d_out), tau, _ptr(g["d_x"]), _ptr(g["d_residual"]),
                                        _ptr(g["dW_r"]), _ptr(g["d_bias"]), _ptr(g["dW_gu"]),
                                        _ptr(g["dW_down"]), _ptr(g["dWs_gu"]), _ptr(g["dWs_down"]),
                                        _ptr(self.ws), self.ws_bytes, _stream(stream)),
               "moe_layer_backward")
        return g


def layer_backward(cfg: Config, w: Weights, x, d_out, d_residual: bool = False,
                   tau: float = math.nan, stream=None) -> dict:
    """Gradients of the layer output for d_out (fresh buffers; tau <= 1 condenses): see Backward."""
    return Backward(cfg, w, d_residual, x.device, condense=tau <= 1.0)(x, d_out, tau, stream)


# ------------------------------------------------------------------ input upload
def upload(cfg: Config, inp: dict, device="cuda") -> tuple[Weights, torch.Tensor, torch.Tensor | None]:
    """Numpy workload arrays -> device tensors in the layer's dtype: (weights, x, residual)."""
    dt = cfg.torch_dtype

    def t(a, dtype=dt):
        if a is None or a.size == 0:
            return None
        return torch.from_numpy(a).to(device=device).to(dtype).contiguous()

    w = Weights(W_r=t(inp["W_r"], torch.float32),
                router_bias=t(inp["bias"], torch.float32) if inp.get("bias") is not None else None,
                W_gu=t(inp["W_gu"]), W_down=t(inp["W_down"]),
                Ws_gu=t(inp["Ws_gu"]) if cfg.n_shared else None,
                Ws_down=t(inp["Ws_down"]) if cfg.n_shared else None)
    x = t(inp["x"])
    r = t(inp["residual"]) if inp.get("residual") is not None else None
    return w, x, r
