"""ctypes binding of libmoe_gb300 (include/moe_gb300.h): same names, argument
marshalling only.  Every step of the layer runs in the library's CUDA kernels;
there is no fallback of any kind, and a missing library is an error.

Tensors are passed as torch tensors (their ``data_ptr``) and checked for device,
dtype and contiguity before the call; ``None`` becomes NULL.  ``stream`` defaults
to torch's current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmoe_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(PKG_DIR), "include", "moe_gb300.h")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_DEVICE_TIMEOUT = -4
MOE_ERR_BAD_INDEX = -5
MOE_ERR_FP16_RANGE = -6


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int

# moe_tuned_gemm_t: index of each token-row GEMM in moe_tuning_t.order
TUNED_GEMMS = ("gate_up", "down", "dA", "bwd_gate_up", "dx")
TUNING_SOURCES = ("default", "table", "override")


class MoeTuning(ctypes.Structure):
    _fields_ = [("order", _I * 5), ("swap_tails", _I), ("da_tile_n", _I),
                ("dw_chunk_rows", _I)]

_SIGS = {
    "moe_abi_version": (_I, []),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_capacity": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "moe_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "moe_workspace_init": (_I, [_P, _P]),
    "moe_route_permute": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_mlp_fwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_expert_mlp_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_get_device_error": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), _P]),
    "moe_route_permute_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                       _P]),
    "moe_debug_drop_next_loads": (_I, []),
    "moe_num_kernels": (_I, []),
    "moe_kernel_name": (ctypes.c_char_p, [_I]),
    "moe_launch_count": (ctypes.c_longlong, [ctypes.POINTER(ctypes.c_longlong)]),
    "moe_timing_enable": (_I, [_I]),
    "moe_router_topk": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_router_weight_grad": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_router_backward": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_timing_enable_mask": (_I, [ctypes.c_ulonglong]),
    "moe_tuning_get": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(MoeTuning), ctypes.POINTER(_I)]),
    "moe_tuning_override": (_I, [ctypes.POINTER(MoeTuning)]),
    "moe_timing_collect": (_I, [ctypes.POINTER(ctypes.c_double),
                                ctypes.POINTER(ctypes.c_longlong)]),
}


def lib():
    """Loads libmoe_gb300.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build(); "
                               "this package has no CPU or PyTorch fallback")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(handle, name)
            f.restype = res
            f.argtypes = args
        _lib = handle
    return _lib


def declared_functions() -> list[str]:
    """Names of the functions include/moe_gb300.h declares."""
    with open(HEADER_PATH) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtype=None, name="tensor", allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status, lib().moe_status_string(status).decode())


def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_capacity(T: int, K: int, E: int, align: int) -> int:
    return lib().moe_capacity(T, K, E, align)


def moe_workspace_bytes(T: int, K: int, E: int, D: int, I: int, align: int) -> int:
    return lib().moe_workspace_bytes(T, K, E, D, I, align)


def moe_workspace_init(workspace, stream=None):
    _check("moe_workspace_init", lib().moe_workspace_init(_ptr(workspace, name="workspace"),
                                                          _stream(stream)))


def moe_route_permute(topk_ids, topk_w, x, T, K, E, D, align, counts, offsets, perm_src,
                      inv_perm, w_perm, x_perm, workspace, stream=None):
    bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
    st = lib().moe_route_permute(
        _ptr(topk_ids, i32, "topk_ids", T == 0), _ptr(topk_w, f32, "topk_w", T == 0),
        _ptr(x, bf, "x", True), T, K, E, D, align,
        _ptr(counts, i32, "counts"), _ptr(offsets, i32, "offsets"),
        _ptr(perm_src, i32, "perm_src"), _ptr(inv_perm, i32, "inv_perm", T == 0),
        _ptr(w_perm, f32, "w_perm"), _ptr(x_perm, bf, "x_perm", x is None),
        _ptr(workspace, name="workspace"), _stream(stream))
    _check("moe_route_permute", st)


def moe_route_permute_noalloc(topk_ids, topk_w, x, T, K, E, D, align, counts, offsets,
                              perm_src, inv_perm, w_perm, x_perm, stream=None):
    """moe_route_permute for callers that cannot allocate a workspace (see the header)."""
    bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
    st = lib().moe_route_permute_noalloc(
        _ptr(topk_ids, i32, "topk_ids", T == 0), _ptr(topk_w, f32, "topk_w", T == 0),
        _ptr(x, bf, "x", True), T, K, E, D, align,
        _ptr(counts, i32, "counts"), _ptr(offsets, i32, "offsets"),
        _ptr(perm_src, i32, "perm_src"), _ptr(inv_perm, i32, "inv_perm", T == 0),
        _ptr(w_perm, f32, "w_perm"), _ptr(x_perm, bf, "x_perm", x is None), _stream(stream))
    _check("moe_route_permute_noalloc", st)


def moe_expert_mlp_fwd(x_perm, w_gate, w_up, w_down, offsets, counts, T, K, E, D, I, align,
                       y_perm, workspace, stream=None):
    bf = torch.bfloat16
    st = lib().moe_expert_mlp_fwd(
        _ptr(x_perm, bf, "x_perm"), _ptr(w_gate, bf, "w_gate"), _ptr(w_up, bf, "w_up"),
        _ptr(w_down, bf, "w_down"), _ptr(offsets, torch.int32, "offsets"),
        _ptr(counts, torch.int32, "counts", True), T, K, E, D, I, align,
        _ptr(y_perm, bf, "y_perm"), _ptr(workspace, name="workspace"), _stream(stream))
    _check("moe_expert_mlp_fwd", st)


def moe_combine(src_perm, inv_perm, topk_w, T, K, D, out, stream=None):
    st = lib().moe_combine(
        _ptr(src_perm, torch.bfloat16, "src_perm", T == 0),
        _ptr(inv_perm, torch.int32, "inv_perm", T == 0),
        _ptr(topk_w, torch.float32, "topk_w", True), T, K, D,
        _ptr(out, torch.bfloat16, "out", T == 0), _stream(stream))
    _check("moe_combine", st)


def moe_expert_mlp_bwd(dy, x, x_perm, perm_src, w_perm, offsets, counts, w_gate, w_up, w_down,
                       T, K, E, D, I, align, dx_perm, dw_gate, dw_up, dw_down, workspace,
                       stream=None, inv_perm=None, dx=None):
    """With inv_perm and dx the call also reduces dx_perm to tokens into dx."""
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    st = lib().moe_expert_mlp_bwd(
        _ptr(dy, bf, "dy", T == 0), _ptr(x, bf, "x", True), _ptr(x_perm, bf, "x_perm"), _ptr(perm_src, i32, "perm_src"),
        _ptr(w_perm, f32, "w_perm"), _ptr(offsets, i32, "offsets"),
        _ptr(counts, i32, "counts", True), _ptr(w_gate, bf, "w_gate"),
        _ptr(w_up, bf, "w_up"), _ptr(w_down, bf, "w_down"), T, K, E, D, I, align,
        _ptr(dx_perm, bf, "dx_perm"), _ptr(dw_gate, f32, "dw_gate"), _ptr(dw_up, f32, "dw_up"),
        _ptr(dw_down, f32, "dw_down"), _ptr(inv_perm, i32, "inv_perm", True),
        _ptr(dx, bf, "dx", True), _ptr(workspace, name="workspace"), _stream(stream))
    _check("moe_expert_mlp_bwd", st)


ROUTERS = {"softmax": 0, "sigmoid_top1": 1}


def moe_router_topk(logits, T, E, K, router, topk_ids, topk_w, stream=None):
    st = lib().moe_router_topk(
        _ptr(logits, torch.float32, "logits", T == 0), T, E, K, ROUTERS[router],
        _ptr(topk_ids, torch.int32, "topk_ids", T == 0),
        _ptr(topk_w, torch.float32, "topk_w", T == 0), _stream(stream))
    _check("moe_router_topk", st)


def moe_router_weight_grad(dy, y_perm, inv_perm, T, K, D, d_topk_w, stream=None):
    st = lib().moe_router_weight_grad(
        _ptr(dy, torch.bfloat16, "dy", T == 0), _ptr(y_perm, torch.bfloat16, "y_perm", T == 0),
        _ptr(inv_perm, torch.int32, "inv_perm", T == 0), T, K, D,
        _ptr(d_topk_w, torch.float32, "d_topk_w", T == 0), _stream(stream))
    _check("moe_router_weight_grad", st)


def moe_router_backward(topk_ids, topk_w, d_topk_w, T, E, K, router, d_logits, stream=None):
    st = lib().moe_router_backward(
        _ptr(topk_ids, torch.int32, "topk_ids", T == 0),
        _ptr(topk_w, torch.float32, "topk_w", T == 0),
        _ptr(d_topk_w, torch.float32, "d_topk_w", T == 0), T, E, K, ROUTERS[router],
        _ptr(d_logits, torch.float32, "d_logits", T == 0), _stream(stream))
    _check("moe_router_backward", st)


def moe_get_device_error(workspace, stream=None):
    """Returns (status, raw device code) and clears the device error word."""
    code, detail = ctypes.c_int(0), ctypes.c_int(0)
    _check("moe_get_device_error", lib().moe_get_device_error(
        _ptr(workspace, name="workspace"), ctypes.byref(code), ctypes.byref(detail),
        _stream(stream)))
    return code.value, detail.value


def moe_debug_drop_next_loads():
    """Test hook: the next gate/up GEMM launch skips its loads so its waits time out."""
    _check("moe_debug_drop_next_loads", lib().moe_debug_drop_next_loads())


def kernel_names() -> list[str]:
    L = lib()
    return [L.moe_kernel_name(i).decode() for i in range(L.moe_num_kernels())]


def moe_launch_count():
    """(total, {kernel name: launches}) since the library was loaded."""
    L = lib()
    n = L.moe_num_kernels()
    arr = (ctypes.c_longlong * n)()
    total = L.moe_launch_count(arr)
    return total, dict(zip(kernel_names(), list(arr)))


def moe_timing_enable(on: bool):
    _check("moe_timing_enable", lib().moe_timing_enable(1 if on else 0))


def moe_timing_enable_only(names):
    """Times only the named kernels (an empty list turns timing off)."""
    ids = kernel_names()
    mask = 0
    for n in names:
        mask |= 1 << ids.index(n)
    _check("moe_timing_enable_mask", lib().moe_timing_enable_mask(mask))


def _tuning_dict(t: MoeTuning) -> dict:
    return {"order": {g: t.order[i] for i, g in enumerate(TUNED_GEMMS)},
            "swap_tails": t.swap_tails, "da_tile_n": t.da_tile_n,
            "dw_chunk_rows": t.dw_chunk_rows}


def moe_tuning_get(T: int, K: int, E: int, D: int, I: int):
    """(choices, source) the forward/backward calls of this shape use; host only."""
    t, src = MoeTuning(), ctypes.c_int(0)
    _check("moe_tuning_get", lib().moe_tuning_get(T, K, E, D, I, ctypes.byref(t),
                                                   ctypes.byref(src)))
    return _tuning_dict(t), TUNING_SOURCES[src.value]


def moe_tuning_override(choices=None):
    """Sets the process-wide override (a dict shaped like moe_tuning_get's), or clears it
    (None).  Missing keys take the defaults."""
    if choices is None:
        _check("moe_tuning_override", lib().moe_tuning_override(None))
        return
    t = MoeTuning()
    order = choices.get("order", {})
    for i, g in enumerate(TUNED_GEMMS):
        t.order[i] = int(order.get(g, 0))
    t.swap_tails = int(choices.get("swap_tails", 1))
    t.da_tile_n = int(choices.get("da_tile_n", 256))
    t.dw_chunk_rows = int(choices.get("dw_chunk_rows", 4096))
    _check("moe_tuning_override", lib().moe_tuning_override(ctypes.byref(t)))


def moe_timing_collect():
    """{kernel name: (total ms, launches)} for the launches recorded since the last collect."""
    L = lib()
    n = L.moe_num_kernels()
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_longlong * n)()
    _check("moe_timing_collect", L.moe_timing_collect(ms, cnt))
    return {name: (ms[i], cnt[i]) for i, name in enumerate(kernel_names()) if cnt[i]}
