"""Python binding of libnvfp4moe.so (argument marshalling only).

Every function here has the name of the C entry point it calls (declared in
``include/nvfp4moe.h``) and does nothing but turn torch tensors into device
pointers, pick the current CUDA stream, call the library and raise
``MoeError`` on a non-OK status.  All computation happens in the library's
CUDA kernels; there is no CPU fallback.  Loading fails loudly when the library
has not been built (``__graft_entry__.build()`` builds it).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvfp4moe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_DEVICE_FLAG = 4
MOE_ERR_WORKSPACE = 5

MOE_W_NVFP4 = 0
MOE_W_BF16 = 1
MOE_PACK_PLAIN = 0
MOE_PACK_GATE_UP = 1

MOE_FLAG_NONFINITE_LOGIT = 1
MOE_FLAG_WAIT_TIMEOUT = 2
MOE_FLAG_BAD_INDEX = 4

HIDDEN = 2048
INTER = 512
EXPERTS = 256
TOPK = 6
MAX_DECODE_T = 8
MAX_CHUNKED_T = 88           # NVFP4 weights
MAX_CHUNKED_T_BF16 = 56
MAX_TOKENS = 65536

# Exported symbols (kept in step with include/nvfp4moe.h; a CPU test checks).
EXPORTS = (
    "moe_abi_version", "moe_status_string", "moe_packed_bytes", "moe_pack_nvfp4",
    "moe_unpack_nvfp4", "moe_dequant_nvfp4", "moe_workspace_bytes", "moe_workspace_init",
    "moe_read_device_flag", "moe_workspace_recover", "moe_route", "moe_read_routing", "moe_layer_forward",
    "moe_layer_forward_static", "moe_static_read_device_flag",
    "moe_layer_forward_prenorm", "moe_stack_workspace_bytes", "moe_stack_forward",
    "moe_dense_gemv_nvfp4", "moe_layer_forward_sink", "moe_read_shared_weights",
)

MOE_STATIC_SCRATCH_BYTES = 7_400_448


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, lib=None):
        name = lib.moe_status_string(status).decode() if lib is not None else str(status)
        super().__init__(f"{fn} failed: {name}")
        self.status = status


class moe_expert_bank(ctypes.Structure):
    _fields_ = [
        ("wtype", ctypes.c_int32),
        ("n_experts", ctypes.c_int32),
        ("w13", ctypes.c_void_p),
        ("w2", ctypes.c_void_p),
        ("tscale13", ctypes.c_void_p),
        ("tscale2", ctypes.c_void_p),
    ]


class moe_layer_weights(ctypes.Structure):
    _fields_ = [
        ("router_w", ctypes.c_void_p),
        ("routed", moe_expert_bank),
        ("shared", moe_expert_bank),
    ]


_lib = None


def _declare(lib):
    vp, i32, sz, u32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32)
    lib.moe_abi_version.argtypes = []
    lib.moe_abi_version.restype = i32
    lib.moe_status_string.argtypes = [i32]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_packed_bytes.argtypes = [i32, i32]
    lib.moe_packed_bytes.restype = sz
    lib.moe_pack_nvfp4.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp]
    lib.moe_pack_nvfp4.restype = i32
    lib.moe_unpack_nvfp4.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp]
    lib.moe_unpack_nvfp4.restype = i32
    lib.moe_dequant_nvfp4.argtypes = [vp, i32, i32, i32, ctypes.c_float, vp, vp]
    lib.moe_dequant_nvfp4.restype = i32
    lib.moe_workspace_bytes.argtypes = [i32]
    lib.moe_workspace_bytes.restype = sz
    lib.moe_workspace_init.argtypes = [vp, sz, vp]
    lib.moe_workspace_init.restype = i32
    lib.moe_read_device_flag.argtypes = [vp, vp, u32p]
    lib.moe_read_device_flag.restype = i32
    lib.moe_route.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.moe_route.restype = i32
    lib.moe_workspace_recover.argtypes = [vp, sz, vp]
    lib.moe_workspace_recover.restype = i32
    lib.moe_static_read_device_flag.argtypes = [vp, u32p]
    lib.moe_static_read_device_flag.restype = i32
    lib.moe_read_routing.argtypes = [vp, sz, i32, vp, vp, vp, vp]
    lib.moe_read_routing.restype = i32
    bank_p = ctypes.POINTER(moe_expert_bank)
    lib.moe_layer_forward.argtypes = [vp, vp, bank_p, bank_p, vp, i32, vp, sz, vp]
    lib.moe_layer_forward.restype = i32
    lib.moe_layer_forward_static.argtypes = [vp, vp, bank_p, bank_p, vp, i32, vp]
    lib.moe_layer_forward_static.restype = i32
    lib.moe_layer_forward_prenorm.argtypes = [vp, vp, vp, vp, ctypes.c_float, vp, bank_p, bank_p, vp, i32, vp,
                                              sz, vp]
    lib.moe_layer_forward_prenorm.restype = i32
    lib.moe_stack_workspace_bytes.argtypes = [i32]
    lib.moe_stack_workspace_bytes.restype = sz
    lib.moe_stack_forward.argtypes = [vp, ctypes.POINTER(moe_layer_weights), i32, i32, ctypes.c_float, vp, sz,
                                      vp]
    lib.moe_stack_forward.restype = i32
    lib.moe_dense_gemv_nvfp4.argtypes = [vp, vp, ctypes.c_float, i32, i32, i32, vp, vp, sz, vp]
    lib.moe_dense_gemv_nvfp4.restype = i32
    lib.moe_layer_forward_sink.argtypes = [vp, vp, bank_p, bank_p, vp, i32, vp, sz, vp]
    lib.moe_layer_forward_sink.restype = i32
    lib.moe_read_shared_weights.argtypes = [vp, sz, i32, i32, vp, vp]
    lib.moe_read_shared_weights.restype = i32
    return lib


def load(path: Optional[str] = None):
    """Load the library (raises if it has not been built)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback implementation)")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status, _lib)


def moe_abi_version() -> int:
    return load().moe_abi_version()


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_packed_bytes(N: int, K: int) -> int:
    return load().moe_packed_bytes(int(N), int(K))


def moe_pack_nvfp4(codes, scales, N: int, K: int, kind: int, count: int, packed, stream=None):
    lib = load()
    _check("moe_pack_nvfp4", lib.moe_pack_nvfp4(_ptr(codes), _ptr(scales), N, K, kind, count,
                                                  _ptr(packed), _stream(stream)))


def moe_unpack_nvfp4(packed, N: int, K: int, kind: int, count: int, codes, scales, stream=None):
    lib = load()
    _check("moe_unpack_nvfp4", lib.moe_unpack_nvfp4(_ptr(packed), N, K, kind, count, _ptr(codes),
                                                      _ptr(scales), _stream(stream)))


def moe_dequant_nvfp4(packed, N: int, K: int, kind: int, tscale: float, out, stream=None):
    lib = load()
    _check("moe_dequant_nvfp4", lib.moe_dequant_nvfp4(_ptr(packed), N, K, kind, float(tscale),
                                                        _ptr(out), _stream(stream)))


def moe_workspace_bytes(T: int) -> int:
    return load().moe_workspace_bytes(int(T))


def moe_workspace_init(workspace, stream=None):
    lib = load()
    _check("moe_workspace_init", lib.moe_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                                          _stream(stream)))


def moe_read_device_flag(workspace, stream=None) -> int:
    """Synchronises the stream; returns the flag bits (0 = no device error)."""
    lib = load()
    v = ctypes.c_uint32(0)
    st = lib.moe_read_device_flag(_ptr(workspace), _stream(stream), ctypes.byref(v))
    if st not in (MOE_OK, MOE_ERR_DEVICE_FLAG):
        raise MoeError("moe_read_device_flag", st, lib)
    return int(v.value)


def moe_workspace_recover(workspace, stream=None):
    """Re-arm a workspace after a wait timeout (keeps its flag bits)."""
    lib = load()
    _check("moe_workspace_recover", lib.moe_workspace_recover(_ptr(workspace),
                                                                workspace.numel() * workspace.element_size(),
                                                                _stream(stream)))


def moe_static_read_device_flag(stream=None) -> int:
    """Synchronises the stream; returns and clears the flag bits of the fixed scratch."""
    lib = load()
    v = ctypes.c_uint32(0)
    st = lib.moe_static_read_device_flag(_stream(stream), ctypes.byref(v))
    if st not in (MOE_OK, MOE_ERR_DEVICE_FLAG):
        raise MoeError("moe_static_read_device_flag", st, lib)
    return int(v.value)


def moe_route(x, router_w, T: int, idx, w, logits=None, workspace=None, stream=None,
              n_experts: int = EXPERTS, top_k: int = TOPK):
    lib = load()
    _check("moe_route", lib.moe_route(_ptr(x), _ptr(router_w), int(T), n_experts, top_k, _ptr(idx),
                                       _ptr(w), _ptr(logits), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_read_routing(workspace, T: int, idx=None, w=None, logits=None, stream=None):
    """Copy the routing the last layer call on ``workspace`` used (device tensors)."""
    lib = load()
    _check("moe_read_routing", lib.moe_read_routing(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                                      int(T), _ptr(idx), _ptr(w), _ptr(logits), _stream(stream)))


def make_bank(wtype: int, n_experts: int, w13, w2, tscale13=None, tscale2=None) -> moe_expert_bank:
    """A host moe_expert_bank pointing at device tensors (the caller keeps them alive)."""
    return moe_expert_bank(int(wtype), int(n_experts), _ptr(w13), _ptr(w2), _ptr(tscale13), _ptr(tscale2))


def moe_layer_forward(x, router_w, routed: moe_expert_bank, shared: Optional[moe_expert_bank], out,
                      T: int, workspace, stream=None):
    lib = load()
    st = lib.moe_layer_forward(_ptr(x), _ptr(router_w), ctypes.byref(routed),
                               ctypes.byref(shared) if shared is not None else None, _ptr(out), int(T),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check("moe_layer_forward", st)


def moe_layer_forward_static(x, router_w, routed: moe_expert_bank, shared: Optional[moe_expert_bank], out,
                             T: int, stream=None):
    lib = load()
    st = lib.moe_layer_forward_static(_ptr(x), _ptr(router_w), ctypes.byref(routed),
                                      ctypes.byref(shared) if shared is not None else None, _ptr(out),
                                      int(T), _stream(stream))
    _check("moe_layer_forward_static", st)


def moe_layer_forward_prenorm(resid, delta, resid_out, xn_out, eps: float, router_w, routed: moe_expert_bank,
                              shared: Optional[moe_expert_bank], out, T: int, workspace, stream=None):
    lib = load()
    st = lib.moe_layer_forward_prenorm(_ptr(resid), _ptr(delta), _ptr(resid_out), _ptr(xn_out), float(eps),
                                       _ptr(router_w), ctypes.byref(routed),
                                       ctypes.byref(shared) if shared is not None else None, _ptr(out), int(T),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    _check("moe_layer_forward_prenorm", st)


def moe_stack_workspace_bytes(T: int) -> int:
    return load().moe_stack_workspace_bytes(int(T))


def layer_weights_array(layers) -> "ctypes.Array":
    """A host moe_layer_weights[n] for objects with router_w, routed, shared."""
    arr = (moe_layer_weights * len(layers))()
    for i, l in enumerate(layers):
        arr[i].router_w = _ptr(l.router_w)
        arr[i].routed = l.routed
        if l.shared is not None:
            arr[i].shared = l.shared
        else:
            arr[i].shared = moe_expert_bank(int(l.routed.wtype), 0, None, None, None, None)
    return arr


def moe_stack_forward(x, layers_arr, n_layers: int, T: int, eps: float, workspace, stream=None):
    lib = load()
    st = lib.moe_stack_forward(_ptr(x), layers_arr, int(n_layers), int(T), float(eps), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check("moe_stack_forward", st)


def moe_dense_gemv_nvfp4(x, w_packed, tscale: float, N: int, K: int, T: int, y, workspace, stream=None):
    """y[T][N] (bf16) = W x for a packed NVFP4 matrix W [N][K] (MOE_PACK_PLAIN)."""
    lib = load()
    st = lib.moe_dense_gemv_nvfp4(_ptr(x), _ptr(w_packed), float(tscale), int(N), int(K), int(T), _ptr(y),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    _check("moe_dense_gemv_nvfp4", st)


def moe_layer_forward_sink(x, router_w, routed: moe_expert_bank, shared: moe_expert_bank, out, T: int, workspace,
                           stream=None):
    """The layer with the shared experts as expert sinks (router_w [E + S][H])."""
    lib = load()
    st = lib.moe_layer_forward_sink(_ptr(x), _ptr(router_w), ctypes.byref(routed), ctypes.byref(shared), _ptr(out),
                                    int(T), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    _check("moe_layer_forward_sink", st)


def moe_read_shared_weights(workspace, T: int, n_shared: int, sw, stream=None):
    lib = load()
    st = lib.moe_read_shared_weights(_ptr(workspace), workspace.numel() * workspace.element_size(), int(T),
                                     int(n_shared), _ptr(sw), _stream(stream))
    _check("moe_read_shared_weights", st)
