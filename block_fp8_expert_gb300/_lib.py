"""ctypes binding of libmoe_fp8.so (include/moe_fp8.h).

Argument marshalling only: every function here passes device pointers, sizes
and the current CUDA stream to the C ABI of the same name and turns a non-zero
status into an exception.  Every step of the layer runs in the library's CUDA
kernels; there is no Python or CPU fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_fp8.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_STATUS = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_NOT_IMPLEMENTED = 7
MOE_DEV_BAD_EXPERT_INDEX = 1
MOE_DEV_WAIT_TIMEOUT = 2
MOE_DEV_FP16_RANGE = 4
MOE_DEV_NONFINITE = 8


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status}: {message}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("I_shared", ctypes.c_int32)]

    def __repr__(self):
        return (f"Dims(T={self.T}, H={self.H}, I={self.I}, E={self.E}, k={self.k}, "
                f"I_shared={self.I_shared})")


class Fp8Mat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class Fp8Ffn(ctypes.Structure):
    _fields_ = [("gate", Fp8Mat), ("up", Fp8Mat), ("down", Fp8Mat)]


_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_st = ctypes.c_int32

_SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_st]),
    "moe_last_error_message": (ctypes.c_char_p, []),
    "moe_version": (ctypes.c_char_p, []),
    "moe_kernel_launches": (ctypes.c_ulonglong, []),
    "moe_expert_uses_gemm": (ctypes.c_int, [Dims]),
    "moe_workspace_bytes": (_st, [Dims, ctypes.POINTER(_sz)]),
    "moe_route": (_st, [_vp, _vp, _vp, Dims, _vp, _vp, _vp, _sz, _vp]),
    "moe_permute": (_st, [_vp, Dims, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_expert_ffn_fp8": (_st, [_vp, _vp, _vp, Fp8Ffn, Dims, _vp, _vp, _sz, _vp]),
    "moe_combine": (_st, [_vp, _vp, _vp, _vp, Dims, _vp, _vp]),
    "moe_layer_forward": (_st, [_vp, _vp, _vp, Fp8Ffn, ctypes.POINTER(Fp8Ffn), Dims, _vp, _vp,
                                _vp, _vp, _sz, _vp]),
    "moe_layer_forward_gated": (_st, [_vp, _vp, _vp, Fp8Ffn, ctypes.POINTER(Fp8Ffn), _vp, Dims,
                                      _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_layer_forward_act8": (_st, [_vp, _vp, _vp, Fp8Ffn, Dims, _vp, _vp, _vp, _vp, _sz,
                                     _vp]),
    "moe_verify_workspace_bytes": (_st, [Dims, ctypes.c_int, ctypes.POINTER(_sz)]),
    "moe_verify_layer": (_st, [_vp, Fp8Ffn, ctypes.POINTER(Fp8Ffn), _vp, Dims, _vp, _vp, _vp,
                               _vp, ctypes.c_int, _vp, _vp, _sz, _vp]),
    "moe_read_device_status": (_st, [_vp, ctypes.POINTER(ctypes.c_int32), _vp]),
    "moe_permute_static_scratch": (_st, [_vp, Dims, _vp, _vp, _vp, _vp]),
}

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with block_fp8_expert_gb300.build.build(); "
                "this package has no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        msg = lib().moe_last_error_message().decode()
        raise MoeError(status, where, msg)


def _ptr(t) -> Optional[int]:
    """Device address of a tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def dims(T: int, H: int, I: int, E: int, k: int, I_shared: int = 0) -> Dims:
    return Dims(T, H, I, E, k, I_shared)


def ffn(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales) -> Fp8Ffn:
    return Fp8Ffn(Fp8Mat(_ptr(gate_codes), _ptr(gate_scales)),
                  Fp8Mat(_ptr(up_codes), _ptr(up_scales)),
                  Fp8Mat(_ptr(down_codes), _ptr(down_scales)))


def version() -> str:
    return lib().moe_version().decode()


def kernel_launches() -> int:
    """Kernel launches this library has issued in this process (diagnostic)."""
    return int(lib().moe_kernel_launches())


def expert_uses_gemm(d) -> bool:
    """True if a layer call with dims d runs its routed experts on the
    tensor-core GEMM (diagnostic; raises on invalid dims)."""
    r = int(lib().moe_expert_uses_gemm(d))
    if r < 0:
        raise ValueError("invalid moe_dims")
    return r == 1


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def workspace_bytes(d: Dims) -> int:
    n = _sz(0)
    _check(lib().moe_workspace_bytes(d, ctypes.byref(n)), "moe_workspace_bytes")
    return n.value


def _nbytes(ws) -> int:
    return ws.numel() * ws.element_size()


def moe_route(x, Wr, bias, d: Dims, topk_idx, topk_w, ws, stream=None) -> None:
    _check(lib().moe_route(_ptr(x), _ptr(Wr), _ptr(bias), d, _ptr(topk_idx), _ptr(topk_w),
                           _ptr(ws), _nbytes(ws), _stream(stream)), "moe_route")


def moe_permute(topk_idx, d: Dims, expert_off, row_token, tok_slot_row, ws, stream=None) -> None:
    _check(lib().moe_permute(_ptr(topk_idx), d, _ptr(expert_off), _ptr(row_token),
                             _ptr(tok_slot_row), _ptr(ws), _nbytes(ws), _stream(stream)),
           "moe_permute")


def moe_permute_static_scratch(topk_idx, d: Dims, expert_off, row_token, tok_slot_row,
                               stream=None) -> None:
    """moe_permute with its scratch in the library's fixed device array
    (no workspace argument; T*k <= 65536, E <= 512)."""
    _check(lib().moe_permute_static_scratch(_ptr(topk_idx), d, _ptr(expert_off),
                                            _ptr(row_token), _ptr(tok_slot_row),
                                            _stream(stream)), "moe_permute_static_scratch")


def moe_expert_ffn_fp8(x, expert_off, row_token, w: Fp8Ffn, d: Dims, y_perm, ws,
                       stream=None) -> None:
    _check(lib().moe_expert_ffn_fp8(_ptr(x), _ptr(expert_off), _ptr(row_token), w, d,
                                    _ptr(y_perm), _ptr(ws), _nbytes(ws), _stream(stream)),
           "moe_expert_ffn_fp8")


def moe_combine(y_perm, tok_slot_row, topk_w, shared_y, d: Dims, out, stream=None) -> None:
    _check(lib().moe_combine(_ptr(y_perm), _ptr(tok_slot_row), _ptr(topk_w), _ptr(shared_y), d,
                             _ptr(out), _stream(stream)), "moe_combine")


def moe_layer_forward(x, Wr, bias, routed: Fp8Ffn, shared: Optional[Fp8Ffn], d: Dims, out,
                      topk_idx_out, topk_w_out, ws, stream=None) -> None:
    sh = ctypes.byref(shared) if shared is not None else None
    _check(lib().moe_layer_forward(_ptr(x), _ptr(Wr), _ptr(bias), routed, sh, d, _ptr(out),
                                   _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(ws), _nbytes(ws),
                                   _stream(stream)), "moe_layer_forward")


def moe_layer_forward_gated(x, Wr, bias, routed: Fp8Ffn, shared: Fp8Ffn, shared_gate, d: Dims,
                            out, topk_idx_out, topk_w_out, ws, stream=None) -> None:
    _check(lib().moe_layer_forward_gated(_ptr(x), _ptr(Wr), _ptr(bias), routed,
                                         ctypes.byref(shared), _ptr(shared_gate), d, _ptr(out),
                                         _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(ws),
                                         _nbytes(ws), _stream(stream)), "moe_layer_forward_gated")


def moe_layer_forward_act8(x, Wr, bias, routed: Fp8Ffn, d: Dims, out, topk_idx_out, topk_w_out,
                           ws, stream=None) -> None:
    _check(lib().moe_layer_forward_act8(_ptr(x), _ptr(Wr), _ptr(bias), routed, d, _ptr(out),
                                        _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(ws),
                                        _nbytes(ws), _stream(stream)), "moe_layer_forward_act8")


def verify_workspace_bytes(d: Dims, n_tokens: int) -> int:
    n = _sz(0)
    _check(lib().moe_verify_workspace_bytes(d, n_tokens, ctypes.byref(n)),
           "moe_verify_workspace_bytes")
    return n.value


def moe_verify_layer(x, routed: Fp8Ffn, shared: Optional[Fp8Ffn], shared_gate, d: Dims, out,
                     topk_idx, topk_w, tokens, result, ws, stream=None) -> None:
    sh = ctypes.byref(shared) if shared is not None else None
    _check(lib().moe_verify_layer(_ptr(x), routed, sh, _ptr(shared_gate), d, _ptr(out),
                                  _ptr(topk_idx), _ptr(topk_w), _ptr(tokens),
                                  int(tokens.numel()), _ptr(result), _ptr(ws), _nbytes(ws),
                                  _stream(stream)), "moe_verify_layer")


def moe_read_device_status(ws, stream=None) -> int:
    """The workspace's device status bits; raises MoeError when any is set.
    ws=None reads the status word of moe_permute_static_scratch's fixed array."""
    v = ctypes.c_int32(0)
    st = lib().moe_read_device_status(_ptr(ws), ctypes.byref(v), _stream(stream))
    if st not in (MOE_OK, MOE_ERR_DEVICE_STATUS):
        _check(st, "moe_read_device_status")
    if st == MOE_ERR_DEVICE_STATUS:
        raise MoeError(st, "moe_read_device_status", f"device status bits 0x{v.value:x}")
    return v.value


EXPORTED = tuple(_SIGNATURES)
