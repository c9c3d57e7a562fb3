"""Device-resident layer weights and a convenience forward call.

PyTorch provides the device memory and the stream; the layer itself runs in
libmoe_fp8.so through the binding in ``_lib``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import _lib


def _dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


@dataclasses.dataclass
class DeviceFfn:
    gate_codes: torch.Tensor
    gate_scales: torch.Tensor
    up_codes: torch.Tensor
    up_scales: torch.Tensor
    down_codes: torch.Tensor
    down_scales: torch.Tensor

    def abi(self) -> _lib.Fp8Ffn:
        return _lib.ffn(self.gate_codes, self.gate_scales, self.up_codes, self.up_scales,
                        self.down_codes, self.down_scales)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in dataclasses.astuple(self))


@dataclasses.dataclass
class DeviceLayer:
    """One MoE layer's weights in HBM (layouts as in include/moe_fp8.h)."""
    H: int
    I: int
    E: int
    k: int
    I_shared: int
    Wr: torch.Tensor
    bias: Optional[torch.Tensor]
    routed: DeviceFfn
    shared: Optional[DeviceFfn]
    # gated shared expert: float32 [H] (None: ungated)
    shared_gate_w: Optional[torch.Tensor] = None

    @classmethod
    def from_host(cls, layer, device="cuda") -> "DeviceLayer":
        """Upload a layer drawn by ``moe_inputs.make_layer`` (or any object
        with the same fields)."""
        def ffn(g, u, d):
            return DeviceFfn(_dev(g.codes, device), _dev(g.scales, device),
                             _dev(u.codes, device), _dev(u.scales, device),
                             _dev(d.codes, device), _dev(d.scales, device))
        shared = None
        if layer.I_shared:
            shared = ffn(layer.shared_gate, layer.shared_up, layer.shared_down)
        gw = getattr(layer, "shared_gate_w", None)
        return cls(H=layer.H, I=layer.I, E=layer.E, k=layer.k, I_shared=layer.I_shared,
                   Wr=_dev(layer.Wr, device),
                   bias=None if layer.bias is None else _dev(layer.bias, device),
                   routed=ffn(layer.gate, layer.up, layer.down), shared=shared,
                   shared_gate_w=None if gw is None else _dev(gw, device))

    def dims(self, T: int) -> _lib.Dims:
        return _lib.dims(T, self.H, self.I, self.E, self.k, self.I_shared)

    def workspace(self, T: int) -> torch.Tensor:
        n = _lib.workspace_bytes(self.dims(T))
        return torch.empty(n, dtype=torch.uint8, device=self.Wr.device)

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None,
                ws: Optional[torch.Tensor] = None, topk_idx: Optional[torch.Tensor] = None,
                topk_w: Optional[torch.Tensor] = None, stream=None,
                act8: bool = False) -> torch.Tensor:
        """out[T, H] (bf16) = the layer applied to x[T, H] (bf16).  act8: the
        routed experts on E4M3 activations (moe_layer_forward_act8)."""
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        if ws is None:
            ws = self.workspace(T)
        if act8:
            _lib.moe_layer_forward_act8(x, self.Wr, self.bias, self.routed.abi(), self.dims(T),
                                        out, topk_idx, topk_w, ws, stream)
        elif self.shared_gate_w is not None:
            _lib.moe_layer_forward_gated(x, self.Wr, self.bias, self.routed.abi(),
                                         self.shared.abi(), self.shared_gate_w, self.dims(T), out,
                                         topk_idx, topk_w, ws, stream)
        else:
            _lib.moe_layer_forward(x, self.Wr, self.bias, self.routed.abi(),
                                   self.shared.abi() if self.shared is not None else None,
                                   self.dims(T), out, topk_idx, topk_w, ws, stream)
        return out


    def verify(self, x: torch.Tensor, out: torch.Tensor, topk_idx: torch.Tensor,
               topk_w: torch.Tensor, tokens, stream=None) -> dict:
        """Runtime cross-check of a forward call on the listed tokens (at most
        64): the worst error in units of the layer tolerance, the worst
        absolute error and rms of the recomputed outputs (see
        moe_verify_layer)."""
        T = x.shape[0]
        tok = torch.as_tensor(tokens, dtype=torch.int32).to(x.device)
        d = self.dims(T)
        ws = torch.empty(_lib.verify_workspace_bytes(d, int(tok.numel())), dtype=torch.uint8,
                         device=x.device)
        res = torch.empty(3, dtype=torch.float32, device=x.device)
        _lib.moe_verify_layer(x, self.routed.abi(),
                              self.shared.abi() if self.shared is not None else None,
                              self.shared_gate_w, d, out, topk_idx, topk_w, tok, res, ws, stream)
        r = res.cpu().tolist()
        return {"max_err_over_tol": r[0], "max_abs_err": r[1], "rms_ref": r[2]}


def x_to_device(x_bits: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (uint16 [T, H]) -> a bf16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(device).view(
        torch.bfloat16)
