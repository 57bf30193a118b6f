"""Device-resident packed layers (marshalling around moe_pack_nvfp4).

``PackedLayer`` takes a layer's canonical arrays (see ``synth``), allocates
the packed banks with torch and packs them with the library's kernels; it
then hands ``moe_layer_forward`` the bank descriptors.  Nothing here computes
any part of the layer.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (HIDDEN, INTER, MOE_PACK_GATE_UP, MOE_PACK_PLAIN, MOE_W_BF16, MOE_W_NVFP4, layer_weights_array,
               make_bank, moe_layer_forward, moe_layer_forward_sink, moe_pack_nvfp4, moe_packed_bytes,
               moe_stack_forward, moe_stack_workspace_bytes, moe_workspace_bytes, moe_workspace_init)


class PackedLayer:
    """Packed NVFP4 weights of one MoE layer (routed bank + optional shared
    experts, packed after the routed ones, or BF16 shared experts given as
    ``shared_w13`` [S, 2I, H] / ``shared_w2`` [S, H, I]).  ``sink``: the shared
    experts are expert sinks (moe_layer_forward_sink)."""

    def __init__(self, router_w: torch.Tensor, codes13, scales13, codes2, scales2, tscale13, tscale2,
                 n_routed: int, n_shared: int, stream=None, shared_w13=None, shared_w2=None, sink: bool = False):
        H, I = HIDDEN, INTER
        self.sink = bool(sink)
        n = n_routed + (0 if shared_w13 is not None else n_shared)
        dev = codes13.device
        self.router_w = router_w.contiguous()
        self.n_routed, self.n_shared = n_routed, n_shared
        self.pb13 = moe_packed_bytes(2 * I, H)
        self.pb2 = moe_packed_bytes(H, I)
        self.w13 = torch.empty(n * self.pb13, dtype=torch.uint8, device=dev)
        self.w2 = torch.empty(n * self.pb2, dtype=torch.uint8, device=dev)
        moe_pack_nvfp4(codes13.contiguous(), scales13.contiguous(), 2 * I, H, MOE_PACK_GATE_UP, n,
                       self.w13, stream)
        moe_pack_nvfp4(codes2.contiguous(), scales2.contiguous(), H, I, MOE_PACK_PLAIN, n, self.w2,
                       stream)
        self.ts13 = tscale13.to(device=dev, dtype=torch.float32).contiguous()
        self.ts2 = tscale2.to(device=dev, dtype=torch.float32).contiguous()
        self.routed = make_bank(MOE_W_NVFP4, n_routed, self.w13, self.w2, self.ts13, self.ts2)
        self.shared = None
        if n_shared and shared_w13 is not None:
            self.sw13 = shared_w13.contiguous()
            self.sw2 = shared_w2.contiguous()
            self.shared = make_bank(MOE_W_BF16, n_shared, self.sw13, self.sw2)
        elif n_shared:
            self.shared = make_bank(MOE_W_NVFP4, n_shared, self.w13.data_ptr() + n_routed * self.pb13,
                                    self.w2.data_ptr() + n_routed * self.pb2,
                                    self.ts13.data_ptr() + 4 * n_routed, self.ts2.data_ptr() + 4 * n_routed)

    @classmethod
    def from_inputs(cls, li, stream=None) -> "PackedLayer":
        return cls(li.router_w, li.codes13, li.scales13, li.codes2, li.scales2, li.tscale13, li.tscale2,
                   li.n_routed, li.n_shared, stream, shared_w13=li.sw13 if li.shared_bf16 else None,
                   shared_w2=li.sw2 if li.shared_bf16 else None, sink=li.sink)

    def bytes_resident(self) -> int:
        return self.w13.numel() + self.w2.numel() + self.router_w.numel() * 2

    def forward(self, x: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, stream=None):
        fwd = moe_layer_forward_sink if self.sink else moe_layer_forward
        fwd(x, self.router_w, self.routed, self.shared, out, x.shape[0], workspace, stream)


class Bf16Layer:
    """BF16 weights of one MoE layer (the W16A16 variant): the banks point at the
    row-major bf16 tensors themselves (W13 [E+S, 2I, H], W2 [E+S, H, I]); no
    packing."""

    def __init__(self, router_w: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, n_routed: int,
                 n_shared: int, sink: bool = False):
        H, I = HIDDEN, INTER
        self.sink = bool(sink)
        n = n_routed + n_shared
        assert w13.dtype == torch.bfloat16 and tuple(w13.shape) == (n, 2 * I, H)
        assert w2.dtype == torch.bfloat16 and tuple(w2.shape) == (n, H, I)
        self.router_w = router_w.contiguous()
        self.w13 = w13.contiguous()
        self.w2 = w2.contiguous()
        self.n_routed, self.n_shared = n_routed, n_shared
        self.routed = make_bank(MOE_W_BF16, n_routed, self.w13, self.w2)
        self.shared = None
        if n_shared:
            self.shared = make_bank(MOE_W_BF16, n_shared, self.w13[n_routed], self.w2[n_routed])

    @classmethod
    def from_inputs(cls, li) -> "Bf16Layer":
        return cls(li.router_w, li.w13, li.w2, li.n_routed, li.n_shared, sink=li.sink)

    def bytes_resident(self) -> int:
        return (self.w13.numel() + self.w2.numel() + self.router_w.numel()) * 2

    def forward(self, x: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, stream=None):
        fwd = moe_layer_forward_sink if self.sink else moe_layer_forward
        fwd(x, self.router_w, self.routed, self.shared, out, x.shape[0], workspace, stream)


def new_workspace(T: int, device="cuda", stream=None) -> torch.Tensor:
    nbytes = moe_workspace_bytes(T)
    if nbytes == 0:
        raise ValueError(f"unsupported token count {T}")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


class Stack:
    """A pre-norm decoder stack of MoE layers (PackedLayer or Bf16Layer
    objects): x <- x + MoE_l(RMSNorm(x)) for each layer, one
    moe_stack_forward call."""

    def __init__(self, layers, eps: float = 1e-6):
        self.layers = list(layers)
        self.eps = float(eps)
        self.arr = layer_weights_array(self.layers)

    def forward(self, x: torch.Tensor, workspace: torch.Tensor, stream=None):
        moe_stack_forward(x, self.arr, len(self.layers), x.shape[0], self.eps, workspace, stream)


def new_stack_workspace(T: int, device="cuda", stream=None) -> torch.Tensor:
    nbytes = moe_stack_workspace_bytes(T)
    if nbytes == 0:
        raise ValueError(f"unsupported token count {T}")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws
