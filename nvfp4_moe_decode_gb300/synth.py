"""Seeded synthetic inputs for the MoE layer (input generation only).

This module holds none of the layer's arithmetic: it only draws random
numbers with torch and casts them to the storage types.  Both the parity tests
(for the CUDA path and for the CPU oracle) and ``bench.py`` take their inputs
from here, so both sides see the same bytes.

Recipe (one ``torch.Generator`` per layer, seeded with ``seed``; draws in
this order):

1. ``x``        [T, H]      ~ N(0, 1), rounded to bf16 (round-to-nearest-even);
2. ``router_w`` [E, H]      ~ N(0, 0.02), rounded to bf16 ([E + S, H] for a
   layer whose S shared experts are expert sinks: their router rows last);
3. for all E routed experts plus the S shared ones (shared last):
   NVFP4: gate/up codes [2I, H/2] uniform bytes (each nibble uniform over the
   16 e2m1 codes), gate/up scales [2I, H/16] = |N(0,1)| * 0.05 rounded to e4m3
   (E4M3FN, round-to-nearest-even, subnormals kept, so some blocks get a zero
   scale), down codes [H, I/2], down scales [H, I/16] likewise; tensor scales
   1.0.  BF16: gate/up [2I, H] and down [H, I] ~ N(0, 0.02) rounded to bf16.
   When the shared experts are BF16 beside NVFP4 routed experts, the E routed
   experts are drawn first (NVFP4), then the S shared ones (BF16).

Dense GEMV inputs (``make_dense``, one generator seeded with ``seed``):
``x`` [T, K] ~ N(0, 1) rounded to bf16, then codes [N, K/2] uniform bytes and
scales [N, K/16] = |N(0,1)| * 0.05 rounded to e4m3, as for an expert matrix.

The canonical NVFP4 byte layout is: byte (n, j) of the codes holds element
(n, 2j) in its low nibble and (n, 2j+1) in its high nibble; scale (n, b)
covers elements (n, 16b .. 16b+15).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

NVFP4 = 0
BF16 = 1


@dataclass
class LayerInputs:
    x: torch.Tensor               # bf16 [T, H]
    router_w: torch.Tensor        # bf16 [E, H]
    wtype: int
    n_routed: int
    n_shared: int
    hidden: int
    inter: int
    # NVFP4 canonical arrays, experts stacked on dim 0 (routed first, shared last)
    codes13: Optional[torch.Tensor] = None   # u8 [E+S, 2I, H/2]
    scales13: Optional[torch.Tensor] = None  # u8 [E+S, 2I, H/16] (e4m3 bits)
    codes2: Optional[torch.Tensor] = None    # u8 [E+S, H, I/2]
    scales2: Optional[torch.Tensor] = None   # u8 [E+S, H, I/16]
    tscale13: Optional[torch.Tensor] = None  # f32 [E+S]
    tscale2: Optional[torch.Tensor] = None   # f32 [E+S]
    # BF16 weights
    w13: Optional[torch.Tensor] = None       # bf16 [E+S, 2I, H]
    w2: Optional[torch.Tensor] = None        # bf16 [E+S, H, I]
    # expert sinks: router_w has E + S rows, the shared experts' last
    sink: bool = False
    # BF16 shared experts beside NVFP4 routed ones (the arrays above then hold
    # the E routed experts only)
    shared_bf16: bool = False
    sw13: Optional[torch.Tensor] = None      # bf16 [S, 2I, H]
    sw2: Optional[torch.Tensor] = None       # bf16 [S, H, I]


def _e4m3_scales(shape, g, device) -> torch.Tensor:
    s = torch.randn(shape, generator=g, device=device).abs_() * 0.05
    return s.to(torch.float8_e4m3fn).view(torch.uint8)


def make_layer(seed: int, T: int, hidden: int = 2048, n_routed: int = 256, inter: int = 512,
               n_shared: int = 1, wtype: int = NVFP4, device="cpu",
               weights: bool = True, sink: bool = False, shared_bf16: bool = False) -> LayerInputs:
    """Draw one layer's inputs.  ``weights=False`` draws only x and the router.
    ``sink``: the shared experts are expert sinks (router rows for them);
    ``shared_bf16``: BF16 shared experts beside NVFP4 routed ones."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    H, E, I, S = hidden, n_routed, inter, n_shared
    x = torch.randn(T, H, generator=g, device=device).to(torch.bfloat16)
    router_w = (torch.randn(E + (S if sink else 0), H, generator=g, device=device) * 0.02).to(torch.bfloat16)
    li = LayerInputs(x=x, router_w=router_w, wtype=wtype, n_routed=E, n_shared=S,
                     hidden=H, inter=I, sink=sink)
    if not weights:
        return li
    if shared_bf16 and wtype != NVFP4:
        raise ValueError("shared_bf16 pairs BF16 shared experts with NVFP4 routed ones")
    li.shared_bf16 = bool(shared_bf16)
    n = E if shared_bf16 else E + S
    if wtype == NVFP4:
        li.codes13 = torch.randint(0, 256, (n, 2 * I, H // 2), generator=g, device=device,
                                   dtype=torch.uint8)
        li.scales13 = _e4m3_scales((n, 2 * I, H // 16), g, device)
        li.codes2 = torch.randint(0, 256, (n, H, I // 2), generator=g, device=device,
                                  dtype=torch.uint8)
        li.scales2 = _e4m3_scales((n, H, I // 16), g, device)
        li.tscale13 = torch.ones(n, dtype=torch.float32, device=device)
        li.tscale2 = torch.ones(n, dtype=torch.float32, device=device)
    elif wtype == BF16:
        li.w13 = (torch.randn(n, 2 * I, H, generator=g, device=device) * 0.02).to(torch.bfloat16)
        li.w2 = (torch.randn(n, H, I, generator=g, device=device) * 0.02).to(torch.bfloat16)
    else:
        raise ValueError(f"unknown wtype {wtype}")
    if shared_bf16:
        li.sw13 = (torch.randn(S, 2 * I, H, generator=g, device=device) * 0.02).to(torch.bfloat16)
        li.sw2 = (torch.randn(S, H, I, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return li


def make_x(seed: int, T: int, hidden: int = 2048, device="cpu") -> torch.Tensor:
    """Activations alone, drawn like step 1 of ``make_layer``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(T, hidden, generator=g, device=device).to(torch.bfloat16)


@dataclass
class DenseInputs:
    x: torch.Tensor        # bf16 [T, K]
    codes: torch.Tensor    # u8 [N, K/2]
    scales: torch.Tensor   # u8 [N, K/16] (e4m3 bits)


def make_dense(seed: int, T: int, N: int, K: int, device="cpu") -> DenseInputs:
    """Draw the activations and one canonical NVFP4 matrix of a dense GEMV."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(T, K, generator=g, device=device).to(torch.bfloat16)
    codes = torch.randint(0, 256, (N, K // 2), generator=g, device=device, dtype=torch.uint8)
    scales = _e4m3_scales((N, K // 16), g, device)
    return DenseInputs(x=x, codes=codes, scales=scales)
