"""Seeded synthetic inputs for the MoE layer (input generation only).

This module holds none of the layer's arithmetic: it only draws random
numbers with torch and casts them to the storage types.  Both the parity tests
(for the CUDA path and for the CPU oracle) and ``bench.py`` take their inputs
from here, so both sides see the same bytes.

Recipe (one ``torch.Generator`` per layer, seeded with ``seed``; draws in
this order):

1. ``x``        [T, H]      ~ N(0, 1), rounded to bf16 (round-to-nearest-even);
2. ``router_w`` [E, H]      ~ N(0, 0.02), rounded to bf16;
3. for all E routed experts plus the S shared ones (shared last):
   NVFP4: gate/up codes [2I, H/2] uniform bytes (each nibble uniform over the
   16 e2m1 codes), gate/up scales [2I, H/16] = |N(0,1)| * 0.05 rounded to e4m3
   (E4M3FN, round-to-nearest-even, subnormals kept, so some blocks get a zero
   scale), down codes [H, I/2], down scales [H, I/16] likewise; tensor scales
   1.0.  BF16: gate/up [2I, H] and down [H, I] ~ N(0, 0.02) rounded to bf16.

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


def _e4m3_scales(shape, g, device) -> torch.Tensor:
    s = torch.randn(shape, generator=g, device=device).abs_() * 0.05
    return s.to(torch.float8_e4m3fn).view(torch.uint8)


def make_layer(seed: int, T: int, hidden: int = 2048, n_routed: int = 256, inter: int = 512,
               n_shared: int = 1, wtype: int = NVFP4, device="cpu",
               weights: bool = True) -> LayerInputs:
    """Draw one layer's inputs.  ``weights=False`` draws only x and the router."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    H, E, I, S = hidden, n_routed, inter, n_shared
    x = torch.randn(T, H, generator=g, device=device).to(torch.bfloat16)
    router_w = (torch.randn(E, H, generator=g, device=device) * 0.02).to(torch.bfloat16)
    li = LayerInputs(x=x, router_w=router_w, wtype=wtype, n_routed=E, n_shared=S,
                     hidden=H, inter=I)
    if not weights:
        return li
    n = E + S
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
    return li


def make_x(seed: int, T: int, hidden: int = 2048, device="cpu") -> torch.Tensor:
    """Activations alone, drawn like step 1 of ``make_layer``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(T, hidden, generator=g, device=device).to(torch.bfloat16)
