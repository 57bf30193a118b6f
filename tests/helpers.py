"""Shared helpers of the GPU parity tests.

Inputs come from ``nvfp4_moe_decode_gb300.synth`` (seeded, drawn on the
device); the expected values come from the fp64 oracle (``oracle``) fed with
the same input bytes copied to the host.  Nothing the CUDA path computes is
ever handed to the oracle.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np
import torch

import oracle
from nvfp4_moe_decode_gb300 import synth

U32 = 2.0 ** -24
U64 = 2.0 ** -53

# The router kernel sums every logit as a tree of exact fp32 products of
# depth 24 (16 sequential per lane, a 5-level butterfly, 3 quarter adds).
ROUTER_DEPTH = 24

# Output tolerances of the layer (the parity target of this project):
#   NVFP4: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3
#   BF16 : max|gpu - ref| <= 5e-3 * max|ref| + 1e-3
TOL_NVFP4 = (1e-2, 1e-3)
TOL_BF16 = (5e-3, 1e-3)


def gamma(n: int, u: float) -> float:
    return n * u / (1.0 - n * u)


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def np_bf16(u16: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def host_expert(li: synth.LayerInputs, e: int) -> oracle.ExpertWeights:
    if li.wtype == synth.NVFP4:
        return oracle.ExpertWeights(0, li.codes13[e].cpu().numpy(), li.scales13[e].cpu().numpy(),
                                    float(li.tscale13[e]), li.codes2[e].cpu().numpy(),
                                    li.scales2[e].cpu().numpy(), float(li.tscale2[e]))
    return oracle.ExpertWeights(1, bits16(li.w13[e]), None, 1.0, bits16(li.w2[e]), None, 1.0)


def oracle_layer(li: synth.LayerInputs, top_k: int = 6, tokens: Optional[Iterable[int]] = None):
    """Run the oracle on (a subset of) the tokens of a device-resident layer.

    The oracle routes first; only the experts it selects are copied to the
    host.  Returns (out [T', H] fp64, idx, w, logits, token list)."""
    x = bits16(li.x)
    if tokens is not None:
        tokens = list(tokens)
        x = np.ascontiguousarray(x[tokens])
    else:
        tokens = list(range(x.shape[0]))
    wr = bits16(li.router_w)
    logits = oracle.router_logits(x, wr)
    idx, _ = oracle.select_topk(logits, top_k)
    needed = sorted(set(idx.reshape(-1).tolist()))
    experts = [None] * li.n_routed
    for e in needed:
        experts[e] = host_expert(li, e)
    shared = host_expert(li, li.n_routed) if li.n_shared else None
    out, idx2, w, lg = oracle.moe_forward(x, wr, experts, top_k, li.inter, shared)
    assert np.array_equal(idx, idx2)
    return out, idx2, w, lg, tokens


# Above MAX_DECODE_T tokens the logits come from a tcgen05 GEMM: 128 MMAs of
# K = 16 accumulate in sequence into fp32.  The rounding inside one MMA is not
# documented; the bound allows 16 further roundings per MMA and takes the
# unit as 2^-23 (truncation) instead of 2^-24.
GEMM_DEPTH = 2 * (2048 // 16 + 16)


def logit_bounds(x_bits: np.ndarray, wr_bits: np.ndarray, depth: int = ROUTER_DEPTH) -> np.ndarray:
    """Per-logit bound on |fp32 router logit - exact|, plus the oracle's own
    fp64 summation error: (gamma_depth(fp32) + gamma_H(fp64)) * sum_k |x_k w_ek|."""
    ax = np.abs(np_bf16(x_bits))
    aw = np.abs(np_bf16(wr_bits))
    H = ax.shape[1]
    return (gamma(depth, U32) + gamma(H, U64)) * (ax @ aw.T) + 1e-300


def classify_selection(logits: np.ndarray, bounds: np.ndarray, oracle_idx: np.ndarray,
                       gpu_idx: np.ndarray):
    """Return (certain_tokens, near_tie_tokens, invalid_tokens).

    A token is certain when every oracle-selected expert's logit interval lies
    strictly above every other expert's; then the GPU set must equal the
    oracle set.  Otherwise (a near tie within the bounds) the GPU set must be
    one that some logits within the bounds would select."""
    certain, near, invalid = [], [], []
    T, E = logits.shape
    for t in range(T):
        o = set(oracle_idx[t].tolist())
        g = set(gpu_idx[t].tolist())
        sel = np.array(sorted(o))
        rest = np.array([e for e in range(E) if e not in o])
        lo = (logits[t, sel] - bounds[t, sel]).min()
        hi = (logits[t, rest] + bounds[t, rest]).max()
        if lo > hi:
            certain.append(t)
            if g != o:
                invalid.append(t)
        else:
            near.append(t)
            gs = np.array(sorted(g))
            grest = np.array([e for e in range(E) if e not in g])
            ok = len(g) == len(o) and (logits[t, gs] + bounds[t, gs]).min() >= \
                (logits[t, grest] - bounds[t, grest]).max()
            if not ok:
                invalid.append(t)
    return certain, near, invalid


def max_abs_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(gpu - ref))) if ref.size else 0.0


def within_tol(gpu: np.ndarray, ref: np.ndarray, tol) -> bool:
    rel, ab = tol
    return max_abs_err(gpu, ref) <= rel * float(np.max(np.abs(ref))) + ab


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def describe_err(gpu: np.ndarray, ref: np.ndarray) -> str:
    m = float(np.max(np.abs(ref))) if ref.size else 0.0
    e = max_abs_err(gpu, ref)
    return f"max|err|={e:.3e} max|ref|={m:.3e} rel={e / m if m else math.nan:.3e}"
