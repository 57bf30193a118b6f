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

# The decode layer kernel's own router: each lane chains 8 exact products per
# token (7 roundings after the first), then two balanced 16-way trees (4 + 4).
LAYER_ROUTER_DEPTH = 15

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


def read_routing(ws: torch.Tensor, T: int):
    """The routing the last layer call on ``ws`` used (the GPU's own), as
    numpy (idx int32 [T, 6], w fp64 [T, 6], logits fp64 [T, 256])."""
    import nvfp4_moe_decode_gb300 as m

    dev = ws.device
    idx = torch.full((T, 6), -1, dtype=torch.int32, device=dev)
    w = torch.full((T, 6), float("nan"), dtype=torch.float32, device=dev)
    lg = torch.full((T, 256), float("nan"), dtype=torch.float32, device=dev)
    m.moe_read_routing(ws, T, idx, w, lg)
    torch.cuda.synchronize(dev)
    return idx.cpu().numpy(), w.cpu().numpy().astype(np.float64), lg.cpu().numpy().astype(np.float64)


def check_gpu_routing(x_bits: np.ndarray, wr_bits: np.ndarray, gidx: np.ndarray, gw: np.ndarray,
                      glg: np.ndarray, depth: int, w_tol: float):
    """Check a GPU routing (indices, weights, fp32 logits) against the oracle.

    * every GPU logit lies within the certified bound for a summation of the
      given depth;
    * on every token whose selection is certain under those bounds, the GPU
      selected exactly the oracle's experts; where the six selected logits
      are also ordered beyond the bounds, in the same order;
    * every near-tie token's GPU selection is one the bounds allow;
    * weights: renormalised, positive, and within ``w_tol`` of the oracle's
      (matched by expert) wherever the two sets agree.
    Returns (certain, near, same): tokens certain, near ties, and tokens whose
    GPU set equals the oracle's (the ones whose outputs are comparable)."""
    T = x_bits.shape[0]
    lg = oracle.router_logits(x_bits, wr_bits)
    bounds = logit_bounds(x_bits, wr_bits, depth)
    err = np.abs(glg - lg)
    assert np.all(err <= bounds), f"logit outside its bound: max ratio {np.max(err / bounds):.3f}"
    oidx, ow = oracle.select_topk(lg, 6)
    certain, near, invalid = classify_selection(lg, bounds, oidx, gidx)
    assert not invalid, f"invalid selections at tokens {invalid[:8]}"
    same = []
    for t in range(T):
        g = gidx[t].tolist()
        assert len(set(g)) == 6 and min(g) >= 0 and max(g) < 256
        assert np.all(gw[t] > 0) and abs(gw[t].sum() - 1.0) <= 1e-5
        if set(g) != set(oidx[t].tolist()):
            continue
        same.append(t)
        o = oidx[t]
        ordered = all(lg[t, o[i]] - bounds[t, o[i]] > lg[t, o[i + 1]] + bounds[t, o[i + 1]] for i in range(5))
        if ordered:
            assert np.array_equal(gidx[t], o), (t, gidx[t], o)
        for i in range(6):
            j = int(np.where(o == gidx[t][i])[0][0])
            assert abs(gw[t][i] - ow[t][j]) <= w_tol, (t, i, gw[t][i], ow[t][j])
    assert set(certain) <= set(same)
    return certain, near, same


def check_decode_layer(li: synth.LayerInputs, x: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, tol,
                       depth: int = LAYER_ROUTER_DEPTH, max_near: int = 1):
    """A decode-path layer call (T <= 8) on ``ws``: its own routing against the
    oracle's (check_gpu_routing), then its output against the oracle on every
    token routed like the oracle.  Returns (gpu out, oracle out) in fp64."""
    T = x.shape[0]
    gidx, gw, glg = read_routing(ws, T)
    _, near, same = check_gpu_routing(bits16(x), bits16(li.router_w), gidx, gw, glg, depth, 2e-6)
    assert len(near) <= max_near, f"{len(near)} near-tie tokens"
    sub = synth.LayerInputs(**{**li.__dict__, "x": x})
    ref, _, _, _, _ = oracle_layer(sub)
    got = to_f64(out)
    assert len(same) >= T - len(near)
    assert within_tol(got[same], ref[same], tol), describe_err(got[same], ref[same])
    return got, ref


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
