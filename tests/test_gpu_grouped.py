"""The grouped path (T above the decode kernel's chunked range, 88 tokens for
NVFP4 weights and 56 for BF16;
moe_route above MOE_MAX_DECODE_T): router GEMM, top-k, expert lists and the
tcgen05 grouped GEMMs, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import nvfp4_moe_decode_gb300 as m
import oracle
from nvfp4_moe_decode_gb300 import synth
from nvfp4_moe_decode_gb300.layer import Bf16Layer, PackedLayer, new_workspace
from tests import helpers as hp

pytestmark = pytest.mark.gpu


def _route(li, dev):
    T = li.x.shape[0]
    ws = new_workspace(T, dev)
    idx = torch.empty(T, 6, dtype=torch.int32, device=dev)
    w = torch.empty(T, 6, dtype=torch.float32, device=dev)
    lg = torch.empty(T, 256, dtype=torch.float32, device=dev)
    m.moe_route(li.x, li.router_w, T, idx, w, lg, ws)
    assert m.moe_read_device_flag(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy().astype(np.float64)


# The tensor-core GEMM's logit bound (GEMM_DEPTH roundings of 2^-23) is about
# 70 times the error actually seen (at most 4.9e-7 of sum|x w| over 8192
# tokens), so 1-3% of random tokens fall inside it as "near ties" (135 of
# 8192).  Those must still be valid selections, and the GPU must pick the
# oracle's own set on all but a few (none so far).
def _max_differ(T: int) -> int:
    return 0 if T <= 512 else 2


@pytest.mark.parametrize("T", [9, 512, 8192])
def test_grouped_routing(cuda_dev, T):
    li = synth.make_layer(60 + T % 97, T, device=cuda_dev, weights=False)
    idx, w, lg_gpu = _route(li, cuda_dev)
    xb, wb = hp.bits16(li.x), hp.bits16(li.router_w)
    certain, near, same = hp.check_gpu_routing(xb, wb, idx, w, lg_gpu, hp.GEMM_DEPTH, 1e-5)
    lg = oracle.router_logits(xb, wb)
    ratio = np.max(np.abs(lg_gpu - lg) / (np.abs(hp.np_bf16(xb)) @ np.abs(hp.np_bf16(wb)).T + 1e-300))
    print(f"T={T}: near ties {len(near)}, GPU set differs on {T - len(same)} tokens, "
          f"max |logit err| / sum|x w| = {ratio:.3e} (bound {hp.gamma(hp.GEMM_DEPTH, 2 ** -23):.3e})")
    assert len(near) <= max(4, T // 20)
    assert T - len(same) <= _max_differ(T)


def _forward(lay, x, dev):
    T = x.shape[0]
    ws = new_workspace(T, dev)
    out = torch.full((T, m.HIDDEN), float("nan"), dtype=torch.bfloat16, device=dev)
    lay.forward(x.contiguous(), out, ws)
    return out, m.moe_read_device_flag(ws), ws


def _check(li, out, ws, tol, tokens=None):
    """The layer's own routing (read back from its workspace, every token)
    against the oracle's, then the outputs of the sampled tokens that the GPU
    routed like the oracle (all but near ties whose GPU set differs)."""
    T = li.x.shape[0]
    tokens = list(range(T)) if tokens is None else list(tokens)
    gidx, gw, glg = hp.read_routing(ws, T)
    xb, wb = hp.bits16(li.x), hp.bits16(li.router_w)
    _, near, same = hp.check_gpu_routing(xb, wb, gidx, gw, glg, hp.GEMM_DEPTH, 1e-5)
    assert len(near) <= max(4, T // 20), f"{len(near)} near-tie tokens"
    assert T - len(same) <= _max_differ(T), f"GPU set differs from the oracle's on {T - len(same)} tokens"
    ref, _, _, _, _ = hp.oracle_layer(li, tokens=tokens)
    got = hp.to_f64(out)[tokens]
    same_set = set(same)
    keep = [i for i, t in enumerate(tokens) if t in same_set]
    assert len(keep) >= len(tokens) - len(near)
    assert hp.within_tol(got[keep], ref[keep], tol), hp.describe_err(got[keep], ref[keep])


@pytest.mark.parametrize("T", [89, 161, 300])
def test_grouped_layer_small(cuda_dev, T):
    """From the first size above the chunked range (89 tokens) up."""
    li = synth.make_layer(70 + T, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    _check(li, out, ws, hp.TOL_NVFP4)


def test_grouped_layer_8192_sampled(cuda_dev):
    """The 8192-token configuration: the routing of all 8192 tokens checked,
    every output finite, and 512 tokens (first, last and random ones)
    compared with the oracle."""
    T = 8192
    li = synth.make_layer(0, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(8192)
    rest = rng.choice(np.arange(2, T - 1), 509, replace=False).tolist()
    toks = sorted(set([0, 1, T - 1] + rest))
    assert len(toks) == 512
    _check(li, out, ws, hp.TOL_NVFP4, toks)


def test_grouped_layer_max_tokens(cuda_dev):
    """The largest batch, MOE_MAX_TOKENS = 65,536 tokens (a 6.2 GB workspace):
    every output finite, every token's own routing valid (six distinct
    experts, positive weights that sum to 1), and 128 tokens (first, last and
    random ones) against the oracle: their routing (indices bit-exact where
    certain) and their outputs."""
    T = m.MAX_TOKENS
    li = synth.make_layer(65, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    assert torch.isfinite(out.float()).all()
    gidx, gw, glg = hp.read_routing(ws, T)
    srt = np.sort(gidx, axis=1)
    assert srt.min() >= 0 and srt.max() < 256 and np.all(srt[:, 1:] != srt[:, :-1])
    assert np.all(gw > 0) and np.all(np.abs(gw.sum(axis=1) - 1.0) <= 1e-5)
    rng = np.random.default_rng(T)
    toks = sorted(set([0, 1, T - 1] + rng.choice(np.arange(2, T - 1), 125, replace=False).tolist()))
    assert len(toks) == 128
    xb, wb = hp.bits16(li.x)[toks], hp.bits16(li.router_w)
    _, near, same = hp.check_gpu_routing(xb, wb, gidx[toks], gw[toks], glg[toks], hp.GEMM_DEPTH, 1e-5)
    assert len(near) <= 4, f"{len(near)} near-tie tokens of 128"
    ref, _, _, _, _ = hp.oracle_layer(li, tokens=toks)
    got = hp.to_f64(out)[toks]
    keep = sorted(same)
    assert len(keep) >= len(toks) - len(near)
    assert hp.within_tol(got[keep], ref[keep], hp.TOL_NVFP4), hp.describe_err(got[keep], ref[keep])


def test_grouped_zero_tokens_route_by_index(cuda_dev):
    """The grouped path with all-zero tokens among the others: experts 0..5
    in that order (a tie goes to the lower index), weights 1/6, and output
    rows exactly 0; the other tokens against the oracle."""
    T = 100
    li = synth.make_layer(430, T, device=cuda_dev)
    zeros = [0, 50, 99]
    li.x[zeros] = 0
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    gidx, gw, _ = hp.read_routing(ws, T)
    for t in zeros:
        assert gidx[t].tolist() == [0, 1, 2, 3, 4, 5]
        assert np.all(np.abs(gw[t] - 1.0 / 6.0) <= 1e-7)
        assert torch.count_nonzero(out[t].float()) == 0
    _check(li, out, ws, hp.TOL_NVFP4)


def test_grouped_nonfinite_router_weight_sets_flag(cuda_dev):
    """The grouped path with a NaN router weight (expert 17's logit NaN for
    every token): the flag is set, expert 17 is never selected, and every
    output is finite."""
    T = 100
    li = synth.make_layer(441, T, device=cuda_dev)
    li.router_w[17, 3] = float("nan")
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag & m.MOE_FLAG_NONFINITE_LOGIT
    gidx, gw, _ = hp.read_routing(ws, T)
    assert not np.any(gidx == 17)
    srt = np.sort(gidx, axis=1)
    assert np.all(srt[:, 1:] != srt[:, :-1]) and srt.min() >= 0 and srt.max() < 256
    assert np.all(gw > 0) and np.all(np.abs(gw.sum(axis=1) - 1.0) <= 1e-5)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("T", [57, 200])
def test_grouped_bf16_weights(cuda_dev, T):
    """BF16 weights, from the first size above their chunked range (57)."""
    li = synth.make_layer(80 + T, T, wtype=synth.BF16, device=cuda_dev)
    bl = Bf16Layer.from_inputs(li)
    out, flag, ws = _forward(bl, li.x, cuda_dev)
    assert flag == 0
    _check(li, out, ws, hp.TOL_BF16)


def test_grouped_without_shared_expert_and_determinism(cuda_dev):
    T = 170
    li = synth.make_layer(81, T, device=cuda_dev)
    li_ns = synth.LayerInputs(**{**li.__dict__, "n_shared": 0,
                                 "codes13": li.codes13[:256], "scales13": li.scales13[:256],
                                 "codes2": li.codes2[:256], "scales2": li.scales2[:256],
                                 "tscale13": li.tscale13[:256], "tscale2": li.tscale2[:256]})
    pl = PackedLayer.from_inputs(li_ns)
    out1, flag, ws = _forward(pl, li.x, cuda_dev)
    out2, _, _ = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    _check(li_ns, out1, ws, hp.TOL_NVFP4)


def test_grouped_expert_with_more_than_256_tokens(cuda_dev):
    """600 copies of one token: six experts get 600 tokens each (three token
    chunks of up to 256), every output row equal."""
    T = 600
    li = synth.make_layer(82, 1, device=cuda_dev)
    li.x = li.x.repeat(T, 1).contiguous()
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    assert torch.equal(out.view(torch.int16), out[:1].repeat(T, 1).view(torch.int16))
    _check(li, out, ws, hp.TOL_NVFP4, tokens=[0, 299, 599])
