"""Shared experts run ahead of the layer kernel (the dense GEMV): expert-sink
routing (moe_layer_forward_sink; TML Inkling, section "MoE") and shared banks
of two experts or of the other weight type (moe_layer_forward), against the
fp64 oracle: the layer's own routing (indices bit-exact on every certain
token, weights and the shared experts' weights within 2e-6) and the output
within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_moe_decode_gb300 as m
from nvfp4_moe_decode_gb300 import synth
from nvfp4_moe_decode_gb300.layer import Bf16Layer, PackedLayer, new_workspace
from tests import helpers as hp

pytestmark = pytest.mark.gpu

E = 256
W_TOL = 2e-6


def shared_experts(li: synth.LayerInputs):
    if li.shared_bf16:
        return [oracle.ExpertWeights(1, hp.bits16(li.sw13[j]), None, 1.0, hp.bits16(li.sw2[j]), None, 1.0)
                for j in range(li.n_shared)]
    return [hp.host_expert(li, E + j) for j in range(li.n_shared)]


def oracle_routing(li: synth.LayerInputs, lg: np.ndarray):
    if li.sink:
        return oracle.select_topk_sink(lg, E, 6)
    idx, w = oracle.select_topk(lg[:, :E], 6)
    return idx, w, np.ones((lg.shape[0], li.n_shared))


def oracle_layer_shared(li: synth.LayerInputs):
    """The oracle layer; only the experts it selects are copied to the host."""
    x, wr = hp.bits16(li.x), hp.bits16(li.router_w)
    idx, _, _ = oracle_routing(li, oracle.router_logits(x, wr))
    experts = [None] * E
    for e in sorted(set(idx.reshape(-1).tolist())):
        experts[e] = hp.host_expert(li, e)
    out, idx2, w, sw, _ = oracle.moe_forward_sinks(x, wr, experts, 6, li.inter, shared_experts(li), li.sink)
    assert np.array_equal(idx, idx2)
    return out, sw


def check_shared_layer(li: synth.LayerInputs, out: torch.Tensor, ws: torch.Tensor, tol):
    T = li.x.shape[0]
    x, wr = hp.bits16(li.x), hp.bits16(li.router_w)
    gidx, gw, glg = hp.read_routing(ws, T)
    gsw = torch.full((T, li.n_shared), float("nan"), dtype=torch.float32, device=ws.device)
    m.moe_read_shared_weights(ws, T, li.n_shared, gsw)
    torch.cuda.synchronize()
    gsw = gsw.cpu().numpy().astype(np.float64)
    # the routed logits within the certified bound of the layer's router
    lg = oracle.router_logits(x, wr)
    bounds = hp.logit_bounds(x, wr, hp.LAYER_ROUTER_DEPTH)
    err = np.abs(glg - lg[:, :E])
    assert np.all(err <= bounds[:, :E]), f"logit outside its bound: {np.max(err / bounds[:, :E]):.3f}"
    oidx, ow, osw = oracle_routing(li, lg)
    certain, near, invalid = hp.classify_selection(lg[:, :E], bounds[:, :E], oidx, gidx)
    assert not invalid, f"invalid selections at tokens {invalid[:8]}"
    assert len(near) <= 1, f"{len(near)} near-tie tokens"
    same = []
    for t in range(T):
        g = gidx[t].tolist()
        assert len(set(g)) == 6 and min(g) >= 0 and max(g) < E
        total = gw[t].sum() + (gsw[t].sum() if li.sink else 0.0)
        assert np.all(gw[t] > 0) and abs(total - 1.0) <= 1e-5
        if set(g) != set(oidx[t].tolist()):
            continue
        same.append(t)
        for i in range(6):
            j = int(np.where(oidx[t] == g[i])[0][0])
            assert abs(gw[t][i] - ow[t][j]) <= W_TOL, (t, i, gw[t][i], ow[t][j])
        assert np.all(np.abs(gsw[t] - osw[t]) <= W_TOL), (t, gsw[t], osw[t])
    assert set(certain) <= set(same)
    ref, _ = oracle_layer_shared(li)
    got = hp.to_f64(out)
    assert hp.within_tol(got[same], ref[same], tol), hp.describe_err(got[same], ref[same])
    return got, ref


def run_layer(li: synth.LayerInputs, dev, repeats: int = 1):
    layer = PackedLayer.from_inputs(li) if li.wtype == synth.NVFP4 else Bf16Layer.from_inputs(li)
    T = li.x.shape[0]
    ws = new_workspace(T, dev)
    out = torch.empty(T, 2048, dtype=torch.bfloat16, device=dev)
    layer.forward(li.x, out, ws)
    assert m.moe_read_device_flag(ws) == 0
    for _ in range(repeats - 1):
        out2 = torch.empty_like(out)
        layer.forward(li.x, out2, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, out2)
    assert m.moe_read_device_flag(ws) == 0
    return out, ws


@pytest.mark.parametrize("T", [1, 3, 8])
def test_sinks_bf16_shared_nvfp4_routed(cuda_dev, T):
    """Two BF16 expert sinks beside NVFP4 routed experts (the Inkling NVFP4 layout)."""
    li = synth.make_layer(300 + T, T, n_shared=2, sink=True, shared_bf16=True, device=cuda_dev)
    out, ws = run_layer(li, cuda_dev, repeats=2)
    check_shared_layer(li, out, ws, hp.TOL_NVFP4)


def test_sinks_nvfp4_shared(cuda_dev):
    li = synth.make_layer(311, 8, n_shared=2, sink=True, device=cuda_dev)
    out, ws = run_layer(li, cuda_dev)
    check_shared_layer(li, out, ws, hp.TOL_NVFP4)


def test_sinks_all_bf16(cuda_dev):
    li = synth.make_layer(312, 4, n_shared=2, sink=True, wtype=synth.BF16, device=cuda_dev)
    out, ws = run_layer(li, cuda_dev)
    check_shared_layer(li, out, ws, hp.TOL_BF16)


def test_single_sink(cuda_dev):
    li = synth.make_layer(313, 8, n_shared=1, sink=True, shared_bf16=True, device=cuda_dev)
    out, ws = run_layer(li, cuda_dev)
    check_shared_layer(li, out, ws, hp.TOL_NVFP4)


@pytest.mark.parametrize("T,S", [(5, 1), (2, 2), (8, 2)])
def test_bf16_shared_without_sinks(cuda_dev, T, S):
    """moe_layer_forward with BF16 shared experts beside NVFP4 routed ones:
    plain routing, each shared expert added with weight 1."""
    li = synth.make_layer(320 + T, T, n_shared=S, shared_bf16=True, device=cuda_dev)
    out, ws = run_layer(li, cuda_dev)
    check_shared_layer(li, out, ws, hp.TOL_NVFP4)


def test_two_nvfp4_shared_without_sinks(cuda_dev):
    li = synth.make_layer(330, 6, n_shared=2, device=cuda_dev)
    out, ws = run_layer(li, cuda_dev)
    check_shared_layer(li, out, ws, hp.TOL_NVFP4)


def test_sinks_then_plain_layer_on_one_workspace(cuda_dev):
    """A sink layer and a plain layer alternating on one workspace: the
    tagged logits of one never leak into the other."""
    T = 8
    a = synth.make_layer(340, T, n_shared=2, sink=True, shared_bf16=True, device=cuda_dev)
    b = synth.make_layer(341, T, device=cuda_dev)
    la, lb = PackedLayer.from_inputs(a), PackedLayer.from_inputs(b)
    ws = new_workspace(T, cuda_dev)
    oa = torch.empty(T, 2048, dtype=torch.bfloat16, device=cuda_dev)
    ob = torch.empty_like(oa)
    for _ in range(2):
        la.forward(a.x, oa, ws)
        lb.forward(b.x, ob, ws)
    assert m.moe_read_device_flag(ws) == 0
    hp.check_decode_layer(b, b.x, ob, ws, hp.TOL_NVFP4)
    la.forward(a.x, oa, ws)
    check_shared_layer(a, oa, ws, hp.TOL_NVFP4)
