"""Pre-norm decoder stacks: moe_layer_forward_prenorm and moe_stack_forward.

Reading of the stack (the pages say only "pre-norm"): layer l maps the bf16
residual stream x to x + MoE_l(RMSNorm(x)), unit-weight RMSNorm.  Parity per
layer: the oracle reruns layer l on the GPU's own input to that layer (the
residual x_l and the previous output), so errors do not compound."""
import numpy as np
import pytest
import torch

import nvfp4_moe_decode_gb300 as m
import oracle
from nvfp4_moe_decode_gb300 import synth
from nvfp4_moe_decode_gb300.layer import Bf16Layer, PackedLayer, Stack, new_stack_workspace, new_workspace
from tests import helpers as hp

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _make(seed, T, wtype, dev):
    li = synth.make_layer(seed, T, wtype=wtype, device=dev)
    lay = PackedLayer.from_inputs(li) if wtype == synth.NVFP4 else Bf16Layer.from_inputs(li)
    return li, lay


def _prenorm_step(lay, resid, delta, ws, dev):
    T = resid.shape[0]
    out = torch.empty(T, m.HIDDEN, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(out)
    xn = torch.empty_like(out)
    m.moe_layer_forward_prenorm(resid, delta, v, xn, EPS, lay.router_w, lay.routed, lay.shared, out, T, ws)
    assert m.moe_read_device_flag(ws) == 0
    return out, v, xn


def _check_layer(li, resid, delta, out, v, xn, tol):
    """Residual add bit-exact; xn within one bf16 ulp of the oracle's (the
    GPU sums the squares in fp32); the MoE output against the oracle run on
    the GPU's own xn."""
    rb = hp.bits16(resid)
    db = None if delta is None else hp.bits16(delta)
    v_ref, xn_ref = oracle.prenorm(rb, db, EPS)
    assert np.array_equal(hp.bits16(v), v_ref)
    got_xn, want_xn = hp.np_bf16(hp.bits16(xn)), hp.np_bf16(xn_ref)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want_xn), 1e-30))) - 7)
    assert np.all(np.abs(got_xn - want_xn) <= ulp)
    assert np.mean(hp.bits16(xn) == xn_ref) >= 0.999
    sub = synth.LayerInputs(**{**li.__dict__, "x": xn.clone()})
    ref, idx, _, lg, _ = hp.oracle_layer(sub)
    bounds = hp.logit_bounds(hp.bits16(xn), hp.bits16(li.router_w))
    certain, _, _ = hp.classify_selection(lg, bounds, idx, idx)
    keep = [t for t in range(resid.shape[0]) if t in certain]
    assert len(keep) >= resid.shape[0] - max(1, resid.shape[0] // 100)
    g = hp.to_f64(out)
    assert hp.within_tol(g[keep], ref[keep], tol), hp.describe_err(g[keep], ref[keep])


@pytest.mark.parametrize("wtype,T", [(synth.NVFP4, 8), (synth.NVFP4, 1), (synth.BF16, 5)])
def test_prenorm_layer_matches_oracle(cuda_dev, wtype, T):
    li, lay = _make(30 + T, T, wtype, cuda_dev)
    g = torch.Generator(device=cuda_dev)
    g.manual_seed(300 + T)
    resid = (torch.randn(T, m.HIDDEN, generator=g, device=cuda_dev) * 3.0).to(torch.bfloat16)
    delta = (torch.randn(T, m.HIDDEN, generator=g, device=cuda_dev) * 40.0).to(torch.bfloat16)
    ws = new_workspace(T, cuda_dev)
    tol = hp.TOL_NVFP4 if wtype == synth.NVFP4 else hp.TOL_BF16
    out, v, xn = _prenorm_step(lay, resid, delta, ws, cuda_dev)
    _check_layer(li, resid, delta, out, v, xn, tol)
    out0, v0, xn0 = _prenorm_step(lay, resid, None, ws, cuda_dev)   # first layer: no delta
    assert torch.equal(v0.view(torch.int16), resid.view(torch.int16))
    _check_layer(li, resid, None, out0, v0, xn0, tol)


def _run_stack_and_steps(layers, x0, dev):
    """moe_stack_forward, and the same stack layer by layer through
    moe_layer_forward_prenorm; returns (stack result, per-layer inputs)."""
    T = x0.shape[0]
    st = Stack(layers, EPS)
    ws = new_stack_workspace(T, dev)
    x = x0.clone()
    st.forward(x, ws)
    assert m.moe_read_device_flag(ws) == 0
    wsl = new_workspace(T, dev)
    resid, delta, steps = x0.clone(), None, []
    for lay in layers:
        out, v, xn = _prenorm_step(lay, resid, delta, wsl, dev)
        steps.append((resid, delta, out, v, xn))
        resid, delta = v, out
    final = (resid.float() + delta.float()).to(torch.bfloat16)
    return x, final, steps


@pytest.mark.parametrize("wtype,T,n", [(synth.NVFP4, 8, 4), (synth.BF16, 3, 3)])
def test_stack_equals_layer_by_layer_and_oracle(cuda_dev, wtype, T, n):
    made = [_make(40 + l, T, wtype, cuda_dev) for l in range(n)]
    x0 = synth.make_x(400, T, device=cuda_dev)
    x, final, steps = _run_stack_and_steps([lay for _, lay in made], x0, cuda_dev)
    assert torch.equal(x.view(torch.int16), final.view(torch.int16))
    tol = hp.TOL_NVFP4 if wtype == synth.NVFP4 else hp.TOL_BF16
    for l in (0, n - 1):
        resid, delta, out, v, xn = steps[l]
        _check_layer(made[l][0], resid, delta, out, v, xn, tol)


def test_stack_47_nvfp4_layers_t1(cuda_dev):
    """The full 47-layer NVFP4 stack at T = 1 (21.4 GB resident); the oracle
    checks the first, a middle and the last layer."""
    n, T = 47, 1
    layers, lis = [], {}
    for l in range(n):
        li, lay = _make(l, T, synth.NVFP4, cuda_dev)
        layers.append(lay)
        if l in (0, 23, 46):
            lis[l] = li
        else:
            del li
    x0 = synth.make_x(0, T, device=cuda_dev)
    x, final, steps = _run_stack_and_steps(layers, x0, cuda_dev)
    assert torch.equal(x.view(torch.int16), final.view(torch.int16))
    assert torch.isfinite(x.float()).all()
    for l, li in lis.items():
        resid, delta, out, v, xn = steps[l]
        _check_layer(li, resid, delta, out, v, xn, hp.TOL_NVFP4)


def test_stack_host_errors(cuda_dev):
    li, lay = _make(50, 2, synth.NVFP4, cuda_dev)
    st = Stack([lay, lay])
    x = synth.make_x(1, 2, device=cuda_dev)
    small = torch.zeros(64, dtype=torch.uint8, device=cuda_dev)
    with pytest.raises(m.MoeError) as ei:
        st.forward(x, small)
    assert ei.value.status == m.MOE_ERR_WORKSPACE
    ws = new_stack_workspace(2, cuda_dev)
    bad = Stack([lay, lay])
    bad.arr[1].routed.n_experts = 255
    with pytest.raises(m.MoeError) as ei:
        bad.forward(x, ws)
    assert ei.value.status == m.MOE_ERR_UNSUPPORTED
