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


def _check_layer(li, resid, delta, out, v, xn, tol, ws):
    """Residual add bit-exact; xn within one bf16 ulp of the oracle's (the
    GPU sums the squares in fp32); the layer's own routing and its MoE output
    against the oracle run on the GPU's own xn (``ws`` holds the routing of
    this layer call)."""
    rb = hp.bits16(resid)
    db = None if delta is None else hp.bits16(delta)
    v_ref, xn_ref = oracle.prenorm(rb, db, EPS)
    assert np.array_equal(hp.bits16(v), v_ref)
    got_xn, want_xn = hp.np_bf16(hp.bits16(xn)), hp.np_bf16(xn_ref)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want_xn), 1e-30))) - 7)
    assert np.all(np.abs(got_xn - want_xn) <= ulp)
    assert np.mean(hp.bits16(xn) == xn_ref) >= 0.999
    hp.check_decode_layer(li, xn.clone(), out, ws, tol)


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
    _check_layer(li, resid, delta, out, v, xn, tol, ws)
    out0, v0, xn0 = _prenorm_step(lay, resid, None, ws, cuda_dev)   # first layer: no delta
    assert torch.equal(v0.view(torch.int16), resid.view(torch.int16))
    _check_layer(li, resid, None, out0, v0, xn0, tol, ws)


def _run_stack_and_steps(layers, x0, dev, keep=None):
    """moe_stack_forward, and the same stack layer by layer through
    moe_layer_forward_prenorm; returns (stack result, the layer-by-layer
    result, per-layer tensors).  For the layers in ``keep`` (default: all)
    each entry also holds a copy of the workspace right after that layer's
    call, which carries the layer's own routing."""
    T = x0.shape[0]
    st = Stack(layers, EPS)
    ws = new_stack_workspace(T, dev)
    x = x0.clone()
    st.forward(x, ws)
    assert m.moe_read_device_flag(ws) == 0
    wsl = new_workspace(T, dev)
    resid, delta, steps = x0.clone(), None, []
    for l, lay in enumerate(layers):
        out, v, xn = _prenorm_step(lay, resid, delta, wsl, dev)
        snap = wsl.clone() if keep is None or l in keep else None
        steps.append((resid, delta, out, v, xn, snap))
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
        resid, delta, out, v, xn, snap = steps[l]
        _check_layer(made[l][0], resid, delta, out, v, xn, tol, snap)


@pytest.mark.parametrize("wtype,T", [(synth.NVFP4, 1), (synth.NVFP4, 8), (synth.BF16, 8)])
def test_stack_47_layers(cuda_dev, wtype, T):
    """The full 47-layer stacks (21.4 GB resident for NVFP4, 76 GB for BF16):
    the stack call equals the layers called one by one, and the oracle checks
    the first, a middle and the last layer, routing included."""
    n = 47
    checked = (0, 23, 46)
    layers, lis = [], {}
    for l in range(n):
        li, lay = _make(l, T, wtype, cuda_dev)
        layers.append(lay)
        if l in checked:
            lis[l] = li
        else:
            del li
    x0 = synth.make_x(0, T, device=cuda_dev)
    x, final, steps = _run_stack_and_steps(layers, x0, cuda_dev, keep=checked)
    assert torch.equal(x.view(torch.int16), final.view(torch.int16))
    assert torch.isfinite(x.float()).all()
    tol = hp.TOL_NVFP4 if wtype == synth.NVFP4 else hp.TOL_BF16
    for l, li in lis.items():
        resid, delta, out, v, xn, snap = steps[l]
        _check_layer(li, resid, delta, out, v, xn, tol, snap)


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
