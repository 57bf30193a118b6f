"""The grouped path (T > MOE_MAX_DECODE_T): router GEMM, top-k, expert lists
and the tcgen05 grouped GEMMs, against the fp64 oracle."""
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


@pytest.mark.parametrize("T", [9, 512, 8192])
def test_grouped_routing(cuda_dev, T):
    li = synth.make_layer(60 + T % 97, T, device=cuda_dev, weights=False)
    idx, w, lg_gpu = _route(li, cuda_dev)
    xb, wb = hp.bits16(li.x), hp.bits16(li.router_w)
    lg = oracle.router_logits(xb, wb)
    bounds = hp.logit_bounds(xb, wb, hp.GEMM_DEPTH)
    # every fp32 logit of the tensor-core GEMM lies within the bound
    assert np.all(np.abs(lg_gpu - lg) <= bounds)
    oidx, ow = oracle.select_topk(lg, 6)
    certain, near, invalid = hp.classify_selection(lg, bounds, oidx, idx)
    assert not invalid
    assert len(near) <= max(2, T // 20)
    c = np.array(certain)
    assert np.array_equal(idx[c], oidx[c])
    assert np.max(np.abs(w[c] - ow[c])) <= 1e-5
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-5)


def _forward(lay, x, dev):
    T = x.shape[0]
    ws = new_workspace(T, dev)
    out = torch.full((T, m.HIDDEN), float("nan"), dtype=torch.bfloat16, device=dev)
    lay.forward(x.contiguous(), out, ws)
    return out, m.moe_read_device_flag(ws)


def _check(li, out, tol, tokens=None):
    T = li.x.shape[0]
    tokens = list(range(T)) if tokens is None else list(tokens)
    ref, idx, _, lg, _ = hp.oracle_layer(li, tokens=tokens)
    xb = np.ascontiguousarray(hp.bits16(li.x)[tokens])
    bounds = hp.logit_bounds(xb, hp.bits16(li.router_w), hp.GEMM_DEPTH)
    certain, _, _ = hp.classify_selection(lg, bounds, idx, idx)
    got = hp.to_f64(out)[tokens]
    assert len(certain) >= len(tokens) - max(2, len(tokens) // 20)
    c = np.array(certain)
    assert hp.within_tol(got[c], ref[c], tol), hp.describe_err(got[c], ref[c])


@pytest.mark.parametrize("T", [9, 64, 300])
def test_grouped_layer_small(cuda_dev, T):
    li = synth.make_layer(70 + T, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    out, flag = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    _check(li, out, hp.TOL_NVFP4)


def test_grouped_layer_8192_sampled(cuda_dev):
    """The 8192-token configuration, all tokens finite, 96 sampled against the
    oracle (first, last, and random ones)."""
    T = 8192
    li = synth.make_layer(0, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    out, flag = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(8192)
    toks = sorted(set([0, 1, T - 1] + rng.choice(T, 93, replace=False).tolist()))
    _check(li, out, hp.TOL_NVFP4, toks)


def test_grouped_bf16_weights(cuda_dev):
    T = 200
    li = synth.make_layer(80, T, wtype=synth.BF16, device=cuda_dev)
    bl = Bf16Layer.from_inputs(li)
    out, flag = _forward(bl, li.x, cuda_dev)
    assert flag == 0
    _check(li, out, hp.TOL_BF16)


def test_grouped_without_shared_expert_and_determinism(cuda_dev):
    T = 100
    li = synth.make_layer(81, T, device=cuda_dev)
    li_ns = synth.LayerInputs(**{**li.__dict__, "n_shared": 0,
                                 "codes13": li.codes13[:256], "scales13": li.scales13[:256],
                                 "codes2": li.codes2[:256], "scales2": li.scales2[:256],
                                 "tscale13": li.tscale13[:256], "tscale2": li.tscale2[:256]})
    pl = PackedLayer.from_inputs(li_ns)
    out1, flag = _forward(pl, li.x, cuda_dev)
    out2, _ = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    _check(li_ns, out1, hp.TOL_NVFP4)


def test_grouped_expert_with_more_than_256_tokens(cuda_dev):
    """600 copies of one token: six experts get 600 tokens each (three token
    chunks of up to 256), every output row equal."""
    T = 600
    li = synth.make_layer(82, 1, device=cuda_dev)
    li.x = li.x.repeat(T, 1).contiguous()
    pl = PackedLayer.from_inputs(li)
    out, flag = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    assert torch.equal(out.view(torch.int16), out[:1].repeat(T, 1).view(torch.int16))
    _check(li, out, hp.TOL_NVFP4, tokens=[0, 299, 599])
