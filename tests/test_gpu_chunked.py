"""Mid-size batches (MOE_MAX_DECODE_T < T <= MOE_MAX_CHUNKED_T, 88 tokens;
BF16 weights up to 56): the decode kernel on
balanced chunks of at most 8 tokens, against the fp64 oracle: every token's
routing read back from the workspace (the decode router's certified bound,
indices bit-exact on certain tokens) and the outputs."""
import numpy as np
import pytest
import torch

import nvfp4_moe_decode_gb300 as m
from nvfp4_moe_decode_gb300 import synth
from nvfp4_moe_decode_gb300.layer import Bf16Layer, PackedLayer, new_workspace
from tests import helpers as hp

pytestmark = pytest.mark.gpu


def _run(layer, x, dev):
    T = x.shape[0]
    ws = new_workspace(T, dev)
    out = torch.full((T, m.HIDDEN), float("nan"), dtype=torch.bfloat16, device=dev)
    layer.forward(x.contiguous(), out, ws)
    assert m.moe_read_device_flag(ws) == 0
    return out, ws


def _check(li, out, ws, tol):
    T = li.x.shape[0]
    gidx, gw, glg = hp.read_routing(ws, T)
    xb, wb = hp.bits16(li.x), hp.bits16(li.router_w)
    _, near, same = hp.check_gpu_routing(xb, wb, gidx, gw, glg, hp.LAYER_ROUTER_DEPTH, 2e-6)
    assert len(near) <= max(1, T // 50), f"{len(near)} near-tie tokens"
    ref, _, _, _, _ = hp.oracle_layer(li)
    got = hp.to_f64(out)
    assert len(same) >= T - len(near)
    assert hp.within_tol(got[same], ref[same], tol), hp.describe_err(got[same], ref[same])


@pytest.mark.parametrize("T", [9, 13, 64, 88])
def test_chunked_layer_nvfp4(cuda_dev, T):
    li = synth.make_layer(90 + T, T, device=cuda_dev)
    out, ws = _run(PackedLayer.from_inputs(li), li.x, cuda_dev)
    _check(li, out, ws, hp.TOL_NVFP4)


@pytest.mark.parametrize("T", [24, 56])
def test_chunked_layer_bf16(cuda_dev, T):
    """BF16 weights up to the largest size of their chunked range (56)."""
    li = synth.make_layer(91 + T, T, wtype=synth.BF16, device=cuda_dev)
    out, ws = _run(Bf16Layer.from_inputs(li), li.x, cuda_dev)
    _check(li, out, ws, hp.TOL_BF16)


def test_chunked_equals_per_chunk_calls(cuda_dev):
    """A chunked call is bit-identical to the same tokens run as separate
    decode calls of the chunk sizes it uses (balanced: 20 tokens -> 7, 7, 6)."""
    T = 20
    li = synth.make_layer(92, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    out, _ = _run(pl, li.x, cuda_dev)
    parts = []
    for t0, t1 in [(0, 6), (6, 13), (13, 20)]:
        o, _ = _run(pl, li.x[t0:t1], cuda_dev)
        parts.append(o)
    assert torch.equal(out.view(torch.int16), torch.cat(parts).view(torch.int16))


def test_chunked_without_shared_expert(cuda_dev):
    T = 17
    li = synth.make_layer(93, T, device=cuda_dev)
    li_ns = synth.LayerInputs(**{**li.__dict__, "n_shared": 0,
                                 "codes13": li.codes13[:256], "scales13": li.scales13[:256],
                                 "codes2": li.codes2[:256], "scales2": li.scales2[:256],
                                 "tscale13": li.tscale13[:256], "tscale2": li.tscale2[:256]})
    out, ws = _run(PackedLayer.from_inputs(li_ns), li.x, cuda_dev)
    _check(li_ns, out, ws, hp.TOL_NVFP4)
