"""moe_layer_forward (NVFP4, T = 1..8) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import nvfp4_moe_decode_gb300 as m
from nvfp4_moe_decode_gb300 import synth
from nvfp4_moe_decode_gb300.layer import PackedLayer, new_workspace
from tests import helpers as hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer0(cuda_dev):
    li = synth.make_layer(0, 8, device=cuda_dev)
    return li, PackedLayer.from_inputs(li)


def _forward(pl, x, dev, ws=None):
    T = x.shape[0]
    ws = ws if ws is not None else new_workspace(T, dev)
    out = torch.empty(T, 2048, dtype=torch.bfloat16, device=dev)
    pl.forward(x.contiguous(), out, ws)
    flag = m.moe_read_device_flag(ws)
    return out, flag, ws


def _check(li_x, li, out, tol=hp.TOL_NVFP4):
    sub = synth.LayerInputs(**{**li.__dict__, "x": li_x})
    ref, idx, w, lg, _ = hp.oracle_layer(sub)
    bounds = hp.logit_bounds(hp.bits16(li_x), hp.bits16(li.router_w))
    # every token must be away from a routing near-tie for a full comparison
    certain, near, invalid = hp.classify_selection(lg, bounds, idx, idx)
    got = hp.to_f64(out)
    keep = [t for t in range(li_x.shape[0]) if t in certain]
    assert len(keep) >= li_x.shape[0] - max(1, li_x.shape[0] // 100)
    assert hp.within_tol(got[keep], ref[keep], tol), hp.describe_err(got[keep], ref[keep])
    return got, ref


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_layer_matches_oracle(layer0, cuda_dev, T):
    li, pl = layer0
    x = li.x[:T].contiguous()
    out, flag, _ = _forward(pl, x, cuda_dev)
    assert flag == 0
    _check(x, li, out)


@pytest.mark.parametrize("seed,T", [(1, 1), (2, 8), (3, 5)])
def test_layer_other_seeds(cuda_dev, seed, T):
    li = synth.make_layer(seed, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    out, flag, _ = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    _check(li.x, li, out)


def test_layer_is_deterministic_and_reuses_workspace(layer0, cuda_dev):
    li, pl = layer0
    out1, _, ws = _forward(pl, li.x, cuda_dev)
    out2, _, _ = _forward(pl, li.x, cuda_dev, ws)
    x1 = li.x[:3].contiguous()
    out3, _, _ = _forward(pl, x1, cuda_dev, ws)       # a different T on the same workspace
    out4, flag, _ = _forward(pl, li.x, cuda_dev, ws)
    assert flag == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(out1.view(torch.int16), out4.view(torch.int16))
    _check(x1, li, out3)


def test_layer_all_tokens_same_experts(layer0, cuda_dev):
    """Eight identical tokens: the union is the 6 experts of one token."""
    li, pl = layer0
    x = li.x[:1].repeat(8, 1).contiguous()
    out, flag, _ = _forward(pl, x, cuda_dev)
    assert flag == 0
    got, ref = _check(x, li, out)
    for t in range(1, 8):
        assert torch.equal(out[t].view(torch.int16), out[0].view(torch.int16))


def test_layer_disjoint_experts(cuda_dev):
    """Router rows built so token t prefers experts 6t..6t+5: 48 distinct experts."""
    li = synth.make_layer(7, 8, device=cuda_dev)
    H = 2048
    g = torch.Generator(device=cuda_dev)
    g.manual_seed(70)
    basis = torch.randn(8, H, generator=g, device=cuda_dev)
    x = basis.to(torch.bfloat16)
    wr = li.router_w.float() * 0.1
    for t in range(8):
        wr[6 * t:6 * t + 6] += basis[t] / basis[t].norm() * 0.05
    li.router_w = wr.to(torch.bfloat16).contiguous()
    li.x = x
    pl = PackedLayer.from_inputs(li)
    out, flag, _ = _forward(pl, x, cuda_dev)
    assert flag == 0
    ref, idx, _, _, _ = hp.oracle_layer(li)
    assert len(set(idx.reshape(-1).tolist())) == 48
    _check(x, li, out)


def test_layer_without_shared_expert(cuda_dev):
    li = synth.make_layer(8, 4, device=cuda_dev)
    li_ns = synth.LayerInputs(**{**li.__dict__, "n_shared": 0,
                                 "codes13": li.codes13[:256], "scales13": li.scales13[:256],
                                 "codes2": li.codes2[:256], "scales2": li.scales2[:256],
                                 "tscale13": li.tscale13[:256], "tscale2": li.tscale2[:256]})
    pl = PackedLayer.from_inputs(li_ns)
    assert pl.shared is None
    out, flag, _ = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    _check(li.x, li_ns, out)


def test_layer_zero_scales_give_zero(cuda_dev):
    li = synth.make_layer(9, 2, device=cuda_dev)
    li.scales2.zero_()
    pl = PackedLayer.from_inputs(li)
    out, flag, _ = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    assert torch.count_nonzero(out.float()) == 0


def test_layer_tensor_scales(cuda_dev):
    """Non-unit per-expert tensor scales (fp32) are applied per expert."""
    li = synth.make_layer(10, 3, device=cuda_dev)
    g = torch.Generator(device=cuda_dev)
    g.manual_seed(100)
    li.tscale13 = (torch.rand(257, generator=g, device=cuda_dev) * 1.5 + 0.25).contiguous()
    li.tscale2 = (torch.rand(257, generator=g, device=cuda_dev) * 1.5 + 0.25).contiguous()
    pl = PackedLayer.from_inputs(li)
    out, flag, _ = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    _check(li.x, li, out)


@pytest.mark.parametrize("seed,T", [(2, 8), (3, 5)])
def test_layer_repeated_calls_are_clean_and_identical(cuda_dev, seed, T):
    """Many calls, each on a fresh workspace and on one reused workspace: no
    device flag (no wait ever runs out) and bit-identical outputs.  The K-split
    hand-over between the four warps of a group once raced when one warp ran
    two units ahead; these cases exposed it."""
    li = synth.make_layer(seed, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    ref, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    for i in range(16):
        out, flag, _ = _forward(pl, li.x, cuda_dev, None if i % 2 else ws)
        assert flag == 0, f"call {i}: device flag {flag}"
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {i}"
