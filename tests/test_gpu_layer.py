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


def _check(li_x, li, out, ws, tol=hp.TOL_NVFP4):
    """The layer's own routing (read back from its workspace) against the
    oracle's, then the output on every token routed like the oracle."""
    return hp.check_decode_layer(li, li_x, out, ws, tol)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_layer_matches_oracle(layer0, cuda_dev, T):
    li, pl = layer0
    x = li.x[:T].contiguous()
    out, flag, ws = _forward(pl, x, cuda_dev)
    assert flag == 0
    _check(x, li, out, ws)


@pytest.mark.parametrize("seed,T", [(1, 1), (2, 8), (3, 5)])
def test_layer_other_seeds(cuda_dev, seed, T):
    li = synth.make_layer(seed, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    _check(li.x, li, out, ws)


def test_layer_is_deterministic_and_reuses_workspace(layer0, cuda_dev):
    li, pl = layer0
    out1, _, ws = _forward(pl, li.x, cuda_dev)
    out2, _, _ = _forward(pl, li.x, cuda_dev, ws)
    x1 = li.x[:3].contiguous()
    out3, _, _ = _forward(pl, x1, cuda_dev, ws)       # a different T on the same workspace
    _check(x1, li, out3, ws)
    out4, flag, _ = _forward(pl, li.x, cuda_dev, ws)
    assert flag == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(out1.view(torch.int16), out4.view(torch.int16))


def test_layer_all_tokens_same_experts(layer0, cuda_dev):
    """Eight identical tokens: the union is the 6 experts of one token."""
    li, pl = layer0
    x = li.x[:1].repeat(8, 1).contiguous()
    out, flag, ws = _forward(pl, x, cuda_dev)
    assert flag == 0
    got, ref = _check(x, li, out, ws)
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
    out, flag, ws = _forward(pl, x, cuda_dev)
    assert flag == 0
    ref, idx, _, _, _ = hp.oracle_layer(li)
    assert len(set(idx.reshape(-1).tolist())) == 48
    _check(x, li, out, ws)


def test_layer_without_shared_expert(cuda_dev):
    li = synth.make_layer(8, 4, device=cuda_dev)
    li_ns = synth.LayerInputs(**{**li.__dict__, "n_shared": 0,
                                 "codes13": li.codes13[:256], "scales13": li.scales13[:256],
                                 "codes2": li.codes2[:256], "scales2": li.scales2[:256],
                                 "tscale13": li.tscale13[:256], "tscale2": li.tscale2[:256]})
    pl = PackedLayer.from_inputs(li_ns)
    assert pl.shared is None
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    _check(li.x, li_ns, out, ws)


@pytest.mark.parametrize("T,zeros", [(8, [0, 5]), (3, [1])])
def test_layer_zero_tokens_route_by_index(cuda_dev, T, zeros):
    """Tokens whose activations are all zero: every logit is exactly 0, so
    the six selected experts are 0..5 in that order (a tie goes to the lower
    index), each weighted 1/6, and the output row is exactly 0 (every expert
    FFN maps 0 to 0).  The other tokens as usual."""
    li = synth.make_layer(420 + T, T, device=cuda_dev)
    li.x[zeros] = 0
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    gidx, gw, _ = hp.read_routing(ws, T)
    for t in zeros:
        assert gidx[t].tolist() == [0, 1, 2, 3, 4, 5]
        assert np.all(np.abs(gw[t] - 1.0 / 6.0) <= 1e-7)
        assert torch.count_nonzero(out[t].float()) == 0
    hp.check_decode_layer(li, li.x, out, ws, hp.TOL_NVFP4, max_near=len(zeros) + 1)


def test_layer_nonfinite_router_weight_sets_flag(cuda_dev):
    """A NaN router weight makes expert 17's logit NaN for every token: the
    layer reports MOE_FLAG_NONFINITE_LOGIT, ranks the NaN last (17 is never
    selected) and still produces finite outputs."""
    T = 4
    li = synth.make_layer(440, T, device=cuda_dev)
    li.router_w[17, 3] = float("nan")
    pl = PackedLayer.from_inputs(li)
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag & m.MOE_FLAG_NONFINITE_LOGIT
    gidx, gw, _ = hp.read_routing(ws, T)
    for t in range(T):
        assert 17 not in gidx[t].tolist() and len(set(gidx[t].tolist())) == 6
        assert np.all(gw[t] > 0) and abs(gw[t].sum() - 1.0) <= 1e-5
    assert torch.isfinite(out.float()).all()


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
    out, flag, ws = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    _check(li.x, li, out, ws)


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


def test_workspace_recover_after_a_timed_out_call(cuda_dev):
    """moe_workspace_recover restores a workspace left as a call that gave up
    on a bounded wait can leave it: the flag word holds MOE_FLAG_WAIT_TIMEOUT
    and the launch tag did not advance, so the stored router logits (here of
    other inputs) carry the tag the next call would use.  The state is
    planted directly in the workspace's control words ([0] device flag,
    [5] launch tag) instead of making a wait run out on the GPU, which would
    leave copies in flight; the layer runs only after the re-arm is seen to
    have advanced the tag."""
    T = 8
    li = synth.make_layer(16, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    want, flag, _ = _forward(pl, li.x, cuda_dev)
    assert flag == 0
    ws = new_workspace(T, cuda_dev)
    other = synth.make_x(99, T, device=cuda_dev)
    junk = torch.empty(T, m.HIDDEN, dtype=torch.bfloat16, device=cuda_dev)
    pl.forward(other, junk, ws)
    torch.cuda.synchronize()
    ctrl = ws[:256].view(torch.int32)
    tag = int(ctrl[5].item())
    ctrl[0] = m.MOE_FLAG_WAIT_TIMEOUT
    ctrl[5] = tag - 1
    m.moe_workspace_recover(ws)
    torch.cuda.synchronize()
    assert int(ctrl[5].item()) == tag, "the re-arm kernel did not advance the launch tag"
    assert int(ctrl[0].item()) == m.MOE_FLAG_WAIT_TIMEOUT
    out = torch.full((T, m.HIDDEN), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    pl.forward(li.x, out, ws)
    assert m.moe_read_device_flag(ws) == m.MOE_FLAG_WAIT_TIMEOUT   # kept for the caller
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    m.moe_workspace_recover(ws)   # no timeout recorded now: nothing to do
    out2, flag, _ = _forward(pl, li.x, cuda_dev, ws)
    assert flag == 0
    assert torch.equal(out2.view(torch.int16), want.view(torch.int16))
