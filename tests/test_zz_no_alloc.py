"""moe_layer_forward_static: the layer for callers that cannot allocate.

Some callers cannot call cudaMalloc or own a workspace: a plugin or custom-op
interface that hands the layer only its inputs and outputs, or a serving
process whose device memory is fixed at start-up.  For them the library keeps
its scratch in a fixed array of its own on each device.  These tests call
that entry point through the C ABI and compare it bit for bit with
moe_layer_forward on a caller-owned workspace (both run the same
deterministic kernel), on calls in a row and alternating with the workspace
path on one stream; and check that a too-large batch is refused.

Named to be collected last, so that it also runs after every other GPU test
has used the device; it passes alone as well (the first call does the
per-device setup).
"""
import pytest
import torch

import nvfp4_moe_decode_gb300 as m
from nvfp4_moe_decode_gb300 import synth
from nvfp4_moe_decode_gb300.layer import PackedLayer, new_workspace

pytestmark = pytest.mark.gpu


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("seed,T", [(11, 8), (12, 1), (13, 5)])
def test_static_scratch_matches_workspace_path(cuda_dev, seed, T):
    li = synth.make_layer(seed, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    x = li.x.contiguous()

    ws = new_workspace(T, cuda_dev)
    want = torch.empty(T, m.HIDDEN, dtype=torch.bfloat16, device=cuda_dev)
    m.moe_layer_forward(x, pl.router_w, pl.routed, pl.shared, want, T, ws)
    assert m.moe_read_device_flag(ws) == 0

    # two calls in a row on the library's scratch: bit-identical results
    for _ in range(2):
        got = torch.full((T, m.HIDDEN), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
        m.moe_layer_forward_static(x, pl.router_w, pl.routed, pl.shared, got, T)
        torch.cuda.synchronize()
        assert _same_bits(got, want)
    assert m.moe_static_read_device_flag() == 0


def test_static_and_workspace_calls_alternate_on_one_stream(cuda_dev):
    """Static and workspace calls interleaved on one stream, with different
    inputs and batch sizes, each bit-identical to its own reference."""
    li = synth.make_layer(15, 8, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    xs = [li.x[:T].contiguous() for T in (8, 3, 1, 8)]
    refs = []
    for x in xs:
        ws = new_workspace(x.shape[0], cuda_dev)
        r = torch.empty(x.shape[0], m.HIDDEN, dtype=torch.bfloat16, device=cuda_dev)
        m.moe_layer_forward(x, pl.router_w, pl.routed, pl.shared, r, x.shape[0], ws)
        refs.append(r)
    torch.cuda.synchronize()
    ws = new_workspace(8, cuda_dev)
    outs = []
    for i, x in enumerate(xs * 2):
        T = x.shape[0]
        o = torch.full((T, m.HIDDEN), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
        if i % 2 == 0:
            m.moe_layer_forward_static(x, pl.router_w, pl.routed, pl.shared, o, T)
        else:
            m.moe_layer_forward(x, pl.router_w, pl.routed, pl.shared, o, T, ws)
        outs.append(o)
    torch.cuda.synchronize()
    assert m.moe_read_device_flag(ws) == 0
    assert m.moe_static_read_device_flag() == 0
    for i, o in enumerate(outs):
        assert _same_bits(o, refs[i % len(xs)]), f"call {i}"


def test_static_scratch_rejects_batches_beyond_its_size(cuda_dev):
    li = synth.make_layer(14, 1, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    x = torch.zeros(m.MAX_DECODE_T + 1, m.HIDDEN, dtype=torch.bfloat16, device=cuda_dev)
    out = torch.empty_like(x)
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer_forward_static(x, pl.router_w, pl.routed, pl.shared, out, m.MAX_DECODE_T + 1)
    assert ei.value.status == m.MOE_ERR_UNSUPPORTED
