"""moe_layer_forward_static (scratch inside the library, no allocation)
against moe_layer_forward with a caller-owned workspace.

Named to be collected last, so that it also runs after every other GPU test
has used the device; it passes alone as well (the first call does the
per-device setup).
"""
import pytest
import torch

import nvfp4_moe_decode_gb300 as m
from nvfp4_moe_decode_gb300 import synth
from nvfp4_moe_decode_gb300.layer import PackedLayer, new_workspace
from tests import helpers as hp

pytestmark = pytest.mark.gpu


def _within(got, want, tol=hp.TOL_NVFP4):
    g, w = hp.to_f64(got), hp.to_f64(want)
    assert hp.within_tol(g, w, tol), hp.describe_err(g, w)


@pytest.mark.parametrize("seed,T", [(11, 8), (12, 1), (13, 5)])
def test_static_scratch_matches_workspace_path(cuda_dev, seed, T):
    li = synth.make_layer(seed, T, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    x = li.x.contiguous()

    ws = new_workspace(T, cuda_dev)
    want = torch.empty(T, m.HIDDEN, dtype=torch.bfloat16, device=cuda_dev)
    m.moe_layer_forward(x, pl.router_w, pl.routed, pl.shared, want, T, ws)
    assert m.moe_read_device_flag(ws) == 0

    # two calls in a row on the library's scratch
    for _ in range(2):
        got = torch.full((T, m.HIDDEN), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
        m.moe_layer_forward_static(x, pl.router_w, pl.routed, pl.shared, got, T)
        torch.cuda.synchronize()
        _within(got, want)


def test_static_scratch_rejects_batches_beyond_its_size(cuda_dev):
    li = synth.make_layer(14, 1, device=cuda_dev)
    pl = PackedLayer.from_inputs(li)
    x = torch.zeros(m.MAX_DECODE_T + 1, m.HIDDEN, dtype=torch.bfloat16, device=cuda_dev)
    out = torch.empty_like(x)
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer_forward_static(x, pl.router_w, pl.routed, pl.shared, out, m.MAX_DECODE_T + 1)
    assert ei.value.status == m.MOE_ERR_UNSUPPORTED
