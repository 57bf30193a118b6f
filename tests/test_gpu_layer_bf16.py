"""moe_layer_forward with BF16 weights (the W16A16 variant, T = 1..8)
against the fp64 oracle, at the BF16 tolerance."""
import pytest
import torch

import nvfp4_moe_decode_gb300 as m
from nvfp4_moe_decode_gb300 import synth
from nvfp4_moe_decode_gb300.layer import Bf16Layer, new_workspace
from tests import helpers as hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer_bf(cuda_dev):
    li = synth.make_layer(20, 8, wtype=synth.BF16, device=cuda_dev)
    return li, Bf16Layer.from_inputs(li)


def _forward(bl, x, dev, ws=None):
    T = x.shape[0]
    ws = ws if ws is not None else new_workspace(T, dev)
    out = torch.empty(T, m.HIDDEN, dtype=torch.bfloat16, device=dev)
    bl.forward(x.contiguous(), out, ws)
    return out, m.moe_read_device_flag(ws), ws


def _check(x, li, out, ws):
    """The layer's own routing against the oracle's, then the output."""
    hp.check_decode_layer(li, x, out, ws, hp.TOL_BF16)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_bf16_layer_matches_oracle(layer_bf, cuda_dev, T):
    li, bl = layer_bf
    x = li.x[:T].contiguous()
    out, flag, ws = _forward(bl, x, cuda_dev)
    assert flag == 0
    _check(x, li, out, ws)


def test_bf16_layer_other_seed_and_determinism(cuda_dev):
    li = synth.make_layer(21, 7, wtype=synth.BF16, device=cuda_dev)
    bl = Bf16Layer.from_inputs(li)
    out1, flag, ws = _forward(bl, li.x, cuda_dev)
    out2, _, _ = _forward(bl, li.x, cuda_dev, ws)
    assert flag == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    _check(li.x, li, out1, ws)


def test_bf16_layer_without_shared_expert(cuda_dev):
    li = synth.make_layer(22, 4, wtype=synth.BF16, device=cuda_dev)
    li_ns = synth.LayerInputs(**{**li.__dict__, "n_shared": 0, "w13": li.w13[:256], "w2": li.w2[:256]})
    bl = Bf16Layer.from_inputs(li_ns)
    assert bl.shared is None
    out, flag, ws = _forward(bl, li.x, cuda_dev)
    assert flag == 0
    _check(li.x, li_ns, out, ws)


def test_bf16_one_hot_row_probe(cuda_dev):
    """Only the shared expert is non-zero and its W2 is a one-hot selector:
    out[t, r] = h[t, j(r)] exactly as the oracle's, which checks the k order
    of the W2 rows (a closed form of the down projection)."""
    li = synth.make_layer(23, 3, wtype=synth.BF16, device=cuda_dev)
    li.w13[:256].zero_()
    li.w2.zero_()
    for r in range(m.HIDDEN):
        li.w2[256, r, (37 * r) % m.INTER] = 1.0
    bl = Bf16Layer.from_inputs(li)
    out, flag, ws = _forward(bl, li.x, cuda_dev)
    assert flag == 0
    _check(li.x, li, out, ws)
