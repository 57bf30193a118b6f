"""moe_route (router GEMV + sigmoid top-6 + renormalise) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_moe_decode_gb300 as m
from nvfp4_moe_decode_gb300 import synth
from tests import helpers as hp

pytestmark = pytest.mark.gpu


def _route(li, T, dev):
    ws = torch.zeros(m.moe_workspace_bytes(T), dtype=torch.uint8, device=dev)
    idx = torch.empty(T, 6, dtype=torch.int32, device=dev)
    w = torch.empty(T, 6, dtype=torch.float32, device=dev)
    lg = torch.empty(T, 256, dtype=torch.float32, device=dev)
    m.moe_route(li.x, li.router_w, T, idx, w, lg, ws)
    flag = m.moe_read_device_flag(ws)
    return idx.cpu().numpy(), w.cpu().numpy().astype(np.float64), lg.cpu().numpy().astype(np.float64), flag


@pytest.mark.parametrize("T", [1, 2, 3, 5, 7, 8])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_route_matches_oracle(cuda_dev, T, seed):
    li = synth.make_layer(seed, T, device=cuda_dev, weights=False)
    gi, gw, glg, flag = _route(li, T, cuda_dev)
    assert flag == 0
    xb, wb = hp.bits16(li.x), hp.bits16(li.router_w)
    lg = oracle.router_logits(xb, wb)
    oi, ow = oracle.select_topk(lg, 6)
    bounds = hp.logit_bounds(xb, wb)
    # logits within the certified summation bound
    assert np.all(np.abs(glg - lg) <= bounds), np.max(np.abs(glg - lg) / bounds)
    certain, near, invalid = hp.classify_selection(lg, bounds, oi, gi)
    assert not invalid, invalid
    for t in certain:
        # same experts; order within the selection may differ only between
        # experts whose logits are within the bound of each other
        assert set(gi[t]) == set(oi[t])
        for i in range(6):
            j = int(np.where(oi[t] == gi[t][i])[0][0])
            assert abs(gw[t][i] - ow[t][j]) <= 2e-6, (t, i, gw[t][i], ow[t][j])
    for t in range(T):
        assert len(set(gi[t].tolist())) == 6
        assert abs(gw[t].sum() - 1.0) <= 1e-6
        assert np.all(gw[t] > 0)
    assert len(near) == 0 or len(near) <= max(1, T // 100)


def test_route_orders_best_first(cuda_dev):
    li = synth.make_layer(3, 8, device=cuda_dev, weights=False)
    gi, gw, glg, _ = _route(li, 8, cuda_dev)
    for t in range(8):
        vals = glg[t][gi[t]]
        assert np.all(np.diff(vals) <= 0)


def test_route_zero_input_picks_lowest_indices(cuda_dev):
    li = synth.make_layer(4, 4, device=cuda_dev, weights=False)
    li.x.zero_()
    gi, gw, _, flag = _route(li, 4, cuda_dev)
    assert flag == 0
    assert np.array_equal(gi, np.tile(np.arange(6, dtype=np.int32), (4, 1)))
    assert np.allclose(gw, 1.0 / 6.0, atol=1e-7)


def test_route_nonfinite_logit_sets_flag(cuda_dev):
    li = synth.make_layer(5, 2, device=cuda_dev, weights=False)
    li.router_w[17, 3] = float("nan")
    gi, gw, _, flag = _route(li, 2, cuda_dev)
    assert flag & m.MOE_FLAG_NONFINITE_LOGIT
    for t in range(2):
        assert 17 not in gi[t].tolist()   # NaN ranks last
