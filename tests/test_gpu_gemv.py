"""The dense small-batch NVFP4 GEMV (moe_dense_gemv_nvfp4) against the fp64
oracle, element by element, with an error bound derived from the kernel's
arithmetic (below)."""
import math

import numpy as np
import pytest
import torch

import oracle
import nvfp4_moe_decode_gb300 as m
from nvfp4_moe_decode_gb300 import synth
from tests import helpers as hp

pytestmark = pytest.mark.gpu


def gemv_bound(W: np.ndarray, x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """Elementwise bound on |y_gpu - y| for y = W x (fp64, [T, N]).

    The kernel: e2m1 x f16 products are exact; each k16 step's 16 products
    are summed by one mma into fp32 (assumed no worse than a sequential fp32
    chain of 16 terms; the factor 2 below is margin for that assumption);
    the block scale is applied by one fma per step into the warp's chain,
    the Q <= 16 warp partials are added in order, and the tensor scale times
    the power of two costs one more rounding: depth K/16 + 33 in all, on
    A = sum_k |W x|.  Then one rounding to bf16 (unit 2^-8).  The f16
    rescale of x is exact except for elements below 2^-31 of the token's
    largest (error under 2^-39 max|x| each)."""
    K = W.shape[1]
    g = 2.0 * hp.gamma(K // 16 + 33, hp.U32)
    A = np.abs(x) @ np.abs(W).T
    ex = (2.0 ** -39) * np.abs(x).max(axis=1, keepdims=True) * np.abs(W).sum(axis=1)[None, :]
    return 2.0 ** -8 * (np.abs(y) + g * A) + g * A + ex


def run_gemv(d: synth.DenseInputs, N: int, K: int, T: int, tscale: float, dev):
    packed = torch.empty(m.moe_packed_bytes(N, K), dtype=torch.uint8, device=dev)
    m.moe_pack_nvfp4(d.codes, d.scales, N, K, m.MOE_PACK_PLAIN, 1, packed)
    y = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    m.moe_dense_gemv_nvfp4(d.x, packed, tscale, N, K, T, y, ws)
    assert m.moe_read_device_flag(ws) == 0
    return y, packed, ws


def check(d: synth.DenseInputs, y: torch.Tensor, tscale: float):
    codes, scales = d.codes.cpu().numpy(), d.scales.cpu().numpy()
    xb = hp.bits16(d.x)
    ref = oracle.dense_gemv_nvfp4(codes, scales, tscale, xb)
    W = oracle.dequant_nvfp4(codes, scales, tscale)
    bound = gemv_bound(W, hp.np_bf16(xb), ref)
    got = hp.to_f64(y)
    bad = np.argwhere(np.abs(got - ref) > bound)
    assert bad.size == 0, f"{len(bad)} outside the bound, first {bad[:4].tolist()}; " + hp.describe_err(got, ref)
    return got, ref


# (N, K, T): the hidden-size projections of a 2048-wide decoder (qkv 5120 x
# 2048, o 2048 x 4096), one band, ragged band counts, K of one stage, a K
# whose stage count is not a power of two, and the two-stage-ring range
@pytest.mark.parametrize("N,K,T", [(2048, 2048, 1), (2048, 2048, 3), (2048, 2048, 8), (5120, 2048, 8),
                                   (2048, 4096, 8), (1024, 8192, 2), (16, 256, 1), (48, 768, 5),
                                   (4112, 512, 8), (304, 1280, 7)])
def test_dense_gemv_matches_oracle(cuda_dev, N, K, T):
    d = synth.make_dense(100 + N + K + T, T, N, K, device=cuda_dev)
    y, _, _ = run_gemv(d, N, K, T, 0.375, cuda_dev)
    torch.cuda.synchronize()
    check(d, y, 0.375)


def test_dense_gemv_repeat_is_bit_identical(cuda_dev):
    N, K, T = 5120, 2048, 8
    d = synth.make_dense(7, T, N, K, device=cuda_dev)
    y, packed, ws = run_gemv(d, N, K, T, 1.0, cuda_dev)
    y2 = torch.empty_like(y)
    for _ in range(3):
        m.moe_dense_gemv_nvfp4(d.x, packed, 1.0, N, K, T, y2, ws)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)
    assert m.moe_read_device_flag(ws) == 0


def test_dense_gemv_wide_activation_range(cuda_dev):
    """Tokens whose magnitudes span many binades (the per-token power-of-two
    rescale into f16), one token all zeros."""
    N, K, T = 256, 2048, 4
    d = synth.make_dense(9, T, N, K, device=cuda_dev)
    sc = torch.tensor([2.0 ** 40, 2.0 ** -30, 1.0, 0.0], device=cuda_dev)[:, None]
    k = torch.arange(K, device=cuda_dev)
    ramp = torch.pow(2.0, -(k % 24).float())[None, :]   # 24 binades within each token
    d.x = (d.x.float() * sc * ramp).to(torch.bfloat16)
    y, _, _ = run_gemv(d, N, K, T, 1.0, cuda_dev)
    torch.cuda.synchronize()
    got, ref = check(d, y, 1.0)
    assert np.all(got[3] == 0.0)


def test_dense_gemv_host_errors(cuda_dev):
    lib = m.load()
    x = torch.zeros(8, 2048, dtype=torch.bfloat16, device=cuda_dev)
    w = torch.zeros(m.moe_packed_bytes(2048, 2048), dtype=torch.uint8, device=cuda_dev)
    y = torch.zeros(8, 2048, dtype=torch.bfloat16, device=cuda_dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda_dev)
    f = lib.moe_dense_gemv_nvfp4
    P = lambda t: t.data_ptr()  # noqa: E731
    assert f(P(x), P(w), 1.0, 2048, 2048, 9, P(y), P(ws), 256, None) == m.MOE_ERR_UNSUPPORTED
    assert f(P(x), P(w), 1.0, 2048, 2048, 0, P(y), P(ws), 256, None) == m.MOE_ERR_UNSUPPORTED
    assert f(P(x), P(w), 1.0, 2040, 2048, 1, P(y), P(ws), 256, None) == m.MOE_ERR_UNSUPPORTED
    assert f(P(x), P(w), 1.0, 2048, 2176, 1, P(y), P(ws), 256, None) == m.MOE_ERR_UNSUPPORTED
    assert f(P(x), P(w), 1.0, 2048, 16384, 1, P(y), P(ws), 256, None) == m.MOE_ERR_UNSUPPORTED
    assert f(P(x), P(w), 1.0, 2048, 2048, 1, P(x), P(ws), 256, None) == m.MOE_ERR_INVALID_ARG
    assert f(P(x), P(w), 1.0, 2048, 2048, 1, P(y), P(ws), 128, None) == m.MOE_ERR_WORKSPACE
    assert f(P(x) + 2, P(w), 1.0, 2048, 2048, 1, P(y), P(ws), 256, None) == m.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.count_nonzero(y) == 0
