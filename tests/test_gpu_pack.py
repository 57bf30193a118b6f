"""Packing on the GPU: exact byte round trip, and the packed layout decoded by
the kernels' in-register decode against the oracle's dequantisation."""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_moe_decode_gb300 as m

pytestmark = pytest.mark.gpu


def _rand_mats(count, N, K, seed, dev):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    codes = torch.randint(0, 256, (count, N, K // 2), generator=g, device=dev, dtype=torch.uint8)
    scales = torch.randint(0, 256, (count, N, K // 16), generator=g, device=dev, dtype=torch.uint8)
    return codes, scales


@pytest.mark.parametrize("N,K,kind", [(1024, 2048, m.MOE_PACK_GATE_UP), (2048, 512, m.MOE_PACK_PLAIN),
                                      (32, 128, m.MOE_PACK_GATE_UP), (16, 128, m.MOE_PACK_PLAIN),
                                      (48, 256, m.MOE_PACK_PLAIN)])
def test_pack_unpack_round_trip(cuda_dev, N, K, kind):
    count = 3
    codes, scales = _rand_mats(count, N, K, 1, cuda_dev)
    codes[0].view(-1)[: 256] = torch.arange(256, device=cuda_dev, dtype=torch.uint8)  # every code pair
    packed = torch.empty(count * m.moe_packed_bytes(N, K), dtype=torch.uint8, device=cuda_dev)
    m.moe_pack_nvfp4(codes, scales, N, K, kind, count, packed)
    c2 = torch.empty_like(codes)
    s2 = torch.empty_like(scales)
    m.moe_unpack_nvfp4(packed, N, K, kind, count, c2, s2)
    torch.cuda.synchronize()
    assert torch.equal(codes, c2)
    assert torch.equal(scales, s2)
    # packing is a permutation: the multiset of bytes' nibbles is kept
    assert not torch.equal(packed[: codes[0].numel()], codes[0].reshape(-1)) or N * K < 4096


@pytest.mark.parametrize("N,K,kind,tscale", [(1024, 2048, m.MOE_PACK_GATE_UP, 1.0),
                                             (2048, 512, m.MOE_PACK_PLAIN, 1.0),
                                             (64, 256, m.MOE_PACK_GATE_UP, 0.3)])
def test_dequant_matches_oracle_bit_exact(cuda_dev, N, K, kind, tscale):
    codes, scales = _rand_mats(1, N, K, 2, cuda_dev)
    # finite e4m3 scales only (0x7F / 0xFF are NaN)
    scales = torch.where((scales & 0x7F) == 0x7F, scales ^ 1, scales)
    packed = torch.empty(m.moe_packed_bytes(N, K), dtype=torch.uint8, device=cuda_dev)
    m.moe_pack_nvfp4(codes, scales, N, K, kind, 1, packed)
    out = torch.empty(N, K, dtype=torch.float32, device=cuda_dev)
    m.moe_dequant_nvfp4(packed, N, K, kind, tscale, out)
    torch.cuda.synchronize()
    ref = oracle.dequant_nvfp4(codes[0].cpu().numpy(), scales[0].cpu().numpy(), tscale)
    ref32 = ref.astype(np.float32)   # exact e2m1*e4m3, one rounding by the tensor scale
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref32.view(np.uint32)), \
        np.argwhere(got.view(np.uint32) != ref32.view(np.uint32))[:5]
