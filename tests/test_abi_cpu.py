"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import nvfp4_moe_decode_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for mt in re.finditer(r"\b(moe_[a-z0-9_]+)\s*\(", text):
            names.add(mt.group(1))
    return names


def test_header_declares_the_binding_exports():
    assert declared_functions() == set(m.EXPORTS)


def header_defines():
    text = open(os.path.join(ROOT, "include", "nvfp4moe.h")).read()
    return {mt.group(1): int(mt.group(2)) for mt in re.finditer(r"#define (MOE_[A-Z0-9_]+) (\d+)u?\b", text)}


def test_binding_constants_match_the_header():
    d = header_defines()
    assert d["MOE_HIDDEN"] == m.HIDDEN and d["MOE_INTER"] == m.INTER
    assert d["MOE_MAX_DECODE_T"] == m.MAX_DECODE_T and d["MOE_MAX_TOKENS"] == m.MAX_TOKENS
    assert d["MOE_MAX_CHUNKED_T"] == m.MAX_CHUNKED_T
    assert d["MOE_MAX_CHUNKED_T_BF16"] == m.MAX_CHUNKED_T_BF16
    assert d["MOE_STATIC_SCRATCH_BYTES"] == m.MOE_STATIC_SCRATCH_BYTES
    assert m.MAX_DECODE_T < m.MAX_CHUNKED_T_BF16 <= m.MAX_CHUNKED_T


def test_library_exports_every_declared_symbol(moe_lib):
    for name in declared_functions():
        assert hasattr(moe_lib, name), name
        assert ctypes.cast(getattr(moe_lib, name), ctypes.c_void_p).value


def test_abi_version_and_status_strings(moe_lib):
    assert m.moe_abi_version() == 1
    assert m.moe_status_string(m.MOE_OK) == "MOE_OK"
    assert m.moe_status_string(m.MOE_ERR_WORKSPACE) == "MOE_ERR_WORKSPACE"
    assert m.moe_status_string(99) == "MOE_UNKNOWN_STATUS"


def test_packed_bytes(moe_lib):
    assert m.moe_packed_bytes(1024, 2048) == 1_179_648
    assert m.moe_packed_bytes(2048, 512) == 589_824
    assert m.moe_packed_bytes(15, 2048) == 0
    assert m.moe_packed_bytes(16, 64) == 0
    assert m.moe_packed_bytes(0, 128) == 0


def test_workspace_bytes(moe_lib):
    for T in range(1, 9):
        assert m.moe_workspace_bytes(T) > 0
    assert m.moe_workspace_bytes(0) == 0
    # above the decode range the grouped path takes over, up to MAX_TOKENS
    assert m.moe_workspace_bytes(9) >= m.moe_workspace_bytes(8)
    assert m.moe_workspace_bytes(8192) > 400_000_000
    assert m.moe_workspace_bytes(m.MAX_TOKENS) > m.moe_workspace_bytes(8192)
    assert m.moe_workspace_bytes(m.MAX_TOKENS + 1) == 0
    # the fixed scratch of moe_layer_forward_static covers the largest batch
    assert m.moe_workspace_bytes(m.MAX_DECODE_T) == m.MOE_STATIC_SCRATCH_BYTES


def test_host_argument_errors_enqueue_nothing(moe_lib):
    lib = moe_lib
    dummy = 1 << 20  # an aligned non-null value; never dereferenced on these paths
    # pack: null pointers, count 0, bad kind, bad shape
    assert lib.moe_pack_nvfp4(None, dummy, 16, 128, 0, 1, dummy, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_nvfp4(dummy, dummy, 16, 128, 0, 0, dummy, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_nvfp4(dummy, dummy, 16, 128, 7, 1, dummy, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_nvfp4(dummy, dummy, 16, 128, 1, 1, dummy, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_unpack_nvfp4(dummy, 16, 100, 0, 1, dummy, dummy, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_dequant_nvfp4(dummy + 4, 16, 128, 0, 1.0, dummy, None) == m.MOE_ERR_INVALID_ARG
    # route / forward: null, misaligned, unsupported T, small workspace
    ws = m.moe_workspace_bytes(1)
    assert lib.moe_route(None, dummy, 1, 256, 6, dummy, dummy, None, dummy, ws, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_route(dummy + 2, dummy, 1, 256, 6, dummy, dummy, None, dummy, ws, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_route(dummy, dummy, m.MAX_TOKENS + 1, 256, 6, dummy, dummy, None, dummy, ws, None) == m.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(dummy, dummy, 8192, 256, 6, dummy, dummy, None, dummy, ws, None) == m.MOE_ERR_WORKSPACE
    assert lib.moe_route(dummy, dummy, 1, 128, 6, dummy, dummy, None, dummy, ws, None) == m.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(dummy, dummy, 1, 256, 6, dummy, dummy, None, dummy, 16, None) == m.MOE_ERR_WORKSPACE
    bank = m.moe_expert_bank(m.MOE_W_NVFP4, 256, dummy, dummy, dummy, dummy)
    bad_n = m.moe_expert_bank(m.MOE_W_NVFP4, 255, dummy, dummy, dummy, dummy)
    bad_w = m.moe_expert_bank(7, 256, dummy, dummy, dummy, dummy)
    null_w = m.moe_expert_bank(m.MOE_W_NVFP4, 256, None, dummy, dummy, dummy)
    fwd = lib.moe_layer_forward
    B = ctypes.byref
    assert fwd(dummy, dummy, B(bank), None, dummy, 0, dummy, ws, None) == m.MOE_ERR_UNSUPPORTED
    assert fwd(dummy, dummy, B(bank), None, dummy, 1, dummy, 8, None) == m.MOE_ERR_WORKSPACE
    assert fwd(dummy, dummy, B(bank), None, dummy, 1, dummy, ws, None) == m.MOE_ERR_INVALID_ARG  # out aliases x
    assert fwd(dummy, dummy, B(bad_n), None, dummy * 2, 1, dummy, ws, None) == m.MOE_ERR_UNSUPPORTED
    assert fwd(dummy, dummy, B(bad_w), None, dummy * 2, 1, dummy, ws, None) == m.MOE_ERR_UNSUPPORTED
    assert fwd(dummy, dummy, B(null_w), None, dummy * 2, 1, dummy, ws, None) == m.MOE_ERR_INVALID_ARG
    assert fwd(dummy, dummy, None, None, dummy * 2, 1, dummy, ws, None) == m.MOE_ERR_INVALID_ARG
    # a shared bank of the other weight type runs ahead on the dense GEMV, on
    # the decode path only
    bf = m.moe_expert_bank(m.MOE_W_BF16, 256, dummy, dummy, None, None)
    sh4 = m.moe_expert_bank(m.MOE_W_NVFP4, 1, dummy, dummy, dummy, dummy)
    ws9 = m.moe_workspace_bytes(9)
    assert fwd(dummy, dummy, B(bf), B(sh4), dummy * 2, 9, dummy, ws9, None) == m.MOE_ERR_UNSUPPORTED
    # up to two shared experts; expert sinks need one, and the decode path
    sh2 = m.moe_expert_bank(m.MOE_W_BF16, 2, dummy, dummy, None, None)
    sh3 = m.moe_expert_bank(m.MOE_W_BF16, 3, dummy, dummy, None, None)
    assert fwd(dummy, dummy, B(bank), B(sh3), dummy * 2, 1, dummy, ws, None) == m.MOE_ERR_UNSUPPORTED
    assert fwd(dummy, dummy, B(bank), B(sh2), dummy * 2, 9, dummy, ws9, None) == m.MOE_ERR_UNSUPPORTED
    snk = lib.moe_layer_forward_sink
    assert snk(dummy, dummy, B(bank), None, dummy * 2, 1, dummy, ws, None) == m.MOE_ERR_INVALID_ARG
    assert snk(dummy, dummy, B(bank), B(sh3), dummy * 2, 1, dummy, ws, None) == m.MOE_ERR_UNSUPPORTED
    assert snk(dummy, dummy, B(bank), B(sh2), dummy * 2, 9, dummy, ws9, None) == m.MOE_ERR_UNSUPPORTED
    assert snk(dummy, dummy, B(bank), B(sh2), dummy, 1, dummy, ws, None) == m.MOE_ERR_INVALID_ARG  # out aliases x
    rsw = lib.moe_read_shared_weights
    assert rsw(None, ws, 1, 2, dummy, None) == m.MOE_ERR_INVALID_ARG
    assert rsw(dummy, ws, 1, 2, None, None) == m.MOE_ERR_INVALID_ARG
    assert rsw(dummy, ws9, 9, 2, dummy, None) == m.MOE_ERR_UNSUPPORTED
    assert rsw(dummy, ws, 1, 3, dummy, None) == m.MOE_ERR_UNSUPPORTED
    assert rsw(dummy, 64, 1, 2, dummy, None) == m.MOE_ERR_WORKSPACE
    # the pre-norm layer takes its shared expert inside the layer kernel only
    pre = lib.moe_layer_forward_prenorm
    assert pre(dummy, None, None, None, 1e-6, dummy, B(bank), B(sh2), dummy * 2, 1, dummy, ws,
               None) == m.MOE_ERR_UNSUPPORTED
    bf_null = m.moe_expert_bank(m.MOE_W_BF16, 256, dummy, None, None, None)
    assert fwd(dummy, dummy, B(bf_null), None, dummy * 2, 1, dummy, ws, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_init(None, ws, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_init(dummy, 8, None) == m.MOE_ERR_WORKSPACE
    assert lib.moe_read_device_flag(None, None, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_recover(None, ws, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_recover(dummy + 8, ws, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_recover(dummy, 8, None) == m.MOE_ERR_WORKSPACE
    assert lib.moe_static_read_device_flag(None, None) == m.MOE_ERR_INVALID_ARG
    # routing read-back: null workspace, no output, T out of range, small workspace
    rr = lib.moe_read_routing
    assert rr(None, ws, 1, dummy, None, None, None) == m.MOE_ERR_INVALID_ARG
    assert rr(dummy, ws, 1, None, None, None, None) == m.MOE_ERR_INVALID_ARG
    assert rr(dummy, ws, 0, dummy, None, None, None) == m.MOE_ERR_UNSUPPORTED
    assert rr(dummy, ws, m.MAX_TOKENS + 1, dummy, None, None, None) == m.MOE_ERR_UNSUPPORTED
    assert rr(dummy, ws, 8192, dummy, None, None, None) == m.MOE_ERR_WORKSPACE
    # dense GEMV: T, N, K outside the supported set, aliasing, small workspace
    gv = lib.moe_dense_gemv_nvfp4
    assert gv(dummy, dummy, 1.0, 2048, 2048, 9, dummy * 2, dummy, 256, None) == m.MOE_ERR_UNSUPPORTED
    assert gv(dummy, dummy, 1.0, 2048, 2048, 0, dummy * 2, dummy, 256, None) == m.MOE_ERR_UNSUPPORTED
    assert gv(dummy, dummy, 1.0, 24, 2048, 1, dummy * 2, dummy, 256, None) == m.MOE_ERR_UNSUPPORTED
    assert gv(dummy, dummy, 1.0, 2048, 384, 1, dummy * 2, dummy, 256, None) == m.MOE_ERR_UNSUPPORTED
    assert gv(dummy, dummy, 1.0, 2048, 8448, 1, dummy * 2, dummy, 256, None) == m.MOE_ERR_UNSUPPORTED
    assert gv(dummy, dummy, 1.0, 2048, 2048, 1, dummy + 64, dummy, 256, None) == m.MOE_ERR_INVALID_ARG
    assert gv(dummy, dummy, 1.0, 2048, 2048, 1, dummy * 2, dummy, 255, None) == m.MOE_ERR_WORKSPACE
    assert gv(None, dummy, 1.0, 2048, 2048, 1, dummy * 2, dummy, 256, None) == m.MOE_ERR_INVALID_ARG
    assert gv(dummy, dummy + 8, 1.0, 2048, 2048, 1, dummy * 2, dummy, 256, None) == m.MOE_ERR_INVALID_ARG
    # the no-allocation variant rejects T beyond its scratch before any CUDA call
    fs = lib.moe_layer_forward_static
    assert fs(dummy, dummy, B(bank), None, dummy * 2, 9, None) == m.MOE_ERR_UNSUPPORTED
    assert fs(dummy, dummy, B(bank), None, dummy * 2, 0, None) == m.MOE_ERR_UNSUPPORTED


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(OSError):
        m.load(str(tmp_path / "missing.so"))
