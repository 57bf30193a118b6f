"""Independent pins for the fp64 oracle (CPU only).

Each ``pin_*`` function checks the oracle loaded as ``lib`` against something
other than itself: exhaustive comparison with torch's float8/bfloat16
decoders, a known-answer table of the e2m1 format, hand-made byte fixtures,
closed forms, invariants, and a brute-force dense evaluation of tiny layers
written here with numpy, scipy and torch (no oracle code).  They raise
AssertionError on a mismatch.  ``tests/test_oracle_pins.py`` runs them on the
real oracle; ``tests/test_oracle_mutants.py`` runs them on builds of the
oracle with a planted mistake and requires that each mistake is caught.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import scipy.special
import torch

import oracle
from nvfp4_moe_decode_gb300 import synth

# The 16 values of the FP4 E2M1 element format (OCP Microscaling Formats
# specification v1.0, FP4 E2M1: exponent bias 1, largest normal 6.0, smallest
# normal 1.0, subnormal 0.5); codes 8..15 are the negatives of 0..7.
E2M1_KNOWN = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


# ---------------------------------------------------------------------------
# independent helpers (numpy / torch / scipy only)
# ---------------------------------------------------------------------------

def np_e4m3(u8: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(u8, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def np_bf16(u16: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def np_dequant(codes: np.ndarray, scales: np.ndarray, tscale: float) -> np.ndarray:
    lo = codes & 0x0F
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)   # (n, 2j), (n, 2j+1)
    vals = np.array(E2M1_KNOWN)[nib]
    sc = np.repeat(np_e4m3(scales), 16, axis=1)
    return vals * sc * float(tscale)


def brute_topk(logits_row: np.ndarray, k: int):
    """The unique k-subset whose members all rank before every non-member
    (rank: larger fp32-rounded logit first, then lower index)."""
    E = len(logits_row)
    f = logits_row.astype(np.float32)

    def before(a, b):
        return (f[a] > f[b]) or (f[a] == f[b] and a < b)

    found = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(before(a, b) for a in S for b in rest):
            found.append(S)
    assert len(found) == 1
    S = sorted(found[0], key=lambda e: (-float(f[e]), e))
    return np.array(S, dtype=np.int32)


def host_inputs(li: synth.LayerInputs):
    """torch CPU LayerInputs -> numpy bit patterns + oracle ExpertWeights."""
    x = li.x.view(torch.int16).numpy().view(np.uint16)
    wr = li.router_w.view(torch.int16).numpy().view(np.uint16)
    E, S = li.n_routed, li.n_shared
    ex = []
    for e in range(E + S):
        if li.wtype == synth.NVFP4:
            ex.append(oracle.ExpertWeights(0, li.codes13[e].numpy(), li.scales13[e].numpy(),
                                           float(li.tscale13[e]), li.codes2[e].numpy(),
                                           li.scales2[e].numpy(), float(li.tscale2[e])))
        else:
            ex.append(oracle.ExpertWeights(1, li.w13[e].view(torch.int16).numpy().view(np.uint16),
                                           None, 1.0,
                                           li.w2[e].view(torch.int16).numpy().view(np.uint16),
                                           None, 1.0))
    return x, wr, ex[:E], (ex[E] if S else None)


def dense_expert_outputs(W13: np.ndarray, W2: np.ndarray, X: np.ndarray, I: int) -> np.ndarray:
    g = X @ W13[:I].T
    u = X @ W13[I:].T
    h = g * scipy.special.expit(g) * u
    return h @ W2.T


def brute_layer(li: synth.LayerInputs, top_k: int):
    """Dense masked evaluation over every expert (no sparsity, no oracle code)."""
    x = np_bf16(li.x.view(torch.int16).numpy())
    wr = np_bf16(li.router_w.view(torch.int16).numpy())
    E, S, I = li.n_routed, li.n_shared, li.inter
    logits = x @ wr.T
    T = x.shape[0]
    gate = np.zeros((T, E))
    idx = np.zeros((T, top_k), dtype=np.int32)
    for t in range(T):
        sel = brute_topk(logits[t], top_k)
        idx[t] = sel
        s = scipy.special.expit(logits[t, sel])
        gate[t, sel] = s / s.sum()

    def weights(e):
        if li.wtype == synth.NVFP4:
            W13 = np_dequant(li.codes13[e].numpy(), li.scales13[e].numpy(), float(li.tscale13[e]))
            W2 = np_dequant(li.codes2[e].numpy(), li.scales2[e].numpy(), float(li.tscale2[e]))
        else:
            W13 = np_bf16(li.w13[e].view(torch.int16).numpy())
            W2 = np_bf16(li.w2[e].view(torch.int16).numpy())
        return W13, W2

    out = np.zeros_like(x)
    for e in range(E):
        W13, W2 = weights(e)
        out += gate[:, e:e + 1] * dense_expert_outputs(W13, W2, x, I)
    for s_ in range(S):
        W13, W2 = weights(E + s_)
        out += dense_expert_outputs(W13, W2, x, I)
    return out, idx, gate, logits


def run_oracle(li: synth.LayerInputs, top_k: int, lib):
    x, wr, routed, shared = host_inputs(li)
    return oracle.moe_forward(x, wr, routed, top_k, li.inter, shared, lib=lib)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_e2m1_known_values(lib):
    for c in range(16):
        v = oracle.e2m1_value(c, lib)
        assert v == E2M1_KNOWN[c] and math.copysign(1, v) == math.copysign(1, E2M1_KNOWN[c]), \
            (c, v, E2M1_KNOWN[c])


def pin_e4m3_matches_torch(lib):
    ref = np_e4m3(np.arange(256, dtype=np.uint8))
    for c in range(256):
        v = oracle.e4m3_value(c, lib)
        if np.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])


def pin_bf16_matches_torch(lib):
    codes = np.arange(65536, dtype=np.uint32)
    ref = np_bf16(codes.astype(np.uint16))
    step = 97  # a stride through all exponents and signs (plus the specials)
    picks = list(range(0, 65536, step)) + [0x0000, 0x8000, 0x0001, 0x7F7F, 0xFF7F, 0x7F80,
                                           0x3F80, 0xBF80, 0x0080]
    for c in picks:
        v = oracle.bf16_value(c, lib)
        if np.isnan(ref[c]):
            assert math.isnan(v)
        else:
            assert v == ref[c], (hex(c), v, ref[c])


def pin_dequant_byte_fixture(lib):
    """Hand-made bytes: row 0 = 0x21 0x8F ..., scale 0x38 (= 1.0), 0x40 (= 2.0)."""
    K = 32
    codes = np.zeros((2, K // 2), dtype=np.uint8)
    scales = np.zeros((2, K // 16), dtype=np.uint8)
    codes[0, 0] = 0x21   # k=0: code 1 (0.5); k=1: code 2 (1.0)
    codes[0, 1] = 0x8F   # k=2: code 15 (-6.0); k=3: code 8 (-0.0)
    codes[0, 8] = 0x07   # k=16: code 7 (6.0); k=17: code 0
    codes[1, 15] = 0xA3  # row 1, k=30: code 3 (1.5); k=31: code 10 (-1.0)
    scales[0, 0] = 0x38  # 1.0 for row 0, k in [0, 16)
    scales[0, 1] = 0x40  # 2.0 for row 0, k in [16, 32)
    scales[1, 1] = 0x30  # 0.5 for row 1, k in [16, 32)
    W = oracle.dequant_nvfp4(codes, scales, 1.0, lib)
    expect = np.zeros((2, K))
    expect[0, 0], expect[0, 1], expect[0, 2], expect[0, 3] = 0.5, 1.0, -6.0, -0.0
    expect[0, 16] = 12.0
    expect[1, 30], expect[1, 31] = 0.75, -0.5
    assert np.array_equal(W, expect), np.argwhere(W != expect)
    W3 = oracle.dequant_nvfp4(codes, scales, 3.0, lib)
    assert np.array_equal(W3, 3.0 * expect)


def pin_dequant_matches_numpy(lib):
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 256, size=(16, 64), dtype=np.uint8)
    codes[0, :] = np.arange(64, dtype=np.uint8) * 4 + 1   # many code pairs
    scales = rng.integers(0, 0x7E, size=(16, 8), dtype=np.uint8)  # finite e4m3
    W = oracle.dequant_nvfp4(codes, scales, 0.75, lib)
    assert np.array_equal(W, np_dequant(codes, scales, 0.75))


def pin_router_logits_numpy(lib):
    li = synth.make_layer(3, 5, hidden=64, n_routed=8, inter=16, weights=False)
    x = li.x.view(torch.int16).numpy().view(np.uint16)
    wr = li.router_w.view(torch.int16).numpy().view(np.uint16)
    lg = oracle.router_logits(x, wr, lib)
    ref = np_bf16(x) @ np_bf16(wr).T
    assert np.allclose(lg, ref, rtol=1e-13, atol=1e-15)


def pin_topk_bruteforce(lib):
    rng = np.random.default_rng(11)
    for E, k in [(4, 2), (6, 3), (8, 6), (7, 1), (5, 5)]:
        lg = rng.normal(size=(20, E))
        lg[0, :] = 0.0                          # all equal: lowest indices win
        lg[1, :] = np.round(lg[1, :] * 2) / 2   # many exact ties
        idx, w = oracle.select_topk(lg, k, lib)
        for t in range(lg.shape[0]):
            assert np.array_equal(idx[t], brute_topk(lg[t], k)), (E, k, t, idx[t])
            s = scipy.special.expit(lg[t, idx[t]])
            assert np.allclose(w[t], s / s.sum(), rtol=1e-14, atol=0)
        assert np.array_equal(idx[0], np.arange(k))


def pin_topk_invariants(lib):
    rng = np.random.default_rng(5)
    lg = rng.normal(scale=0.9, size=(64, 256))
    idx, w = oracle.select_topk(lg, 6, lib)
    for t in range(64):
        sel = idx[t]
        assert len(set(sel.tolist())) == 6 and sel.min() >= 0 and sel.max() < 256
        assert np.all(w[t] > 0) and abs(w[t].sum() - 1.0) <= 1e-12
        rest = np.setdiff1d(np.arange(256), sel)
        assert lg[t, sel].astype(np.float32).min() >= lg[t, rest].astype(np.float32).max()


def pin_layer_bruteforce_nvfp4(lib):
    li = synth.make_layer(1, 5, hidden=32, n_routed=6, inter=16, n_shared=1)
    out, idx, w, _ = run_oracle(li, 2, lib)
    ref, ridx, _, _ = brute_layer(li, 2)
    assert np.array_equal(idx, ridx)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def pin_layer_bruteforce_bf16(lib):
    li = synth.make_layer(2, 4, hidden=32, n_routed=5, inter=16, n_shared=1, wtype=synth.BF16)
    out, idx, w, _ = run_oracle(li, 3, lib)
    ref, ridx, _, _ = brute_layer(li, 3)
    assert np.array_equal(idx, ridx)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def pin_layer_bruteforce_larger_k(lib):
    li = synth.make_layer(4, 3, hidden=48, n_routed=8, inter=32, n_shared=1)
    out, idx, w, _ = run_oracle(li, 6, lib)
    ref, ridx, _, _ = brute_layer(li, 6)
    assert np.array_equal(idx, ridx)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def pin_zero_input(lib):
    """x = 0: every logit is 0, experts 0..k-1 are chosen with weight 1/k, and
    every expert output is 0 (g = u = 0)."""
    li = synth.make_layer(5, 3, hidden=32, n_routed=6, inter=16)
    li.x.zero_()
    out, idx, w, _ = run_oracle(li, 3, lib)
    assert np.all(out == 0.0)
    assert np.array_equal(idx, np.tile(np.arange(3, dtype=np.int32), (3, 1)))
    assert np.allclose(w, 1.0 / 3.0, rtol=0, atol=1e-15)


def pin_zero_scales(lib):
    li = synth.make_layer(6, 2, hidden=32, n_routed=4, inter=16)
    li.scales13.zero_()
    out, _, _, _ = run_oracle(li, 2, lib)
    assert np.all(out == 0.0)


def pin_routed_off_leaves_shared(lib):
    """Routed tensor scales 0: the output is the shared expert alone, which
    for a one-hot x reduces to a closed form."""
    li = synth.make_layer(8, 1, hidden=32, n_routed=4, inter=16)
    li.tscale13[:4] = 0.0
    H, I = 32, 16
    # Shared expert: every gate/up code 2 (1.0) in column 0 only; x = e_0 * 1.5.
    li.x.zero_()
    li.x[0, 0] = 1.5
    sh = 4
    li.codes13[sh].zero_()
    li.codes13[sh][:, 0] = 0x02          # element (n, 0) = code 2 = 1.0, (n, 1) = 0
    li.scales13[sh].fill_(0x38)          # 1.0
    li.codes2[sh].zero_()
    li.codes2[sh][:, 0] = 0x02 | (0x0A << 4)   # element (n,0) = 1.0, (n,1) = -1.0
    li.scales2[sh].fill_(0x40)           # 2.0
    out, _, _, _ = run_oracle(li, 2, lib)
    g = 1.5
    h0 = g * (1.0 / (1.0 + math.exp(-g))) * 1.5     # every row i: g_i = u_i = 1.5
    # y_n = sum_i W2[n][i] h_i = 2.0 * (1.0 * h0 - 1.0 * h0) = 0 for column pair;
    # rows n: only columns 0 and 1 are nonzero -> y_n = 2*h0 - 2*h0 = 0.
    assert np.allclose(out, 0.0, atol=1e-15)
    li.codes2[sh][:, 0] = 0x02           # now only element (n, 0) = 1.0
    out, _, _, _ = run_oracle(li, 2, lib)
    assert np.allclose(out, 2.0 * h0, rtol=1e-15, atol=0), (out[0, :4], 2 * h0)


def pin_combine_linear_in_down_scale(lib):
    """Doubling every routed down tensor scale doubles the routed part."""
    li = synth.make_layer(9, 3, hidden=32, n_routed=5, inter=16)
    base, _, _, _ = run_oracle(li, 2, lib)
    li.tscale2[:5] = 0.0
    shared_only, _, _, _ = run_oracle(li, 2, lib)
    li.tscale2[:5] = 2.0
    doubled, _, _, _ = run_oracle(li, 2, lib)
    routed = base - shared_only
    assert np.allclose(doubled - shared_only, 2.0 * routed, rtol=1e-12,
                       atol=1e-12 * np.abs(routed).max())


def pin_expert_permutation_invariance(lib):
    """Relabelling the routed experts (router rows permuted with them) leaves
    the output unchanged when no two logits tie."""
    li = synth.make_layer(10, 4, hidden=32, n_routed=6, inter=16)
    base, idx, _, _ = run_oracle(li, 2, lib)
    perm = torch.tensor([3, 0, 5, 1, 4, 2])
    li.router_w = li.router_w[perm].contiguous()
    full = torch.cat([perm, torch.tensor([6])])
    for name in ("codes13", "scales13", "codes2", "scales2", "tscale13", "tscale2"):
        setattr(li, name, getattr(li, name)[full].contiguous())
    out, idx2, _, _ = run_oracle(li, 2, lib)
    assert np.allclose(out, base, rtol=1e-12, atol=1e-12 * np.abs(base).max())
    assert np.array_equal(perm.numpy()[idx2], idx)


# ---------------------------------------------------------------------------
# expert sinks (shared experts in the normalisation, not in the top-k)
# ---------------------------------------------------------------------------

def host_inputs_sinks(li: synth.LayerInputs):
    """LayerInputs with S shared experts -> bits + routed and shared ExpertWeights lists."""
    x = li.x.view(torch.int16).numpy().view(np.uint16)
    wr = li.router_w.view(torch.int16).numpy().view(np.uint16)
    E, S = li.n_routed, li.n_shared

    def nv(e):
        return oracle.ExpertWeights(0, li.codes13[e].numpy(), li.scales13[e].numpy(), float(li.tscale13[e]),
                                    li.codes2[e].numpy(), li.scales2[e].numpy(), float(li.tscale2[e]))

    def bf(w13, w2):
        return oracle.ExpertWeights(1, w13.view(torch.int16).numpy().view(np.uint16), None, 1.0,
                                    w2.view(torch.int16).numpy().view(np.uint16), None, 1.0)

    if li.wtype == synth.NVFP4:
        routed = [nv(e) for e in range(E)]
        shared = ([bf(li.sw13[j], li.sw2[j]) for j in range(S)] if li.shared_bf16
                  else [nv(E + j) for j in range(S)])
    else:
        routed = [bf(li.w13[e], li.w2[e]) for e in range(E)]
        shared = [bf(li.w13[E + j], li.w2[E + j]) for j in range(S)]
    return x, wr, routed, shared


def brute_layer_sinks(li: synth.LayerInputs, top_k: int):
    """Dense masked evaluation with S shared experts (numpy/scipy only)."""
    x = np_bf16(li.x.view(torch.int16).numpy())
    wr = np_bf16(li.router_w.view(torch.int16).numpy())
    E, S, I = li.n_routed, li.n_shared, li.inter
    logits = x @ wr.T
    T = x.shape[0]
    gate = np.zeros((T, E))
    sw = np.ones((T, S))
    idx = np.zeros((T, top_k), dtype=np.int32)
    for t in range(T):
        sel = brute_topk(logits[t, :E], top_k)
        idx[t] = sel
        s_ = scipy.special.expit(logits[t, sel])
        d = s_.sum()
        if li.sink:
            ss = scipy.special.expit(logits[t, E:E + S])
            d += ss.sum()
            sw[t] = ss / d
        gate[t, sel] = s_ / d

    def nv(e):
        return (np_dequant(li.codes13[e].numpy(), li.scales13[e].numpy(), float(li.tscale13[e])),
                np_dequant(li.codes2[e].numpy(), li.scales2[e].numpy(), float(li.tscale2[e])))

    def bf(w13, w2):
        return np_bf16(w13.view(torch.int16).numpy()), np_bf16(w2.view(torch.int16).numpy())

    out = np.zeros_like(x)
    for e in range(E):
        W13, W2 = nv(e) if li.wtype == synth.NVFP4 else bf(li.w13[e], li.w2[e])
        out += gate[:, e:e + 1] * dense_expert_outputs(W13, W2, x, I)
    for j in range(S):
        if li.shared_bf16:
            W13, W2 = bf(li.sw13[j], li.sw2[j])
        elif li.wtype == synth.NVFP4:
            W13, W2 = nv(E + j)
        else:
            W13, W2 = bf(li.w13[E + j], li.w2[E + j])
        out += sw[:, j:j + 1] * dense_expert_outputs(W13, W2, x, I)
    return out, idx, gate, sw


def pin_topk_sink_bruteforce(lib):
    """Top-k over the routed columns only (brute force over k-subsets); the
    sinks' scores join the denominator.  Half of the rows give the sinks
    the largest logits, so a sink taken as a candidate would be selected."""
    rng = np.random.default_rng(13)
    for E, S, k in [(6, 2, 3), (8, 2, 6), (5, 1, 2), (7, 2, 1)]:
        lg = rng.normal(size=(20, E + S))
        lg[::2, E:] += 4.0
        idx, w, sw = oracle.select_topk_sink(lg, E, k, lib=lib)
        for t in range(lg.shape[0]):
            sel = brute_topk(lg[t, :E], k)
            assert np.array_equal(idx[t], sel), (E, S, k, t)
            s_ = scipy.special.expit(lg[t, sel])
            ss = scipy.special.expit(lg[t, E:])
            d = s_.sum() + ss.sum()
            assert np.allclose(w[t], s_ / d, rtol=1e-14, atol=0)
            assert np.allclose(sw[t], ss / d, rtol=1e-14, atol=0)
            assert abs(w[t].sum() + sw[t].sum() - 1.0) < 1e-14


def pin_topk_sink_limits(lib):
    """Sink logits -inf: the sinks absorb nothing and the routing is the plain
    sigmoid top-k.  +inf: each sink scores exactly 1."""
    rng = np.random.default_rng(17)
    E, S, k = 12, 2, 4
    lg = rng.normal(size=(16, E + S))
    lo = lg.copy()
    lo[:, E:] = -np.inf
    idx, w, sw = oracle.select_topk_sink(lo, E, k, lib=lib)
    idx0, w0 = oracle.select_topk(lg[:, :E], k, lib=lib)
    assert np.array_equal(idx, idx0) and np.all(sw == 0.0)
    assert np.allclose(w, w0, rtol=1e-15, atol=0)
    hi = lg.copy()
    hi[:, E:] = np.inf
    idx, w, sw = oracle.select_topk_sink(hi, E, k, lib=lib)
    for t in range(lg.shape[0]):
        s_ = scipy.special.expit(lg[t, idx[t]])
        d = s_.sum() + S
        assert np.allclose(w[t], s_ / d, rtol=1e-14, atol=0)
        assert np.allclose(sw[t], 1.0 / d, rtol=1e-14, atol=0)


def _check_sink_layer(lib, li, top_k):
    x, wr, routed, shared = host_inputs_sinks(li)
    out, idx, w, sw, _ = oracle.moe_forward_sinks(x, wr, routed, top_k, li.inter, shared, li.sink, lib=lib)
    ref, ridx, _, rsw = brute_layer_sinks(li, top_k)
    assert np.array_equal(idx, ridx)
    assert np.allclose(sw, rsw, rtol=1e-12, atol=0)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12 * np.abs(ref).max())


def pin_layer_sinks_bruteforce(lib):
    """Two BF16 shared experts as sinks beside NVFP4 routed experts, and the
    same layer shape without sinks (shared weight 1)."""
    _check_sink_layer(lib, synth.make_layer(12, 3, hidden=32, n_routed=6, inter=16, n_shared=2, sink=True,
                                            shared_bf16=True), 2)
    _check_sink_layer(lib, synth.make_layer(13, 2, hidden=32, n_routed=7, inter=16, n_shared=2, sink=False,
                                            shared_bf16=True), 3)
    _check_sink_layer(lib, synth.make_layer(14, 2, hidden=48, n_routed=5, inter=32, n_shared=1, sink=True,
                                            wtype=synth.BF16), 2)


# ---------------------------------------------------------------------------
# the dense GEMV
# ---------------------------------------------------------------------------

def _bf16_bits(v: torch.Tensor) -> np.ndarray:
    return v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def pin_dense_gemv_one_hot(lib):
    """One non-zero code (6.0 at row 17, column 45, block scale 2.0) and a
    tensor scale of 0.5: y[t][17] = 6 * 2 * 0.5 * x[t][45], every other y is 0."""
    N, K, T = 32, 64, 3
    codes = np.zeros((N, K // 2), dtype=np.uint8)
    codes[17, 45 // 2] = 0x7 << 4            # odd column: the high nibble; e2m1 code 7 = 6.0
    scales = np.full((N, K // 16), 0x38, dtype=np.uint8)   # e4m3 1.0
    scales[17, 45 // 16] = 0x40                           # e4m3 2.0
    x = _bf16_bits(torch.randn(T, K, generator=torch.Generator().manual_seed(3)))
    y = oracle.dense_gemv_nvfp4(codes, scales, 0.5, x, lib=lib)
    xv = np_bf16(x)
    want = np.zeros((T, N))
    want[:, 17] = 6.0 * xv[:, 45]
    assert np.array_equal(y, want)


def pin_dense_gemv_row_sums(lib):
    """Every code 1.0, every scale 1.0, tensor scale 1: y[t][n] is the sum of
    token t's activations (math.fsum, correctly rounded)."""
    N, K, T = 16, 256, 4
    codes = np.full((N, K // 2), 0x22, dtype=np.uint8)    # both nibbles e2m1 1.0
    scales = np.full((N, K // 16), 0x38, dtype=np.uint8)
    x = _bf16_bits(torch.randn(T, K, generator=torch.Generator().manual_seed(4)) * 3)
    y = oracle.dense_gemv_nvfp4(codes, scales, 1.0, x, lib=lib)
    xv = np_bf16(x)
    for t in range(T):
        s_ = math.fsum(xv[t])
        bound = 1e-13 * np.abs(xv[t]).sum()
        assert np.all(np.abs(y[t] - s_) <= bound), (t, y[t, 0], s_)


def pin_dense_gemv_bruteforce(lib):
    """Tiny random matrix: loops over the e2m1 table and torch's e4m3 decode."""
    N, K, T = 16, 32, 2
    rng = np.random.default_rng(21)
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = (np.abs(rng.standard_normal((N, K // 16))) * 0.3).astype(np.float32)
    scales = torch.from_numpy(scales).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    x = _bf16_bits(torch.randn(T, K, generator=torch.Generator().manual_seed(5)))
    ts = 0.75
    y = oracle.dense_gemv_nvfp4(codes, scales, ts, x, lib=lib)
    xv = np_bf16(x)
    sv = np_e4m3(scales)
    for t in range(T):
        for n in range(N):
            terms = []
            for k in range(K):
                byte = int(codes[n, k // 2])
                code = (byte >> 4) if k % 2 else (byte & 0xF)
                terms.append(E2M1_KNOWN[code] * float(sv[n, k // 16]) * ts * float(xv[t, k]))
            want = math.fsum(terms)
            assert abs(y[t, n] - want) <= 1e-13 * sum(abs(v) for v in terms), (t, n)


# ---------------------------------------------------------------------------
# the pre-norm step of a decoder stack and bf16 rounding
# ---------------------------------------------------------------------------

def _torch_bf16_bits(v32: np.ndarray) -> np.ndarray:
    """float32 values -> bf16 bit patterns by torch's float32 -> bfloat16 cast
    (one round-to-nearest-even)."""
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _near_bf16_tie(v: float) -> bool:
    """True when v lies within 2^-20 of a quantum of the midpoint between two
    bf16 neighbours (where a float32 intermediate could round twice)."""
    if v == 0.0 or not math.isfinite(v):
        return False
    m, e = math.frexp(abs(v))
    q = m * 256.0
    return abs((q - math.floor(q)) - 0.5) < 2.0 ** -20


def pin_round_bf16_known_answers(lib):
    rb = lambda v: oracle.round_bf16(v, lib=lib)  # noqa: E731
    # exact ties go to the even neighbour
    assert rb(1.0 + 2.0 ** -8) == 0x3F80
    assert rb(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert rb(-(1.0 + 2.0 ** -8)) == 0xBF80
    # just above a tie (below float32 resolution) rounds up: no double rounding
    assert rb(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert rb(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    # the largest finite bf16, overflow, zero signs, subnormals
    assert rb(3.3895313892515355e38) == 0x7F7F
    assert rb(3.5e38) == 0x7F80 and rb(-3.5e38) == 0xFF80
    assert rb(0.0) == 0x0000 and rb(-0.0) == 0x8000
    assert rb(2.0 ** -130) == 0x0008 and rb(2.0 ** -133) == 0x0001
    # random float32 values: the same single rounding as torch's cast
    rng = np.random.default_rng(5)
    vals = (rng.standard_normal(4000) * np.exp2(rng.integers(-60, 60, 4000))).astype(np.float32)
    want = _torch_bf16_bits(vals)
    got = np.array([rb(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def pin_prenorm_constant_vector(lib):
    """A constant token c: RMSNorm gives c / sqrt(c^2 + eps) in every entry."""
    H, eps = 256, 1e-3
    for c in (0.0625, -3.0, 0.75, 40.0):
        bits = int(_torch_bf16_bits(np.array([c], dtype=np.float32))[0])
        x = np.full((1, H), bits, dtype=np.uint16)
        v, xn = oracle.prenorm(x, None, eps, lib=lib)
        assert np.all(v == bits)
        val = c / math.sqrt(c * c + eps)
        assert not _near_bf16_tie(val)
        want = int(_torch_bf16_bits(np.array([val], dtype=np.float32))[0])
        assert np.all(xn == want), (c, hex(int(xn[0, 0])), hex(want))


def pin_prenorm_matches_torch(lib):
    """Random tokens: v against torch's bf16 add, xn against
    torch.nn.functional.rms_norm in float64, rounded once to bf16."""
    T, H, eps = 3, 512, 1e-6
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(T, H, generator=g) * 2.0).to(torch.bfloat16)
    d = (torch.randn(T, H, generator=g) * 0.5).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    db = d.view(torch.int16).numpy().view(np.uint16)
    v, xn = oracle.prenorm(xb, db, eps, lib=lib)
    v_t = (x.float() + d.float()).to(torch.bfloat16)
    assert np.array_equal(v, v_t.view(torch.int16).numpy().view(np.uint16))
    ref = torch.nn.functional.rms_norm(v_t.double(), (H,), eps=eps).numpy()
    got = np_bf16(xn)
    flat_ref = ref.reshape(-1)
    ok = np.array([not _near_bf16_tie(float(r)) for r in flat_ref])
    want = _torch_bf16_bits(flat_ref.astype(np.float32))
    assert np.array_equal(xn.reshape(-1)[ok], want[ok])
    ulp = np.exp2(np.floor(np.log2(np.abs(ref))) - 7)
    assert np.all(np.abs(got - ref) <= 0.5 * ulp * (1 + 1e-9))
    # delta = None is the same as a zero delta
    v0, xn0 = oracle.prenorm(xb, None, eps, lib=lib)
    vz, xnz = oracle.prenorm(xb, np.zeros_like(xb), eps, lib=lib)
    assert np.array_equal(v0, vz) and np.array_equal(xn0, xnz) and np.array_equal(v0, xb)


ALL_PINS = [
    pin_e2m1_known_values,
    pin_e4m3_matches_torch,
    pin_bf16_matches_torch,
    pin_dequant_byte_fixture,
    pin_dequant_matches_numpy,
    pin_router_logits_numpy,
    pin_topk_bruteforce,
    pin_topk_invariants,
    pin_layer_bruteforce_nvfp4,
    pin_layer_bruteforce_bf16,
    pin_layer_bruteforce_larger_k,
    pin_zero_input,
    pin_zero_scales,
    pin_routed_off_leaves_shared,
    pin_combine_linear_in_down_scale,
    pin_expert_permutation_invariance,
    pin_topk_sink_bruteforce,
    pin_topk_sink_limits,
    pin_layer_sinks_bruteforce,
    pin_dense_gemv_one_hot,
    pin_dense_gemv_row_sums,
    pin_dense_gemv_bruteforce,
    pin_round_bf16_known_answers,
    pin_prenorm_constant_vector,
    pin_prenorm_matches_torch,
]
