"""Pins of the oracle's layer steps (CPU only).

Router logits against numpy's fp64 matmul; top-k against a stable numpy sort;
gates against scipy's softmax over the selected logits; dispatch against
bincount / stable argsort; the expert FFN against a numpy dense SwiGLU on the
oracle's own dequantised weights; combine against zero-gate, linearity and
token-permutation invariants; the whole layer against the textbook dense
SwiGLU when E = 1, k = 1.
"""
import numpy as np
import pytest
from scipy.special import softmax

import gen
import oracle


def _bf16_bits(a):
    a = np.ascontiguousarray(a, np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _bf16_vals(bits):
    return gen.bf16_to_f32(bits).astype(np.float64)


def _tiny_layer(fmt=oracle.FMT_NVFP4, H=64, I=32, E=6, k=2, shared=1, bias=True, seed=0):
    if fmt == oracle.FMT_FP6:
        H, I = max(H, 128), max(I, 128)
    rng = np.random.default_rng(seed)
    router = _bf16_bits(rng.standard_normal((E, H)) * 0.2)
    b = (rng.standard_normal(E) * 0.1).astype(np.float32) if bias else None
    L = oracle.Layer(fmt, H, I, E, k, shared, router, b)
    for e in range(E + shared):
        for m in range(3):
            rows, K = L.shape(m)
            L.quantize_matrix(e, m, (rng.standard_normal((rows, K)) * 0.05).astype(np.float32))
    x = _bf16_bits(rng.standard_normal((5, H)))
    return L, x


def _silu(v):
    return v / (1.0 + np.exp(-v))


def _dense_swiglu(L, e, x_vals):
    Wg, Wu, Wd = (L.dequant(e, m).astype(np.float64) for m in range(3))
    a = _silu(x_vals @ Wg.T) * (x_vals @ Wu.T)
    return a @ Wd.T


def test_router_logits_match_numpy():
    L, x = _tiny_layer()
    got = L.logits(x)
    ref = (_bf16_vals(x) @ _bf16_vals(L.router).T).astype(np.float32) + L.bias
    assert np.array_equal(got, ref.astype(np.float32))


def test_topk_matches_stable_sort_and_softmax():
    rng = np.random.default_rng(7)
    T, E, k = 40, 16, 4
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[3, 5] = lg[3, 9] = lg[3].max() + 1  # an exact tie: the lower index goes first
    L = oracle.Layer(1, 16, 16, E, k, 0, np.zeros((E, 16), np.uint16))
    idx, gates = L.topk(lg)
    for t in range(T):
        order = np.lexsort((np.arange(E), -lg[t].astype(np.float64)))[:k]
        assert list(idx[t]) == list(order)
        ref = softmax(lg[t, order].astype(np.float64))
        assert np.allclose(gates[t], ref, rtol=0, atol=2e-7)
        assert abs(float(gates[t].astype(np.float64).sum()) - 1.0) <= k * 2.0 ** -23
    assert list(idx[3][:2]) == [5, 9]


def test_topk_single_expert_gate_is_one():
    L = oracle.Layer(1, 16, 16, 1, 1, 0, np.zeros((1, 16), np.uint16))
    idx, gates = L.topk(np.array([[0.3], [-7.0]], np.float32))
    assert np.all(idx == 0) and np.all(gates == 1.0)


def test_dispatch_matches_numpy():
    rng = np.random.default_rng(8)
    T, k, E = 33, 3, 10
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = oracle.dispatch(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(counts))
    assert offsets[-1] == T * k
    assert np.array_equal(perm, np.argsort(idx.ravel(), kind="stable"))
    assert np.array_equal(np.sort(perm), np.arange(T * k))


@pytest.mark.parametrize("fmt", [oracle.FMT_NVFP4, oracle.FMT_FP6, oracle.FMT_MXFP4])
def test_expert_ffn_matches_dense_swiglu(fmt):
    L, x = _tiny_layer(fmt=fmt)
    for e in (0, L.E):  # a routed expert and the shared one
        got = L.expert_ffn(e, x)
        ref = _dense_swiglu(L, e, _bf16_vals(x))
        assert np.allclose(got, ref, rtol=1e-6, atol=1e-9), np.abs(got - ref).max()


def test_combine_zero_gates_is_zero_without_shared():
    L, x = _tiny_layer(shared=0)
    idx = np.tile(np.array([[0, 3]], np.int32), (x.shape[0], 1))
    out = L.combine(x, idx, np.zeros(idx.shape, np.float32))
    assert np.all(out == 0.0)


def test_combine_is_linear_in_gates_and_sums_the_shared_expert():
    L, x = _tiny_layer(shared=1)
    T = x.shape[0]
    idx = np.tile(np.array([[1, 4]], np.int32), (T, 1))
    xv = _bf16_vals(x)
    y1, y4, ys = (_dense_swiglu(L, e, xv) for e in (1, 4, L.E))
    g = np.array([[0.75, 0.25]] * T, np.float32)
    out = L.combine(x, idx, g)
    ref = 0.75 * y1 + 0.25 * y4 + ys
    assert np.allclose(out, ref, rtol=1e-6, atol=1e-9)
    g2 = np.array([[0.5, 2.0]] * T, np.float32)
    out2 = L.combine(x, idx, g2)
    both = L.combine(x, idx, g + g2)
    assert np.allclose(both, out + out2 - ys, rtol=1e-6, atol=1e-7)


def test_forward_token_permutation_equivariance():
    L, x = _tiny_layer()
    lg, idx, gates, out = L.forward(x)
    p = np.array([3, 0, 4, 1, 2])
    lg2, idx2, gates2, out2 = L.forward(x[p])
    assert np.array_equal(lg2, lg[p]) and np.array_equal(idx2, idx[p])
    assert np.array_equal(gates2, gates[p]) and np.array_equal(out2, out[p])


def test_single_expert_top1_is_dense_swiglu():
    L, x = _tiny_layer(E=1, k=1, shared=0, bias=False)
    lg, idx, gates, out = L.forward(x)
    assert np.all(idx == 0) and np.all(gates == 1.0)
    ref = _dense_swiglu(L, 0, _bf16_vals(x))
    assert np.allclose(out, ref, rtol=1e-6, atol=1e-9)


def test_whole_layer_matches_numpy_composition():
    L, x = _tiny_layer(E=8, k=3, shared=1)
    lg, idx, gates, out = L.forward(x)
    xv = _bf16_vals(x)
    ref_lg = ((xv @ _bf16_vals(L.router).T).astype(np.float32) + L.bias).astype(np.float64)
    p = softmax(ref_lg, axis=1)
    ys = {e: _dense_swiglu(L, e, xv) for e in range(L.E + 1)}
    for t in range(x.shape[0]):
        sel = np.lexsort((np.arange(L.E), -p[t]))[:L.k]
        assert list(idx[t]) == list(sel)
        g = p[t, sel] / p[t, sel].sum()
        ref = sum(g[j] * ys[sel[j]][t] for j in range(L.k)) + ys[L.E][t]
        assert np.allclose(out[t], ref, rtol=1e-6, atol=1e-9)


def test_workload_inputs_are_seeded_and_shaped():
    w = gen.get_workload(0)
    x1, x2 = gen.x_tokens(w), gen.x_tokens(w)
    assert x1.shape == (w.T, w.H) and np.array_equal(x1, x2)
    xs = _bf16_vals(x1)
    assert abs(xs.mean()) < 0.1 and 0.9 < xs.std() < 1.1
    W = gen.expert_weight(w, 0, 2)
    assert W.shape == (w.H, w.I) and 0.018 < W.std() < 0.022
    # a slice drawn on its own equals the same slice of the whole tensor
    assert np.array_equal(gen.x_tokens(w, T=2, first=2), x1[2:4])
    zb = gen.router_bias(gen.get_workload(1))
    assert sorted(zb)[-1] == np.float32(0.5) and np.all(zb > 0)


# ---------------------------------------------------------------- sigmoid router (R19)
def test_sigmoid_router_selection_and_gates_against_numpy():
    rng = np.random.default_rng(21)
    T, E, k = 7, 40, 6
    lg = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    b = (rng.standard_normal(E) * 0.3).astype(np.float32)
    idx, gates = oracle.topk_gates_sigmoid(lg, b, k)
    s = 1.0 / (1.0 + np.exp(-lg.astype(np.float64)))
    key = s + b.astype(np.float64)
    for t in range(T):
        order = np.lexsort((np.arange(E), -key[t]))[:k]  # key descending, ties to the lower index
        assert np.array_equal(idx[t], order)
        g = s[t, order] / s[t, order].sum()
        assert np.allclose(gates[t], g, rtol=1e-6, atol=0)
        assert abs(float(gates[t].sum()) - 1.0) < 1e-6


def test_sigmoid_router_without_bias_picks_like_the_softmax_router():
    # sigmoid is increasing, so with b = 0 the picks are the top-k logits
    rng = np.random.default_rng(22)
    lg = rng.standard_normal((5, 64)).astype(np.float32)
    lg[2, 10] = lg[2, 20]  # an exact tie: the lower index first
    idx_s, _ = oracle.topk_gates_sigmoid(lg, None, 8)
    L = oracle.Layer(oracle.FMT_NVFP4, 64, 64, 64, 8, 0, np.zeros((64, 64), np.uint16))
    idx_m, _ = L.topk(lg)
    assert np.array_equal(idx_s, idx_m)


def test_sigmoid_router_bias_selects_but_does_not_weight():
    lg = np.array([[3.0, 2.0, -4.0, 1.0]], np.float32)
    b = np.array([0.0, 0.0, 2.0, 0.0], np.float32)  # lifts expert 2 into the top 2
    idx, gates = oracle.topk_gates_sigmoid(lg, b, 2)
    assert list(idx[0]) == [2, 0]
    s0, s2 = 1 / (1 + np.exp(-3.0)), 1 / (1 + np.exp(4.0))
    assert np.allclose(gates[0], [s2 / (s0 + s2), s0 / (s0 + s2)], rtol=1e-6)


# ---------------------------------------------------------------- W4A4 (R20)
def _fp4_rows(v):
    """Rows of v through the NVFP4 recipe and back, with the oracle's (pinned)
    quantiser and dequantiser, one row at a time."""
    v32 = np.ascontiguousarray(v, np.float32)
    out = np.empty_like(v32)
    for r in range(v32.shape[0]):
        c, s, ts = oracle.quantize_nvfp4(v32[r:r + 1])
        out[r] = oracle.dequant_nvfp4(c, s, ts, 1, v32.shape[1])[0]
    return out.astype(np.float64)


@pytest.mark.parametrize("fmt", [oracle.FMT_NVFP4, oracle.FMT_MXFP4, oracle.FMT_FP6])
def test_w4a4_expert_ffn_matches_numpy_composition(fmt):
    """The W4A4 expert (R20) against numpy over the oracle's pinned quantiser:
    x per token through NVFP4, the dense gate / up, a rounded to fp32 and per
    row through NVFP4, then the down projection."""
    L, x = _tiny_layer(fmt=fmt)
    L.act_fp4 = True
    xq = _fp4_rows(_bf16_vals(x))
    for e in (0, L.E):
        Wg, Wu, Wd = (L.dequant(e, m).astype(np.float64) for m in range(3))
        a = (_silu(xq @ Wg.T) * (xq @ Wu.T)).astype(np.float32)
        ref = _fp4_rows(a) @ Wd.T
        got = L.expert_ffn(e, x)
        assert np.allclose(got, ref, rtol=1e-6, atol=1e-9), np.abs(got - ref).max()


def test_w4a4_layer_differs_from_w4a16_by_activation_rounding_only():
    """The whole W4A4 layer: routing unchanged (the router keeps bf16 x), the
    output off the W4A16 one by the activation rounding (a few per cent for
    Gaussian activations, never zero), and exactly zero with zero down
    weights and no shared expert."""
    L, x = _tiny_layer(E=8, k=3, shared=1, seed=2)
    lg16, idx16, g16, out16 = L.forward(x)
    L.act_fp4 = True
    lg4, idx4, g4, out4 = L.forward(x)
    assert np.array_equal(lg16, lg4) and np.array_equal(idx16, idx4) and np.array_equal(g16, g4)
    rel = np.linalg.norm(out4 - out16, axis=1) / np.linalg.norm(out16, axis=1)
    assert np.all(rel > 1e-4) and np.all(rel < 0.3), rel
    # zero down weights: both give exactly zero (no shared expert)
    Z, xz = _tiny_layer(E=4, k=1, shared=0, seed=3)
    for e in range(4):
        Z.set_matrix(e, 2, np.zeros_like(Z.mats[(e, 2)][0]), np.zeros_like(Z.mats[(e, 2)][1]), 1.0)
    Z.act_fp4 = True
    assert np.all(Z.forward(xz)[3] == 0.0)


def test_w4a4_tie_evaluation_matches_the_oracle():
    """The tie-tolerant W4A4 comparison of the GPU tests (tests/parity.py,
    w4a4_tie_rel) re-evaluates a token in numpy with a scaled by 1 +- eta
    before its quantisation.  Against the oracle's own output it gives ~0
    (the smallest eta leaves the codes of a non-tie token alone), and against
    an output off by 1% it reports about 1%."""
    import parity
    L, x = _tiny_layer(E=8, k=3, shared=1, seed=4)
    L.act_fp4 = True
    lg, idx, gates, out = L.forward(x)
    for t in range(x.shape[0]):
        assert parity.w4a4_tie_rel(L, x[t], idx[t], gates[t], out[t]) < 1e-6
        r = parity.w4a4_tie_rel(L, x[t], idx[t], gates[t], out[t] * 1.01)
        assert 0.009 < r < 0.011
