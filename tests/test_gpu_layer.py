"""GPU: the whole layer against the oracle on the seeded workloads, plus the
properties that hold at any size (determinism, batch invariance, every output
written, zero gates, linearity) and the error paths of the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_moe_expert_layer_gb300 as moe
from quantized_moe_expert_layer_gb300.synthetic import build_layer

from parity import compare_layer, logit_bound, run_gpu, to_dev_bf16, valid_near_tie

pytestmark = pytest.mark.gpu

_layers = {}


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    gen.build(device=True)
    moe.build()
    yield
    for L in _layers.values():
        L.close()
    _layers.clear()


def layer(w, T_max=None):
    key = (w.H, w.I, w.E, w.k, w.shared, w.fmt, w.seed, w.bias, w.bias_scale)
    if key not in _layers:
        _layers[key] = build_layer(w, T_max=T_max or 4096)
    return _layers[key]


def small(fmt=1, H=256, I=128, E=8, k=2, shared=1, T=13, bias="normal", seed=3):
    return gen.Workload(f"small-{fmt}-{H}-{I}-{E}-{k}-{shared}", H, I, E, k, shared, T, fmt, bias,
                        0.0, 0.1, seed)


# ---------------------------------------------------------------- parity per workload
def test_tiny_workload():
    w = gen.get_workload(0)
    rel, ties = compare_layer(w, layer(w), gen.x_tokens(w))
    assert ties == 0


@pytest.mark.parametrize("fmt", [1, 2, 3])
@pytest.mark.parametrize("T", [1, 5, 13, 64, 70, 200])
def test_small_layers_ragged_token_counts(fmt, T):
    """Several tiles, ragged last entries, the routing paths (T = 1 in-CTA,
    T <= 16 top-k inside the dispatch kernel, larger T the top-k kernel whose
    last CTA dispatches), all formats, with a shared expert."""
    w = small(fmt=fmt, H=384 if fmt == 2 else 320, I=256 if fmt == 2 else 192, E=24, k=3, T=T)
    compare_layer(w, layer(w), gen.x_tokens(w, T))


@pytest.mark.parametrize("T", [128, 300, 700])
def test_tensor_core_path_small_layer(T):
    """Enough tokens per expert for the tcgen05 grouped GEMMs (T*k >= 16 E): ragged
    per-expert counts (N from 1 to ~250, padded to 16), several shared-expert
    work items of up to 256 tokens."""
    w = small(fmt=1, H=256, I=128, E=8, k=2, T=T, seed=5)
    L = layer(w)
    # router, top-k + dispatch (one kernel), row gather, tc gate/up, tc down, combine
    assert L.launches(T) == 6
    compare_layer(w, L, gen.x_tokens(w, T))


@pytest.mark.parametrize("T", [2731, 3000])
def test_several_cta_dispatch_ragged_chunks(T):
    """T*k above one CTA's dispatch (8192 slots): per-chunk counts, then a
    placement CTA per 1024 slots that sums the earlier chunks' counts itself,
    the last chunk ragged (1 slot at T = 2731); the top-k takes a warp per
    token (T >= 1024);
    counts / offsets / perm bit-exact against the oracle's dispatch of the same
    picks (compare_layer), the output on sampled tokens."""
    w = small(fmt=1, H=256, I=128, E=24, k=3, T=T, seed=9)
    L = layer(w)
    # router, top-k, count, scan + place, row gather, tc gate/up, tc down, combine
    assert L.launches(T) == 8
    compare_layer(w, L, gen.x_tokens(w, T), sample=[0, 1, T // 2, T - 2, T - 1])


@pytest.mark.parametrize("T", [1024, 1100])
def test_tensor_core_router_small_layer(T):
    """128 experts: the router runs as a bf16 tcgen05 GEMM (one 128-expert block,
    token tiles of 128 with a ragged last one), ahead of the grouped expert GEMMs."""
    w = small(fmt=1, H=256, I=128, E=128, k=2, T=T, seed=7)
    L = layer(w)
    # tc router, top-k, dispatch, row gather (with the x conversion), tc gate/up, tc down, combine
    assert L.launches(T) == 7
    compare_layer(w, L, gen.x_tokens(w, T))


def test_decode_nvfp4_full_size():
    w = gen.get_workload(1)
    L = layer(w)
    assert L.launches(1) == 3  # router, gate/up (routing inside), down + combine (routing inside)
    rel, ties = compare_layer(w, L, gen.x_tokens(w))
    print(f"decode nvfp4: rel-L2 {rel:.2e}, near ties {ties}")


@pytest.mark.parametrize("T", [1, 3, 8])
def test_self_routed_and_dispatched_paths_agree_bit_for_bit(T):
    """For T <= 8 the expert kernels take the top-k and the dispatch themselves;
    given the same picks and gates, the explicitly dispatched path (dispatch
    kernel, then the expert kernels) gives the same bits."""
    w = gen.get_workload(1)
    L = layer(w)
    x_np = gen.x_tokens(w, T)
    a = run_gpu(L, x_np, w)
    x = to_dev_bf16(x_np)
    idx = torch.from_numpy(a["idx"]).cuda()
    gates = torch.from_numpy(a["gates"]).cuda()
    out = torch.empty((T, w.H), device="cuda")
    L.forward_routed(x, idx, gates, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), a["out"])


def test_decode_fp6_full_size():
    w = gen.get_workload(2)
    L = build_layer(w, T_max=8)
    try:
        rel, ties = compare_layer(w, L, gen.x_tokens(w))
        print(f"decode fp6: rel-L2 {rel:.2e}, near ties {ties}")
    finally:
        L.close()


def test_batched_decode_full_size():
    w = gen.get_workload(3)
    rel, ties = compare_layer(w, layer(w), gen.x_tokens(w))
    print(f"batched T=64: rel-L2 {rel:.2e}, near ties {ties}")


def test_prefill_full_size_sampled():
    """Routing (logits, top-k, gates) of all 4096 tokens against the oracle;
    the layer output on sampled tokens (the expert FFNs dominate the oracle's
    time)."""
    w = gen.get_workload(4)
    sample = [0, 1, 7, 8, 511, 1024, 2047, 2048, 3000, 4093, 4094, 4095]
    rel, ties = compare_layer(w, layer(w), gen.x_tokens(w), sample=sample, route_all=True)
    print(f"prefill T=4096 (routing of every token, output sampled): rel-L2 {rel:.2e}, "
          f"near ties {ties}")


def test_tiny_mxfp4_workload():
    w = gen.get_workload(5)
    rel, ties = compare_layer(w, layer(w), gen.x_tokens(w))
    assert ties == 0


def test_deepseek_shape_mxfp4_decode_full_size():
    """The wide-expert decode (128 tile pairs an expert): more CTAs than fit the
    GPU at once, so a routed CTA takes several tile pairs in turn; T = 1 and a
    batch of 8 against the oracle, and for T = 3 the self-routed kernel gives
    the bits of the explicitly dispatched one (one tile pair per CTA)."""
    w = gen.get_workload(6)
    L = build_layer(w, T_max=8)
    try:
        assert L.launches(1) == 3
        rel, ties = compare_layer(w, L, gen.x_tokens(w))
        print(f"decode mxfp4 (H 4096, I 2048, E 256, k 6): rel-L2 {rel:.2e}, near ties {ties}")
        rel8, _ = compare_layer(w, L, gen.x_tokens(w, 8))
        print(f"the same, 8 tokens: rel-L2 {rel8:.2e}")
        x_np = gen.x_tokens(w, 3, first=5)
        a = run_gpu(L, x_np, w)
        out = torch.empty((3, w.H), device="cuda")
        L.forward_routed(to_dev_bf16(x_np), torch.from_numpy(a["idx"]).cuda(),
                         torch.from_numpy(a["gates"]).cuda(), out)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), a["out"])
    finally:
        L.close()


def test_deepseek_shape_mxfp4_prefill_sampled():
    """T = 4096 over 256 experts (96 tokens per expert): the tcgen05 grouped
    GEMMs on MXFP4 weights packed as e4m3 powers of two."""
    w = gen.get_workload(7)
    L = build_layer(w, T_max=w.T)
    try:
        # tc router, top-k, dispatch (count, scan + place: T*k > 8192), row gather (with the x
        # conversion), tc gate/up, tc down, combine
        assert L.launches(w.T) == 8
        sample = [0, 1, 100, 2047, 2048, 4095]
        rel, ties = compare_layer(w, L, gen.x_tokens(w), sample=sample, route_all=True)
        print(f"prefill mxfp4 T=4096 (sampled): rel-L2 {rel:.2e}, near ties {ties}")
    finally:
        L.close()


# ---------------------------------------------------------------- properties
def test_deterministic_and_batch_invariant():
    w = gen.get_workload(1)
    L = layer(w)
    x8 = gen.x_tokens(w, 8)
    a = run_gpu(L, x8, w, want_routing=False)["out"]
    b = run_gpu(L, x8, w, want_routing=False)["out"]
    assert np.array_equal(a, b), "two runs differ"
    for t in (0, 3, 7):
        one = run_gpu(L, x8[t:t + 1], w, want_routing=False)["out"]
        assert np.array_equal(one[0], a[t]), f"token {t} alone differs from its batch of 8"


def test_zero_gates_and_linearity_with_given_routing():
    w = small(shared=0, T=9)
    L = layer(w)
    x = to_dev_bf16(gen.x_tokens(w, 9))
    rng = np.random.default_rng(5)
    idx_np = np.stack([rng.choice(w.E, w.k, replace=False) for _ in range(9)]).astype(np.int32)
    idx = torch.from_numpy(idx_np).cuda()
    out = torch.full((9, w.H), float("nan"), device="cuda")
    L.forward_routed(x, idx, torch.zeros((9, w.k), device="cuda"), out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)
    g1 = torch.rand((9, w.k), device="cuda")
    g2 = torch.rand((9, w.k), device="cuda")
    o1, o2, o12 = (torch.empty((9, w.H), device="cuda") for _ in range(3))
    L.forward_routed(x, idx, g1, o1)
    L.forward_routed(x, idx, g2, o2)
    L.forward_routed(x, idx, g1 + g2, o12)
    torch.cuda.synchronize()
    assert torch.allclose(o12, o1 + o2, rtol=1e-5, atol=1e-7)
    # and against the oracle with the same given routing
    ol = oracle.layer_for_workload(w, sorted(set(idx_np.ravel().tolist())))
    ref = ol.combine(gen.x_tokens(w, 9), idx_np, g1.cpu().numpy())
    got = o1.cpu().numpy()
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert np.all(rel <= 2e-3)


def test_forward_host_matches_device_forward():
    """The host-buffer call gives the device forward's bits: pinned buffers
    (read and written by the kernels in place) with new contents, another
    token count, other buffers, both router modes; and pageable buffers (the
    staged copies)."""
    w = dataclasses.replace(gen.get_workload(0), bias="normal", bias_scale=0.1, seed=11)
    L = build_layer(w, T_max=16)
    try:
        xh = torch.empty((16, w.H), dtype=torch.int16).pin_memory()
        oh = torch.empty((16, w.H), dtype=torch.float32).pin_memory()
        for T, first, mode in [(4, 0, 0), (4, 4, 0), (13, 0, 0), (13, 3, 1), (4, 8, 1)]:
            L.set_router_mode(mode)
            x_np = gen.x_tokens(w, T, first=first)
            dev = run_gpu(L, x_np, w, want_routing=False)["out"]
            xh[:T].copy_(torch.from_numpy(x_np.view(np.int16)))
            L.forward_host(xh, oh[:T], T=T)
            assert np.array_equal(oh[:T].numpy(), dev), (T, first, mode)
        other = torch.from_numpy(gen.x_tokens(w, 4, first=2).view(np.int16)).pin_memory()
        o2 = torch.empty((4, w.H), dtype=torch.float32).pin_memory()
        L.forward_host(other, o2)
        dev = run_gpu(L, gen.x_tokens(w, 4, first=2), w, want_routing=False)["out"]
        assert np.array_equal(o2.numpy(), dev)
        xp = np.ascontiguousarray(gen.x_tokens(w, 5, first=1)).view(np.int16)  # pageable
        op = np.zeros((5, w.H), np.float32)
        L.forward_host(xp, op)
        dev = run_gpu(L, gen.x_tokens(w, 5, first=1), w, want_routing=False)["out"]
        assert np.array_equal(op, dev)
    finally:
        L.close()


def test_error_paths():
    w = gen.get_workload(0)
    L = moe.MoeLayer(w.fmt, w.H, w.I, w.E, w.k, w.shared)
    x = to_dev_bf16(gen.x_tokens(w))
    out = torch.empty((w.T, w.H), device="cuda")
    with pytest.raises(moe.MoeError) as e:
        L.forward(x, out)  # no workspace yet
    assert e.value.code == moe.ESTATE
    L.reserve(2)
    with pytest.raises(moe.MoeError) as e:
        L.forward(x, out)  # router not set
    assert e.value.code == moe.ESTATE
    L.set_router(gen.router_weights(w))
    with pytest.raises(moe.MoeError) as e:
        L.forward(x, out)  # T = 4 > T_max = 2
    assert e.value.code == moe.ESTATE and "T_max" in str(e.value)
    with pytest.raises(moe.MoeError) as e:
        moe.check(moe.lib().moe_forward(L.h, x.data_ptr() + 2, 1, out.data_ptr(), None))
    assert e.value.code == moe.EINVAL
    bad = torch.full((1, w.k), 99, dtype=torch.int32, device="cuda")
    L.forward_routed(x[:1], bad, torch.ones((1, w.k), device="cuda"), out[:1])
    assert L.status(reset=True) == moe.EINVAL  # the device bounds check caught the expert id
    assert L.status() == 0
    L.close()


# ---------------------------------------------------------------- top-k: exact ties
def _tie_biases(case, E, rng):
    b = rng.uniform(-1.0, 0.9, E).astype(np.float32)
    if case == "all_equal":          # every logit equal: the picks are experts 0..k-1
        b[:] = 0.5
    elif case == "tied_group":       # 20 experts tied at the top: their 10 lowest ids
        b[rng.choice(E, 20, replace=False)] = 1.0
    elif case == "straddle":         # 8 clear winners, then 5 tied for the last 2 places
        ids = rng.choice(E, 13, replace=False)
        b[ids[:8]] = np.linspace(2.0, 1.3, 8, dtype=np.float32)
        b[ids[8:]] = 1.0
    elif case == "one_share":        # the whole top 10 inside one 64-expert share
        b[64:74] = np.linspace(3.0, 2.1, 10, dtype=np.float32)
    elif case == "negative":         # all negative, ties among the best
        b = -np.abs(b) - 0.25
        b[rng.choice(E, 12, replace=False)] = -0.125
    return b


TIE_CASES = ["all_equal", "tied_group", "straddle", "one_share", "negative", "signed_zero"]


def _tie_bias(case, E, k, rng):
    if case == "signed_zero":  # +0 and -0 tied for the last places, the rest below
        b = -rng.uniform(0.5, 1.0, E).astype(np.float32)
        ids = rng.choice(E, k + 4, replace=False)
        b[ids[: k - 2]] = np.linspace(2.0, 1.0, k - 2, dtype=np.float32)
        b[ids[k - 2:]] = np.array([0.0, -0.0, -0.0, 0.0, -0.0, 0.0], np.float32)
        return b
    return _tie_biases(case, E, rng)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("T,E", [(1, 512), (13, 512), (64, 512), (300, 512), (1100, 128)])
@pytest.mark.parametrize("case", TIE_CASES)
def test_topk_exact_ties_every_path(case, T, E, mode):
    """Exact ties at and around the k-th pick on every routing path: T = 1 in
    the gate/up CTAs, T = 13 in the dispatch CTA, T = 64 and 300 in the top-k
    kernel, T = 1100 after the tensor-core router (128 experts; several-CTA
    dispatch), for the softmax and the sigmoid router.  Zero router weights
    make every logit the bias exactly (the sigmoid router's keys are then
    sigmoid(0) + bias); +0 and -0 compare equal.  Picks, order and gates equal
    the oracle's."""
    k = 10
    w = small(fmt=1, H=256, I=128, E=E, k=k, shared=1, T=T, seed=11)
    L = layer(w, T_max=1100)
    rng = np.random.default_rng(1000 * TIE_CASES.index(case) + T)
    bias = _tie_bias(case, E, k, rng)
    zeros = np.zeros((E, w.H), np.uint16)
    L.set_router(zeros, bias)
    L.set_router_mode(mode)
    try:
        a = run_gpu(L, gen.x_tokens(w, T), w)
        if mode == 0:
            np.testing.assert_array_equal(a["logits"], np.broadcast_to(bias + np.float32(0), (T, E)))
            ol = oracle.Layer(w.fmt, w.H, w.I, w.E, w.k, w.shared, zeros, bias)
            idx, gates = ol.topk(np.broadcast_to(bias + np.float32(0), (T, E)).copy())
        else:
            np.testing.assert_array_equal(a["logits"], np.zeros((T, E), np.float32))
            idx, gates = oracle.topk_gates_sigmoid(np.zeros((T, E), np.float32), bias, k)
        np.testing.assert_array_equal(a["idx"], idx)
        np.testing.assert_allclose(a["gates"], gates, rtol=1e-6, atol=0)
        assert L.status() == 0
    finally:
        L.set_router_mode(0)
        L.set_router(gen.router_weights(w), gen.router_bias(w))


# ---------------------------------------------------------------- sigmoid router with selection bias
@pytest.mark.parametrize("T", [1, 5, 13, 64, 200, 1100])
def test_sigmoid_router_layer(T):
    """The sigmoid router (scores sigmoid(x . Wr_e), top-k by score + bias,
    gates = the picked scores renormalised) on every routing path: T = 1 in
    the gate/up CTAs, T <= 16 in the dispatch kernel, the top-k kernel, and
    the tensor-core router (T = 1100, 128 experts)."""
    E = 128 if T == 1100 else 64
    w = small(fmt=1, H=256, I=128, E=E, k=6, shared=1, T=T, seed=13)
    L = build_layer(w, T_max=T)
    try:
        L.set_router_mode(moe.ROUTER_SIGMOID)
        x_np = gen.x_tokens(w, T)
        g = run_gpu(L, x_np, w)
        router, bias = gen.router_weights(w), gen.router_bias(w)
        base = oracle.Layer(w.fmt, w.H, w.I, w.E, w.k, w.shared, router, None)
        lg = base.logits(x_np)  # without the bias
        assert np.allclose(g["logits"], lg, rtol=1e-5, atol=1e-5)
        idx_o, gates_o = oracle.topk_gates_sigmoid(lg, bias, w.k)
        # Where the GPU's picks differ from the oracle's, they must be a valid
        # top-k of score + bias up to the rounding of the scores: the GPU's
        # fp32 logit is within `bound` of the oracle's, the fp32 sigmoid moves
        # it by at most a quarter of that plus its own rounding, and adding the
        # bias rounds once more.
        bound_l = logit_bound(x_np, router, None)
        s = 1.0 / (1.0 + np.exp(-lg.astype(np.float64)))
        key = s + bias.astype(np.float64)
        kb = 0.25 * bound_l + 4 * 2.0 ** -24 * (np.abs(key) + 1.0)
        near = 0
        for t in range(T):
            if not np.array_equal(g["idx"][t], idx_o[t]):
                assert valid_near_tie(key[t], kb[t], g["idx"][t], idx_o[t]), \
                    f"token {t}: {g['idx'][t]} vs {idx_o[t]}"
                near += 1
            # gates: the oracle's scores of the GPU's own picks, renormalised
            sg = s[t, g["idx"][t]]
            assert np.allclose(g["gates"][t], sg / sg.sum(), rtol=0, atol=2e-6), t
        print(f"sigmoid router T={T}: {near} near-tie tokens")
        ol = oracle.layer_for_workload(w, sorted(set(g["idx"].ravel().tolist()) | {w.E}))
        ref = ol.combine(x_np, g["idx"], g["gates"])
        rel = np.linalg.norm(g["out"] - ref, axis=1) / np.linalg.norm(ref, axis=1)
        assert np.all(rel <= 2e-3), rel.max()
    finally:
        L.close()
