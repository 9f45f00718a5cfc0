"""GPU: the two-tier expert placement (HBM slots and the pinned host mirror the
kernels read over the CPU-GPU link).  The placement moves bytes, not
arithmetic: a layer gives the same bits whichever tier each expert sits in
(for the token counts whose path does not change with it), and matches the
oracle either way."""
import numpy as np
import pytest
import torch

import gen
import quantized_moe_expert_layer_gb300 as moe
from quantized_moe_expert_layer_gb300.synthetic import build_layer

from parity import compare_layer, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    gen.build(device=True)
    moe.build()


def forward(L, x_np):
    x = to_dev_bf16(x_np)
    out = torch.empty((x_np.shape[0], L.H), device="cuda")
    L.forward(x, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def half_mask(n, seed):
    rng = np.random.default_rng(seed)
    m = rng.random(n) < 0.5
    m[-1] = False  # the shared expert in the host mirror too
    return m


def test_decode_shapes_bit_identical_across_placements():
    """Full decode shape (H=2048, I=512, E=512, k=10 + shared, NVFP4): all in
    HBM, half in the host mirror, all in the mirror, back to HBM; T = 1, 3, 8,
    64 give the same bits each time, and the tiers hold what was asked."""
    w = gen.get_workload(1)
    L = build_layer(w, T_max=64)
    try:
        n = w.n_experts_total
        _, eb = L.info()
        xs = {T: gen.x_tokens(w, T) for T in (1, 3, 8, 64)}
        ref = {T: forward(L, x) for T, x in xs.items()}
        for mask in (half_mask(n, 1), np.zeros(n, bool), np.ones(n, bool)):
            L.place_experts(mask)
            got, hbm, host = L.placement()
            assert np.array_equal(got, mask)
            assert hbm == int(mask.sum()) * eb and host == int((~mask).sum()) * eb
            for T, x in xs.items():
                assert np.array_equal(forward(L, x), ref[T]), f"T={T}, {int(mask.sum())} in HBM"
        assert L.status() == 0
    finally:
        L.close()


def test_packed_into_the_mirror_matches_the_oracle():
    """Experts packed straight into the host mirror (placement before packing):
    the decode output against the oracle, and the same bits as the all-HBM
    layer."""
    w = gen.get_workload(1)
    mask = half_mask(w.n_experts_total, 2)
    L = build_layer(w, T_max=8, in_hbm=mask)
    ref = build_layer(w, T_max=8)
    try:
        assert np.array_equal(L.placement()[0], mask)
        x = gen.x_tokens(w, 8)
        assert np.array_equal(forward(L, x), forward(ref, x))
        rel, ties = compare_layer(w, L, gen.x_tokens(w))
        print(f"decode, half the experts in the host mirror: rel-L2 {rel:.2e}")
    finally:
        L.close()
        ref.close()


@pytest.mark.parametrize("fmt", [1, 2, 3])
def test_mirror_dequant_bit_exact(fmt):
    """The packed bytes of a host-mirror expert dequantise to the oracle's
    weights exactly, like an HBM one."""
    w = gen.Workload(f"place-{fmt}", 384 if fmt == 2 else 256, 256 if fmt == 2 else 128, 6, 2, 1,
                     5, fmt, "normal", 0.0, 0.1, 4)
    import oracle
    mask = np.array([1, 0, 1, 0, 0, 1, 0], bool)
    L = build_layer(w, T_max=8, in_hbm=mask)
    try:
        orc = oracle.layer_for_workload(w)
        for e in (0, 1, 6):
            for m in range(3):
                rows, K = gen.matrix_shape(w, m)
                out = torch.empty((rows, K), device="cuda")
                L.debug_dequant(e, m, out)
                torch.cuda.synchronize()
                want = orc.dequant(e, m)
                assert np.array_equal(out.cpu().numpy().view(np.uint32),
                                      want.astype(np.float32).view(np.uint32)), (e, m)
    finally:
        L.close()


@pytest.mark.parametrize("fmt", [1, 2, 3])
@pytest.mark.parametrize("T", [1, 13, 300])
def test_small_layer_mirror_against_oracle(fmt, T):
    """A small layer with most experts in the host mirror, in every format, at
    the self-routed decode (1), the streamed small-N path (13) and a token
    count that takes the tensor-core path while every expert is in HBM (300,
    NVFP4 / MXFP4) but the streamed path with any in the mirror; against the
    oracle, then again with every expert back in HBM."""
    H, I = (384, 256) if fmt == 2 else (256, 128)
    w = gen.Workload("place-small", H, I, 8, 2, 1, T, fmt, "normal", 0.0, 0.1, 5)
    mask = np.array([0, 0, 1, 0, 0, 0, 1, 0, 0], bool)
    L = build_layer(w, T_max=T, in_hbm=mask)
    try:
        compare_layer(w, L, gen.x_tokens(w, T))
        L.place_experts(np.ones(w.n_experts_total, bool))
        compare_layer(w, L, gen.x_tokens(w, T))
    finally:
        L.close()


def test_placement_errors():
    w = gen.get_workload(0)
    L = build_layer(w, T_max=4)
    try:
        with pytest.raises(ValueError):
            L.place_experts(np.ones(w.n_experts_total + 1, bool))
        with pytest.raises(moe.MoeError) as e:
            moe.check(moe.lib().moe_place_experts(L.h, None))
        assert e.value.code == moe.EINVAL
        # a failed call leaves the layer usable
        x = gen.x_tokens(w)
        a = forward(L, x)
        L.place_experts(np.zeros(w.n_experts_total, bool))
        assert np.array_equal(forward(L, x), a)
    finally:
        L.close()
