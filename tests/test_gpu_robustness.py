"""GPU: the layer's failure handling, driven from the host without faulting
the GPU.

  * allocation failure: moe_debug_fail_alloc makes the n-th allocation of the
    library fail, so every MOE_ENOMEM path (creation, workspace, staging of a
    host pack, placement) runs on a GPU with memory to spare; each leaves the
    layer usable or cleanly destroyed;
  * bounded waits: a tiny wait budget makes the tensor-core kernels' waits run
    out; the kernels drain their copies and MMAs, free their tensor memory and
    record MOE_ETIMEOUT, and a forward with the default budget is then correct;
  * workspace guard regions: no kernel of any path writes past its buffers;
  * value range: an element of x, or of the SwiGLU output a, beyond f16's
    range records MOE_ERANGE in the status word on every path.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_moe_expert_layer_gb300 as moe
from quantized_moe_expert_layer_gb300.synthetic import build_layer

from parity import compare_layer, f32_to_bf16, run_gpu, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    gen.build(device=True)
    moe.build()
    yield
    moe.fail_alloc(0)


def small(fmt=1, H=256, I=128, E=8, k=2, shared=1, T=13, bias="normal", seed=3):
    return gen.Workload(f"small-{fmt}-{H}-{I}-{E}-{k}-{shared}", H, I, E, k, shared, T, fmt, bias,
                        0.0, 0.1, seed)


# ---------------------------------------------------------------- allocation failures
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_create_fails_cleanly_at_each_allocation(n):
    """moe_layer_create makes five device allocations; failing any of them
    returns MOE_ENOMEM with the size in the message, leaves no handle and
    nothing allocated, and the next create succeeds."""
    w = gen.get_workload(1)  # the decode shape: a 908 MB arena, so a leak would show
    for rep in range(4):
        if rep == 1:
            torch.cuda.synchronize()
            before = torch.cuda.mem_get_info()[0]
        moe.fail_alloc(n)
        with pytest.raises(moe.MoeError) as e:
            moe.MoeLayer(w.fmt, w.H, w.I, w.E, w.k, w.shared)
        assert e.value.code == moe.ENOMEM and "allocation failed" in str(e.value)
    moe.fail_alloc(0)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= before - (64 << 20)  # nothing leaked
    L = moe.MoeLayer(w.fmt, w.H, w.I, w.E, w.k, w.shared)
    L.close()


def test_reserve_pack_and_place_fail_without_breaking_the_layer():
    w = gen.get_workload(0)
    L = build_layer(w, T_max=4)
    try:
        x_np = gen.x_tokens(w)
        ref = run_gpu(L, x_np, w, want_routing=False)["out"]
        # growing the workspace fails: the old one stays and still serves T <= 4
        moe.fail_alloc(1)
        with pytest.raises(moe.MoeError) as e:
            L.reserve(64)
        assert e.value.code == moe.ENOMEM
        assert np.array_equal(run_gpu(L, x_np, w, want_routing=False)["out"], ref)
        # a host pack needs a staging buffer: its failure leaves the packed weights alone
        ol = oracle.layer_for_workload(w, [0])
        c, s, ts = ol.mats[(0, 0)]
        moe.fail_alloc(1)
        with pytest.raises(moe.MoeError) as e:
            L.pack_matrix(0, 0, c, s, ts)
        assert e.value.code == moe.ENOMEM
        assert np.array_equal(run_gpu(L, x_np, w, want_routing=False)["out"], ref)
        # placement: the HBM slots, the pinned mirror, or the address table fails
        mask = np.array([e % 2 == 0 for e in range(w.n_experts_total)])
        for n in (1, 2, 3):
            moe.fail_alloc(n)
            with pytest.raises(moe.MoeError) as e:
                L.place_experts(mask)
            assert e.value.code == moe.ENOMEM
            in_hbm, _, host = L.placement()
            assert in_hbm.all() and host == 0  # the old placement stays
        moe.fail_alloc(0)
        assert np.array_equal(run_gpu(L, x_np, w, want_routing=False)["out"], ref)
        L.reserve(64)  # and the workspace grows once memory is there
        assert np.array_equal(run_gpu(L, x_np, w, want_routing=False)["out"], ref)
        assert L.status() == 0 and L.check_workspace() == 0
    finally:
        moe.fail_alloc(0)
        L.close()


def test_host_forward_before_reserve_is_a_state_error():
    w = gen.get_workload(0)
    L = moe.MoeLayer(w.fmt, w.H, w.I, w.E, w.k, w.shared)
    try:
        xh = np.zeros((w.T, w.H), np.int16)
        oh = np.zeros((w.T, w.H), np.float32)
        with pytest.raises(moe.MoeError) as e:
            L.forward_host(xh, oh)
        assert e.value.code == moe.ESTATE and "reserve" in str(e.value)
        with pytest.raises(moe.MoeError) as e:
            L.check_workspace()
        assert e.value.code == moe.ESTATE
    finally:
        L.close()


# ---------------------------------------------------------------- bounded waits
@pytest.mark.parametrize("T", [128, 1100])
def test_tiny_wait_budget_times_out_and_the_layer_recovers(T):
    """With a wait budget of a few cycles the tensor-core kernels give up:
    MOE_ETIMEOUT in the status word, no fault, tensor memory freed (later
    launches allocate it again).  With the default budget the next forward
    matches the oracle and the guard regions are intact."""
    E = 128 if T == 1100 else 8  # T = 1100 also runs the tensor-core router
    w = small(fmt=1, H=256, I=128, E=E, k=2, T=T, seed=5)
    L = build_layer(w, T_max=T)
    try:
        x_np = gen.x_tokens(w, T)
        L.set_wait_budget(1)
        for _ in range(3):
            run_gpu(L, x_np, w, want_routing=False)
            assert L.status(reset=True) == moe.ETIMEOUT
        L.set_wait_budget(0)
        compare_layer(w, L, x_np)
        assert L.status() == 0
        assert L.check_workspace() == 0
    finally:
        L.close()


# ---------------------------------------------------------------- workspace guard regions
@pytest.mark.parametrize("T,E", [(1, 64), (5, 24), (13, 24), (64, 24), (300, 24), (2731, 24),
                                 (1100, 128)])
def test_no_kernel_writes_past_its_workspace_buffers(T, E):
    """Every path (decode T <= 8, top-k in the dispatch CTA, the top-k kernel,
    the tensor-core GEMMs, the several-CTA dispatch, the tensor-core router)
    and the given-routing forward leave the guard regions between the
    workspace buffers untouched."""
    w = small(fmt=1, H=256, I=128, E=E, k=3, T=T, seed=9)
    L = build_layer(w, T_max=T)
    try:
        assert L.check_workspace() == 0
        g = run_gpu(L, gen.x_tokens(w, T), w)
        assert L.check_workspace() == 0
        out = torch.empty((T, w.H), device="cuda")
        L.forward_routed(to_dev_bf16(gen.x_tokens(w, T)), torch.from_numpy(g["idx"]).cuda(),
                         torch.from_numpy(g["gates"]).cuda(), out)
        assert L.check_workspace() == 0
        assert L.status() == 0
    finally:
        L.close()


# ---------------------------------------------------------------- value range
@pytest.mark.parametrize("T", [1, 13, 300])
def test_values_beyond_f16_range_are_flagged(T):
    """x has bf16's range but the experts multiply f16 copies: an element of x
    above 65504, or an a = silu(g) u above it, records MOE_ERANGE (decode,
    small-batch and tensor-core paths, and the given-routing forward); inputs
    inside the range record nothing."""
    w = small(fmt=1, H=256, I=128, E=8, k=2, T=T, seed=5)
    L = build_layer(w, T_max=T)
    try:
        x_np = gen.x_tokens(w, T)
        run_gpu(L, x_np, w, want_routing=False)
        assert L.status() == 0
        xf = gen.bf16_to_f32(x_np).copy()
        big = xf.copy()
        big[T // 2, 7] = 70000.0          # beyond 65504: x itself does not fit f16
        run_gpu(L, f32_to_bf16(big), w, want_routing=False)
        assert L.status(reset=True) == moe.ERANGE
        loud = xf * np.float32(6000.0)    # |x| < 65504, but a = silu(g) u ~ |x|^2 overflows
        assert np.abs(loud).max() < 65504
        x_loud = f32_to_bf16(loud)
        run_gpu(L, x_loud, w, want_routing=False)
        assert L.status(reset=True) == moe.ERANGE
        idx = torch.zeros((T, w.k), dtype=torch.int32, device="cuda")
        idx[:, 1] = 1
        out = torch.empty((T, w.H), device="cuda")
        L.forward_routed(to_dev_bf16(f32_to_bf16(big)), idx,
                         torch.full((T, w.k), 0.5, device="cuda"), out)
        assert L.status(reset=True) == moe.ERANGE
        run_gpu(L, x_np, w, want_routing=False)
        assert L.status() == 0
    finally:
        L.close()
