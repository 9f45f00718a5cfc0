"""GPU: moe_route_noalloc, the routing entry point for callers that may not
allocate device memory (code whose GPU memory belongs to a serving runtime's
own pre-planned pool), against the oracle's router and top-k on the same
inputs, on two calls in a row.  Its scratch is a fixed array inside the
library, so the second call must not depend on what the first left there.

This file is collected last on purpose: it needs nothing from the other tests
and passes alone in a fresh process as well as after them."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_moe_expert_layer_gb300 as moe

from parity import check_routing, logit_bound, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    gen.build(device=True)
    moe.build()


@pytest.mark.parametrize("widx", [0, 1, 3])  # T=4 E=8; T=1 E=512 (4-way K-split); T=64 E=512
def test_route_noalloc_matches_the_oracle(widx):
    """Two calls in a row against the oracle's router and top-k on the same
    inputs: logits within the fp32 dot-product bound, top-k indices equal
    (up to near ties, none expected), gates the softmax of the picks."""
    w = gen.get_workload(widx)
    T = w.T
    x_np = gen.x_tokens(w)
    router, b = gen.router_weights(w), gen.router_bias(w)
    base = oracle.Layer(w.fmt, w.H, w.I, w.E, w.k, w.shared, router, b)
    lg_o = base.logits(x_np)
    idx_o, gates_o = base.topk(lg_o)
    bound = logit_bound(x_np, router, b)
    x = to_dev_bf16(x_np)
    wr = torch.from_numpy(router.view(np.int16)).cuda()
    bias = None if b is None else torch.from_numpy(b).cuda()
    for call in range(2):
        logits = torch.full((T, w.E), float("nan"), device="cuda")
        idx = torch.full((T, w.k), -1, dtype=torch.int32, device="cuda")
        gates = torch.full((T, w.k), float("nan"), device="cuda")
        moe.route_noalloc(x, wr, bias, w.E, w.k, logits, idx, gates)
        torch.cuda.synchronize()
        lg, ix, gt = logits.cpu().numpy(), idx.cpu().numpy(), gates.cpu().numpy()
        ties = check_routing(lg, ix, lg_o, idx_o, bound)
        assert not ties, f"call {call}: near ties {ties}"
        assert np.allclose(gt, gates_o, rtol=0, atol=2e-5), f"call {call}: gates"


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    H, E, k, T = 2048, 1024, 8, 2048  # one K slice: T * E = 2^21 floats > 2^20
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, E), device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.route_noalloc(x, wr, None, E, k, out, idx, out)
    assert e.value.code == moe.EINVAL and "scratch" in str(e.value)


@pytest.mark.parametrize("T,H", [(1, 65536 + 64), (524281, 64)])
def test_route_noalloc_rejects_shapes_beyond_its_limits(T, H):
    """H above 65536 (the router's K slices would not cover it) and T whose
    token groups exceed the grid's y limit are rejected before any launch."""
    E, k = 8, 2
    x = torch.zeros(16, dtype=torch.int16, device="cuda")
    out = torch.empty(16, device="cuda")
    idx = torch.empty(16, dtype=torch.int32, device="cuda")
    rc = moe.lib().moe_route_noalloc(x.data_ptr(), T, H, x.data_ptr(), None, E, k, out.data_ptr(),
                                     idx.data_ptr(), out.data_ptr(), None)
    assert rc == moe.EINVAL
