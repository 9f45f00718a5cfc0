"""GPU: moe_route_noalloc, the routing entry point for callers that may not
allocate device memory (code whose GPU memory belongs to a serving runtime's
own pre-planned pool), against the routing moe_forward computes on the same
inputs, on two calls in a row.  Its scratch is a fixed array inside the
library, so the second call must not depend on what the first left there.

This file is collected last on purpose: it needs nothing from the other tests
and passes alone in a fresh process as well as after them."""
import numpy as np
import pytest
import torch

import gen
import quantized_moe_expert_layer_gb300 as moe
from quantized_moe_expert_layer_gb300.synthetic import build_layer

from parity import to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    gen.build(device=True)
    moe.build()


@pytest.mark.parametrize("widx", [0, 1, 3])  # T=4 E=8; T=1 E=512 (4-way K-split); T=64 E=512
def test_route_noalloc_matches_forward_routing(widx):
    w = gen.get_workload(widx)
    T = w.T
    L = build_layer(w, experts=[])  # routing does not depend on the expert weights
    x = to_dev_bf16(gen.x_tokens(w))
    out = torch.empty((T, w.H), device="cuda")
    L.forward(x, out)
    ref = {"logits": torch.empty((T, w.E), device="cuda"),
           "idx": torch.empty((T, w.k), dtype=torch.int32, device="cuda"),
           "gates": torch.empty((T, w.k), device="cuda")}
    L.debug_routing(**ref)
    torch.cuda.synchronize()
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    L.close()

    wr = torch.from_numpy(gen.router_weights(w).view(np.int16)).cuda()
    b = gen.router_bias(w)
    bias = None if b is None else torch.from_numpy(b).cuda()
    for call in range(2):
        logits = torch.full((T, w.E), float("nan"), device="cuda")
        idx = torch.full((T, w.k), -1, dtype=torch.int32, device="cuda")
        gates = torch.full((T, w.k), float("nan"), device="cuda")
        moe.route_noalloc(x, wr, bias, w.E, w.k, logits, idx, gates)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ref["idx"]), f"call {call}: top-k differs"
        assert np.allclose(gates.cpu().numpy(), ref["gates"], rtol=0, atol=2e-5), f"call {call}"
        assert np.allclose(logits.cpu().numpy(), ref["logits"], rtol=1e-6, atol=1e-6), f"call {call}"


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    H, E, k, T = 2048, 1024, 8, 2048  # one K slice: T * E = 2^21 floats > 2^20
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, E), device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.route_noalloc(x, wr, None, E, k, out, idx, out)
    assert e.value.code == moe.EINVAL and "scratch" in str(e.value)
