"""GPU: the W4A4 forward (moe_set_act_format(MOE_ACT_NVFP4)) against the
oracle's act_fp4 contract: x of every token and a of every (token, expert)
row quantised to NVFP4 per row with the weights' recipe before their products.

  * the activation quantiser (moe_quantize_act_nvfp4) gives the oracle's
    quantiser's codes, scales and tensor scale for every row, bit for bit
    (bf16 rows of x, fp32 rows with ties, zero rows and one huge value);
  * the layer on every path (decode T <= 8 with the self-routed and fused
    kernels, the top-k inside the dispatch CTA, the streamed GEMVs, the
    tensor-core GEMMs and router, a full-size decode and prefill) within the
    2e-3 relative L2 bar of the oracle evaluated with act_fp4;
  * x beyond f16's range is fine in this mode (no MOE_ERANGE);
  * switching back to MOE_ACT_BF16 gives the W4A16 bits again.
The routing does not change (the router keeps bf16 x): compare_layer checks
it against the oracle as for W4A16."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_moe_expert_layer_gb300 as moe
from quantized_moe_expert_layer_gb300.synthetic import build_layer

from parity import compare_layer, f32_to_bf16, run_gpu, to_dev_bf16

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


def small(fmt=1, H=256, I=128, E=8, k=2, shared=1, T=13, bias="normal", seed=3):
    return gen.Workload(f"small-{fmt}-{H}-{I}-{E}-{k}-{shared}", H, I, E, k, shared, T, fmt, bias,
                        0.0, 0.1, seed)


def layer(w, T_max):
    key = (w.H, w.I, w.E, w.k, w.shared, w.fmt, w.seed)
    if key not in _layers:
        _layers[key] = build_layer(w, T_max=T_max)
    return _layers[key]


# ---------------------------------------------------------------- the quantiser
def _gpu_quant_rows(A):
    rows, K = A.shape
    codes = torch.empty(rows * K // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows * K // 16, dtype=torch.uint8, device="cuda")
    ts = torch.empty(rows, dtype=torch.float32, device="cuda")
    moe.quantize_act_nvfp4(A, codes, scales, ts)
    torch.cuda.synchronize()
    return (codes.cpu().numpy().reshape(rows, K // 2), scales.cpu().numpy().reshape(rows, K // 16),
            ts.cpu().numpy())


@pytest.mark.parametrize("K", [256, 2048, 6144])
def test_activation_quantiser_bit_exact_bf16_rows(K):
    w = small(H=K)
    x = gen.x_tokens(w, 37)
    x[3] = 0  # an all-zero row: tensor scale 0, codes 0
    c, s, ts = _gpu_quant_rows(to_dev_bf16(x))
    xf = gen.bf16_to_f32(x)
    for r in range(x.shape[0]):
        oc, osc, ots = oracle.quantize_nvfp4(xf[r:r + 1])
        assert np.array_equal(c[r], oc[0]) and np.array_equal(s[r], osc[0]), r
        assert np.float32(ts[r]).tobytes() == np.float32(ots).tobytes(), r


def test_activation_quantiser_bit_exact_fp32_rows():
    rng = np.random.default_rng(4)
    A = (rng.standard_normal((24, 512)) * 3).astype(np.float32)
    A[1] = 0.0
    A[2, :16] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2, np.float32) * 2.0 ** -4
    A[2, 16] = np.float32(6 * 448 * 2.0 ** -4)  # tensor scale 2^-4: the e2m1 midpoints are exact
    A[3, 5] = np.float32(1e30)                  # one huge value: the rest of the row underflows
    A[4, :] = np.float32(1e-38)                 # subnormal scales
    c, s, ts = _gpu_quant_rows(torch.from_numpy(A).cuda())
    for r in range(A.shape[0]):
        oc, osc, ots = oracle.quantize_nvfp4(A[r:r + 1])
        assert np.array_equal(c[r], oc[0]) and np.array_equal(s[r], osc[0]), r
        assert np.float32(ts[r]).tobytes() == np.float32(ots).tobytes(), r


# ---------------------------------------------------------------- the layer
@pytest.mark.parametrize("T", [1, 4, 13, 40, 64, 300])
def test_w4a4_layer_every_path(T):
    """T = 1 and 4: decode (self-routed gate/up, fused down + combine); 13:
    top-k in the dispatch CTA; 40: streamed GEMVs; 64 and 300 (T k >= 16 E):
    the block-scaled FP4 tensor-core GEMMs (kind::mxf4nvf4)."""
    w = small(fmt=1, H=256, I=128, E=8, k=2, T=T, seed=5)
    L = layer(w, T_max=300)
    L.set_act_format(moe.ACT_NVFP4)
    try:
        want = {1: moe.PATH_DECODE, 4: moe.PATH_DECODE, 13: moe.PATH_STREAM, 40: moe.PATH_STREAM,
                64: moe.PATH_TC_FP4, 300: moe.PATH_TC_FP4}[T]
        assert L.path(T) == want
        n16 = L.launches(T)
        rel, ties = compare_layer(w, L, gen.x_tokens(w, T), act_fp4=True)
        assert L.status() == 0 and L.check_workspace() == 0
        print(f"W4A4 T={T}: rel-L2 {rel:.2e} ({n16} launches)")
    finally:
        L.set_act_format(moe.ACT_BF16)


@pytest.mark.parametrize("T", [1100])
def test_w4a4_tensor_core_router(T):
    w = small(fmt=1, H=256, I=128, E=128, k=2, T=T, seed=7)
    L = build_layer(w, T_max=T)
    try:
        L.set_act_format(moe.ACT_NVFP4)
        rel, _ = compare_layer(w, L, gen.x_tokens(w, T), sample=list(range(0, T, 37)), act_fp4=True)
        assert L.status() == 0
    finally:
        L.close()


def test_w4a4_fp6_and_mxfp4_weights():
    for fmt, H, I in [(2, 384, 256), (3, 320, 192)]:
        w = small(fmt=fmt, H=H, I=I, E=24, k=3, T=13)
        L = build_layer(w, T_max=64)
        try:
            L.set_act_format(moe.ACT_NVFP4)
            for T in (3, 13, 64):
                compare_layer(w, L, gen.x_tokens(w, T), act_fp4=True)
            assert L.status() == 0
        finally:
            L.close()


def test_w4a4_x_beyond_f16_range():
    """The quantised activations stay within f16 and the tensor scales stay
    fp32, so an x element of 70000 needs no f16 copy of itself."""
    w = small(fmt=1, H=256, I=128, E=8, k=2, T=13, seed=5)
    L = layer(w, T_max=300)
    L.set_act_format(moe.ACT_NVFP4)
    try:
        xf = gen.bf16_to_f32(gen.x_tokens(w, 13)).copy()
        xf[4, 9] = 70000.0
        compare_layer(w, L, f32_to_bf16(xf), act_fp4=True)
        assert L.status() == 0
    finally:
        L.set_act_format(moe.ACT_BF16)


def test_switching_back_restores_w4a16_bits():
    w = small(fmt=1, H=256, I=128, E=8, k=2, T=13, seed=5)
    L = layer(w, T_max=300)
    x = gen.x_tokens(w, 13)
    a = run_gpu(L, x, w, want_routing=False)["out"]
    L.set_act_format(moe.ACT_NVFP4)
    b = run_gpu(L, x, w, want_routing=False)["out"]
    L.set_act_format(moe.ACT_BF16)
    c = run_gpu(L, x, w, want_routing=False)["out"]
    assert np.array_equal(a, c) and not np.array_equal(a, b)


def test_w4a4_decode_full_size():
    w = gen.get_workload(1)
    L = build_layer(w, T_max=8)
    try:
        L.set_act_format(moe.ACT_NVFP4)
        rel, ties = compare_layer(w, L, gen.x_tokens(w), act_fp4=True)
        rel8, _ = compare_layer(w, L, gen.x_tokens(w, 8), act_fp4=True)
        print(f"W4A4 decode: rel-L2 {rel:.2e}, 8 tokens {rel8:.2e}")
    finally:
        L.close()


def test_w4a4_prefill_full_size_sampled():
    w = gen.get_workload(4)
    L = build_layer(w, T_max=w.T)
    try:
        assert L.path(w.T) == moe.PATH_TC_F16
        L.set_act_format(moe.ACT_NVFP4)
        assert L.path(w.T) == moe.PATH_TC_FP4
        sample = [0, 1, 7, 8, 511, 1024, 2047, 2048, 3000, 4093, 4094, 4095]
        rel, ties = compare_layer(w, L, gen.x_tokens(w), sample=sample, act_fp4=True)
        assert L.status() == 0
        print(f"W4A4 prefill (sampled): rel-L2 {rel:.2e}")
    finally:
        L.close()


@pytest.mark.parametrize("H,I,E,T", [(256, 128, 8, 300), (512, 256, 16, 600), (384, 192, 24, 700)])
def test_block_scaled_gemms_ragged_shapes(H, I, E, T):
    """The FP4 GEMMs on shapes whose K is not a multiple of a 256-column stage
    (I = 192: a down stage of 3 K-steps; H = 384) and with items of every
    token count: against the act_fp4 oracle, bit-identical over repeats,
    every output element written."""
    w = small(fmt=1, H=H, I=I, E=E, k=3, T=T, seed=11)
    L = build_layer(w, T_max=T)
    try:
        L.set_act_format(moe.ACT_NVFP4)
        assert L.path(T) == moe.PATH_TC_FP4
        x = gen.x_tokens(w, T)
        compare_layer(w, L, x, sample=list(range(0, T, 5)), act_fp4=True)
        a = run_gpu(L, x, w, want_routing=False)["out"]
        b = run_gpu(L, x, w, want_routing=False)["out"]
        assert np.array_equal(a, b)
        assert L.status() == 0 and L.check_workspace() == 0
    finally:
        L.close()


def test_block_scaled_gemms_follow_a_repack():
    """Packing new weights into the layer after W4A4 is on rebuilds the MMA
    layout before the next forward."""
    w = small(fmt=1, H=256, I=128, E=8, k=2, T=300, seed=5)
    L = build_layer(w, T_max=300)
    try:
        L.set_act_format(moe.ACT_NVFP4)
        x = gen.x_tokens(w, 300)
        compare_layer(w, L, x, sample=list(range(0, 300, 7)), act_fp4=True)
        w2 = small(fmt=1, H=256, I=128, E=8, k=2, T=300, seed=6)  # other expert weights
        ol = oracle.layer_for_workload(w2, list(range(w2.n_experts_total)))
        for e in range(w2.n_experts_total):
            for m in range(3):
                c, sc, ts = ol.mats[(e, m)]
                L.pack_matrix(e, m, c, sc, ts)
        # (the router stays w's: the oracle routes with it and combines w2's experts)
        compare_layer(w, L, x, sample=list(range(0, 300, 7)), orc_layer=ol, act_fp4=True)
    finally:
        L.close()
