"""GPU: the device quantisers, the packer and the packed decode, bit-exact
against the oracle on the same seeded inputs."""
import dataclasses

import numpy as np
import pytest
import torch

import gen
import oracle
import quantized_moe_expert_layer_gb300 as moe
from quantized_moe_expert_layer_gb300.synthetic import build_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    gen.build(device=True)
    moe.build()


def test_device_generator_matches_host():
    k = gen.key(7, gen.T_WEIGHT, 3, 1)
    n = 1 << 20
    d = torch.empty(n, dtype=torch.float32, device="cuda")
    gen.fill_normal_dev(k, n, 0.02, d.data_ptr(), bf16=False, offset=12345)
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy(), gen.normal_f32(k, n, 0.02, offset=12345))
    b = torch.empty(n, dtype=torch.int16, device="cuda")
    gen.fill_normal_dev(k, n, 1.0, b.data_ptr(), bf16=True)
    torch.cuda.synchronize()
    assert np.array_equal(b.cpu().numpy().view(np.uint16), gen.normal_bf16(k, n, 1.0))


def _tie_matrix_nvfp4():
    """A matrix whose quantisation hits e2m1 and e4m3 rounding ties exactly:
    ts = 2^-10 (tensor amax 2688 * 2^-10); a block with amax 24 * 2^-10 gets
    s = 4, so w / (s ts) = w * 256 and the e2m1 midpoints are exact."""
    W = np.zeros((32, 64), np.float32)
    W[0, 0] = 2688.0 * 2.0 ** -10
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    W[1, :8] = mids * 2.0 ** -8
    W[1, 8:16] = -mids * 2.0 ** -8
    W[2, :16] = np.float32(6 * 4.25 * 2.0 ** -10)      # sv = 4.25: e4m3 tie between 4 and 4.5
    W[3, :16] = np.float32(6 * 4.75 * 2.0 ** -10)      # tie between 4.5 and 5
    W[4, 16:32] = np.float32(1e-9)                      # block scale underflows to 0
    rng = np.random.default_rng(0)
    W[5:] = (rng.standard_normal((27, 64)) * 0.05).astype(np.float32)
    return W


def _gpu_quant_nvfp4(W):
    rows, K = W.shape
    Wd = torch.from_numpy(W).cuda()
    c = torch.empty(rows * K // 2, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows * K // 16, dtype=torch.uint8, device="cuda")
    ts = torch.empty(1, dtype=torch.float32, device="cuda")
    moe.quantize_nvfp4(Wd, c, s, ts)
    torch.cuda.synchronize()
    return c.cpu().numpy().reshape(rows, K // 2), s.cpu().numpy().reshape(rows, K // 16), float(ts.item())


def _gpu_quant_fp6(W):
    rows, K = W.shape
    Wd = torch.from_numpy(W).cuda()
    c = torch.empty(rows * K, dtype=torch.uint8, device="cuda")
    e = torch.empty(rows * K // 128, dtype=torch.uint8, device="cuda")
    moe.quantize_fp6(Wd, c, e)
    torch.cuda.synchronize()
    return c.cpu().numpy().reshape(rows, K), e.cpu().numpy().reshape(rows, K // 128)


@pytest.mark.parametrize("case", ["ties", "random", "workload"])
def test_quantize_nvfp4_bit_exact(case):
    if case == "ties":
        W = _tie_matrix_nvfp4()
    elif case == "random":
        rng = np.random.default_rng(1)
        W = (rng.standard_normal((48, 192)) * np.exp(rng.standard_normal((48, 1)))).astype(np.float32)
        W[7] = 0.0
    else:
        W = gen.expert_weight(gen.get_workload(1), 17, 2)
    c, s, ts = _gpu_quant_nvfp4(W)
    rc, rs, rts = oracle.quantize_nvfp4(W)
    assert ts == rts
    assert np.array_equal(s, rs)
    assert np.array_equal(c, rc)


@pytest.mark.parametrize("case", ["ties", "random", "workload"])
def test_quantize_fp6_bit_exact(case):
    if case == "ties":
        W = np.zeros((16, 256), np.float32)
        grid = np.array([0.0625, 0.1875, 1.9375, 2.125, 3.875, 4.25, 7.25, 7.5], np.float32)
        W[0, :8] = grid * 2.0 ** -6
        W[0, 8:16] = -grid * 2.0 ** -6
        W[1, :128] = np.float32(1e-40)                 # subnormal block
        W[2, 128:] = np.float32(7.5 * 2.0 ** 3)        # amax exactly on 7.5 * 2^E
        W[3, 5] = np.float32(7.5 * 2.0 ** 3 * 1.0000001)
    elif case == "random":
        rng = np.random.default_rng(2)
        W = (rng.standard_normal((32, 384)) * np.exp(2 * rng.standard_normal((32, 1)))).astype(np.float32)
    else:
        W = gen.expert_weight(gen.get_workload(2), 3, 0)[:256]
    c, e = _gpu_quant_fp6(W)
    rc, re_ = oracle.quantize_fp6(W)
    assert np.array_equal(e, re_)
    assert np.array_equal(c, rc)


def _gpu_quant_mxfp4(W):
    rows, K = W.shape
    Wd = torch.from_numpy(W).cuda()
    c = torch.empty(rows * K // 2, dtype=torch.uint8, device="cuda")
    e = torch.empty(rows * K // 32, dtype=torch.uint8, device="cuda")
    moe.quantize_mxfp4(Wd, c, e)
    torch.cuda.synchronize()
    return c.cpu().numpy().reshape(rows, K // 2), e.cpu().numpy().reshape(rows, K // 32)


@pytest.mark.parametrize("case", ["ties", "random", "workload"])
def test_quantize_mxfp4_bit_exact(case):
    if case == "ties":
        W = np.zeros((16, 128), np.float32)
        grid = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 7.99], np.float32)
        W[0, :10] = grid                               # amax 7.99: E = 0, ties and saturation
        W[0, 32:42] = -grid * 2.0 ** -20
        W[1, :32] = np.float32(1e-40)                  # subnormal block
        W[2, 64:96] = np.float32(2.0 ** 100)           # huge, exactly a power of two
        W[3, 96] = np.float32(3e38)
    elif case == "random":
        rng = np.random.default_rng(3)
        W = (rng.standard_normal((32, 256)) * np.exp(3 * rng.standard_normal((32, 1)))).astype(np.float32)
        W[5] = 0.0
    else:
        W = gen.expert_weight(gen.get_workload(6), 3, 0)[:256]
    c, e = _gpu_quant_mxfp4(W)
    rc, re_ = oracle.quantize_mxfp4(W)
    assert np.array_equal(e, re_)
    assert np.array_equal(c, rc)


def test_mxfp4_pack_rejects_exponents_beyond_the_tile_scale_range():
    """The tile layout holds a block scale as an e4m3 power of two within 17
    binades of the matrix's largest one; a wider spread is an error, and so is
    a NaN scale byte."""
    H, I = 128, 64
    L = moe.MoeLayer(moe.FMT_MXFP4, H, I, 2, 1, 0)
    c = np.full((I, H // 2), 0x22, np.uint8)            # every code 1.0
    e = np.full((I, H // 32), 127, np.uint8)
    e[3, 1] = 127 - 17                                  # 17 binades below: fine
    L.pack_matrix(0, 0, c, e)
    e[3, 1] = 127 - 18                                  # 18 binades: rejected
    with pytest.raises(moe.MoeError) as err:
        L.pack_matrix(0, 0, c, e)
    assert err.value.code == moe.EINVAL
    e[3, 1] = 127
    c[3, 16:32] = 0                                     # an all-zero block may have any exponent
    e[3, 1] = 0
    L.pack_matrix(0, 0, c, e)
    e[5, 0] = 255
    with pytest.raises(moe.MoeError):
        L.pack_matrix(0, 0, c, e)
    L.close()


def _dequant_gpu(L, expert, matrix, rows, K):
    out = torch.full((rows, K), float("nan"), device="cuda")
    L.debug_dequant(expert, matrix, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("name,fmt,H,I", [("nvfp4", 1, 256, 128), ("nvfp4-ragged", 1, 320, 192),
                                           ("fp6", 2, 256, 128), ("fp6-ragged", 2, 1152, 384),
                                           ("mxfp4", 3, 256, 128), ("mxfp4-ragged", 3, 320, 192)])
def test_pack_from_host_and_dequant_bit_exact(name, fmt, H, I):
    """Oracle-quantised canonical bytes, packed from the host, decode bit-exactly
    (super-chunks with a partial tail in the ragged shapes)."""
    w = gen.Workload(f"pack-{name}", H, I, 4, 2, 1, 3, fmt, "none", seed=11)
    ol = oracle.layer_for_workload(w)
    L = moe.MoeLayer(fmt, H, I, w.E, w.k, 1)
    for (e, m), (c, s, ts) in ol.mats.items():
        L.pack_matrix(e, m, c, s, ts if fmt == 1 else None)
    for (e, m) in ol.mats:
        rows, K = gen.matrix_shape(w, m)
        got = _dequant_gpu(L, e, m, rows, K)
        assert np.array_equal(got, ol.dequant(e, m)), (e, m)
    L.close()


@pytest.mark.parametrize("widx,experts", [(0, None), (1, [0, 5, 511, 512]), (2, [0, 255, 256]),
                                          (5, None), (6, [0, 255, 256])])
def test_device_built_layer_dequant_bit_exact(widx, experts):
    """The full device pipeline (generator -> device quantiser -> packer) gives
    the weights the oracle's own quantiser gives, bit for bit."""
    w = gen.get_workload(widx)
    ids = list(range(w.n_experts_total)) if experts is None else experts
    L = build_layer(dataclasses.replace(w, T=1), experts=ids)
    ol = oracle.layer_for_workload(w, ids)
    for e in ids:
        for m in range(3):
            rows, K = gen.matrix_shape(w, m)
            assert np.array_equal(_dequant_gpu(L, e, m, rows, K), ol.dequant(e, m)), (e, m)
    arena, per_expert = L.info()
    assert arena == per_expert * w.n_experts_total
    L.close()


@pytest.mark.parametrize("fmt,shared", [(1, 0), (1, 1), (2, 1), (3, 1)])
def test_pack_weights_whole_layer_from_host(fmt, shared):
    """moe_pack_weights: router, bias and every expert's three matrices (the
    shared expert last) packed from host arrays in the canonical format, here
    the oracle's own quantisation.  Every matrix decodes bit-exactly to the
    oracle's dequantisation, and the forward gives the bits of the same layer
    built on the device (device quantiser + per-matrix packer)."""
    H, I = (256, 128)
    w = gen.Workload(f"pack-{fmt}-{shared}", H, I, 8, 2, shared, 5, fmt, "normal", 0.0, 0.1, 21)
    ol = oracle.layer_for_workload(w)
    L = moe.MoeLayer(w.fmt, w.H, w.I, w.E, w.k, w.shared)
    ref = build_layer(w, T_max=w.T)
    try:
        L.reserve(w.T)
        L.pack_weights(gen.router_weights(w), gen.router_bias(w), ol.mats)
        for e in range(w.n_experts_total):
            for m in range(3):
                rows, K = gen.matrix_shape(w, m)
                got = torch.empty((rows, K), dtype=torch.float32, device="cuda")
                L.debug_dequant(e, m, got)
                torch.cuda.synchronize()
                assert np.array_equal(got.cpu().numpy(), ol.dequant(e, m)), (e, m)
        x = torch.from_numpy(gen.x_tokens(w).view(np.int16)).cuda()
        a = torch.full((w.T, w.H), float("nan"), device="cuda")
        b = torch.full((w.T, w.H), float("nan"), device="cuda")
        L.forward(x, a)
        ref.forward(x, b)
        torch.cuda.synchronize()
        assert torch.equal(a, b)
        assert L.status() == 0
    finally:
        L.close()
        ref.close()
