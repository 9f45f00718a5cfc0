"""Helpers shared by the GPU parity tests: run the CUDA layer and the oracle on
the same seeded inputs and compare them.

Tolerances:
  * dequantised weights, quantiser codes / scales, dispatch: bit-exact;
  * top-k indices: exact, except where the oracle's own logits are closer than
    twice the rounding bound of an fp32 dot product (a near tie: either choice
    is a correct routing; the token is then compared with the oracle evaluated
    on the GPU's selection);
  * layer output: relative L2 error per token <= 2e-3 (fp32 accumulation).
"""
from __future__ import annotations

import numpy as np
import torch

import gen
import oracle

REL_L2 = 2e-3


def to_dev_bf16(x_np: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).cuda()


def logit_bound(x_np, wr_np, bias):
    """Per (token, expert) bound on |fp32 logit - exact logit|: any summation
    order of H products is within H * u * sum|x w| (u = 2^-23, allowing
    truncating accumulation), plus the rounding of the bias add."""
    xv = gen.bf16_to_f32(x_np).astype(np.float64)
    wv = gen.bf16_to_f32(wr_np).astype(np.float64)
    H = xv.shape[1]
    s = np.abs(xv) @ np.abs(wv).T
    b = 0.0 if bias is None else np.abs(bias.astype(np.float64))[None, :]
    return H * 2.0 ** -23 * s + 2.0 ** -22 * (s + b)


def gates_for(logits_row, sel):
    v = logits_row[sel].astype(np.float64)
    e = np.exp(v - v.max())
    return (e / e.sum()).astype(np.float32)


def check_routing(lg_gpu, idx_gpu, lg_orc, idx_orc, bound):
    """Returns the tokens whose selection differs (all of them valid near ties)."""
    assert np.all(np.abs(lg_gpu.astype(np.float64) - lg_orc) <= bound), \
        f"logit error {np.max(np.abs(lg_gpu - lg_orc) - bound)} above bound"
    ties = []
    k = idx_gpu.shape[1]
    for t in range(idx_gpu.shape[0]):
        if np.array_equal(idx_gpu[t], idx_orc[t]):
            continue
        o = lg_orc[t].astype(np.float64)
        kth = o[idx_orc[t, k - 1]]
        slack = 2 * bound[t].max()
        assert len(set(idx_gpu[t].tolist())) == k, f"token {t}: repeated expert"
        assert np.all(o[idx_gpu[t]] >= kth - slack), f"token {t}: invalid selection"
        missing = [e for e in idx_orc[t] if e not in set(idx_gpu[t].tolist())]
        assert all(o[e] <= o[idx_gpu[t]].min() + slack for e in missing), f"token {t}"
        ties.append(t)
    return ties


def run_gpu(L, x_np, w, want_routing=True):
    T = x_np.shape[0]
    x = to_dev_bf16(x_np)
    out = torch.full((T, w.H), float("nan"), device="cuda")
    L.forward(x, out)
    res = {}
    if want_routing:
        res["logits"] = torch.empty((T, w.E), dtype=torch.float32, device="cuda")
        res["idx"] = torch.empty((T, w.k), dtype=torch.int32, device="cuda")
        res["gates"] = torch.empty((T, w.k), dtype=torch.float32, device="cuda")
        res["counts"] = torch.empty(w.E, dtype=torch.int32, device="cuda")
        res["offsets"] = torch.empty(w.E + 1, dtype=torch.int32, device="cuda")
        res["perm"] = torch.empty(T * w.k, dtype=torch.int32, device="cuda")
        L.debug_routing(**res)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in res.items()}
    res["out"] = out.cpu().numpy()
    return res


def compare_layer(w, L, x_np, sample=None, orc_layer=None):
    """Full forward on the GPU; oracle on the sampled tokens (default: all).
    Returns (max rel-L2, near-tie token count)."""
    g = run_gpu(L, x_np, w)
    T = x_np.shape[0]
    assert not np.isnan(g["out"]).any(), "some output elements were not written"
    # dispatch of the GPU's own selection, against the oracle's dispatch, bit-exact
    counts, offsets, perm = oracle.dispatch(g["idx"], w.E)
    assert np.array_equal(g["counts"], counts)
    assert np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["perm"], perm)
    rows = np.arange(T) if sample is None else np.asarray(sample)
    xs = x_np[rows]
    router = gen.router_weights(w)
    bias = gen.router_bias(w)
    base = oracle.Layer(w.fmt, w.H, w.I, w.E, w.k, w.shared, router, bias)
    lg_o = base.logits(xs)
    idx_o, gates_o = base.topk(lg_o)
    bound = logit_bound(xs, router, bias)
    ties = check_routing(g["logits"][rows], g["idx"][rows], lg_o, idx_o, bound)
    idx_use = idx_o.copy()
    gates_use = gates_o.copy()
    for i in ties:
        idx_use[i] = g["idx"][rows[i]]
        gates_use[i] = gates_for(lg_o[i], idx_use[i])
    same = [i for i in range(len(rows)) if i not in ties]
    assert np.allclose(g["gates"][rows[same]], gates_o[same], rtol=0, atol=2e-5)
    need = set(idx_use.ravel().tolist()) | ({w.E} if w.shared else set())
    ol = orc_layer if orc_layer is not None else oracle.layer_for_workload(w, sorted(need))
    ref = ol.combine(xs, idx_use, gates_use)
    got = g["out"][rows]
    rel = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert np.all(rel <= REL_L2), f"rel-L2 {rel.max():.3e} > {REL_L2} (token {rows[rel.argmax()]})"
    return float(rel.max()), len(ties)
