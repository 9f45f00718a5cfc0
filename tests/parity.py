"""Helpers shared by the GPU parity tests: run the CUDA layer and the oracle on
the same seeded inputs and compare them.

Tolerances:
  * dequantised weights, quantiser codes / scales, dispatch: bit-exact;
  * top-k indices: exact, except where the oracle's own logits of a picked
    and a passed-over expert are closer than the sum of their fp32 rounding
    bounds (delta = gamma_H * sum_h |x_h w_h| each, gamma_H = H u / (1 - H u),
    u = 2^-24: the standard bound of an fp32 dot product in any summation
    order, plus the bias add).  Such a near tie makes either choice a correct
    routing; the token is then compared with the oracle evaluated on the GPU's
    selection, and its gates with the softmax of the oracle's logits over it;
  * layer output: relative L2 error per token <= 2e-3 (fp32 accumulation).
"""
from __future__ import annotations

import numpy as np
import torch

import gen
import oracle

REL_L2 = 2e-3


def f32_to_bf16(f: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def to_dev_bf16(x_np: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).cuda()


U = 2.0 ** -24


def logit_bound(x_np, wr_np, bias):
    """Per (token, expert) bound on |fp32 logit - exact logit|: the products
    x_h w_h of bf16 values are exact in fp32, and any order of summing H of
    them in fp32 is within gamma_H * sum_h |x_h w_h| of the exact sum
    (gamma_H = H u / (1 - H u)); the bias add rounds once more (u |dot + b|).
    The oracle's own logit (an fp64 sum rounded once) is within u |l| of the
    exact one, which the same terms cover."""
    xv = gen.bf16_to_f32(x_np).astype(np.float64)
    wv = gen.bf16_to_f32(wr_np).astype(np.float64)
    H = xv.shape[1]
    s = np.abs(xv) @ np.abs(wv).T
    gamma = H * U / (1.0 - H * U)
    b = 0.0 if bias is None else np.abs(bias.astype(np.float64))[None, :]
    return gamma * s + 2 * U * (s + b)


def gates_for(logits_row, sel):
    v = logits_row[sel].astype(np.float64)
    e = np.exp(v - v.max())
    return (e / e.sum()).astype(np.float32)


def valid_near_tie(key, bound, sel_gpu, sel_orc):
    """True when the selection sel_gpu differs from sel_orc (the oracle's top-k
    of `key`) only by near ties: every expert the GPU picked in place of one
    the oracle picked is within the two experts' rounding bounds of it, and
    the GPU's order of its picks is by descending key up to the same slack."""
    k = len(sel_orc)
    if len(set(sel_gpu.tolist())) != k or np.any(sel_gpu < 0) or np.any(sel_gpu >= len(key)):
        return False
    extra = [e for e in sel_gpu if e not in set(sel_orc.tolist())]
    missing = [e for e in sel_orc if e not in set(sel_gpu.tolist())]
    for a in extra:
        for b in missing:
            if key[b] - key[a] > bound[a] + bound[b]:
                return False
    # every passed-over expert is at most a near tie above every pick
    for a in sel_gpu:
        others = np.setdiff1d(np.arange(len(key)), sel_gpu)
        if np.any(key[others] - key[a] > bound[others] + bound[a]):
            return False
    for j in range(k - 1):  # pick order: descending, ties to the lower id
        a, b = sel_gpu[j], sel_gpu[j + 1]
        if key[b] - key[a] > bound[a] + bound[b]:
            return False
    return True


def check_routing(lg_gpu, idx_gpu, lg_orc, idx_orc, bound):
    """Returns the tokens whose selection differs from the oracle's (every one
    of them a valid near tie, else the assertion fails)."""
    err = np.abs(lg_gpu.astype(np.float64) - lg_orc)
    assert np.all(err <= bound), f"logit error {np.max(err - bound)} above bound"
    ties = []
    for t in range(idx_gpu.shape[0]):
        if np.array_equal(idx_gpu[t], idx_orc[t]):
            continue
        assert valid_near_tie(lg_orc[t].astype(np.float64), bound[t], idx_gpu[t], idx_orc[t]), \
            f"token {t}: GPU picks {idx_gpu[t]} vs oracle {idx_orc[t]} are not a near tie"
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


def compare_layer(w, L, x_np, sample=None, orc_layer=None, route_all=False, act_fp4=False):
    """Full forward on the GPU; the oracle's layer output on the sampled tokens
    (default: all; act_fp4: the W4A4 oracle).  The routing (logits, top-k, gates) is compared on the
    sampled tokens, or on every token with route_all (the router and top-k
    are cheap next to the expert FFNs).  Returns (max rel-L2, near-tie token
    count over the routed rows)."""
    g = run_gpu(L, x_np, w)
    T = x_np.shape[0]
    assert not np.isnan(g["out"]).any(), "some output elements were not written"
    # dispatch of the GPU's own selection, against the oracle's dispatch, bit-exact
    counts, offsets, perm = oracle.dispatch(g["idx"], w.E)
    assert np.array_equal(g["counts"], counts)
    assert np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["perm"], perm)
    rows = np.arange(T) if sample is None else np.asarray(sample)
    rrows = np.arange(T) if route_all else rows
    router = gen.router_weights(w)
    bias = gen.router_bias(w)
    base = oracle.Layer(w.fmt, w.H, w.I, w.E, w.k, w.shared, router, bias)
    lg_r = base.logits(x_np[rrows])
    idx_r, gates_r = base.topk(lg_r)
    bound = logit_bound(x_np[rrows], router, bias)
    ties_r = check_routing(g["logits"][rrows], g["idx"][rrows], lg_r, idx_r, bound)
    same_r = np.array([i for i in range(len(rrows)) if i not in set(ties_r)], dtype=np.int64)
    if len(same_r):
        assert np.allclose(g["gates"][rrows[same_r]], gates_r[same_r], rtol=0, atol=2e-5)
    for i in ties_r:  # near ties: the GPU's gates are the softmax over its own picks
        assert np.allclose(g["gates"][rrows[i]], gates_for(lg_r[i], g["idx"][rrows[i]]),
                           rtol=0, atol=2e-5)
    # output rows: the oracle's routing, or the GPU's picks where they are a near tie
    pos = {int(r): i for i, r in enumerate(rrows)}
    sel = np.array([pos[int(r)] for r in rows], dtype=np.int64)
    xs = x_np[rows]
    lg_o, idx_o = lg_r[sel], idx_r[sel]
    ties = [i for i, r in enumerate(sel) if r in set(ties_r)]
    idx_use = idx_o.copy()
    gates_use = gates_r[sel].copy()
    for i in ties:
        idx_use[i] = g["idx"][rows[i]]
        gates_use[i] = gates_for(lg_o[i], idx_use[i])
    need = set(idx_use.ravel().tolist()) | ({w.E} if w.shared else set())
    ol = orc_layer if orc_layer is not None else oracle.layer_for_workload(w, sorted(need))
    ol.act_fp4 = act_fp4  # W4A4: the oracle quantises the activations of every product too
    ref = ol.combine(xs, idx_use, gates_use)
    got = g["out"][rows]
    rel = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    if act_fp4:  # near ties of the activation quantiser: either rounding is the contract's
        for i in np.nonzero(rel > REL_L2)[0]:
            rel[i] = w4a4_tie_rel(ol, xs[i], idx_use[i], gates_use[i], got[i])
    assert np.all(rel <= REL_L2), f"rel-L2 {rel.max():.3e} > {REL_L2} (token {rows[rel.argmax()]})"
    return float(rel.max()), len(ties_r)


W4A4_ETA = (3e-6, -3e-6, 3e-5, -3e-5)


def w4a4_tie_rel(ol, x_row, idx_row, gates_row, got_row):
    """W4A4 (R20) quantises a = silu(g) u, computed in fp64 by the oracle and in
    fp32 by the GPU (another summation order), to NVFP4: where an element of a
    (or its block's amax, which sets the e4m3 scale) lies within the fp32
    rounding of a rounding decision, both codes follow the contract.  The
    token is evaluated again in fp64 (numpy, independent of the oracle's C
    loops) with each row of a scaled by (1 + eta) before its quantisation, for
    eta of either sign (3e-6: a few fp32 roundings of K = 2048 sums; 3e-5);
    returns the smallest rel-L2 of the GPU row against those evaluations."""
    xf = gen.bf16_to_f32(np.asarray(x_row)[None, :])
    xq = _q_dq(xf)[0].astype(np.float64)
    experts = [int(e) for e in idx_row] + ([ol.E] if ol.shared else [])
    gts = [float(v) for v in gates_row] + ([1.0] if ol.shared else [])
    mats = {e: [ol.dequant(e, m).astype(np.float64) for m in range(3)] for e in experts}
    best = np.inf
    for eta in W4A4_ETA:
        out = np.zeros(ol.H)
        for e, gt in zip(experts, gts):
            wg, wu, wd = mats[e]
            gv, uv = wg @ xq, wu @ xq
            a = gv / (1.0 + np.exp(-gv)) * uv
            # (the quantised row scaled back: eta moves the rounding decisions only)
            aq = _q_dq((a * (1.0 + eta)).astype(np.float32)[None, :])[0].astype(np.float64) / (1.0 + eta)
            out += gt * (wd @ aq)
        r = np.linalg.norm(got_row - out) / max(np.linalg.norm(out), 1e-30)
        best = min(best, r)
    return best


def _q_dq(rows_f32):
    """NVFP4 quantise-and-dequantise of fp32 rows with the oracle's quantiser."""
    c, sc, ts = oracle.quantize_nvfp4(np.ascontiguousarray(rows_f32, dtype=np.float32))
    return oracle.dequant_nvfp4(c, sc, ts, rows_f32.shape[0], rows_f32.shape[1])
