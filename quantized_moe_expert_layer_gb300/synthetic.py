"""Build a device layer of a synthetic workload.

The fp32 expert weights come from the seeded generator (``gen``) straight
into device memory, are quantised by the library's device quantiser and
packed by its packer; router weights and bias come from the same generator.
No host copy of the expert weights is made, so full-size layers (7.35 GB of
packed FP6 weights) build in seconds.
"""
from __future__ import annotations

import dataclasses

import torch

import gen

from . import FMT_MXFP4, FMT_NVFP4, MoeLayer, quantize_fp6, quantize_mxfp4, quantize_nvfp4


def build_layer(w, T_max=None, seed=None, experts=None, stream=None, in_hbm=None) -> MoeLayer:
    """Create, pack and reserve a layer for workload ``w``.

    seed: overrides the workload's seed (distinct layer instances);
    experts: iterable of expert ids to fill (default: all, E = shared expert);
    the others keep zero weights;
    in_hbm: per-expert placement (see MoeLayer.place_experts), applied before
    packing, so the packer writes host-mirror experts in place.
    """
    s = w.seed if seed is None else seed
    L = MoeLayer(w.fmt, w.H, w.I, w.E, w.k, w.shared)
    L.reserve(T_max or w.T)
    if in_hbm is not None:
        L.place_experts(in_hbm)
    ws = dataclasses.replace(w, seed=s)
    L.set_router(gen.router_weights(ws), gen.router_bias(ws))
    dev = torch.device("cuda")
    st = torch.cuda.current_stream() if stream is None else stream
    n_max = max(w.I * w.H, w.H * w.I)
    W = torch.empty(n_max, dtype=torch.float32, device=dev)
    codes = torch.empty(n_max, dtype=torch.uint8, device=dev)
    scales = torch.empty(n_max // 16, dtype=torch.uint8, device=dev)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    ids = range(w.n_experts_total) if experts is None else experts
    with torch.cuda.stream(st):
        for e in ids:
            for m in range(3):
                rows, K = gen.matrix_shape(w, m)
                Wm = W[: rows * K].view(rows, K)
                gen.fill_expert_weight_dev(w, e, m, Wm.data_ptr(), st.cuda_stream, seed=s)
                if w.fmt == FMT_NVFP4:
                    c = codes[: rows * K // 2]
                    sc = scales[: rows * K // 16]
                    quantize_nvfp4(Wm, c, sc, ts, stream=st)
                    L.pack_matrix(e, m, c, sc, ts, stream=st)
                elif w.fmt == FMT_MXFP4:
                    c = codes[: rows * K // 2]
                    sc = scales[: rows * K // 32]
                    quantize_mxfp4(Wm, c, sc, stream=st)
                    L.pack_matrix(e, m, c, sc, None, stream=st)
                else:
                    c = codes[: rows * K]
                    sc = scales[: rows * K // 128]
                    quantize_fp6(Wm, c, sc, stream=st)
                    L.pack_matrix(e, m, c, sc, None, stream=st)
    st.synchronize()
    return L
