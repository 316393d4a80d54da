"""Shared test helpers: convert synthetic torch inputs for the oracle."""
import numpy as np
import torch

import synthetic
from oracle import quant


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").float().numpy()


def oracle_model(model: dict):
    glob = {k: to_np(model[k]) for k in ("embed", "lm_head", "final_norm")}
    layers = [{k: to_np(v) for k, v in lw.items()} for lw in model["layers"]]
    return glob, layers


def oracle_draft_layers(cfg, layers, bits=4, hqq_iters=0):
    """Draft weights: resident layers shared, the rest replaced by the
    dequantised substitutes (oracle quantiser); bits: 2, 3 or 4 for every
    substitute, or a list with one entry per layer (mixed precision);
    hqq_iters > 0: HQQ-optimised zero points."""
    out = []
    for i, lw in enumerate(layers):
        if i < cfg.n_resident:
            out.append(lw)
            continue
        b = bits[i] if isinstance(bits, (list, tuple)) else bits
        d = dict(lw)
        for name in synthetic.LAYER_TENSORS:
            w = lw[name]
            if hqq_iters > 0:
                q, s, z = quant.wq_pack_hqq(w, b, hqq_iters)
                d[name] = quant.wq_dequant(q, s, z, w.shape[1], b)
            elif b == 4:
                q, s, z = quant.w4_pack(w)
                d[name] = quant.w4_dequant(q, s, z, w.shape[1])
            else:
                q, s, z = quant.wq_pack(w, b)
                d[name] = quant.wq_dequant(q, s, z, w.shape[1], b)
        out.append(d)
    return out
