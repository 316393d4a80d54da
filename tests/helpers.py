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


def oracle_draft_layers(cfg, layers):
    """Draft weights: resident layers shared, the rest replaced by the
    dequantised int4 substitutes (oracle quantiser)."""
    out = []
    for i, lw in enumerate(layers):
        if i < cfg.n_resident:
            out.append(lw)
            continue
        d = dict(lw)
        for name in synthetic.LAYER_TENSORS:
            w = lw[name]
            q, s, z = quant.w4_pack(w)
            d[name] = quant.w4_dequant(q, s, z, w.shape[1])
        out.append(d)
    return out
