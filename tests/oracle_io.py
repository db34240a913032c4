"""Test helpers: turn synthetic torch inputs into the oracle's numpy form, and
enforce the router margin by redrawing router weights (oracle-driven)."""

import numpy as np
import torch

from moe_decode_layer_persistent_gb300 import synth
import oracle
from oracle import layer as ol

MARGIN = 1e-2


def np64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def np_weights(W):
    out = {}
    for k, v in W.items():
        if v.dtype in (torch.uint8,):
            out[k] = v.detach().cpu().numpy()
        elif v.dtype == torch.float32:
            out[k] = v.detach().cpu().numpy()
        else:
            out[k] = np64(v)
    return out


def oracle_cfg(c):
    return dict(n_q_heads=c["n_q_heads"], n_kv_heads=c["n_kv_heads"], head_dim=c["head_dim"],
                window=c["window"], ffn=c["ffn"], top_k=c.get("top_k", 0))


def router_margin(logits, k):
    s = -np.sort(-logits.astype(np.float64), axis=1)
    return s[:, k - 1] - s[:, k]


def enforce_margin_single(work, x_np=None, q_np=None, first_layer=True, max_draws=400):
    """Redraw layer 0's router (draw 0, 1, ...) until every token's gap between
    the k-th and (k+1)-th float32 logit is >= MARGIN.  Mutates work['Ws'][0]
    (torch) and returns the numpy weights and the draw used."""
    wl = work["wl"]
    c = work["cfgs"][0]
    W = work["Ws"][0]
    Wn = np_weights(W)
    x = np64(work["x_in"]) if x_np is None else x_np
    kc, vc = (np64(t) for t in work["caches"][0])
    cfg = oracle_cfg(c)
    # the router input h depends only on the attention half of the layer
    T = x.shape[0]
    if first_layer:
        q, kn, vn = ol.qkv_project(x, Wn["attn_norm_w"], Wn["w_qkv"], c["n_q_heads"],
                                   c["n_kv_heads"], c["head_dim"])
        kc[work["wl"]["ctx"]:work["wl"]["ctx"] + T] = kn
        vc[work["wl"]["ctx"]:work["wl"]["ctx"] + T] = vn
    else:
        q = q_np
    from oracle.numerics import bf16_round
    o = bf16_round(ol.attention(q, kc, vc, wl["ctx"], c["window"])).reshape(T, -1)
    x_mid = bf16_round(x + o @ Wn["w_o"].T)
    h = bf16_round(ol.rmsnorm(x_mid, Wn["ffn_norm_w"]))
    dev = W["w_router"].device
    for draw in range(max_draws):
        wr = synth.router_weight(wl, work["seed"], 0, draw, dev)
        logits, _, _ = ol.router(h, np64(wr), c["top_k"])
        if np.all(router_margin(logits, c["top_k"]) >= MARGIN):
            W["w_router"] = wr
            Wn["w_router"] = np64(wr)
            return Wn, draw
    raise RuntimeError("no router draw met the margin")
