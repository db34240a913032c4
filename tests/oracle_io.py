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


def enforce_margin_single(work, x_np=None, q_np=None, first_layer=True, max_draws=400, tree=None):
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
    o = bf16_round(ol.attention(q, kc, vc, wl["ctx"], c["window"], tree)).reshape(T, -1)
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


def _quantize_dequantize_row(x):
    from oracle import numerics as n
    q, s, r = n.nvfp4_quantize_rows(x[None, :])
    return n.nvfp4_dequantize(q, s, r)[0]


def _ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.frexp(np.where(x > 0, x, 1.0))[1]
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def _ambiguous_alternatives(row):
    """Dequantized alternatives of an NVFP4 row quantisation that a one-ulp
    change of one bf16 input element would select (the element's own code,
    or its block's scale, or -- for the row maximum -- the row scale)."""
    from oracle.numerics import bf16_round
    base = _quantize_dequantize_row(row)
    alts = []
    for i in range(row.size):
        for sgn in (-1.0, 1.0):
            r2 = row.copy()
            r2[i] = bf16_round(row[i] + sgn * _ulp(row[i]))
            d = _quantize_dequantize_row(r2)
            if not np.array_equal(d, base):
                alts.append(d)
                break
    return base, alts


def flip_tolerance(cfg, W, ref):
    """Per-token bound on how far x_out moves when one NVFP4 activation
    decision takes its other admissible value.

    An expert-input decision is admissible either way when a one-ulp change of
    a bf16 input element -- the size of the rounding differences between two
    correct evaluations -- selects the other code (or block / row scale).  For
    every such decision of the pooled rows p and the SwiGLU rows a, the oracle
    recomputes the affected token with the alternative and records
    max |x_out' - x_out| of that token.  Returns an array [T] of the largest
    such change per token.  (Small shapes only: the cost grows with P and I.)"""
    from oracle import numerics as n
    from oracle.layer import silu
    idx, w = ref["idx"], np.asarray(ref["w"], dtype=np.float64)
    T, k = idx.shape
    deq = {}

    def mats(e):
        if e not in deq:
            deq[e] = tuple(n.nvfp4_dequantize(W["exp_%s_q" % m][e], W["exp_%s_s" % m][e],
                                              W["exp_%s_ts" % m][e]) for m in ("gate", "up", "down"))
        return deq[e]

    wun = np.asarray(W["w_unpool"], dtype=np.float64)

    def x_row(t, z_rows):
        y = n.bf16_round(sum(w[t, r] * z_rows[r] for r in range(k)))
        return n.bf16_round(ref["x_mid"][t] + wun @ y)

    out = np.zeros(T)
    for t in range(T):
        x0 = ref["x_out"][t]
        z_base = [ref["z"][t, r] for r in range(k)]
        # pooled-row decisions
        _, alts = _ambiguous_alternatives(ref["p"][t])
        for ph in alts:
            zr = []
            for r in range(k):
                wg, wu, wd = mats(int(idx[t, r]))
                a = n.bf16_round(silu(wg @ ph) * (wu @ ph))
                zr.append(n.bf16_round(wd @ _quantize_dequantize_row(a)))
            out[t] = max(out[t], np.max(np.abs(x_row(t, zr) - x0)))
        # SwiGLU-row decisions
        for r in range(k):
            _, alts = _ambiguous_alternatives(ref["a"][t, r])
            wd = mats(int(idx[t, r]))[2]
            for ah in alts:
                zr = list(z_base)
                zr[r] = n.bf16_round(wd @ ah)
                out[t] = max(out[t], np.max(np.abs(x_row(t, zr) - x0)))
    return out


def _row_decisions(row):
    """All alternative dequantized rows reachable by moving one bf16 element of
    `row` by one ulp (each returned as (indices, new values) of the changed
    dequantized elements).  Vectorised: an element's own code for ordinary
    elements, its block re-quantised when it is the block maximum, the whole
    row re-quantised when it is the row maximum."""
    from oracle import numerics as n
    x = np.asarray(row, dtype=np.float64)
    K = x.size
    q, s, r = n.nvfp4_quantize_rows(x[None])
    base = n.nvfp4_dequantize(q, s, r)[0]
    codes = n.unpack_nibbles(q)[0]
    sb = n.e4m3_decode(s[0]).astype(np.float32)
    c = np.repeat((sb * r[0]).astype(np.float32), 16)
    ax = np.abs(x)
    blk_max = np.repeat(ax.reshape(-1, 16).max(axis=1), 16)
    row_max = ax.max()
    out = []
    ul = _ulp(x)
    for sgn in (-1.0, 1.0):
        x2 = n.bf16_round(x + sgn * ul)
        # ordinary elements: own code only
        ordinary = (ax < blk_max) & (c > 0)
        ratio = (x2.astype(np.float32) / np.where(c > 0, c, 1).astype(np.float32)).astype(np.float32)
        c2 = n.e2m1_encode(ratio)
        hit = np.nonzero(ordinary & (c2 != codes))[0]
        for i in hit:
            out.append((np.array([i]), np.array([n.e2m1_decode(c2[i]) * float(c[i])])))
        # block maxima (not the row maximum): re-quantise the block
        for i in np.nonzero((ax == blk_max) & (ax < row_max))[0]:
            xr = x.copy()
            xr[i] = x2[i]
            d = _quantize_dequantize_row(xr)
            b0 = (i // 16) * 16
            ch = np.nonzero(d[b0:b0 + 16] != base[b0:b0 + 16])[0] + b0
            if ch.size:
                out.append((ch, d[ch]))
        # row maximum: re-quantise the row
        for i in np.nonzero(ax == row_max)[0]:
            xr = x.copy()
            xr[i] = x2[i]
            d = _quantize_dequantize_row(xr)
            ch = np.nonzero(d != base)[0]
            if ch.size:
                out.append((ch, d[ch]))
    return base, out


def flip_tolerance_fast(cfg, W, ref):
    """Same bound as flip_tolerance, computed by propagating each single
    decision change through the token's expert path with the float64 sums the
    oracle kept (gate/up sums, down sums, unpooler sums): exact for the one
    changed decision; the candidates of a token are propagated together as
    matrix products."""
    from oracle import numerics as n
    from oracle.layer import silu
    idx, w = ref["idx"], np.asarray(ref["w"], dtype=np.float64)
    T, k = idx.shape
    deq = {}

    def mats(e):
        if e not in deq:
            deq[e] = tuple(n.nvfp4_dequantize(W["exp_%s_q" % m][e], W["exp_%s_s" % m][e],
                                              W["exp_%s_ts" % m][e]) for m in ("gate", "up", "down"))
        return deq[e]

    wun = np.asarray(W["w_unpool"], dtype=np.float64)
    out = np.zeros(T)
    for t in range(T):
        zb = np.stack([ref["z"][t, r] for r in range(k)])          # [k, P]
        Z = []                                                      # candidate z rows [k, P]
        # pooled-row decisions: every expert of the token sees the change
        _, alts = _row_decisions(ref["p"][t])
        for ii, vals in alts:
            dp = vals - ref["p_hat"][t][ii]
            zr = zb.copy()
            for r in range(k):
                wg, wu, wd = mats(int(idx[t, r]))
                g = ref["gu"][t, r, 0] + wg[:, ii] @ dp
                u = ref["gu"][t, r, 1] + wu[:, ii] @ dp
                a2 = n.bf16_round(silu(g) * u)
                if np.array_equal(a2, ref["a"][t, r]):
                    continue
                da = _quantize_dequantize_row(a2) - ref["a_hat"][t, r]
                nz = np.nonzero(da)[0]
                zr[r] = n.bf16_round(ref["z_acc"][t, r] + wd[:, nz] @ da[nz])
            Z.append(zr)
        # SwiGLU-row decisions: one expert's z changes
        for r in range(k):
            _, alts = _row_decisions(ref["a"][t, r])
            if not alts:
                continue
            wd = mats(int(idx[t, r]))[2]
            DA = np.zeros((len(alts), ref["a_hat"].shape[2]))
            for ci, (ii, vals) in enumerate(alts):
                DA[ci, ii] = vals - ref["a_hat"][t, r][ii]
            zr_all = n.bf16_round(ref["z_acc"][t, r][None, :] + DA @ wd.T)
            for ci in range(len(alts)):
                zr = zb.copy()
                zr[r] = zr_all[ci]
                Z.append(zr)
        if not Z:
            continue
        Z = np.stack(Z)                                             # [c, k, P]
        Y = n.bf16_round(np.einsum("r,crp->cp", w[t], Z))
        DY = Y - ref["y"][t][None, :]
        X = n.bf16_round(ref["x_acc"][t][None, :] + DY @ wun.T)
        out[t] = float(np.max(np.abs(X - ref["x_out"][t][None, :])))
    return out
