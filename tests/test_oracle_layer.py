"""Pins for the oracle's layer steps (CPU only): library routines, closed
forms, invariants and brute force on tiny inputs."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import layer as ol
from oracle import numerics as n


def bf(rng, *shape, scale=1.0):
    return n.bf16_round(rng.standard_normal(shape) * scale)


# ---------------------------------------------------------------- RMSNorm ---

def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((5, 96))
    g = 1 + 0.1 * rng.standard_normal(96)
    ref = F.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), eps=1e-6).numpy()
    assert np.allclose(ol.rmsnorm(x, g), ref, rtol=1e-14, atol=1e-14)


def test_rmsnorm_constant_row_and_scale_invariance():
    g = np.linspace(0.5, 1.5, 32)
    for c in (3.0, -0.25):
        y = ol.rmsnorm(np.full((1, 32), c), g)
        assert np.allclose(y, c / math.sqrt(c * c + 1e-6) * g, rtol=1e-15)
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 64))
    assert np.allclose(ol.rmsnorm(7.5 * x, g[:1].repeat(64)), ol.rmsnorm(x, g[:1].repeat(64)), rtol=1e-6)


# -------------------------------------------------------------- attention ---

def _sdpa_reference(q, kc, vc, ctx, window):
    T, Hq, d = q.shape
    Hkv = kc.shape[1]
    S = ctx + T
    K = torch.from_numpy(kc[:S]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    V = torch.from_numpy(vc[:S]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    Q = torch.from_numpy(q).permute(1, 0, 2)
    pos = torch.arange(T)[:, None] + ctx
    j = torch.arange(S)[None, :]
    mask = j <= pos
    if window:
        mask &= (pos - j) < window
    o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("T,ctx,window,Hq,Hkv,d", [
    (1, 7, 0, 4, 1, 8), (4, 5, 0, 4, 2, 4), (16, 40, 8, 8, 2, 16), (3, 2, 4, 2, 2, 4),
    (5, 0, 0, 4, 4, 8), (16, 100, 32, 32, 8, 16)])
def test_attention_matches_torch_sdpa(T, ctx, window, Hq, Hkv, d):
    rng = np.random.default_rng(T * 100 + ctx)
    q = bf(rng, T, Hq, d)
    kc = bf(rng, ctx + T, Hkv, d)
    vc = bf(rng, ctx + T, Hkv, d)
    got = ol.attention(q, kc, vc, ctx, window)
    assert np.allclose(got, _sdpa_reference(q, kc, vc, ctx, window), rtol=1e-12, atol=1e-12)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(12)
    T, ctx, W, Hq, Hkv, d = 3, 4, 3, 4, 2, 2
    q = bf(rng, T, Hq, d)
    kc = bf(rng, ctx + T, Hkv, d)
    vc = bf(rng, ctx + T, Hkv, d)
    got = ol.attention(q, kc, vc, ctx, W)
    for i in range(T):
        p = ctx + i
        for h in range(Hq):
            g = h // (Hq // Hkv)
            js = [j for j in range(ctx + T) if j <= p and p - j < W]
            sc = [sum(q[i, h, c] * kc[j, g, c] for c in range(d)) / math.sqrt(d) for j in js]
            m = max(sc)
            ws = [math.exp(s - m) for s in sc]
            tot = sum(ws)
            for c in range(d):
                want = sum(w * vc[j, g, c] for w, j in zip(ws, js)) / tot
                assert abs(got[i, h, c] - want) < 1e-12


def test_attention_identical_keys_average_visible_values():
    # identical keys -> uniform weights -> output = mean of the visible V rows
    rng = np.random.default_rng(13)
    T, ctx, W, d = 6, 20, 9, 8
    q = bf(rng, T, 4, d)
    kc = np.tile(bf(rng, 1, 1, d), (ctx + T, 1, 1))
    vc = bf(rng, ctx + T, 1, d)
    for window in (0, W):
        got = ol.attention(q, kc, vc, ctx, window)
        for i in range(T):
            p = ctx + i
            lo = 0 if window == 0 else p - window + 1
            want = vc[lo:p + 1, 0].mean(axis=0)
            assert np.allclose(got[i], want[None, :], rtol=1e-13, atol=1e-13)


def test_swa_equals_global_when_context_fits_window():
    rng = np.random.default_rng(14)
    T, W = 16, 64
    ctx = W - T                       # ctx + T <= W: every key is inside the window
    q = bf(rng, T, 4, 8)
    kc = bf(rng, ctx + T, 1, 8)
    vc = bf(rng, ctx + T, 1, 8)
    assert np.array_equal(ol.attention(q, kc, vc, ctx, W), ol.attention(q, kc, vc, ctx, 0))
    ctx2 = W - T + 1                  # one more position: the first token loses key 0
    kc2 = bf(rng, ctx2 + T, 1, 8)
    vc2 = bf(rng, ctx2 + T, 1, 8)
    assert not np.array_equal(ol.attention(q, kc2, vc2, ctx2, W), ol.attention(q, kc2, vc2, ctx2, 0))


def test_attention_ignores_nan_outside_window_and_future():
    rng = np.random.default_rng(15)
    T, ctx, W = 4, 30, 10
    q = bf(rng, T, 2, 8)
    kc = bf(rng, ctx + T + 5, 1, 8)
    vc = bf(rng, ctx + T + 5, 1, 8)
    base = ol.attention(q, kc, vc, ctx, W)
    kp, vp = kc.copy(), vc.copy()
    kp[: ctx - W + 1] = np.nan        # outside every token's window
    vp[: ctx - W + 1] = np.nan
    kp[ctx + T:] = np.nan             # beyond the verify tokens
    vp[ctx + T:] = np.nan
    assert np.array_equal(ol.attention(q, kp, vp, ctx, W), base)


def test_attention_single_query_and_causality():
    rng = np.random.default_rng(16)
    T, ctx = 5, 12
    q = bf(rng, T, 2, 4)
    kc = bf(rng, ctx + T, 1, 4)
    vc = bf(rng, ctx + T, 1, 4)
    full = ol.attention(q, kc, vc, ctx, 0)
    one = ol.attention(q[:1], kc[:ctx + 1], vc[:ctx + 1], ctx, 0)
    assert np.array_equal(full[:1], one)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[ctx + 3] += 1.0               # change token 3's key/value
    vc2[ctx + 3] -= 2.0
    other = ol.attention(q, kc2, vc2, ctx, 0)
    assert np.array_equal(other[:3], full[:3])
    assert not np.array_equal(other[3:], full[3:])


# ------------------------------------------------------------------ router ---

def test_topk_matches_stable_sort():
    rng = np.random.default_rng(17)
    x = rng.integers(-5, 5, size=(30, 40)).astype(np.float32)      # many ties
    got = ol.topk_select(x, 8)
    ref = np.argsort(-x, axis=1, kind="stable")[:, :8]
    assert np.array_equal(got, ref)


def test_router_softmax_and_weights():
    rng = np.random.default_rng(18)
    h = bf(rng, 6, 64)
    wr = bf(rng, 32, 64, scale=0.125)
    logits, idx, w = ol.router(h, wr, 4)
    p = ol.softmax(logits.astype(np.float64))
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)
    tp = torch.softmax(torch.from_numpy(logits.astype(np.float64)), dim=1).numpy()
    assert np.allclose(p, tp, rtol=1e-12)
    assert np.array_equal(idx, torch.topk(torch.from_numpy(logits), 4, dim=1).indices.numpy())
    assert np.array_equal(w, np.take_along_axis(p, idx, axis=1).astype(np.float32))
    _, _, wn = ol.router(h, wr, 4, renorm=True)
    assert np.allclose(wn.sum(axis=1), 1.0, atol=1e-6)
    # logits are the float32 rounding of the float64 product
    assert np.array_equal(logits, (h @ wr.T).astype(np.float32))


# ------------------------------------------------------ token-tree attention ---

# A 16-token tree in topological order, written as parent indices (-1: the
# root, i.e. the token after the committed prefix): a root with three
# branches, branches of different depth, siblings at several levels.
TREE_PARENTS = [-1, 0, 0, 0, 1, 1, 2, 4, 4, 5, 6, 7, 3, 12, 9, 13]


def tree_masks(parents):
    """Ancestor-or-self bitmasks from parent indices (independent of the oracle)."""
    m = []
    for i, p in enumerate(parents):
        m.append((1 << i) | (m[p] if p >= 0 else 0))
    return m


def test_tree_masks_of_a_chain_and_of_the_test_tree():
    assert ol.chain_tree(4) == tree_masks([-1, 0, 1, 2]) == [1, 3, 7, 15]
    m = tree_masks(TREE_PARENTS)
    assert ol.tree_depths(m)[:7] == [0, 1, 1, 1, 2, 2, 2]
    assert ol.tree_depths(m)[15] == 4             # 15 -> 13 -> 12 -> 3 -> 0


@pytest.mark.parametrize("window", [0, 5, 3, 2048])
def test_tree_chain_mask_equals_the_causal_chain(window):
    """The chain given as a tree reproduces the causal attention bit for bit,
    also with windows shorter than the verify tokens."""
    rng = np.random.default_rng(30)
    T, ctx = 16, 23
    q = bf(rng, T, 4, 8)
    kc = bf(rng, ctx + T, 2, 8)
    vc = bf(rng, ctx + T, 2, 8)
    assert np.array_equal(ol.attention(q, kc, vc, ctx, window, tree_masks(list(range(-1, T - 1)))),
                          ol.attention(q, kc, vc, ctx, window))


@pytest.mark.parametrize("window", [0, 9])
def test_tree_token_equals_chain_attention_over_its_path(window):
    """Verify token i of a tree attends exactly like the last token of the
    causal chain made of the prefix and i's root-to-i path: rebuild that chain
    (its rows at positions ctx .. ctx + depth_i) and compare bit for bit."""
    rng = np.random.default_rng(31)
    T, ctx, Hq, Hkv, d = len(TREE_PARENTS), 12, 4, 2, 8
    q = bf(rng, T, Hq, d)
    kc = bf(rng, ctx + T, Hkv, d)
    vc = bf(rng, ctx + T, Hkv, d)
    got = ol.attention(q, kc, vc, ctx, window, tree_masks(TREE_PARENTS))
    for i in range(T):
        path = []
        j = i
        while j >= 0:
            path.append(j)
            j = TREE_PARENTS[j]
        path.reverse()
        kp = np.concatenate([kc[:ctx], kc[[ctx + j for j in path]]])
        vp = np.concatenate([vc[:ctx], vc[[ctx + j for j in path]]])
        qp = np.zeros((len(path), Hq, d))
        qp[-1] = q[i]
        chain = ol.attention(qp, kp, vp, ctx, window)
        assert np.array_equal(got[i], chain[-1]), i


def test_tree_attention_brute_force_and_siblings_unseen():
    """Textbook loop over the visible keys of a small tree; changing a token
    that is not an ancestor of i leaves i's output unchanged."""
    rng = np.random.default_rng(32)
    parents = [-1, 0, 0, 1, 2]
    T, ctx, W, Hq, Hkv, d = 5, 6, 4, 2, 1, 3
    m = tree_masks(parents)
    depth = [0, 1, 1, 2, 2]
    q = bf(rng, T, Hq, d)
    kc = bf(rng, ctx + T, Hkv, d)
    vc = bf(rng, ctx + T, Hkv, d)
    got = ol.attention(q, kc, vc, ctx, W, m)
    for i in range(T):
        pos = ctx + depth[i]
        js = [j for j in range(ctx) if pos - j < W]
        js += [ctx + j for j in range(T) if (m[i] >> j) & 1 and depth[i] - depth[j] < W]
        for h in range(Hq):
            sc = [sum(q[i, h, c] * kc[j, 0, c] for c in range(d)) / math.sqrt(d) for j in js]
            mx = max(sc)
            ws = [math.exp(s - mx) for s in sc]
            for c in range(d):
                want = sum(w * vc[j, 0, c] for w, j in zip(ws, js)) / sum(ws)
                assert abs(got[i, h, c] - want) < 1e-12
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[ctx + 2] += 1.0                       # token 2: not an ancestor of 1 or 3
    vc2[ctx + 2] -= 1.0
    other = ol.attention(q, kc2, vc2, ctx, W, m)
    for i in (0, 1, 3):
        assert np.array_equal(other[i], got[i])
    for i in (2, 4):
        assert not np.array_equal(other[i], got[i])


# -------------------------------------------------------------------- MoE ---

def _moe_weights(rng, E, H, P, I):
    from moe_decode_layer_persistent_gb300.synth import encode_nvfp4
    W = {"w_pool": bf(rng, P, H, scale=H ** -0.5), "w_unpool": bf(rng, H, P, scale=P ** -0.5)}
    for name, (N, K) in (("gate", (I, P)), ("up", (I, P)), ("down", (P, I))):
        q, s, ts = encode_nvfp4(torch.from_numpy(rng.standard_normal((E, N, K)) * K ** -0.5).float())
        W["exp_%s_q" % name], W["exp_%s_s" % name], W["exp_%s_ts" % name] = q.numpy(), s.numpy(), ts.numpy()
    return W


def test_moe_identical_experts_independent_of_routing():
    rng = np.random.default_rng(19)
    E, H, P, I, T, k = 6, 64, 32, 32, 3, 2
    W = _moe_weights(rng, E, H, P, I)
    for key in ("gate", "up", "down"):
        for part in ("q", "s", "ts"):
            arr = W["exp_%s_%s" % (key, part)]
            arr[:] = arr[0]
    h = bf(rng, T, H)
    w = np.full((T, k), 0.5, dtype=np.float32)
    r1 = ol.moe_ffn(h, W, np.array([[0, 1], [2, 3], [4, 5]]), w)
    r2 = ol.moe_ffn(h, W, np.array([[5, 4], [1, 0], [3, 2]]), w)
    assert np.array_equal(r1["y"], r2["y"])


def test_swiglu_orientation_and_activation_quantisation():
    # gate = 2*I, up = I (as NVFP4): a = SiLU(2 p) * p elementwise
    P = I = 16
    rng = np.random.default_rng(20)
    h = bf(rng, 1, 16)
    W = {"w_pool": np.eye(16), "w_unpool": np.eye(16)}
    eye_codes = n.pack_nibbles(np.where(np.eye(16) > 0, 2, 0).astype(np.uint8))  # code 2 = 1.0
    sc = np.full((16, 1), 0x38, dtype=np.uint8)                                  # e4m3 1.0
    for name, ts in (("gate", 2.0), ("up", 1.0), ("down", 1.0)):
        W["exp_%s_q" % name] = eye_codes[None]
        W["exp_%s_s" % name] = sc[None]
        W["exp_%s_ts" % name] = np.float32([ts])
    r = ol.moe_ffn(h, W, np.array([[0]]), np.float32([[1.0]]))
    p_hat = r["p_hat"][0]
    want_a = n.bf16_round(F.silu(torch.from_numpy(2 * p_hat)).numpy() * p_hat)
    assert np.allclose(r["a"][0, 0], want_a, rtol=1e-15)
    assert np.array_equal(r["p"], h)                        # identity pooler
    aq, as_, ar = n.nvfp4_quantize_rows(r["a"][0])
    assert np.array_equal(r["z"][0, 0], n.bf16_round(n.nvfp4_dequantize(aq, as_, ar)[0]))
    assert np.array_equal(r["y"][0], r["z"][0, 0])          # weight 1, one expert


def test_combine_is_weighted_sum_in_rank_order():
    rng = np.random.default_rng(21)
    E, H, P, I, T, k = 5, 32, 32, 16, 2, 3
    W = _moe_weights(rng, E, H, P, I)
    h = bf(rng, T, H)
    idx = np.array([[0, 3, 1], [4, 2, 0]])
    w = np.float32([[0.5, 0.25, 0.125], [0.3, 0.2, 0.1]])
    r = ol.moe_ffn(h, W, idx, w)
    for t in range(T):
        acc = sum(float(w[t, j]) * r["z"][t, j] for j in range(k))
        assert np.array_equal(r["y"][t], n.bf16_round(acc))


def test_combine_pairs_each_weight_with_its_expert():
    """Experts identical except for a power-of-two down tensor scale 2^e, so
    that every z of token t is 2^e times one vector z0_t (exactly: scaling by a
    power of two commutes with every rounding).  Then y_t must be
    bf16(sum_r w_tr 2^idx_tr z0_t) summed in rank order; a combine that pairs a
    weight with another rank's expert, reorders the weights or renormalises
    them gives another value on these inputs (checked)."""
    rng = np.random.default_rng(22)
    E, H, P, I, T, k = 5, 32, 32, 16, 3, 3
    W = _moe_weights(rng, E, H, P, I)
    for key in ("gate", "up", "down"):
        for part in ("q", "s", "ts"):
            arr = W["exp_%s_%s" % (key, part)]
            arr[:] = arr[0]
    h = bf(rng, T, H)
    idx = np.array([[0, 3, 1], [4, 2, 0], [2, 1, 3]])
    w = np.float32([[0.5, 0.25, 0.125], [0.375, 0.3125, 0.0625], [0.6, 0.2, 0.15]])
    z0 = ol.moe_ffn(h, W, idx, w)["z"][:, 0]          # all experts alike: z of any rank
    W["exp_down_ts"] = W["exp_down_ts"][0] * np.float32([2.0 ** e for e in range(E)])
    r = ol.moe_ffn(h, W, idx, w)
    for t in range(T):
        want = np.zeros(P)
        for j in range(k):
            want = want + float(w[t, j]) * (2.0 ** idx[t, j]) * z0[t]
        assert np.array_equal(r["y"][t], n.bf16_round(want)), t
        # the inputs tell the correct pairing from a rotated one and from renormalised weights
        rot = sum(float(w[t, (j + 1) % k]) * (2.0 ** idx[t, j]) * z0[t] for j in range(k))
        assert not np.array_equal(n.bf16_round(want), n.bf16_round(rot))
        assert not np.array_equal(n.bf16_round(want), n.bf16_round(want / float(w[t].sum())))


# ------------------------------------------------------------ whole layer ---

def _tiny_layer_inputs(rng, ffn="moe"):
    cfg = dict(n_q_heads=4, n_kv_heads=1, head_dim=16, window=0, ffn=ffn, top_k=2)
    H, E, P, I, T, ctx = 64, 6, 32, 32, 3, 9
    W = _moe_weights(rng, E, H, P, I) if ffn == "moe" else {
        "w_gate": bf(rng, 48, H, scale=H ** -0.5), "w_up": bf(rng, 48, H, scale=H ** -0.5),
        "w_down": bf(rng, H, 48, scale=48 ** -0.5)}
    W.update(attn_norm_w=n.bf16_round(1 + 0.1 * rng.standard_normal(H)),
             ffn_norm_w=n.bf16_round(1 + 0.1 * rng.standard_normal(H)),
             w_qkv=bf(rng, 6 * 16, H, scale=H ** -0.5), w_o=bf(rng, H, 64, scale=0.125),
             w_router=bf(rng, E, H, scale=H ** -0.5))
    x = bf(rng, T, H)
    kc = np.zeros((ctx + T, 1, 16))
    vc = np.zeros((ctx + T, 1, 16))
    kc[:ctx] = bf(rng, ctx, 1, 16)
    vc[:ctx] = bf(rng, ctx, 1, 16)
    return cfg, W, x, kc, vc, ctx


def _torch_layer(cfg, W, x, kc, vc, ctx):
    """The same layer composed from torch library routines (float64)."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    r16 = lambda a: t(n.bf16_round(a.numpy()))
    T, H = x.shape
    d = cfg["head_dim"]
    nrm = r16(F.rms_norm(t(x), (H,), t(W["attn_norm_w"]), eps=1e-6))
    qkv = r16(F.linear(nrm, t(W["w_qkv"])))
    q = qkv[:, :64].reshape(T, 4, d)
    kc = kc.copy(); vc = vc.copy()
    kc[ctx:ctx + T] = qkv[:, 64:80].reshape(T, 1, d).numpy()
    vc[ctx:ctx + T] = qkv[:, 80:96].reshape(T, 1, d).numpy()
    o = r16(torch.from_numpy(_sdpa_reference(q.numpy(), kc, vc, ctx, 0)).reshape(T, 64))
    x_mid = r16(t(x) + F.linear(o, t(W["w_o"])))
    h = r16(F.rms_norm(x_mid, (H,), t(W["ffn_norm_w"]), eps=1e-6))
    if cfg["ffn"] == "dense":
        a = r16(F.silu(F.linear(h, t(W["w_gate"]))) * F.linear(h, t(W["w_up"])))
        return r16(x_mid + F.linear(a, t(W["w_down"]))).numpy(), None
    logits = F.linear(h, t(W["w_router"])).float()
    top = torch.topk(logits, cfg["top_k"], dim=1)
    probs = torch.softmax(logits.double(), dim=1)
    w = torch.gather(probs, 1, top.indices).float().double()
    p = r16(F.linear(h, t(W["w_pool"])))
    pq = n.nvfp4_quantize_rows(p.numpy())
    p_hat = t(n.nvfp4_dequantize(*pq))
    y = torch.zeros(T, p.shape[1], dtype=torch.float64)
    for i in range(T):
        acc = torch.zeros(p.shape[1], dtype=torch.float64)
        for j in range(cfg["top_k"]):
            e = int(top.indices[i, j])
            deq = lambda nm: t(n.nvfp4_dequantize(W["exp_%s_q" % nm][e], W["exp_%s_s" % nm][e],
                                                  W["exp_%s_ts" % nm][e]))
            a = r16(F.silu(F.linear(p_hat[i], deq("gate"))) * F.linear(p_hat[i], deq("up")))
            aq = n.nvfp4_quantize_rows(a.numpy()[None])
            z = r16(F.linear(t(n.nvfp4_dequantize(*aq)[0]), deq("down")))
            acc = acc + w[i, j] * z
        y[i] = r16(acc)
    return r16(x_mid + F.linear(y, t(W["w_unpool"]))).numpy(), top.indices.numpy()


@pytest.mark.parametrize("ffn", ["moe", "dense"])
def test_layer_matches_torch_composition(ffn):
    rng = np.random.default_rng(22 if ffn == "moe" else 23)
    cfg, W, x, kc, vc, ctx = _tiny_layer_inputs(rng, ffn)
    r = ol.layer_forward(cfg, W, x, kc, vc, ctx)
    want, idx = _torch_layer(cfg, W, x, kc, vc, ctx)
    if idx is not None:
        assert np.array_equal(r["idx"], idx)
    # same rounding points, float64 sums: identical up to a rare one-ulp flip
    assert np.max(np.abs(r["x_out"] - want)) <= 2 ** -8 * np.max(np.abs(want))
    assert np.mean(r["x_out"] == want) > 0.99


def test_layer_zero_ffn_gives_x_mid_and_zero_attention_out_gives_x():
    rng = np.random.default_rng(24)
    cfg, W, x, kc, vc, ctx = _tiny_layer_inputs(rng, "moe")
    W["w_unpool"] = np.zeros_like(W["w_unpool"])
    r = ol.layer_forward(cfg, W, x, kc, vc, ctx)
    assert np.array_equal(r["x_out"], r["x_mid"])
    W["w_o"] = np.zeros_like(W["w_o"])
    r = ol.layer_forward(cfg, W, x, kc, vc, ctx)
    assert np.array_equal(r["x_out"], x)


def test_layer_expert_permutation_invariance():
    rng = np.random.default_rng(25)
    cfg, W, x, kc, vc, ctx = _tiny_layer_inputs(rng, "moe")
    r1 = ol.layer_forward(cfg, W, x, kc, vc, ctx)
    perm = np.array([3, 0, 5, 1, 4, 2])
    W2 = dict(W)
    W2["w_router"] = W["w_router"][perm]
    for key in ("gate", "up", "down"):
        for part in ("q", "s", "ts"):
            W2["exp_%s_%s" % (key, part)] = W["exp_%s_%s" % (key, part)][perm]
    r2 = ol.layer_forward(cfg, W2, x, kc, vc, ctx)
    assert np.array_equal(r1["x_out"], r2["x_out"])
    assert np.array_equal(perm[r2["idx"]], r1["idx"])


def test_stack_chains_layers_like_single_layers():
    # a two-layer stack equals layer 0 with fused next QKV, then layer 1 on q_next
    rng = np.random.default_rng(26)
    cfg, W0, x, kc0, vc0, ctx = _tiny_layer_inputs(rng, "moe")
    _, W1, _, kc1, vc1, _ = _tiny_layer_inputs(rng, "moe")
    xo, per, kcs, vcs = ol.stack_forward([cfg, cfg], [W0, W1], x, [kc0, kc1], [vc0, vc1], ctx)
    a = ol.layer_forward(cfg, W0, x, kc0, vc0, ctx)
    b = ol.layer_forward(cfg, W1, a["x_out"], kc1, vc1, ctx, first_layer=True)
    assert np.array_equal(xo, b["x_out"])
    assert np.array_equal(kcs[1], b["k_cache"]) and np.array_equal(vcs[1], b["v_cache"])
