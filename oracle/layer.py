"""The decode layer, one operation at a time, in float64 with bf16 storage.

Op order of one MoE decoder layer (canonical form) and where each step comes
from.  Page names:
  [ORCA] "Muse Spark Open: 1,109 Tokens a Second Is a Kernel Change, Not a
         Model Change" (orcarouter.ai)
  [AIC]  "LMSYS Details SGLang Megakernel: Muse Spark Open Decodes at 1,109
         tok/s on 8x GB300 at Batch 1" (aicoder.com news)

  1. n = bf16(RMSNorm(x) * g1); [q|k|v] = bf16(n W_qkv^T); k, v written to the
     KV cache at positions ctx .. ctx+T-1.              [ORCA "Where the kernel
     boundary sits": the launch ends with the next layer's qkv projection and
     KV write; AIC "Architecture and how it works"]
  2. GQA attention over the bf16 KV cache, sliding window of 2,048 tokens or
     global, causal over the T verify tokens.           [ORCA same section]
  3. x_mid = bf16(x + o W_o^T)                          [ORCA same section:
     "the dense GEMMs"]
  4. h = bf16(RMSNorm(x_mid) * g2)
  5. router: logits = h W_r^T (float32), softmax over all experts, top-k
     ("routing every token to 8 of 256 experts")        [ORCA same section]
  6. p = bf16(h W_pool^T)  ("a pooler projection that shrinks each token
     vector before the experts")                        [ORCA same section]
  7. expert gate/up on NVFP4 p, a = bf16(SiLU(g) * u), re-quantised to NVFP4
     ("an fp4 all-gather after the first" MoE GEMM)     [ORCA same section]
  8. expert down, z = bf16(a W_d^T) ("a bf16 one after the second")
  9. y_t = bf16(sum_r w_{t,r} z_{t,r}), summed in rank order  [ORCA "What the
     5.9 ms is still spent on": the combine]
 10. x_out = bf16(x_mid + y W_unpool^T) ("an unpooler that restores it")
 11. optionally the next layer's step 1 on x_out (fused next QKV + KV write).

Readings where the pages are silent: RMSNorm y = x * (mean(x^2) + eps)^-1/2 * g
with eps = 1e-6; no positional rotation and no QK-norm; q head h reads KV head
floor(h / (Hq/Hkv)); scale 1/sqrt(d); key j is visible to the query at
position p iff j <= p and (window == 0 or p - j < window); top-k by descending
float32 logit, an exact tie going to the lower expert index; combine weights
are the softmax probabilities of the chosen experts (renormalised over the
top-k only when ``renorm`` is set); pooler and unpooler are plain linear maps.

Dense variant (draft layers, [AIC] "Key Takeaways" / ORCA "The draft model got
faster too": Qwen3-style GQA layers): steps 4-10 become
  h = bf16(RMSNorm(x_mid) * g2); a = bf16(SiLU(h W_g^T) * (h W_u^T));
  x_out = bf16(x_mid + a W_d^T).
The down projection's output is added to the residual before its one
rounding, as the o-proj (step 3) and the unpooler (step 10) are: rounding it
to bf16 first would add a second rounding after which x_out depends on which
side of a bf16 boundary each product lands.

Weight layouts (all "output rows x input columns", input contiguous):
  w_qkv [Hq*d + 2*Hkv*d, H] (q heads, then k heads, then v heads), w_o [H, Hq*d],
  w_router [E, H], w_pool [P, H], w_unpool [H, P], expert gate/up codes
  [E, I, P/2] + scales [E, I, P/16] + tensor scale [E], expert down codes
  [E, P, I/2] + scales [E, P, I/16] + tensor scale [E]; dense w_gate/w_up
  [F, H], w_down [H, F].  KV cache [positions, Hkv, d].
"""

import math

import numpy as np

from .numerics import bf16_round, f32, nvfp4_dequantize, nvfp4_quantize_rows

RMS_EPS = 1e-6


def rmsnorm(x, gamma, eps=RMS_EPS):
    """x * (mean(x^2) + eps)^-1/2 * gamma, per row, float64 (not rounded)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def qkv_project(x, gamma1, w_qkv, n_q_heads, n_kv_heads, head_dim, eps=RMS_EPS):
    """Step 1: returns q [T, Hq, d], k [T, Hkv, d], v [T, Hkv, d] (bf16 values)."""
    T = x.shape[0]
    n = bf16_round(rmsnorm(x, gamma1, eps))
    qkv = bf16_round(n @ np.asarray(w_qkv, dtype=np.float64).T)
    nq = n_q_heads * head_dim
    nk = n_kv_heads * head_dim
    q = qkv[:, :nq].reshape(T, n_q_heads, head_dim)
    k = qkv[:, nq:nq + nk].reshape(T, n_kv_heads, head_dim)
    v = qkv[:, nq + nk:nq + 2 * nk].reshape(T, n_kv_heads, head_dim)
    return q, k, v


def visible_range(pos, window):
    """Key positions [lo, pos] visible to the query at ``pos``."""
    lo = 0 if window == 0 else max(0, pos - window + 1)
    return lo, pos


def chain_tree(T):
    """The causal chain as a token tree: token i's ancestors are 0 .. i-1."""
    return [(1 << (i + 1)) - 1 for i in range(T)]


def tree_depths(tree):
    """Depth of each verify token in a token tree: the number of its ancestors.
    tree[i] has bit j set iff verify token j is i itself or an ancestor of i
    (tokens in topological order: ancestors come first)."""
    return [bin(int(m)).count("1") - 1 for m in tree]


def visible_keys(i, ctx, window, tree):
    """Cache positions visible to verify token i, ascending.

    Token-tree verification ([EXPL] "What the README says the kernels do":
    the draft proposes a tree of candidates instead of a chain; ORCA "The
    draft model got faster too": 16 tokens verified): verify token i sits at
    sequence position ctx + depth_i and its K/V row at cache position ctx + i.
    It sees the committed prefix j < ctx within the window counted from its
    sequence position (ctx + depth_i - j < window), and each verify token j
    that is i or an ancestor of i, within the window counted in depth
    (depth_i - depth_j < window).  For the chain, depth_i = i and this is the
    causal rule: key j visible iff j <= ctx + i and ctx + i - j < window."""
    depth = tree_depths(tree)
    lo, _ = visible_range(ctx + depth[i], window)
    keys = list(range(lo, ctx))
    for j in range(i + 1):
        if (int(tree[i]) >> j) & 1 and (window == 0 or depth[i] - depth[j] < window):
            keys.append(ctx + j)
    return keys


def attention(q, k_cache, v_cache, ctx, window, tree=None):
    """Step 2.  q [T, Hq, d]; caches [>= ctx+T, Hkv, d] holding the new rows.

    Verify token i sees the keys visible_keys(i, ...) gives; tree = None is
    the causal chain (token i at position ctx + i).  Returns o [T, Hq, d]
    (float64, not rounded)."""
    T, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    o = np.zeros((T, Hq, d))
    scale = 1.0 / math.sqrt(d)
    tree = chain_tree(T) if tree is None else tree
    for i in range(T):
        keys = visible_keys(i, ctx, window, tree)
        for g in range(Hkv):
            K = np.asarray(k_cache[keys, g, :], dtype=np.float64)
            V = np.asarray(v_cache[keys, g, :], dtype=np.float64)
            Q = q[i, g * group:(g + 1) * group, :]
            s = (Q @ K.T) * scale                       # [group, n]
            s = s - s.max(axis=1, keepdims=True)
            e = np.exp(s)
            p = e / e.sum(axis=1, keepdims=True)
            o[i, g * group:(g + 1) * group, :] = p @ V
    return o


def topk_select(logits, k):
    """Indices of the k largest entries per row: descending value, an exact
    tie going to the lower index.  Plain repeated selection."""
    logits = np.asarray(logits)
    rows, n = logits.shape
    idx = np.zeros((rows, k), dtype=np.int32)
    for r in range(rows):
        taken = np.zeros(n, dtype=bool)
        for j in range(k):
            best = -1
            for c in range(n):
                if taken[c]:
                    continue
                if best < 0 or logits[r, c] > logits[r, best]:
                    best = c
            taken[best] = True
            idx[r, j] = best
    return idx


def softmax(x):
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def router(h, w_router, top_k, renorm=False):
    """Step 5.  Returns (logits float32 [T, E], idx int32 [T, k], w float32 [T, k]).

    Logits are summed in float64 and stored as float32; the top-k decision is
    taken on the float32 logits; the softmax is over all E experts."""
    logits = f32(np.asarray(h, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T)
    idx = topk_select(logits, top_k)
    probs = softmax(logits.astype(np.float64))
    w = np.take_along_axis(probs, idx, axis=1)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return logits, idx, f32(w)


def silu(x):
    return x / (1.0 + np.exp(-x))


def moe_ffn(h, W, idx, w):
    """Steps 6-10 (without the residual).  Returns a dict with p, p_hat, a,
    z [T, k, P], y [T, P] (bf16 values, float64 arrays)."""
    T = h.shape[0]
    k = idx.shape[1]
    p = bf16_round(h @ np.asarray(W["w_pool"], dtype=np.float64).T)
    pq, ps, prow = nvfp4_quantize_rows(p)
    p_hat = nvfp4_dequantize(pq, ps, prow)
    P = p.shape[1]
    I = W["exp_gate_q"].shape[1]
    a = np.zeros((T, k, I))
    a_hat = np.zeros((T, k, I))
    gu = np.zeros((T, k, 2, I))      # gate / up sums before SiLU (float64)
    z = np.zeros((T, k, P))
    z_acc = np.zeros((T, k, P))      # down sums before rounding (float64)
    for e in sorted(set(int(v) for v in idx.ravel())):
        wg = nvfp4_dequantize(W["exp_gate_q"][e], W["exp_gate_s"][e], W["exp_gate_ts"][e])
        wu = nvfp4_dequantize(W["exp_up_q"][e], W["exp_up_s"][e], W["exp_up_ts"][e])
        wd = nvfp4_dequantize(W["exp_down_q"][e], W["exp_down_s"][e], W["exp_down_ts"][e])
        for t in range(T):
            for r in range(k):
                if int(idx[t, r]) != e:
                    continue
                g = wg @ p_hat[t]
                u = wu @ p_hat[t]
                gu[t, r, 0], gu[t, r, 1] = g, u
                a[t, r] = bf16_round(silu(g) * u)
                aq, as_, arow = nvfp4_quantize_rows(a[t, r][None, :])
                a_hat[t, r] = nvfp4_dequantize(aq, as_, arow)[0]
                z_acc[t, r] = wd @ a_hat[t, r]
                z[t, r] = bf16_round(z_acc[t, r])
    wf = np.asarray(w, dtype=np.float32).astype(np.float64)
    y = np.zeros((T, P))
    for t in range(T):
        acc = np.zeros(P)
        for r in range(k):
            acc = acc + wf[t, r] * z[t, r]
        y[t] = bf16_round(acc)
    return dict(p=p, p_hat=p_hat, a=a, a_hat=a_hat, gu=gu, z=z, z_acc=z_acc, y=y)


def dense_ffn(h, W):
    """Steps 6-10 of the dense variant: the SwiGLU activation a (bf16 values)
    and the down projection's output before the residual (not rounded)."""
    g = h @ np.asarray(W["w_gate"], dtype=np.float64).T
    u = h @ np.asarray(W["w_up"], dtype=np.float64).T
    a = bf16_round(silu(g) * u)
    return dict(a=a, ffn_out=a @ np.asarray(W["w_down"], dtype=np.float64).T)


def layer_forward(cfg, W, x_in, k_cache, v_cache, ctx, q_in=None, first_layer=True,
                  next_W=None, next_k_cache=None, next_v_cache=None, renorm=False, tree=None):
    """One layer launch's worth of work.

    cfg: dict with n_q_heads, n_kv_heads, head_dim, window, ffn ('moe'|'dense'),
         top_k (moe), eps (optional).
    W:   dict of weights (numpy; bf16 tensors as float64 values, NVFP4 as bytes).
    x_in [T, H]; caches [max_ctx, Hkv, d] (copied, not modified in place).
    first_layer: run step 1 on x_in; otherwise ``q_in`` [T, Hq, d] is used and
         the caches must already hold rows ctx .. ctx+T-1.
    next_W: if given, step 11 with next_W's attn_norm_w and w_qkv, writing
         rows ctx .. ctx+T-1 of copies of next_k_cache / next_v_cache.
    tree: token-tree masks (see visible_keys); None = the causal chain.
    Returns a dict of every intermediate (bf16 values as float64 arrays).
    """
    eps = cfg.get("eps", RMS_EPS)
    Hq, Hkv, d = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    x_in = np.asarray(x_in, dtype=np.float64)
    T = x_in.shape[0]
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    out = {}
    if first_layer:
        q, k_new, v_new = qkv_project(x_in, W["attn_norm_w"], W["w_qkv"], Hq, Hkv, d, eps)
        kc[ctx:ctx + T] = k_new
        vc[ctx:ctx + T] = v_new
        out.update(k_new=k_new, v_new=v_new)
    else:
        q = np.asarray(q_in, dtype=np.float64).reshape(T, Hq, d)
    out["q"] = q
    o = bf16_round(attention(q, kc, vc, ctx, cfg["window"], tree)).reshape(T, Hq * d)
    out["o"] = o
    x_mid = bf16_round(x_in + o @ np.asarray(W["w_o"], dtype=np.float64).T)
    out["x_mid"] = x_mid
    h = bf16_round(rmsnorm(x_mid, W["ffn_norm_w"], eps))
    out["h"] = h
    if cfg["ffn"] == "moe":
        logits, idx, w = router(h, W["w_router"], cfg["top_k"], renorm)
        out.update(logits=logits, idx=idx, w=w)
        m = moe_ffn(h, W, idx, w)
        out.update(m)
        out["x_acc"] = x_mid + m["y"] @ np.asarray(W["w_unpool"], dtype=np.float64).T
        x_out = bf16_round(out["x_acc"])
    else:
        dres = dense_ffn(h, W)
        out["a"] = dres["a"]
        x_out = bf16_round(x_mid + dres["ffn_out"])
    out["x_out"] = x_out
    out["k_cache"] = kc
    out["v_cache"] = vc
    if next_W is not None:
        qn, kn, vn = qkv_project(x_out, next_W["attn_norm_w"], next_W["w_qkv"], Hq, Hkv, d, eps)
        nkc = np.array(next_k_cache, dtype=np.float64, copy=True)
        nvc = np.array(next_v_cache, dtype=np.float64, copy=True)
        nkc[ctx:ctx + T] = kn
        nvc[ctx:ctx + T] = vn
        out.update(q_next=qn, k_next=kn, v_next=vn, next_k_cache=nkc, next_v_cache=nvc)
    return out


def stack_forward(cfgs, Ws, x_in, k_caches, v_caches, ctx, renorm=False, keep=None, tree=None):
    """A chain of layers: layer 0 runs step 1 itself, layer l < L-1 fuses layer
    l+1's step 1, the last layer has no next QKV.  Returns (x_out, per-layer
    list of dicts restricted to the keys in ``keep``), and the updated caches.
    """
    L = len(Ws)
    keep = keep or ("idx", "w", "k_new", "v_new", "k_next", "v_next", "x_out")
    x = np.asarray(x_in, dtype=np.float64)
    q = None
    kcs = list(k_caches)
    vcs = list(v_caches)
    per = []
    for l in range(L):
        nxt = Ws[l + 1] if l + 1 < L else None
        r = layer_forward(cfgs[l], Ws[l], x, kcs[l], vcs[l], ctx, q_in=q,
                          first_layer=(l == 0), next_W=nxt,
                          next_k_cache=kcs[l + 1] if nxt is not None else None,
                          next_v_cache=vcs[l + 1] if nxt is not None else None,
                          renorm=renorm, tree=tree)
        kcs[l] = r["k_cache"]
        vcs[l] = r["v_cache"]
        if nxt is not None:
            kcs[l + 1] = r["next_k_cache"]
            vcs[l + 1] = r["next_v_cache"]
            q = r["q_next"]
        x = r["x_out"]
        per.append({k: r[k] for k in keep if k in r})
    return x, per, kcs, vcs
