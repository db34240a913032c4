"""Seeded synthetic inputs for the decode layer (weights, activations, KV).

This module only draws and encodes INPUTS; it holds none of the layer's own
arithmetic.  Both the CUDA library and the CPU oracle consume exactly the
tensors produced here.

Recipe (the same for every workload):
  * activations x_in ~ N(0, 1), stored bf16;
  * KV cache rows [0, ctx) ~ N(0, 1), stored bf16; rows >= ctx start at 0
    (the layer writes rows ctx .. ctx+T-1);
  * norm gains g ~ 1 + 0.1 N(0, 1), bf16;
  * dense weights ~ N(0, 1/fan_in), bf16, stored [out, in];
  * expert weights ~ N(0, 1/fan_in) encoded to NVFP4 once, here: one float32
    tensor scale per matrix (amax / (6 * 448)), one E4M3 scale per 16 inputs
    (block amax / (6 * tensor scale), rounded to nearest even by torch's
    float8_e4m3fn cast), E2M1 codes by round-to-nearest-even of w / (block
    scale * tensor scale).  Codes are packed two per byte, element 2i in the
    low nibble.
Every tensor draws from its own torch.Generator seeded by splitmix64 of
(seed, layer, tensor name), so a tensor does not depend on which others were
drawn.  CPU and CUDA generators give different streams: a workload is always
generated on one device.
"""

import zlib

import torch

SEED_BASE = 20261111

# Workloads (shapes from the five configurations this library is measured on).
WORKLOADS = {
    "tiny_layer": dict(
        index=0, layers=1, T=1, ctx=128, hidden=256, n_q_heads=4, n_kv_heads=1,
        head_dim=64, window=0, ffn="moe", n_experts=16, top_k=2, pooled_dim=128,
        expert_inter=128, fuse_next=False),
    "swa_layer": dict(
        index=1, layers=1, T=16, ctx=8192, hidden=4096, n_q_heads=32, n_kv_heads=8,
        head_dim=128, window=2048, ffn="moe", n_experts=256, top_k=8,
        pooled_dim=2048, expert_inter=1024, fuse_next=False),
    "global_layer_fused": dict(
        index=2, layers=1, T=16, ctx=32768, hidden=4096, n_q_heads=32, n_kv_heads=8,
        head_dim=128, window=0, ffn="moe", n_experts=256, top_k=8,
        pooled_dim=2048, expert_inter=1024, fuse_next=True),
    "dense_draft_stack": dict(
        index=3, layers=5, T=16, ctx=4096, hidden=4096, n_q_heads=32, n_kv_heads=8,
        head_dim=128, window=0, ffn="dense", dense_inter=12288, fuse_next=False),
    "moe_stack": dict(
        index=4, layers=62, T=16, ctx=16384, hidden=4096, n_q_heads=32, n_kv_heads=8,
        head_dim=128, window="pattern", ffn="moe", n_experts=256, top_k=8,
        pooled_dim=2048, expert_inter=1024, fuse_next=False),
}


def stack_window(layer, n_layers, swa=2048):
    """Window of layer ``layer`` in the 62-layer stack: 46 sliding-window and 16
    global layers.  Layers 0..59 are global iff layer % 4 == 3 (45 SWA, 15
    global); then one SWA layer (60) and one global layer (61)."""
    if n_layers == 62:
        if layer < 60:
            return 0 if layer % 4 == 3 else swa
        return swa if layer == 60 else 0
    return 0 if layer % 4 == 3 else swa


def layer_cfg(wl, layer=0):
    """Per-layer shape dict (window resolved) for workload dict ``wl``."""
    c = dict(wl)
    if wl["window"] == "pattern":
        c["window"] = stack_window(layer, wl["layers"])
    return c


def _splitmix64(x):
    x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return x ^ (x >> 31)


def sub_seed(seed, layer, name):
    s = _splitmix64(seed)
    s = _splitmix64(s ^ (layer * 0x100000001B3))
    s = _splitmix64(s ^ zlib.crc32(name.encode()))
    return s & 0x7FFFFFFFFFFFFFFF


def _gen(seed, layer, name, device):
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, layer, name))
    return g


def randn(shape, seed, layer, name, device="cpu", std=1.0):
    g = _gen(seed, layer, name, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.mul_(std) if std != 1.0 else x


# Round-to-nearest-even onto the E2M1 magnitudes {0,.5,1,1.5,2,3,4,6}: the
# midpoints between neighbouring codes, and whether an exact midpoint goes up.
_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)
_E2M1_TIE_UP = (False, True, False, True, False, True, False)


def _e2m1_codes(r):
    mag = r.abs()
    mids = torch.tensor(_E2M1_MID, device=r.device, dtype=torch.float32)
    code = torch.bucketize(mag, mids, right=False)          # ties go down
    at_mid = torch.zeros_like(mag, dtype=torch.bool)
    for m, tie_up in zip(_E2M1_MID, _E2M1_TIE_UP):
        if tie_up:
            at_mid |= mag == m
    code = (code + at_mid.to(code.dtype)).clamp(max=7)
    return (code | torch.where(r < 0, 8, 0)).to(torch.uint8)


def encode_nvfp4(w):
    """[..., N, K] float32 -> (codes [..., N, K/2] u8, scales [..., N, K/16] u8,
    tensor scale [...] f32), one tensor scale per trailing [N, K] matrix."""
    *lead, N, K = w.shape
    assert K % 16 == 0
    amax = w.abs().amax(dim=(-2, -1))
    ts = torch.where(amax > 0, amax / 2688.0, torch.ones_like(amax))
    blk = w.reshape(*lead, N, K // 16, 16)
    a16 = blk.abs().amax(dim=-1)
    tsb = ts.reshape(*lead, 1, 1)
    sb = (a16 / (6.0 * tsb)).clamp(max=448.0).to(torch.float8_e4m3fn)
    c = sb.to(torch.float32) * tsb
    r = blk / torch.where(c > 0, c, torch.ones_like(c)).unsqueeze(-1)
    codes = _e2m1_codes(r)
    codes = torch.where((c > 0).unsqueeze(-1), codes, torch.zeros_like(codes))
    codes = codes.reshape(*lead, N, K)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).contiguous()
    return packed, sb.view(torch.uint8).contiguous(), ts.to(torch.float32).contiguous()


def make_qkv_weights(wl, seed, layer, device="cpu"):
    """The attention-input norm gain and QKV weight of one layer."""
    H, Hq, Hkv, d = wl["hidden"], wl["n_q_heads"], wl["n_kv_heads"], wl["head_dim"]
    bf = torch.bfloat16
    nqkv = Hq * d + 2 * Hkv * d
    return {
        "attn_norm_w": (1.0 + randn((H,), seed, layer, "attn_norm_w", device, 0.1)).to(bf),
        "w_qkv": randn((nqkv, H), seed, layer, "w_qkv", device, H ** -0.5).to(bf),
    }


def make_layer_weights(wl, seed, layer, device="cpu", expert_chunk=32):
    """All weights of one layer (torch tensors on ``device``)."""
    H, Hq, d = wl["hidden"], wl["n_q_heads"], wl["head_dim"]
    bf = torch.bfloat16
    W = make_qkv_weights(wl, seed, layer, device)
    W["w_o"] = randn((H, Hq * d), seed, layer, "w_o", device, (Hq * d) ** -0.5).to(bf)
    W["ffn_norm_w"] = (1.0 + randn((H,), seed, layer, "ffn_norm_w", device, 0.1)).to(bf)
    if wl["ffn"] == "moe":
        E, P, I = wl["n_experts"], wl["pooled_dim"], wl["expert_inter"]
        W["w_router"] = router_weight(wl, seed, layer, 0, device)
        W["w_pool"] = randn((P, H), seed, layer, "w_pool", device, H ** -0.5).to(bf)
        W["w_unpool"] = randn((H, P), seed, layer, "w_unpool", device, P ** -0.5).to(bf)
        for name, (N, K) in (("gate", (I, P)), ("up", (I, P)), ("down", (P, I))):
            q = torch.empty((E, N, K // 2), dtype=torch.uint8, device=device)
            s = torch.empty((E, N, K // 16), dtype=torch.uint8, device=device)
            ts = torch.empty((E,), dtype=torch.float32, device=device)
            g = _gen(seed, layer, "exp_" + name, device)
            for e0 in range(0, E, expert_chunk):
                e1 = min(E, e0 + expert_chunk)
                w = torch.randn((e1 - e0, N, K), generator=g, device=device,
                                dtype=torch.float32).mul_(K ** -0.5)
                q[e0:e1], s[e0:e1], ts[e0:e1] = encode_nvfp4(w)
                del w
            W["exp_%s_q" % name], W["exp_%s_s" % name], W["exp_%s_ts" % name] = q, s, ts
    else:
        F = wl["dense_inter"]
        W["w_gate"] = randn((F, H), seed, layer, "w_gate", device, H ** -0.5).to(bf)
        W["w_up"] = randn((F, H), seed, layer, "w_up", device, H ** -0.5).to(bf)
        W["w_down"] = randn((H, F), seed, layer, "w_down", device, F ** -0.5).to(bf)
    return W


def router_weight(wl, seed, layer, draw, device="cpu"):
    """Router weight draw number ``draw`` (0, 1, ...).  A caller that needs a
    minimum gap between the k-th and (k+1)-th logit redraws with draw + 1."""
    H, E = wl["hidden"], wl["n_experts"]
    return randn((E, H), seed, layer, "w_router#%d" % draw, device, H ** -0.5).to(torch.bfloat16)


def make_activations(wl, seed, device="cpu", T=None, ctx=None, step=0):
    T = wl["T"] if T is None else T
    H = wl["hidden"]
    return randn((T, H), seed, 1000 + step, "x_in", device).to(torch.bfloat16)


def make_kv_cache(wl, seed, layer, device="cpu", ctx=None, max_ctx=None):
    """(k_cache, v_cache) bf16 [max_ctx, Hkv, d]: rows [0, ctx) drawn, the rest 0."""
    ctx = wl["ctx"] if ctx is None else ctx
    max_ctx = ctx + wl["T"] if max_ctx is None else max_ctx
    Hkv, d = wl["n_kv_heads"], wl["head_dim"]
    out = []
    for name in ("k_cache", "v_cache"):
        c = torch.zeros((max_ctx, Hkv, d), dtype=torch.bfloat16, device=device)
        if ctx > 0:
            c[:ctx] = randn((ctx, Hkv, d), seed, layer, name, device).to(torch.bfloat16)
        out.append(c)
    return tuple(out)


def make_workload(name_or_wl, device="cpu", layers=None, T=None, ctx=None, seed=None):
    """Weights, KV caches and x_in for a workload.  ``layers`` truncates a
    stack; ``T``/``ctx`` override the token count / context."""
    wl = dict(WORKLOADS[name_or_wl]) if isinstance(name_or_wl, str) else dict(name_or_wl)
    if T is not None:
        wl["T"] = T
    if ctx is not None:
        wl["ctx"] = ctx
    seed = SEED_BASE + wl["index"] if seed is None else seed
    L = wl["layers"] if layers is None else layers
    cfgs = [layer_cfg(wl, l) for l in range(L)]
    Ws = [make_layer_weights(wl, seed, l, device) for l in range(L)]
    caches = [make_kv_cache(wl, seed, l, device) for l in range(L)]
    x_in = make_activations(wl, seed, device)
    nxt = None
    if wl.get("fuse_next") and L == 1:
        nxt = make_qkv_weights(wl, seed, 1, device)
        nxt["k_cache"], nxt["v_cache"] = make_kv_cache(wl, seed, 1, device)
    return dict(wl=wl, seed=seed, cfgs=cfgs, Ws=Ws, caches=caches, x_in=x_in, next=nxt)
