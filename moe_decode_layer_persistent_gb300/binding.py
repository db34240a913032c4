"""ctypes binding of libmk.so: the mk_* C ABI with the same names.

Argument marshalling only: every step of the decode layer runs in the CUDA
library.  Tensors are passed as device pointers (torch tensors are accepted
for convenience; only ``data_ptr()`` is read).  Loading fails loudly if the
library has not been built -- there is no CPU fallback.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmk.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libmk.so not built (run __graft_entry__.build()): %s" % LIB_PATH)
_lib = ctypes.CDLL(LIB_PATH)

MK_OK = 0
STATUS_NAMES = {0: "MK_OK", 1: "MK_ERR_INVALID_ARG", 2: "MK_ERR_UNSUPPORTED", 3: "MK_ERR_CUDA",
                4: "MK_ERR_OOM", 5: "MK_ERR_TIMEOUT", 6: "MK_ERR_DEVICE_FAULT"}
MK_FFN_MOE_NVFP4 = 0
MK_FFN_DENSE_SWIGLU_BF16 = 1
MK_FIRST_LAYER = 0x1
MK_FUSE_NEXT_QKV = 0x2
MK_TOPK_RENORM = 0x4
MK_PREFETCH_NEXT_KV = 0x8

_vp = ctypes.c_void_p


class MkError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s -> %s" % (fn, STATUS_NAMES.get(status, status)))


class mk_layer_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("window", ctypes.c_int32), ("ffn_kind", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("pooled_dim", ctypes.c_int32), ("expert_inter", ctypes.c_int32),
                ("dense_inter", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("max_ctx", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("flags", ctypes.c_uint32), ("prefetch_experts", ctypes.c_int32),
                ("wait_timeout_ns", ctypes.c_uint64)]


class mk_prefetch_stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("predicted", ctypes.c_uint64),
                ("active", ctypes.c_uint64), ("hits", ctypes.c_uint64)]


_WEIGHT_FIELDS = ["attn_norm_w", "w_qkv", "w_o", "ffn_norm_w", "w_router", "w_pool", "w_unpool",
                  "exp_gate_q", "exp_gate_s", "exp_gate_ts", "exp_up_q", "exp_up_s", "exp_up_ts",
                  "exp_down_q", "exp_down_s", "exp_down_ts", "w_gate", "w_up", "w_down",
                  "next_attn_norm_w", "next_w_qkv"]


class mk_layer_weights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in _WEIGHT_FIELDS]


class mk_step_io(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("ctx_len", ctypes.c_int32),
                ("x_in", _vp), ("x_out", _vp), ("q_in", _vp), ("k_cache", _vp),
                ("v_cache", _vp), ("next_k_cache", _vp), ("next_v_cache", _vp),
                ("q_out", _vp), ("topk_idx_out", _vp), ("topk_w_out", _vp),
                ("tree_mask", ctypes.POINTER(ctypes.c_uint16))]


class mk_stack_io(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("ctx_len", ctypes.c_int32),
                ("x_in", _vp), ("x_out", _vp), ("k_caches", ctypes.POINTER(_vp)),
                ("v_caches", ctypes.POINTER(_vp)), ("topk_idx_out", _vp), ("topk_w_out", _vp),
                ("tree_mask", ctypes.POINTER(ctypes.c_uint16))]


class mk_layer_info(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("tmem_cols", ctypes.c_int32),
                ("scratch_bytes", ctypes.c_int64)]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_c = ctypes
_lib_mk_layer_create = _sig("mk_layer_create", _c.c_int,
                            [_c.POINTER(mk_layer_config), _c.POINTER(mk_layer_weights),
                             _c.POINTER(_vp)])
_lib_mk_decode_step = _sig("mk_decode_step", _c.c_int, [_vp, _c.POINTER(mk_step_io), _vp])
_lib_mk_layer_status = _sig("mk_layer_status", _c.c_int, [_vp])
_lib_mk_layer_clear_status = _sig("mk_layer_clear_status", _c.c_int, [_vp])
_lib_mk_layer_destroy = _sig("mk_layer_destroy", None, [_vp])
_lib_mk_stack_create = _sig("mk_stack_create", _c.c_int, [_c.POINTER(_vp), _c.c_int32, _c.POINTER(_vp)])
_lib_mk_stack_step = _sig("mk_stack_step", _c.c_int, [_vp, _c.POINTER(mk_stack_io), _vp])
_lib_mk_stack_status = _sig("mk_stack_status", _c.c_int, [_vp])
_lib_mk_layer_prefetch_stats = _sig("mk_layer_prefetch_stats", _c.c_int, [_vp, _vp])
_lib_mk_stack_prefetch_stats = _sig("mk_stack_prefetch_stats", _c.c_int, [_vp, _vp])
_lib_mk_stack_destroy = _sig("mk_stack_destroy", None, [_vp])
_lib_mk_status_string = _sig("mk_status_string", _c.c_char_p, [_c.c_int])
_lib_mk_layer_get_info = _sig("mk_layer_get_info", _c.c_int, [_vp, _c.POINTER(mk_layer_info)])
_lib_mk_selftest_quantize = _sig("mk_selftest_quantize", _c.c_int,
                                 [_vp, _c.c_int32, _c.c_int32, _vp, _vp, _vp, _vp])
_lib_mk_selftest_mma = _sig("mk_selftest_mma", _c.c_int,
                            [_c.c_int32, _vp, _vp, _vp, _vp, _c.c_int32, _vp, _vp])

_lib_mk_get_timestamps = _sig("mk_get_timestamps", _c.c_int, [_vp, _c.c_void_p, _c.c_size_t])

_lib_mk_selftest_sync = _sig("mk_selftest_sync", _c.c_int,
                             [_c.c_int32, _c.c_int32, _c.POINTER(_c.c_double)])

_lib_mk_decode_step_noalloc = _sig("mk_decode_step_noalloc", _c.c_int,
                                   [_c.POINTER(mk_layer_config), _c.POINTER(mk_layer_weights),
                                    _c.POINTER(mk_step_io), _vp])

EXPORTED = ["mk_layer_create", "mk_decode_step", "mk_decode_step_noalloc", "mk_layer_status", "mk_layer_clear_status",
            "mk_layer_destroy", "mk_stack_create", "mk_stack_step", "mk_stack_status",
            "mk_stack_destroy", "mk_status_string", "mk_layer_get_info", "mk_get_timestamps",
            "mk_layer_prefetch_stats", "mk_stack_prefetch_stats",
            "mk_selftest_quantize", "mk_selftest_mma", "mk_selftest_sync"]


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, st):
    if st != MK_OK:
        raise MkError(fn, st)


def mk_status_string(status):
    return _lib_mk_status_string(int(status)).decode()


def make_config(wl, flags=0, max_ctx=None, timeout_ns=0, window=None, prefetch_experts=None):
    """mk_layer_config from a workload/layer shape dict.  prefetch_experts:
    experts of the previous step prefetched into L2 (MoE; None = 0, off)."""
    c = mk_layer_config()
    c.hidden = wl["hidden"]
    c.n_q_heads = wl["n_q_heads"]
    c.n_kv_heads = wl["n_kv_heads"]
    c.head_dim = wl["head_dim"]
    c.window = wl["window"] if window is None else window
    if wl["ffn"] == "moe":
        c.ffn_kind = MK_FFN_MOE_NVFP4
        c.n_experts, c.top_k = wl["n_experts"], wl["top_k"]
        c.pooled_dim, c.expert_inter = wl["pooled_dim"], wl["expert_inter"]
    else:
        c.ffn_kind = MK_FFN_DENSE_SWIGLU_BF16
        c.dense_inter = wl["dense_inter"]
    c.max_tokens = 16
    c.max_ctx = max_ctx if max_ctx is not None else wl["ctx"] + 16
    c.rms_eps = 1e-6
    c.flags = flags
    if prefetch_experts is None:
        prefetch_experts = 0
    c.prefetch_experts = prefetch_experts
    c.wait_timeout_ns = timeout_ns
    return c


def mk_layer_create(cfg, weights):
    """cfg: mk_layer_config; weights: dict name -> tensor (missing = NULL)."""
    w = mk_layer_weights()
    for n in _WEIGHT_FIELDS:
        setattr(w, n, _ptr(weights.get(n)))
    h = _vp()
    _check("mk_layer_create", _lib_mk_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)))
    return h.value


def _tree(io, tree_mask):
    """Host array of the token-tree masks (kept alive with the io struct)."""
    if tree_mask is None:
        return
    arr = (ctypes.c_uint16 * len(tree_mask))(*[int(m) for m in tree_mask])
    io.tree_mask = ctypes.cast(arr, ctypes.POINTER(ctypes.c_uint16))
    io._tree = arr


def make_step_io(T, ctx, x_in, x_out, k_cache, v_cache, q_in=None, next_k_cache=None,
                 next_v_cache=None, q_out=None, topk_idx_out=None, topk_w_out=None, tree_mask=None):
    """tree_mask: optional list of T ancestor-or-self bitmasks (token tree)."""
    io = mk_step_io()
    io.n_tokens, io.ctx_len = T, ctx
    io.x_in, io.x_out, io.q_in = _ptr(x_in), _ptr(x_out), _ptr(q_in)
    io.k_cache, io.v_cache = _ptr(k_cache), _ptr(v_cache)
    io.next_k_cache, io.next_v_cache, io.q_out = _ptr(next_k_cache), _ptr(next_v_cache), _ptr(q_out)
    io.topk_idx_out, io.topk_w_out = _ptr(topk_idx_out), _ptr(topk_w_out)
    _tree(io, tree_mask)
    return io


def mk_decode_step(layer, io, stream=None):
    _check("mk_decode_step", _lib_mk_decode_step(layer, ctypes.byref(io), _stream(stream)))


def mk_decode_step_noalloc(cfg, weights, io, stream=None):
    """One decode step without any device allocation (scratch in the
    library's fixed static array; small layers only)."""
    w = mk_layer_weights()
    for n in _WEIGHT_FIELDS:
        setattr(w, n, _ptr(weights.get(n)))
    _check("mk_decode_step_noalloc", _lib_mk_decode_step_noalloc(
        ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(io), _stream(stream)))


def mk_layer_status(layer):
    return _lib_mk_layer_status(layer)


def mk_layer_clear_status(layer):
    _check("mk_layer_clear_status", _lib_mk_layer_clear_status(layer))


def mk_layer_destroy(layer):
    _lib_mk_layer_destroy(layer)


def mk_layer_get_info(layer):
    info = mk_layer_info()
    _check("mk_layer_get_info", _lib_mk_layer_get_info(layer, ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in mk_layer_info._fields_}


def mk_stack_create(layers):
    arr = (_vp * len(layers))(*layers)
    h = _vp()
    _check("mk_stack_create", _lib_mk_stack_create(arr, len(layers), ctypes.byref(h)))
    return h.value


def make_stack_io(T, ctx, x_in, x_out, k_caches, v_caches, topk_idx_out=None, topk_w_out=None,
                  tree_mask=None):
    io = mk_stack_io()
    io.n_tokens, io.ctx_len = T, ctx
    io.x_in, io.x_out = _ptr(x_in), _ptr(x_out)
    kc = (_vp * len(k_caches))(*[_ptr(t) for t in k_caches])
    vc = (_vp * len(v_caches))(*[_ptr(t) for t in v_caches])
    io.k_caches = ctypes.cast(kc, ctypes.POINTER(_vp))
    io.v_caches = ctypes.cast(vc, ctypes.POINTER(_vp))
    io._keep = (kc, vc)
    io.topk_idx_out, io.topk_w_out = _ptr(topk_idx_out), _ptr(topk_w_out)
    _tree(io, tree_mask)
    return io


def mk_stack_step(stack, io, stream=None):
    _check("mk_stack_step", _lib_mk_stack_step(stack, ctypes.byref(io), _stream(stream)))


def mk_stack_status(stack):
    return _lib_mk_stack_status(stack)


def _stats_dict(st):
    return {f: int(getattr(st, f)) for f, _ in mk_prefetch_stats._fields_}


def mk_layer_prefetch_stats(layer):
    st = mk_prefetch_stats()
    _check("mk_layer_prefetch_stats", _lib_mk_layer_prefetch_stats(layer, ctypes.byref(st)))
    return _stats_dict(st)


def mk_stack_prefetch_stats(stack):
    st = mk_prefetch_stats()
    _check("mk_stack_prefetch_stats", _lib_mk_stack_prefetch_stats(stack, ctypes.byref(st)))
    return _stats_dict(st)


def mk_stack_destroy(stack):
    _lib_mk_stack_destroy(stack)


def mk_selftest_quantize(x, codes, scales, s_row, stream=None):
    rows, K = x.shape
    _check("mk_selftest_quantize", _lib_mk_selftest_quantize(
        _ptr(x), rows, K, _ptr(codes), _ptr(scales), _ptr(s_row), _stream(stream)))


def mk_selftest_mma(fp4, a, a_scales, b, b_scales, K, out, stream=None):
    _check("mk_selftest_mma", _lib_mk_selftest_mma(
        int(fp4), _ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales), K, _ptr(out), _stream(stream)))


def mk_get_timestamps(layer, grid):
    """Self-timing stamps of the layer's last step: uint64 array [grid, 10, 16]."""
    import numpy as np
    buf = np.zeros((grid, 10, 16), dtype=np.uint64)
    _check("mk_get_timestamps", _lib_mk_get_timestamps(layer, buf.ctypes.data, buf.size))
    return buf


SYNC_MODES = {"flag_hop": 0, "sentinel_hop": 1, "acquire_poll": 2, "fence": 3}


def mk_selftest_sync(mode, iters=10000):
    """ns per operation of an intra-GPU synchronisation primitive (see mk_selftest.h)."""
    m = SYNC_MODES[mode] if isinstance(mode, str) else mode
    out = _c.c_double()
    _check("mk_selftest_sync", _lib_mk_selftest_sync(m, iters, _c.byref(out)))
    return out.value
