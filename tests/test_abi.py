"""Host-only checks of the C ABI: the library loads, exports every function
the headers declare, and rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "moe_decode_layer_persistent_gb300", "libmk.so")


def _declared():
    names = set()
    for h in ("mk.h", "mk_selftest.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def test_headers_declare_the_entry_points():
    d = _declared()
    for n in ("mk_layer_create", "mk_decode_step", "mk_stack_step", "mk_layer_status",
              "mk_stack_create", "mk_layer_destroy", "mk_stack_destroy", "mk_status_string"):
        assert n in d


def test_library_exports_every_declared_symbol(lib):
    for name in sorted(_declared()):
        assert hasattr(lib, name), name


def test_binding_exports_match_headers(lib):
    from moe_decode_layer_persistent_gb300 import binding
    assert set(binding.EXPORTED) == _declared()


def test_status_strings(lib):
    from moe_decode_layer_persistent_gb300 import binding
    for code, name in binding.STATUS_NAMES.items():
        assert binding.mk_status_string(code) == name
    assert binding.mk_status_string(99) == "MK_ERR_UNKNOWN"


def test_create_rejects_bad_arguments_without_a_gpu(lib):
    from moe_decode_layer_persistent_gb300 import binding as b
    wl = dict(hidden=256, n_q_heads=4, n_kv_heads=1, head_dim=64, window=0, ffn="moe",
              n_experts=16, top_k=2, pooled_dim=128, expert_inter=128, ctx=128)
    cfg = b.make_config(wl, flags=b.MK_FIRST_LAYER)
    # missing weights
    with pytest.raises(b.MkError) as e:
        b.mk_layer_create(cfg, {})
    assert e.value.status == 1
    fake = {n: 0x10000 for n in b._WEIGHT_FIELDS}
    # unsupported shapes
    for field, value in (("head_dim", 96), ("n_q_heads", 8), ("max_tokens", 17),
                         ("hidden", 200), ("top_k", 9), ("pooled_dim", 96)):
        c2 = b.make_config(wl, flags=b.MK_FIRST_LAYER)
        setattr(c2, field, value)
        with pytest.raises(b.MkError) as e:
            b.mk_layer_create(c2, fake)
        assert e.value.status == 2, field
    # misaligned weight pointer
    bad = dict(fake, w_o=0x10008)
    with pytest.raises(b.MkError) as e:
        b.mk_layer_create(cfg, bad)
    assert e.value.status == 1
    # unknown flag
    c3 = b.make_config(wl, flags=0x80)
    with pytest.raises(b.MkError) as e:
        b.mk_layer_create(c3, fake)
    assert e.value.status == 1
    # expert prefetch count outside 0..16
    for n in (-1, 17):
        c4 = b.make_config(wl, flags=b.MK_FIRST_LAYER, prefetch_experts=n)
        with pytest.raises(b.MkError) as e:
            b.mk_layer_create(c4, fake)
        assert e.value.status == 1, n


def test_null_handles(lib):
    from moe_decode_layer_persistent_gb300 import binding as b
    with pytest.raises(b.MkError):
        b.mk_layer_prefetch_stats(None)
    with pytest.raises(b.MkError):
        b.mk_stack_prefetch_stats(None)
    io = b.make_step_io(1, 0, 0, 0, 0, 0)
    with pytest.raises(b.MkError):
        b.mk_decode_step(None, io)
    assert b.mk_layer_status(None) == 1
    assert b.mk_stack_status(None) == 1
    b.mk_layer_destroy(None)
    b.mk_stack_destroy(None)
    with pytest.raises(b.MkError):
        b.mk_stack_create([])
