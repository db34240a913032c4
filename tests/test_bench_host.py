"""Host arithmetic behind bench.py's numbers (no GPU): the algorithmic bytes of
a layer launch, the kernel-source hash that ties the profiled DRAM traffic to
the code it was measured on, and the expert-prefetch summary."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from moe_decode_layer_persistent_gb300 import synth  # noqa: E402


def _cfg(name):
    return synth.layer_cfg(synth.WORKLOADS[name])


def test_algorithmic_bytes_tiny_layer():
    # T=1, ctx=128, H=256, 4q/1kv, d=64, E=16 top-2, P=I=128, prologue on:
    # QKV 196,608 + o 131,072 + router 8,192 + pooler/unpooler 131,072
    # + 2 experts x 27,648 (+ 12 B of tensor scales each) + KV read (129 rows
    # x 256 B) + KV write (1 row x 256 B) + x in/out (2 x 512 B)
    b = bench.algorithmic_bytes(_cfg("tiny_layer"), 1, 128, 2, True, False)
    want = 196608 + 131072 + 8192 + 131072 + 2 * (27648 + 12) + 129 * 256 + 256 + 1024
    assert b == want


def test_algorithmic_bytes_swa_layer_matches_the_per_unit_figures():
    c = _cfg("swa_layer")
    n_exp = 101
    b = bench.algorithmic_bytes(c, 16, 8192, n_exp, True, False)
    dense = 2 * 6144 * 4096 + 2 * 4096 * 4096 + 2 * 256 * 4096 + 2 * 2 * 2048 * 4096
    per_expert = 3 * (1024 * 2048 // 2 + 1024 * 2048 // 16) + 12  # gate, up, down + tensor scales
    kv_read = 2 * 2 * (8192 + 16 - (8192 - 2048 + 1)) * 8 * 128
    kv_write = 2 * 2 * 16 * 8 * 128
    acts = 2 * 2 * 16 * 4096
    assert per_expert - 12 == 3538944          # the expert size the pages' sizing uses
    assert abs(dense - 119.5e6) < 0.1e6        # "119.5 MB dense (incl. QKV)"
    assert b == dense + n_exp * per_expert + kv_read + kv_write + acts


def test_algorithmic_bytes_global_fused_adds_next_qkv_and_full_kv():
    c = _cfg("global_layer_fused")
    b_fused = bench.algorithmic_bytes(c, 16, 32768, 100, True, True)
    b_plain = bench.algorithmic_bytes(c, 16, 32768, 100, True, False)
    assert b_fused - b_plain == 2 * 6144 * 4096 + 2 * 16 * 2 * 8 * 128
    kv_read = 2 * 2 * (32768 + 16) * 8 * 128
    assert abs(kv_read - 134.2e6) < 0.1e6      # "KV 134.2 MB"


def test_source_hash_ignores_comments_and_layout(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text('int f(int x) { return x + 1; }  // one\n/* block */\nconst char* s = "// kept";\n')
    b.write_text('// other comment\nint f(int x) {\n  return x + 1;\n}\nconst char* s = "// kept";\n')
    c.write_text('int f(int x) { return x + 2; }\nconst char* s = "// kept";\n')
    h = bench.kernel_source_hash
    assert h([str(a)]) == h([str(b)])
    assert h([str(a)]) != h([str(c)])


def test_profiled_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "mk_layer_kernel_w.md").write_text("notes\nsource_hash: abc\ntraffic_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=None: "abc")
    assert bench.profiled_traffic("w") == 123
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=None: "def")
    assert bench.profiled_traffic("w") is None
    assert bench.profiled_traffic("missing") is None


def test_expert_prefetch_line():
    a = dict(steps=2, predicted=10, active=100, hits=5)
    b = dict(steps=4, predicted=38, active=300, hits=29)
    d = bench.expert_prefetch_line(a, b)
    assert d == {"predicted_per_step": 14.0, "hit_rate": 0.12, "precision": round(24 / 28, 4)}
    assert bench.expert_prefetch_line(a, a)["hit_rate"] is None
