"""Benchmark: latency of the persistent decode layer / layer stack on one GPU.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl mk|reference]

Prints ONE JSON line (rank 0).  A step is one decode step of the workload:
one layer launch (single-layer workloads) or one launch per layer (stacks),
16 verify tokens.  value = microseconds per step (device time, CUDA events on
the launching stream, inputs resident in HBM); e2e = the same through the C
ABI with host buffers (pinned H2D of x_in and D2H of x_out inside the timed
region).  roofline: algorithmic bytes of one layer launch (dense weights +
the distinct experts this step routed to + KV read + KV/activation writes)
over the average launch duration, against the measured HBM copy bandwidth.
cpu_baseline: the CPU oracle on a bounded sample of the same workload.
Multi-GPU: replicas only (one independent replica per rank, no collective).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per decode layer & per step (16-token verify); HBM GB/s vs roofline"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        self.path = "/tmp/mk_clocks_%d.csv" % os.getpid()
        q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[2]), max=float(parts[3]), power=float(parts[4]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            if r["hw"].lower() == "active":
                reasons.add("hw_slowdown")
            if r["hwt"].lower() == "active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"].lower() == "active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"].lower() == "active":
                reasons.add("sw_power_cap")
        loaded = [r["sm"] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ replicas
def replica_seed(workload, rank):
    """Seed of rank `rank`'s inputs: replicas run independent problems."""
    from moe_decode_layer_persistent_gb300 import synth
    return synth.SEED_BASE + synth.WORKLOADS[workload]["index"] + 1000 * rank


def max_over_ranks(x, device):
    """The slowest rank's time (every rank gets it)."""
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def expert_prefetch_line(a, b):
    """Expert-prefetch statistics of the timed steps: hit_rate = share of the
    active experts that were prefetched, precision = share of the prefetched
    experts that were active."""
    d = {k: b[k] - a[k] for k in b}
    return {"predicted_per_step": round(d["predicted"] / max(d["steps"], 1), 2),
            "hit_rate": round(d["hits"] / d["active"], 4) if d["active"] else None,
            "precision": round(d["hits"] / d["predicted"], 4) if d["predicted"] else None}


# ------------------------------------------------------------------ ncu traffic
def _code_only(text):
    """C++ source without comments and whitespace (string literals kept)."""
    import re
    pat = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"', re.S)
    text = pat.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return "".join(text.split())


def kernel_source_hash(files=None):
    """Hash of the kernel sources' code (comments and layout do not count)."""
    import glob
    import hashlib
    if files is None:
        files = sorted(glob.glob(os.path.join(ROOT, "moe_decode_layer_persistent_gb300", "csrc", "*")))
    h = hashlib.sha256()
    for f in files:
        h.update(_code_only(open(f, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def profiled(workload):
    """Figures per launch from the committed ncu summary of this workload
    (profiles/mk_layer_kernel_<workload>.md): DRAM bytes read + written
    (traffic_bytes_per_launch) and the tensor pipe's share of the launch's
    cycles (tensor_pipe), or {} when there is none or the kernel sources
    changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "mk_layer_kernel_%s.md" % workload)
    if not os.path.exists(path):
        return {}
    fields = {}
    for ln in open(path):
        if ":" in ln:
            k, v = ln.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("source_hash") != kernel_source_hash():
        return {}
    out = {}
    if "traffic_bytes_per_launch" in fields:
        out["traffic_bytes_per_launch"] = int(fields["traffic_bytes_per_launch"])
    if "tensor_pipe" in fields:
        out["tensor_pipe"] = fields["tensor_pipe"]
    return out


def profiled_traffic(workload):
    """DRAM bytes (read + write) per launch from the committed ncu summary, or
    None (see profiled)."""
    return profiled(workload).get("traffic_bytes_per_launch")


# ------------------------------------------------------------------ workloads
def algorithmic_bytes(c, T, ctx, n_experts_touched, first, fuse):
    """Bytes one layer launch must move at least (weights read once, KV read
    once, new rows and activations written once)."""
    H, Hq, Hkv, d = c["hidden"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"]
    nqkv = (Hq + 2 * Hkv) * d
    b = 2 * H * Hq * d                              # o-proj
    if first:
        b += 2 * nqkv * H
    if fuse:
        b += 2 * nqkv * H + 2 * T * 2 * Hkv * d     # next QKV + next K/V rows
    if c["ffn"] == "moe":
        E, P, I = c["n_experts"], c["pooled_dim"], c["expert_inter"]
        b += 2 * E * H + 2 * P * H + 2 * H * P       # router, pooler, unpooler
        per_expert = 2 * (I * P // 2 + I * P // 16) + (P * I // 2 + P * I // 16) + 12
        b += n_experts_touched * per_expert
    else:
        F = c["dense_inter"]
        b += 2 * 3 * F * H
    lo = max(0, ctx - c["window"] + 1) if c["window"] else 0
    b += 2 * 2 * (ctx + T - lo) * Hkv * d           # K and V rows read
    b += 2 * 2 * T * Hkv * d                        # K and V rows written
    b += 2 * 2 * T * H + (0 if first else 2 * T * Hq * d)   # x in/out, q in
    return b


def build_layers(B, work, prefetch_experts=None, prefetch_next_kv=False):
    cfgs, Ws = work["cfgs"], work["Ws"]
    L = len(Ws)
    max_ctx = work["caches"][0][0].shape[0]
    layers = []
    for l in range(L):
        fuse = l + 1 < L or (L == 1 and work["next"] is not None)
        flags = (B.MK_FIRST_LAYER if l == 0 else 0) | (B.MK_FUSE_NEXT_QKV if fuse else 0)
        if prefetch_next_kv and l + 1 < L:
            flags |= B.MK_PREFETCH_NEXT_KV
        cfg = B.make_config(cfgs[l], flags=flags, max_ctx=max_ctx, prefetch_experts=prefetch_experts)
        wd = dict(Ws[l])
        nxt = Ws[l + 1] if l + 1 < L else work["next"]
        if fuse:
            wd["next_attn_norm_w"], wd["next_w_qkv"] = nxt["attn_norm_w"], nxt["w_qkv"]
        layers.append(B.mk_layer_create(cfg, wd))
    return layers


class Runner:
    """Holds the device state of one replica and runs steps."""

    def __init__(self, B, work, stream, prefetch_experts=None, prefetch_next_kv=False):
        self.B, self.work, self.stream = B, work, stream
        wl = work["wl"]
        self.T, self.ctx = wl["T"], wl["ctx"]
        self.layers = build_layers(B, work, prefetch_experts, prefetch_next_kv)
        self.L = len(self.layers)
        self.stack = B.mk_stack_create(self.layers) if self.L > 1 else None
        self.kcs = [c[0] for c in work["caches"]]
        self.vcs = [c[1] for c in work["caches"]]
        self.x_in = work["x_in"].contiguous()
        self.x_out = torch.zeros_like(self.x_in)
        k = wl.get("top_k", 0)
        self.moe = wl["ffn"] == "moe"
        self.idx = torch.zeros((self.L, self.T, max(k, 1)), dtype=torch.int32, device="cuda")
        if self.L == 1:
            nx = work["next"]
            self.q_out = torch.zeros((self.T, wl["n_q_heads"] * wl["head_dim"]),
                                     dtype=torch.bfloat16, device="cuda") if nx else None
            self.io = B.make_step_io(self.T, self.ctx, self.x_in, self.x_out, self.kcs[0], self.vcs[0],
                                     next_k_cache=nx["k_cache"] if nx else None,
                                     next_v_cache=nx["v_cache"] if nx else None, q_out=self.q_out,
                                     topk_idx_out=self.idx[0] if self.moe else None)
        else:
            self.io = B.make_stack_io(self.T, self.ctx, self.x_in, self.x_out, self.kcs, self.vcs,
                                      topk_idx_out=self.idx if self.moe else None)

    @property
    def launches_per_step(self):
        return self.L

    def step(self):
        if self.stack is not None:
            self.B.mk_stack_step(self.stack, self.io, self.stream)
        else:
            self.B.mk_decode_step(self.layers[0], self.io, self.stream)

    def status(self):
        return self.B.mk_stack_status(self.stack) if self.stack is not None else \
            self.B.mk_layer_status(self.layers[0])

    def drift(self, gen, mode="drift"):
        """Next step's input of a MoE workload.  drift: x <- 0.9 x + sqrt(0.19) n,
        n ~ N(0, 1), so that consecutive steps route partly alike (the previous
        step's most-used experts are the prefetch's prediction); independent:
        x <- n; fixed: unchanged."""
        if not self.moe or mode == "fixed":
            return
        n = torch.randn(self.x_in.shape, generator=gen, device="cuda", dtype=torch.float32)
        a = 0.9 if mode == "drift" else 0.0
        self.x_in.copy_((a * self.x_in.float() + (1.0 - a * a) ** 0.5 * n).to(torch.bfloat16))

    def experts_touched(self, hist=None):
        """Distinct experts per layer, averaged over the recorded steps."""
        if not self.moe:
            return [0] * self.L
        h = (self.idx[None] if hist is None else hist).cpu().numpy()
        return [float(np.mean([len(set(h[i, l].ravel().tolist())) for i in range(h.shape[0])]))
                for l in range(self.L)]

    def prefetch_stats(self):
        if self.stack is not None:
            return self.B.mk_stack_prefetch_stats(self.stack)
        return self.B.mk_layer_prefetch_stats(self.layers[0])

    def close(self):
        if self.stack is not None:
            self.B.mk_stack_destroy(self.stack)
        for lay in self.layers:
            self.B.mk_layer_destroy(lay)


def cpu_baseline(work, samples_layers):
    """Oracle wall time on the host cores for a bounded sample: the listed
    layers of the workload (single tokens of work are not sampled: every
    sampled layer runs all 16 verify tokens).  Returns seconds per sampled
    layer."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle_io as oio
    from oracle import layer as ol
    out = {}
    for l in samples_layers:
        c = work["cfgs"][l]
        Wn = oio.np_weights(work["Ws"][l])
        kc, vc = (oio.np64(t) for t in work["caches"][l])
        x = oio.np64(work["x_in"])
        q = None
        if l > 0:  # a non-first layer needs q: use the layer's own QKV as the sample input
            q, kn, vn = ol.qkv_project(x, Wn["attn_norm_w"], Wn["w_qkv"], c["n_q_heads"],
                                       c["n_kv_heads"], c["head_dim"])
            ctx = work["wl"]["ctx"]
            kc[ctx:ctx + x.shape[0]], vc[ctx:ctx + x.shape[0]] = kn, vn
        t0 = time.perf_counter()
        ol.layer_forward(oio.oracle_cfg(c), Wn, x, kc, vc, work["wl"]["ctx"], q_in=q,
                         first_layer=(l == 0))
        out[l] = time.perf_counter() - t0
    return out


def per_step_from_layer_sample(work, tl):
    """Per-step oracle time of a workload from sampled layer times: each layer
    takes the time of the sampled layer of its attention kind (sliding window
    or global)."""
    L = len(work["cfgs"])
    kind = {l: work["cfgs"][l]["window"] == 0 for l in tl}
    total = 0.0
    for l in range(L):
        g = work["cfgs"][l]["window"] == 0
        same = [tl[s] for s in tl if kind[s] == g] or list(tl.values())
        total += sum(same) / len(same)
    return total


def host_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def percentiles(ms):
    """median, p10, p90 and mean of per-step times (ms) -> microseconds."""
    a = np.asarray(ms, dtype=np.float64) * 1e3
    return dict(median=round(float(np.median(a)), 3), p10=round(float(np.percentile(a, 10)), 3),
                p90=round(float(np.percentile(a, 90)), 3), mean=round(float(np.mean(a)), 3))


def timed_steps(R, steps, warmup, gen, inputs, stream, flush, hist=None):
    """`warmup` untimed steps, then `steps` steps each bracketed by CUDA events
    on the launching stream.  Single-layer workloads flush L2 (a 512 MB
    write) before every step, outside its events.  MoE inputs move between
    steps as `inputs` says (outside the events).  Returns per-step ms."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            R.drift(gen, inputs)
            if flush is not None:
                flush.fill_(1.0)
            R.step()
    torch.cuda.synchronize()
    st = R.status()
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            R.drift(gen, inputs)
            if flush is not None:
                flush.fill_(float(i))
            evs[i][0].record(stream)
            R.step()
            evs[i][1].record(stream)
            if hist is not None:
                hist[i].copy_(R.idx)
    torch.cuda.synchronize()
    st = R.status()
    if st != 0:
        raise RuntimeError("device status %d in timed steps" % st)
    return [a.elapsed_time(b) for a, b in evs]


def launch_bytes(work, R, touched):
    """Algorithmic bytes of each layer launch of one step."""
    first = [l == 0 for l in range(R.L)]
    fuse = [(l + 1 < R.L) or (R.L == 1 and work["next"] is not None) for l in range(R.L)]
    return [algorithmic_bytes(work["cfgs"][l], R.T, R.ctx, touched[l], first[l], fuse[l])
            for l in range(R.L)]


def prefetch_hit_rate_host(hist, n):
    """Share of each step's active experts that the previous step's n most-used
    experts cover (the prediction the expert prefetch fetches), per layer,
    averaged: computed from recorded routing, for any input sequence."""
    h = hist.cpu().numpy()
    hits = act = 0
    for i in range(1, h.shape[0]):
        for l in range(h.shape[1]):
            prev = h[i - 1, l].ravel()
            cnt = np.bincount(prev, minlength=256)
            order = sorted(range(len(cnt)), key=lambda e: (-cnt[e], e))
            pred = {e for e in order[:n] if cnt[e] > 0}
            a = set(h[i, l].ravel().tolist())
            hits += len(a & pred)
            act += len(a)
    return round(hits / act, 4) if act else None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="moe_stack")
    ap.add_argument("--layers", type=int, default=None,
                    help="stacks: run only the first N layers (a short stack for profiling)")
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the secondary measurements (single SWA layer, expert-prefetch variants)")
    ap.add_argument("--inputs", default="drift", choices=["drift", "independent", "fixed"],
                    help="MoE inputs between steps: x <- 0.9x + 0.436n (drift), a fresh "
                         "draw (independent) or the same x (fixed)")
    ap.add_argument("--prefetch-next-kv", type=int, default=0,
                    help="stacks: 1 = each layer fetches the next layer's old KV rows into L2 "
                         "during its last weight phases (MK_PREFETCH_NEXT_KV)")
    ap.add_argument("--prefetch-experts", type=int, default=None,
                    help="MoE: experts of the previous step prefetched into L2 (default 0: "
                         "off, measured faster on these inputs)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "mk" else "gloo")
    from moe_decode_layer_persistent_gb300 import synth

    if args.impl == "reference":
        return run_reference(args, rank, world)

    torch.cuda.set_device(local_rank)
    from moe_decode_layer_persistent_gb300 import binding as B
    # each replica draws its own inputs (seed offset by rank)
    work = synth.make_workload(args.workload, device="cuda", seed=replica_seed(args.workload, rank),
                               layers=args.layers)
    stream = torch.cuda.Stream()
    R = Runner(B, work, stream, prefetch_experts=args.prefetch_experts,
               prefetch_next_kv=bool(args.prefetch_next_kv))
    wl = work["wl"]
    single = R.L == 1
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    gen = torch.Generator(device="cuda")
    gen.manual_seed(replica_seed(args.workload, rank) + 7)
    hist = torch.zeros((args.steps,) + tuple(R.idx.shape), dtype=torch.int32, device="cuda")

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    pf0 = R.prefetch_stats() if R.moe else None
    t_wall0 = time.perf_counter()
    ms = timed_steps(R, args.steps, args.warmup, gen, args.inputs, stream,
                     flush if single else None, hist)
    t_wall = time.perf_counter() - t_wall0
    pf1 = R.prefetch_stats() if R.moe else None
    if world > 1:
        torch.distributed.barrier()
    ck = clocks.stop()
    pc = percentiles(ms)
    ms_step = pc["median"] / 1e3
    ms_mean = pc["mean"] / 1e3
    if world > 1:
        ms_step = max_over_ranks(ms_step, "cuda")
        ms_mean = max_over_ranks(ms_mean, "cuda")

    # e2e: host buffers, pinned H2D of x_in and D2H of x_out inside every
    # step's events; the L2 flush (single-layer workloads) stays outside them
    x_host = work["x_in"].cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    evs2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            if single:
                flush.fill_(float(i))
            evs2[i][0].record(stream)
            R.x_in.copy_(x_host, non_blocking=True)
            R.step()
            y_host.copy_(R.x_out, non_blocking=True)
            evs2[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = float(np.median([a.elapsed_time(b) for a, b in evs2]))
    bytes_io = x_host.numel() * x_host.element_size()

    # roofline of the layer kernel (the only kernel of the step): algorithmic
    # bytes per launch over the average launch duration of the timed steps
    touched = R.experts_touched(hist)
    alg = launch_bytes(work, R, touched)
    alg_per_launch = sum(alg) / R.L
    launch_s = ms_mean / 1e3 / R.L
    peak, peak_kind = load_peaks()
    achieved = alg_per_launch / launch_s / 1e9
    prof = profiled(args.workload)

    us_step = ms_step * 1e3
    line = {
        "metric": METRIC, "value": round(us_step, 3),
        "unit": "us/step", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 + nvfp4 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": args.workload, "layers": R.L, "T": R.T, "ctx": R.ctx,
                   "hidden": wl["hidden"], "ffn": wl["ffn"],
                   "prefetch_next_kv": bool(args.prefetch_next_kv) and R.L > 1,
                   "l2": "flushed between steps (512 MB write)" if single else
                         "inputs larger than L2 (%.1f GB read per step)" % (sum(alg) / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "statistic": "median of the timed steps",
        "us_per_step": pc,
        "us_per_layer": round(us_step / R.L, 3),
        "experts_touched_mean": round(float(np.mean(touched)), 2) if R.moe else None,
        "inputs": ({"drift": "x_{s+1} = 0.9 x_s + 0.436 n_s per step (consecutive steps route partly alike)",
                    "independent": "a fresh x_in per step",
                    "fixed": "the same x_in every step"}[args.inputs]
                   if R.moe else "the same x_in every step"),
        "expert_prefetch": expert_prefetch_line(pf0, pf1) if R.moe else None,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_of_8TBs": round(achieved / 8000.0, 4),
                     "algorithmic_bytes_per_launch": int(alg_per_launch),
                     "launch_us_mean": round(launch_s * 1e6, 3),
                     "traffic": prof.get("traffic_bytes_per_launch"),
                     "tensor_pipe": prof.get("tensor_pipe")},
        "e2e": {"value": round(e2e_ms * 1e3, 3), "unit": "us/step",
                "h2d_bytes_per_step": bytes_io, "d2h_bytes_per_step": bytes_io},
        "gpu_launches": args.steps * R.launches_per_step,
        "timed_wall_s": round(t_wall, 4),
        "clocks": ck,
    }

    if R.moe and not single and not args.no_extras:
        # the expert prefetch of the pages (the previous step's 14 most-used
        # experts into L2) on both input sequences, on the same weights
        var = {}
        for inputs in ("drift", "independent"):
            Rv = Runner(B, work, stream, prefetch_experts=14)
            hv = torch.zeros((10,) + tuple(Rv.idx.shape), dtype=torch.int32, device="cuda")
            a0 = Rv.prefetch_stats()
            mv = timed_steps(Rv, 10, 3, gen, inputs, stream, None, hv)
            a1 = Rv.prefetch_stats()
            var[inputs] = dict(us_per_step=percentiles(mv), prefetch=expert_prefetch_line(a0, a1),
                               host_hit_rate_of_prediction=prefetch_hit_rate_host(hv, 14))
            Rv.close()
        line["expert_prefetch_14"] = var
        line["expert_prefetch_14"]["note"] = ("prefetch on; the headline runs with it off "
                                              "(prefetch_experts=0)")
    if not args.no_extras:
        # intra-GPU synchronisation costs (the pages measure the cross-GPU ones)
        line["sync_ns"] = {m: round(B.mk_selftest_sync(m, 20000), 1) for m in B.SYNC_MODES}
    if not single and not args.no_extras and args.workload == "moe_stack":
        # config 2 per layer: one sliding-window layer, L2 flushed between steps
        sw = synth.make_workload("swa_layer", device="cuda", seed=replica_seed("swa_layer", rank))
        Rs = Runner(B, sw, stream)
        hs = torch.zeros((args.steps,) + tuple(Rs.idx.shape), dtype=torch.int32, device="cuda")
        msw = timed_steps(Rs, args.steps, args.warmup, gen, "drift", stream, flush, hs)
        psw = percentiles(msw)
        asw = launch_bytes(sw, Rs, Rs.experts_touched(hs))[0]
        gsw = asw / (psw["mean"] * 1e-6) / 1e9
        line["swa_layer"] = {"us": psw, "algorithmic_bytes": int(asw),
                             "achieved_gbs": round(gsw, 1), "frac": round(gsw / peak, 4),
                             "l2": "flushed between steps (512 MB write)"}
        Rs.close()
        del sw

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        samples = [0] if R.L == 1 else sorted({0, next(l for l in range(R.L) if work["cfgs"][l]["window"] == 0)})
        tl = cpu_baseline(work, samples)
        per_step = per_step_from_layer_sample(work, tl)
        if R.L == 1:
            sample = "layer 0 of %s, all %d tokens (the whole step)" % (args.workload, R.T)
        else:
            sample = ("layers %s of %s (all %d tokens each), scaled to %d layers by window kind"
                      % (samples, args.workload, R.T, R.L))
        line["cpu_baseline"] = {"value": round(per_step * 1e6, 1), "unit": "us/step",
                                "cores": host_threads(), "kind": "oracle", "sample": sample}
    R.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle as the reference arm, on the host cores: each timed step is
    one whole layer of the workload (all verify tokens), taking the
    workload's layer kinds in turn (first layer, then the first global one);
    `value` is the per-step time of the whole workload built from the
    measured layer times by kind, `ms_per_step` the mean measured sample."""
    if rank != 0:
        return
    from moe_decode_layer_persistent_gb300 import synth
    L = synth.WORKLOADS[args.workload]["layers"]
    work = synth.make_workload(args.workload, device="cpu", layers=min(L, 4))
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    full_cfgs = [synth.layer_cfg(work["wl"], l) for l in range(L)]
    kinds = sorted({0} | ({next(l for l in range(len(work["cfgs"])) if work["cfgs"][l]["window"] == 0)}
                          if any(c["window"] == 0 for c in work["cfgs"]) and L > 1 else set()))
    # a bounded run: at most 10 timed layers and 1 warm-up
    steps = min(args.steps, 10)
    warm = min(args.warmup, 1)
    for i in range(warm):
        cpu_baseline(work, [kinds[i % len(kinds)]])
    times = {k: [] for k in kinds}
    t0 = time.perf_counter()
    for i in range(steps):
        l = kinds[i % len(kinds)]
        times[l].append(cpu_baseline(work, [l])[l])
    wall = time.perf_counter() - t0
    tl = {l: float(np.mean(v)) for l, v in times.items() if v}
    per_step = per_step_from_layer_sample(dict(work, cfgs=full_cfgs), tl)
    us = per_step * 1e6
    line = {"metric": METRIC, "value": round(us, 1), "unit": "us/step", "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": round(wall / steps * 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "layers": L, "T": work["wl"]["T"],
                       "ctx": work["wl"]["ctx"]},
            "value_from": "sum over the workload's %d layers of the measured oracle time of a "
                          "layer of the same attention kind (ms_per_step: one measured layer)" % L,
            "cpu_baseline": {"value": round(us, 1), "unit": "us/step", "cores": host_threads(),
                             "kind": "oracle",
                             "sample": "per step: one whole layer (all %d verify tokens) of %s, "
                                       "layers %s in turn" % (work["wl"]["T"], args.workload, kinds)},
            "e2e": {"value": round(us, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
