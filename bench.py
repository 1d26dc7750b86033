#!/usr/bin/env python
"""Benchmark of the LegoLink link step (position-independent KV link) at the Llama-3-8B shape.

One step = one pic_link call over one request of the workload (default: 10 compiled
chunks x 512 tokens + a 64-token query, k = 16, bf16, random-init weights): host
metadata, request-private block copies, 32 layers of the selected rows, final norm
and LM head. The chunks are compiled once before timing (compile is reported
separately). Metric: linked prompt tokens per second (chunk + query tokens / link
latency). Inputs (15 GB of weights, 0.68 GB of KV) are far larger than L2.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--config 8b_10x512]

Under torchrun each rank runs an independent replica (requests are independent, so
the link step shards by request with no collective); value = all ranks' tokens / the
slowest rank's time. `--impl reference` times the fp64 CPU oracle on a bounded sample
of the same workload.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import pic_inputs as pi  # noqa: E402

METRIC = "linked prompt tokens/sec (link step, 8B shape)"
UNIT = "tokens/s"

# ncu dram__bytes_read.sum + dram__bytes_write.sum of the tcgen05 GEMM over all its launches of
# one 8B link step (10 x 512 + 64 query, k = 16: 224 rows), per launch: measured on a 2-layer
# model of the same width (every layer's four projections are the same launches), scaled to 32
# layers + the LM head (32 x 475.29 MB + 1051.71 MB over 129 launches), on the kernel source
# whose sha256 prefix is recorded beside it; reported as null once that source changes.
GEMM_TRAFFIC = {"src_sha256_12": "6937abbb0ec2", "bytes_per_launch": 125962442, "shape": "all launches of an 8B 10x512 link step"}


def kernel_sha() -> str:
    p = os.path.join(ROOT, "position_independent_kv_link_gb300", "csrc", "k_gemm_tc.cu")
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:12]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- setup

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def slowest_rank(x: float, world: int, device: str = "cuda") -> float:
    """Max over ranks of a per-rank elapsed time: the whole job's time in a weak-scaled run."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job rate: every rank processed units_per_rank; seconds is the slowest rank's time."""
    return world * units_per_rank / seconds


def workload(name: str) -> pi.Workload:
    return pi.config_workloads()[name]


def roofline_link(wl: pi.Workload, pk) -> dict:
    """Roofline of one link: max(weights + KV bytes / HBM, FLOPs / bf16 peak)."""
    sp = wl.spec
    H, G, D = sp.n_heads, sp.n_kv_heads, sp.head_dim
    per_layer_w = (sp.qkv_dim * sp.d_model + sp.d_model * H * D + 3 * sp.d_model * sp.ffn_dim) * 2
    W = sp.n_layers * per_layer_w + sp.vocab * sp.d_model * 2
    kv = 0
    flops_attn = 0.0
    rows = 0
    for r in wl.requests:
        lens = [len(wl.chunks[c]) for c in r.chunk_ids]
        n = sum(lens) + len(r.query)
        kv += n * G * D * 2 * 2 * sp.n_layers
        off = 0
        sel = []
        for L in lens:
            sel += list(range(off, off + min(wl.k, L)))
            off += L
        sel += list(range(off, off + len(r.query)))
        rows += len(sel)
        flops_attn += sum(p + 1 for p in sel) * H * D * 4.0 * sp.n_layers
    flops = 2.0 * rows * (sp.n_layers * per_layer_w / 2) + 2.0 * len(wl.requests) * sp.vocab * sp.d_model + flops_attn
    t_mem = (W + kv) / (pk["hbm_gbs"] * 1e9)
    t_flop = flops / (pk["bf16_tflops_sustained"] * 1e12)   # a link step is a long run of back-to-back GEMMs
    return {"bytes": W + kv, "flops": flops, "t_mem_ms": t_mem * 1e3, "t_flop_ms": t_flop * 1e3,
            "roofline_ms": max(t_mem, t_flop) * 1e3, "bound": "hbm" if t_mem >= t_flop else "tensor",
            "peaks": "HBM copy and sustained dense bf16, measured"}


# ----------------------------------------------------------------------------- CPU oracle (baseline / reference arm)

def oracle_sample(wl: pi.Workload, weights, n_layers: int):
    """Oracle link of the workload restricted to its first n_layers layers.

    Compiled chunk KV is drawn from the seeded generator (the link's cost does not
    depend on its values). Returns (seconds, OracleStore, cids) for repeated timing.
    """
    from oracle import pic_oracle as po
    spec = wl.spec.with_layers(n_layers)
    w = {k: v for k, v in weights.items() if not k.startswith("layers.") or int(k.split(".")[1]) < n_layers}
    model = po.OracleModel(spec, w, cache_all=True)
    need = sum(-(-len(wl.chunks[c]) // 16) for r in wl.requests for c in r.chunk_ids) + 4 * wl.selected_rows // 16 + 64
    st = po.OracleStore(model, need)
    cids = {}
    for c in sorted({c for r in wl.requests for c in r.chunk_ids}):
        k, v = pi.gen_chunk_kv(spec, len(wl.chunks[c]), c)
        cids[c] = st.import_chunk(wl.chunks[c], [k[l] for l in range(n_layers)], [v[l] for l in range(n_layers)])
    for l in range(n_layers):
        model.layer(l)          # upcast once, outside the timed calls
    return model, st, cids


def oracle_link_time(st, cids, wl) -> float:
    t0 = time.perf_counter()
    out = st.link([([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests], wl.k)
    dt = time.perf_counter() - t0
    for rid in list(st.requests):
        st.release_request(rid)
    for c in cids.values():
        st.chunks[c].refs = max(st.chunks[c].refs, 1)
    del out
    return dt


def cpu_threads() -> int:
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max((i.get("num_threads", 0) for i in info if i.get("user_api") == "blas"), default=0)
        if n:
            return n
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    wl = workload(args.config)
    n_layers = args.cpu_layers
    weights = pi.gen_weights(wl.spec, layers=range(n_layers))
    model, st, cids = oracle_sample(wl, weights, n_layers)
    # A step is the oracle link of the workload through its first n_layers layers (+ final norm
    # and LM head): n_layers / all of a link step's work, so it counts that share of the step's
    # linked tokens. ms_per_step is the measured time of that step.
    frac = n_layers / wl.spec.n_layers
    for _ in range(args.warmup):
        oracle_link_time(st, cids, wl)
    ts = [oracle_link_time(st, cids, wl) for _ in range(args.steps)]
    step_s = statistics.mean(ts)
    tokens = wl.linked_tokens
    value = tokens * frac / step_s
    sample = (f"each step: the oracle link of '{wl.name}' over the first {n_layers} of {wl.spec.n_layers} layers "
              f"(+ final norm and LM head), counted as {frac:g} of the step's {tokens} linked tokens; "
              f"chunk KV from the seeded generator; a full step would take ~{step_s / frac:.1f} s")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": wl.name, "k": wl.k, "linked_tokens": tokens, "selected_rows": wl.selected_rows},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def make_store(model, wl, extra_positions=0):
    """A store sized for the workload: its chunks, one private block per chunk per request and
    the query pages (with slack), a private copy of every chunk block, every request's
    positions, and rows for a compile call of 4 chunks behind their dummy prefix (LegoLink-0)."""
    from position_independent_kv_link_gb300 import PicStore
    n_pos = max(sum(len(wl.chunks[c]) for c in r.chunk_ids) + len(r.query) for r in wl.requests)
    chunk_blocks = sum(-(-len(c) // 16) for c in wl.chunks)
    # room for every chunk block made private once (a dynamic-selection link may choose a token
    # in each of them), plus the static links' private and query blocks
    n_blocks = 2 * chunk_blocks + 4 * (wl.selected_rows // 16 + 2 * len(wl.requests) * 10)
    compile_rows = max(sum(len(c) + wl.n_dummy for c in wl.chunks[i:i + 4]) for i in range(0, len(wl.chunks), 4))
    return PicStore(model, num_blocks=n_blocks, max_rows=max(wl.selected_rows, compile_rows, 2048),
                    max_requests=max(len(wl.requests), 64), max_positions=n_pos + 80 + extra_positions,
                    max_logit_rows=max(64, len(wl.requests)))


def compile_all(store, wl):
    """Every chunk of the workload compiled, 4 per call (LegoLink-0 dummies when the workload has them)."""
    cids = []
    for i in range(0, len(wl.chunks), 4):
        cids += store.compile(wl.chunks[i:i + 4], n_dummy=wl.n_dummy)
    store.sync()
    return cids


def kernel_classes(prof, steps):
    """Per-class event times of an instrumented run, per step."""
    return {k: {"ms_per_step": v["ms"] / steps, "launches_per_step": v["launches"] / steps,
                "GBs": v["bytes"] / (v["ms"] / 1e3) / 1e9 if v["ms"] > 0 else None,
                "TFs": v["flops"] / (v["ms"] / 1e3) / 1e12 if v["ms"] > 0 else None}
            for k, v in prof.items() if isinstance(v, dict)}


def attention_roofline(prof, n_layers, pk, steps):
    """The fused-RoPE paged attention (kernel + split merge) against its own floor: the slower of
    its FLOPs (4 per head dim and visible query-key pair) at the sustained bf16 tensor peak (it
    runs inside a long step) and its KV + q + output bytes at the HBM peak. Per step."""
    a = prof.get("attention")
    if not a or a["ms"] <= 0:
        return None
    ms = a["ms"] / steps
    t_flop = a["flops"] / steps / (pk["bf16_tflops_sustained"] * 1e12) * 1e3
    t_mem = a["bytes"] / steps / (pk["hbm_gbs"] * 1e9) * 1e3
    floor = max(t_flop, t_mem)
    return {"bound": "tensor" if t_flop >= t_mem else "hbm", "ms_per_step": ms, "floor_ms": floor,
            "frac": floor / ms, "us_per_layer": ms * 1e3 / n_layers,
            "achieved_tflops": a["flops"] / (a["ms"] / 1e3) / 1e12, "achieved_gbs": a["bytes"] / (a["ms"] / 1e3) / 1e9,
            "peak_tflops": pk["bf16_tflops_sustained"], "peak_gbs": pk["hbm_gbs"],
            "peak_kind": "bf16 dense sustained / HBM copy, measured"}


def measure_config(model, name, pk, steps, warmup):
    """One evaluated configuration: compile its chunks, time `steps` link steps (all requests in
    one pic_link call) after `warmup`, then the same steps under per-launch profiling."""
    wl = workload(name)
    store = make_store(model, wl)
    try:
        cids = compile_all(store, wl)
        reqs = [([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests]

        def step():
            res = store.link(reqs, wl.k)
            for r in res.requests:
                store.release_request(r)
        for _ in range(max(3, warmup)):
            step()
        store.sync()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        store.sync()
        ms = e0.elapsed_time(e1) / steps
        store.profile_begin()
        for _ in range(steps):
            step()
        prof = store.profile_end()
        store.sync()
    finally:
        store.close()
    rl = roofline_link(wl, pk)
    return {"workload": wl.name, "k": wl.k, "requests": len(wl.requests), "linked_tokens": wl.linked_tokens,
            "selected_rows": wl.selected_rows, "steps": steps, "ms_per_step": ms,
            "tokens_per_s": wl.linked_tokens / (ms / 1e3),
            "link_roofline": {"bound": rl["bound"], "roofline_ms": rl["roofline_ms"], "frac": rl["roofline_ms"] / ms,
                              "t_mem_ms": rl["t_mem_ms"], "t_flop_ms": rl["t_flop_ms"]},
            "attention_roofline": attention_roofline(prof, wl.spec.n_layers, pk, steps),
            "kernels": kernel_classes(prof, steps)}


def run_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from position_independent_kv_link_gb300 import PicModel, PicStore

    wl = workload(args.config)
    spec = wl.spec
    pk = peaks()
    t0 = time.time()
    weights = pi.gen_weights(spec)
    t_gen = time.time() - t0
    model = PicModel(spec, weights)
    cpu_weights = weights if (rank == 0 and not args.no_cpu_baseline) else None
    if cpu_weights is None:
        del weights
    store = make_store(model, wl, extra_positions=2 * args.steps)
    # compile every chunk once (timed separately; batches of up to 4 chunks)
    torch.cuda.synchronize()
    c0 = time.perf_counter()
    cids = compile_all(store, wl)
    compile_s = time.perf_counter() - c0
    compiled_tokens = sum(len(c) for c in wl.chunks)

    reqs = [([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests]
    n_q = sum(len(r.query) for r in wl.requests)
    hid = torch.empty((n_q, spec.d_model), dtype=torch.float32, device="cuda")
    lg = torch.empty((len(wl.requests), spec.vocab), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        res = store.link(reqs, wl.k, hidden_out=hid, logits_out=lg)
        for r in res.requests:
            store.release_request(r)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    store.sync()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # timed region: K steps, no instrumentation
    launches0 = store.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    launches = store.launch_count() - launches0
    ms = e0.elapsed_time(e1)
    # the same K steps again with CUDA events around every kernel launch (per-kernel times)
    store.profile_begin()
    for _ in range(args.steps):
        step()
    prof = store.profile_end()
    torch.cuda.synchronize()
    clk = clocks.stop()
    store.sync()
    ms = slowest_rank(ms, world)
    ms_step = ms / args.steps
    tokens = wl.linked_tokens
    value = job_throughput(tokens * args.steps, world, ms / 1e3)

    # end to end through the public API: host query tokens in, hidden + logits to pinned host
    hid_h = torch.empty(hid.shape, dtype=hid.dtype, pin_memory=True)
    lg_h = torch.empty(lg.shape, dtype=lg.dtype, pin_memory=True)
    def e2e_step():
        res = store.link(reqs, wl.k, hidden_out=hid, logits_out=lg)
        hid_h.copy_(hid, non_blocking=True)
        lg_h.copy_(lg, non_blocking=True)
        stream.synchronize()
        for r in res.requests:
            store.release_request(r)
    for _ in range(3):
        e2e_step()
    barrier()
    w0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    w_s = slowest_rank(time.perf_counter() - w0, world)
    e2e_value = job_throughput(tokens * args.steps, world, w_s)
    h2d = sum(4 * (len(r.query) + len(r.chunk_ids)) for r in wl.requests)
    d2h = hid.numel() * 4 + lg.numel() * 4

    dec = time_decode(store, reqs, wl, 3, args.steps, stream, world, barrier)
    dyn = time_dynamic(store, reqs, wl, 15, 3, args.steps, stream, world, barrier)
    cpool = time_compile_pool(model, spec, pk, world, barrier) if spec.n_layers == 32 else None

    rl = roofline_link(wl, pk)
    dec_roof_ms = rl["bytes"] / (pk["hbm_gbs"] * 1e9) * 1e3   # weights + the requests' KV, read once
    dec_ms = dec["ms"]
    n_r = dec["requests"]
    # dominant kernel: the tcgen05 GEMM over ALL its launches of the step (QKV, O, gate/up, down,
    # LM head); achieved = their algorithmic bytes (weights + activations read once, fp32 result
    # written once) / their summed event-timed launch durations
    gl = [prof[k] for k in ("gemm", "gemm_gate_up") if k in prof]
    g_ms, g_bytes, g_n = sum(v["ms"] for v in gl), sum(v["bytes"] for v in gl), sum(v["launches"] for v in gl)
    achieved = g_bytes / (g_ms / 1e3) / 1e9 if g_ms > 0 else None
    traffic = None
    if GEMM_TRAFFIC["src_sha256_12"] == kernel_sha() and GEMM_TRAFFIC.get("shape") == "all launches of an 8B 10x512 link step":
        traffic = GEMM_TRAFFIC["bytes_per_launch"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded random-init weights and uniform token ids)",
        "config": {"workload": wl.name, "k": wl.k, "linked_tokens": tokens, "selected_rows": wl.selected_rows,
                   "l2": "inputs larger than L2 (15 GB weights + 0.68 GB KV per step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "tc_gemm_kernel (tcgen05), all launches of the step: QKV, O, gate/up, "
                                                 "down projections and the LM head",
                     "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": (achieved / pk["hbm_gbs"]) if achieved else None, "traffic": traffic,
                     "algorithmic_bytes_per_launch": g_bytes / g_n if g_n else None,
                     "launches_per_step": g_n / args.steps, "peak_source": pk["source"]},
        "attention_roofline": attention_roofline(prof, spec.n_layers, pk, args.steps),
        "link_roofline": {"roofline_ms": rl["roofline_ms"], "bound": rl["bound"], "measured_ms": ms_step,
                          "frac": rl["roofline_ms"] / ms_step, "bytes": rl["bytes"], "flops": rl["flops"],
                          "t_mem_ms": rl["t_mem_ms"], "t_flop_ms": rl["t_flop_ms"]},
        "kernels_note": "per-kernel times from a second, event-instrumented run of the same steps",
        "kernels": {k: {"ms_per_step": v["ms"] / args.steps, "launches_per_step": v["launches"] / args.steps,
                        "GBs": v["bytes"] / (v["ms"] / 1e3) / 1e9 if v["ms"] > 0 else None,
                        "TFs": v["flops"] / (v["ms"] / 1e3) / 1e12 if v["ms"] > 0 else None}
                    for k, v in prof.items() if isinstance(v, dict)},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk,
        "compile": {"tokens_per_s": compiled_tokens / compile_s, "ms": compile_s * 1e3, "chunks": len(wl.chunks)},
        "compile_pool": cpool,
        "dynamic": {"what": "pic_link_dynamic at r = 15 % (CacheBlend-15, the pages' comparison point): layer-0 "
                            "query attention scores for every prompt token, the top 15 % chosen on the GPU, the "
                            "link over the chosen rows and the query; against the LegoLink-16 step above",
                    **dyn, "static_ms_per_step": ms_step, "ratio_to_static": dyn["ms_per_step"] / ms_step},
        "decode": {"what": "pic_decode after the link: one generated token per request per step, attending to "
                           "the request's linked KV (RoPE inside the attention)",
                   "requests": n_r, "steps": args.steps, "ms_per_step": dec_ms / args.steps,
                   "tokens_per_s": job_throughput(n_r * args.steps, world, dec_ms / 1e3),
                   "roofline_ms": dec_roof_ms, "frac": dec_roof_ms / (dec_ms / args.steps),
                   "bound": "hbm: every weight and the requests' KV read once per step",
                   "gpu_launches_per_step": dec["launches"] / args.steps, "kernels": dec["kernels"]},
        "setup_s": {"weights_gen": t_gen},
    }
    # the other evaluated configurations on the same model (the 8B shape): link throughput, the
    # link roofline and per-class kernel times; the k sweep at k = 16 is the headline workload itself
    if not args.no_configs and spec.n_layers == 32:
        cfgs = {}
        for name, n in (("8b_98x512", 5), ("8b_32req", 5), ("8b_10x512_k0", 10), ("8b_10x512_k2", 10),
                        ("8b_10x512_k32", 10), ("8b_10x512_k512", 5)):
            try:
                cfgs[name] = measure_config(model, name, pk, min(n, args.steps), 3)
            except Exception as e:   # reported in the line, never fatal to it
                cfgs[name] = {"error": repr(e)[:300]}
        cfgs["8b_10x512_k16"] = {"same_as": "the headline workload (8b_10x512)"}
        line["configs"] = cfgs
    if cpu_weights is not None:
        try:
            # the oracle as it stands, on this host's cores: the same sample of the link (its first
            # --cpu-layers layers) repeated until about 10 s of CPU work, the mean scaled to all layers
            n_l = args.cpu_layers
            model_o, st_o, cids_o = oracle_sample(wl, cpu_weights, n_l)
            ts = []
            while sum(ts) < 10.0 and len(ts) < 30:
                ts.append(oracle_link_time(st_o, cids_o, wl))
            t = statistics.mean(ts)
            cpu_step = t * wl.spec.n_layers / n_l
            line["cpu_baseline"] = {
                "value": tokens / cpu_step, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                "sample": f"fp64 oracle link of this workload over the first {n_l} of {spec.n_layers} layers (+ LM head), "
                          f"mean of {len(ts)} runs ({sum(ts):.1f} s of CPU work), {t:.2f} s each, scaled "
                          f"x{spec.n_layers / n_l:g}; chunk KV from the seeded generator"}
        except Exception as e:   # reported in the line, never fatal to it
            line["cpu_baseline"] = {"error": repr(e)[:200], "kind": "oracle"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def time_decode(store, reqs, wl, warmup, steps, stream, world, barrier):
    """Links the workload's requests once, then times `steps` decode steps (one generated token
    per request each, pic_decode over the linked KV) with CUDA events after `warmup` steps, and
    the same number again under the store's per-launch profiling. Releases the requests."""
    spec = wl.spec
    res = store.link(reqs, wl.k)
    n_r = len(res.requests)
    dh = torch.empty((n_r, spec.d_model), dtype=torch.float32, device="cuda")
    dl = torch.empty((n_r, spec.vocab), dtype=torch.float32, device="cuda")
    dtok = pi.gen_tokens((warmup + 2 * steps) * n_r, spec.vocab, 7, "decode").reshape(-1, n_r)
    for i in range(warmup):
        store.decode(res.requests, dtok[i], hidden_out=dh, logits_out=dl)
    store.sync()
    barrier()
    n0 = store.launch_count()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for i in range(steps):
        store.decode(res.requests, dtok[warmup + i], hidden_out=dh, logits_out=dl)
    d1.record(stream)
    torch.cuda.synchronize()
    store.sync()
    barrier()
    ms = slowest_rank(d0.elapsed_time(d1), world)
    launches = store.launch_count() - n0
    store.profile_begin()
    for i in range(steps):
        store.decode(res.requests, dtok[warmup + steps + i], hidden_out=dh, logits_out=dl)
    prof = store.profile_end()
    store.sync()
    for r in res.requests:
        store.release_request(r)
    kernels = {k: {"ms_per_step": v["ms"] / steps, "launches_per_step": v["launches"] / steps,
                   "GBs": v["bytes"] / (v["ms"] / 1e3) / 1e9 if v["ms"] > 0 else None}
               for k, v in prof.items() if isinstance(v, dict)}
    return {"ms": ms, "requests": n_r, "launches": launches, "kernels": kernels}


def time_dynamic(store, reqs, wl, r_percent, warmup, steps, stream, world, barrier):
    """Times `steps` links of the workload's requests with dynamic (attention-based) token
    selection at r % (pic_link_dynamic: the layer-0 scoring pass, the wait for its choice, then
    the link over the chosen rows) after `warmup`, then the same steps under per-launch
    profiling. Every request is released after its step."""
    def step():
        res = store.link_dynamic(reqs, r_percent)
        for h in res.requests:
            store.release_request(h)
        return res
    for _ in range(warmup):
        step()
    store.sync()
    barrier()
    n0 = store.launch_count()
    t0 = time.perf_counter()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for _ in range(steps):
        res = step()
    d1.record(stream)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) * 1e3 / steps
    store.sync()
    barrier()
    ms = slowest_rank(d0.elapsed_time(d1), world) / steps
    launches = (store.launch_count() - n0) / steps
    store.profile_begin()
    for _ in range(steps):
        step()
    prof = store.profile_end()
    store.sync()
    rows = sum(int(r_percent * sum(len(wl.chunks[c]) for c in q.chunk_ids) // 100) + len(q.query)
               for q in wl.requests)
    kernels = {k: {"ms_per_step": v["ms"] / steps, "launches_per_step": v["launches"] / steps}
               for k, v in prof.items() if isinstance(v, dict) and v["launches"] > 0}
    return {"r_percent": r_percent, "ms_per_step": ms, "wall_ms_per_step": wall, "selected_rows": rows,
            "gpu_launches_per_step": launches, "kernels": kernels}


def compile_flops_per_token(spec, L: int) -> float:
    """FLOPs of pic_compile per token of an L-token chunk: every projection of all layers but
    the last, whose QKV alone is needed (its K/V are the last stored rows), plus causal
    attention within the chunk (QK and PV, 4 FLOPs per head dim and visible key)."""
    H, D, d, F = spec.n_heads, spec.head_dim, spec.d_model, spec.ffn_dim
    per_layer = spec.qkv_dim * d + H * D * d + 3 * d * F
    gemm = 2.0 * ((spec.n_layers - 1) * per_layer + spec.qkv_dim * d)
    attn = (L + 1) / 2 * H * D * 4.0 * (spec.n_layers - 1)
    return gemm + attn


def time_compile_pool(model, spec, pk, world, barrier):
    """Batched compile throughput over the chunk pool of the batched workload (64 chunks x 512
    tokens), 4 chunks (2048 rows) per pic_compile call after one warm-up call; every chunk's KV
    stays resident until the end. CUDA events around the 16 timed calls."""
    from position_independent_kv_link_gb300 import PicStore
    wl4 = pi.config_workloads(spec)["8b_32req"]
    pool = wl4.chunks
    L = len(pool[0])
    per_call = 4
    # sized for the batched link as well (HBM use of the shared pool, below)
    n_pos = max(sum(len(pool[c]) for c in r.chunk_ids) + len(r.query) for r in wl4.requests)
    st = PicStore(model, num_blocks=sum(-(-len(c) // 16) for c in pool) + 16 * len(wl4.requests) + 8 * per_call,
                  max_rows=max(per_call * L, wl4.selected_rows), max_requests=max(per_call, len(wl4.requests)),
                  max_positions=n_pos + 16, max_logit_rows=max(64, len(wl4.requests)))
    warm = st.compile(pool[:per_call])
    st.sync()
    for c in warm:
        st.release_chunk(c)
    barrier()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    ids = []
    for i in range(0, len(pool), per_call):
        ids += st.compile_cached(pool[i:i + per_call])[0]
    e1.record(stream)
    torch.cuda.synchronize()
    st.sync()
    barrier()
    ms = slowest_rank(e0.elapsed_time(e1), world)
    hbm = None
    try:   # MEPIC's metric: KV pages resident for the batched workload, shared vs per request
        again, hits = st.compile_cached(pool)             # every chunk is found resident
        res = st.link([([ids[c] for c in r.chunk_ids], r.query) for r in wl4.requests], wl4.k)
        st.sync()
        cs = st.cache_stats()
        unshared = sum(sum(-(-len(pool[c]) // 16) for c in r.chunk_ids) + -(-len(r.query) // 16)
                       for r in wl4.requests)
        hbm = {"workload": wl4.name, "blocks_in_use": cs["blocks_in_use"], "block_bytes": cs["block_bytes"],
               "kv_gb": cs["blocks_in_use"] * cs["block_bytes"] / 1e9,
               "kv_gb_unshared": unshared * cs["block_bytes"] / 1e9,
               "reduction": unshared / cs["blocks_in_use"], "recompile_hits": int(sum(hits)),
               "note": "pool chunks resident once, one private block per chunk per request (k = 16) and the "
                       "query pages; unshared = every request holding its whole prompt's pages"}
        for r in res.requests:
            st.release_request(r)
    except Exception as e:   # reported, never fatal to the benchmark line
        hbm = {"error": repr(e)[:200]}
    st.close()
    tokens = sum(len(c) for c in pool)
    tf = tokens * compile_flops_per_token(spec, L) / (ms / 1e3) / 1e12
    peak = pk["bf16_tflops_sustained"]
    return {"what": "pic_compile_cached of the batched workload's chunk pool, 4 chunks (2048 rows) per call",
            "hbm_use": hbm,
            "chunks": len(pool), "tokens": tokens, "ms": ms, "ms_per_call": ms / (len(pool) // per_call),
            "tokens_per_s": job_throughput(tokens, world, ms / 1e3),
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_kind": "bf16 dense, sustained (a ~0.4 s run of back-to-back GEMMs)",
                         "flops_per_token": compile_flops_per_token(spec, L)}}


def run_compile(args):
    """Compile calls only (for launch lists): the batched workload's chunk pool, 4 chunks (2048
    rows) per pic_compile call; W warm-up calls, then K timed calls. Prints the event-timed call
    and the library's launches per call."""
    from position_independent_kv_link_gb300 import PicModel, PicStore
    torch.cuda.set_device(0)
    spec = workload(args.config).spec
    model = PicModel(spec, pi.gen_weights(spec))
    pool = pi.config_workloads(spec)["8b_32req"].chunks
    per_call, n_calls = 4, max(1, args.warmup) + args.steps
    batch = lambda i: [pool[(per_call * i + j) % len(pool)] for j in range(per_call)]
    st = PicStore(model, num_blocks=n_calls * sum(-(-len(c) // 16) for c in batch(0)) + 8,
                  max_rows=per_call * len(pool[0]), max_requests=per_call, max_positions=len(pool[0]) + 16)
    for i in range(max(1, args.warmup)):
        st.compile(batch(i))
    st.sync()
    n0 = st.launch_count()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        st.compile(batch(max(1, args.warmup) + i))
    e1.record(stream)
    torch.cuda.synchronize()
    st.sync()
    ms = e0.elapsed_time(e1) / args.steps
    tokens = per_call * len(pool[0])
    print(json.dumps({"kernel": "compile", "chunks_per_call": per_call, "tokens_per_call": tokens, "ms_per_call": ms,
                      "tokens_per_s": tokens / (ms / 1e3), "launches_per_call": (st.launch_count() - n0) / args.steps,
                      "steps": args.steps, "warmup": max(1, args.warmup)}), flush=True)
    return 0


def run_decode(args):
    """Decode steps only (for launch lists): compile and link the workload once, then W + K
    decode steps; prints the event-timed step and the library's launches per step."""
    from position_independent_kv_link_gb300 import PicModel, PicStore
    torch.cuda.set_device(0)
    wl = workload(args.config)
    spec = wl.spec
    model = PicModel(spec, pi.gen_weights(spec))
    n_pos = max(sum(len(wl.chunks[c]) for c in r.chunk_ids) + len(r.query) for r in wl.requests)
    chunk_blocks = sum(-(-len(c) // 16) for c in wl.chunks)
    # room for every chunk block made private once (a dynamic-selection link may choose a token
    # in each of them), plus the static links' private and query blocks
    n_blocks = 2 * chunk_blocks + 4 * (wl.selected_rows // 16 + 2 * len(wl.requests) * 10)
    store = PicStore(model, num_blocks=n_blocks, max_rows=max(wl.selected_rows, 2048),
                     max_requests=max(len(wl.requests), 64), max_positions=n_pos + 80 + 2 * args.steps + args.warmup,
                     max_logit_rows=max(64, len(wl.requests)))
    cids = []
    for i in range(0, len(wl.chunks), 4):
        cids += store.compile(wl.chunks[i:i + 4], n_dummy=wl.n_dummy)
    reqs = [([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests]
    d = time_decode(store, reqs, wl, args.warmup, args.steps, torch.cuda.current_stream(), 1, lambda: None)
    print(json.dumps({"kernel": "decode", "workload": wl.name, "requests": d["requests"],
                      "ms_per_step": d["ms"] / args.steps, "launches_per_step": d["launches"] / args.steps,
                      "steps": args.steps, "warmup": args.warmup, "kernels": d["kernels"]}), flush=True)
    return 0


def run_link_only(args):
    """Link steps only (for launch lists and per-kernel captures): compile the workload's chunks,
    then W warm-up and K timed pic_link calls; prints the event-timed step and the launches per
    step. --layers sets the model depth of this run (the 8B width is kept), so that a capture of
    every kernel of a step holds a few GB instead of 16."""
    from position_independent_kv_link_gb300 import PicModel
    torch.cuda.set_device(0)
    spec = workload(args.config).spec
    if args.layers:
        spec = spec.with_layers(args.layers)
    wl = pi.config_workloads(spec)[args.config]
    model = PicModel(spec, pi.gen_weights(spec))
    store = make_store(model, wl)
    cids = compile_all(store, wl)
    reqs = [([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests]

    def step():
        res = store.link(reqs, wl.k)
        for r in res.requests:
            store.release_request(r)
    for _ in range(max(1, args.warmup)):
        step()
    store.sync()
    n0 = store.launch_count()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    store.sync()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"kernel": "link", "workload": wl.name, "layers": spec.n_layers, "ms_per_step": ms,
                      "launches_per_step": (store.launch_count() - n0) / args.steps, "steps": args.steps,
                      "warmup": max(1, args.warmup)}), flush=True)
    return 0


def run_kernel(args):
    """Times one kernel-level call at its shape in the 8B link (for ncu captures and sweeps).

    gemm:      gate/up projection, 28672 x 4096 weights, 224 selected rows (tcgen05).
    attention: the link's paged attention, 10 x 512 chunks + 64 query, k = 16
               (224 query rows, 324 pages, 32 Q / 8 KV heads), fused RoPE; --shape
               n_chunks,k,query_len for other prompts of 512-token chunks.
    """
    import ctypes as C
    from position_independent_kv_link_gb300 import _lib as L, api
    torch.cuda.set_device(0)
    lib = L.load()
    st = torch.cuda.current_stream()
    sp = C.c_void_p(st.cuda_stream)
    g = torch.Generator(device="cuda").manual_seed(0)
    if args.kernel == "gemm":
        N, K, T = (int(x) for x in args.shape.split(",")) if args.shape else (28672, 4096, 224)
        W = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        X = torch.randn(T, K, device="cuda", generator=g).to(torch.bfloat16)
        Y = torch.empty(T, N, device="cuda")
        if not args.unpacked:
            X = X.to(torch.float16)   # the packed (model) path runs fp16 operands
        if args.unpacked:
            call = lambda: L.check(lib.pic_op_gemm(L.PIC_BF16, W.data_ptr(), X.data_ptr(), Y.data_ptr(), N, K, T, sp))
        else:   # the tile layout the model repacks its matrices into
            Wp = api.pack_weight(W)
            del W
            call = lambda: L.check(lib.pic_op_gemm_packed(Wp.data_ptr(), X.data_ptr(), Y.data_ptr(), N, K, T, sp))
        nbytes, flops = N * K * 2 + T * K * 2 + T * N * 4, 2.0 * N * K * T
    else:
        n_chunks, k, qlen = (int(x) for x in args.shape.split(",")) if args.shape else (10, 16, 64)
        lens = [512] * n_chunks
        pblk, ppos, plen, sel, off = [], [], [], [], 0
        for i, Ln in enumerate(lens + [qlen]):
            for j in range(-(-Ln // 16)):
                pblk.append(len(pblk))
                ppos.append(off + 16 * j)
                plen.append(min(16, Ln - 16 * j))
            sel += list(range(off, off + (min(k, Ln) if i < len(lens) else Ln)))
            off += Ln
        i32 = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.int32))
        qpos, blk, pp, pl = i32(sel), i32(pblk), i32(ppos), i32(plen)
        T, n_pages = len(sel), len(pblk)
        Kp = torch.randn(n_pages, 8, 16, 128, device="cuda", generator=g).to(torch.bfloat16)
        Vp = torch.randn(n_pages, 8, 16, 128, device="cuda", generator=g).to(torch.bfloat16)
        q = torch.randn(T, 32, 128, device="cuda", generator=g)
        out = torch.empty(q.shape, dtype=torch.float16, device="cuda")
        rope = api.rope_table(off + 16, 128, 500000.0)
        nb = lib.pic_op_attention_scratch_bytes(T, 32, 8, 128, n_pages)
        scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
        P = lambda a: a.ctypes.data_as(L.PI32)
        call = lambda: L.check(lib.pic_op_attention(L.PIC_BF16, T, 32, 8, 128, q.data_ptr(), P(qpos), Kp.data_ptr(),
                                                    Vp.data_ptr(), P(blk), P(pp), P(pl), n_pages, n_pages,
                                                    rope.data_ptr(), rope.shape[0], out.data_ptr(),
                                                    scratch.data_ptr(), nb, sp))
        pairs = sum(p + 1 for p in sel)
        nbytes, flops = n_pages * 16 * 8 * 128 * 2 * 2 + 2 * T * 32 * 128 * 2, pairs * 32 * 128 * 4.0
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(args.steps):
        call()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"kernel": args.kernel, "shape": args.shape, "ms": ms, "GBs": nbytes / ms / 1e6, "TFs": flops / ms / 1e9,
                      "steps": args.steps}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="8b_10x512",
                    help="tiny, 8b_10x512, 8b_98x512, 8b_32req, 8b_10x512_k{0,2,16,32,512}")
    ap.add_argument("--cpu-layers", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configurations' link measurements")
    ap.add_argument("--kernel", choices=["gemm", "attention", "decode", "compile", "link"], default=None,
                    help="time one kernel-level call at its 8B link shape instead of the link step "
                         "(decode: decode steps after one link of --config; compile: calls of 4 x 512-token "
                         "chunks)")
    ap.add_argument("--shape", default=None, help="gemm N,K,T for --kernel gemm (default 28672,4096,224); "
                                                  "attention n_chunks,k,query_len of 512-token chunks (default 10,16,64)")
    ap.add_argument("--unpacked", action="store_true", help="--kernel gemm on the plain [N][K] layout")
    ap.add_argument("--layers", type=int, default=0, help="--kernel link: model depth of the run (8B width kept)")
    args = ap.parse_args()
    if args.kernel == "decode":
        return run_decode(args)
    if args.kernel == "compile":
        return run_compile(args)
    if args.kernel == "link":
        return run_link_only(args)
    if args.kernel:
        return run_kernel(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
