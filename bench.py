"""Benchmark of the MAC-Attention decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--band-r R] [--amend-band 0|1]

Workloads: gqa_128k_b1_hetero (default), gqa_32k_b8_paged, gqa_4k_b1_contig,
qwen_stack_120k_b4 (48-layer stack, --tau 0.3|0.45), sweep (forced hit rate x
context x batch, MQA and GQA), match_windows (Match latency vs window and GQA
setting), rectification (output error vs reuse gap and band; hit rate and
skipped prefix vs threshold and window) -- the last three print one JSON line
per point.

A step is one MAC decode step (KV append, Match, planning, split-KV
Complete, merge, Amend) for every request of the workload, on inputs already
resident in HBM.  The default workload is the 128K-context one the metric is
quoted on: 1 request x 131072 tokens, 32 q / 8 KV heads, d 128, bf16 paged KV
(page 16, random page permutation), per-head AR(1) rho ~ U[0.5, 0.99], ring
32, r 64, tau 0.3.  KV (537 MB) is larger than L2, so no flush is needed.

Rank 0 prints one JSON line.  N > 1 runs independent replicas (one process
per GPU, no collective on the data path; the path has no exchange step).

--impl reference times the fp64 CPU oracle on the host cores on the same
workload, metric and unit (each step a bounded sample of query heads, scaled
to the whole step).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn us/step & HBM GB/s (frac of 8 TB/s) at 128K ctx; KV bytes read vs full"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
BYTES_PER_KV_TOKEN = 128 * 2 * 2        # K + V, bf16, d = 128, one KV head


def workload(name, band_r, steps):
    from kv_cache_computation_gb300 import workloads as W
    table = {
        "gqa_128k_b1_hetero": lambda: W.llama_gqa_128k_b1_hetero(steps=steps, band_r=band_r),
        "gqa_32k_b8_paged": lambda: W.llama_gqa_32k_b8_paged(steps=steps),
        "gqa_4k_b1_contig": lambda: W.llama_gqa_4k_b1_contig(steps=steps),
    }
    if name not in table:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(table)}")
    return table[name]()


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def launches_per_step(cfg, amend_band):
    """Kernels one decode step launches: Match (after the grid-wide ring scan
    when rings are longer than 32 entries), split-KV attention, Combine, and
    the side-stream Amend when it recomputes the band."""
    wide = cfg.ring_len > 32
    return 3 + (1 if wide else 0) + (1 if amend_band else 0)


def kernel_source_sha(files):
    """First 16 hex digits of the SHA-256 of the kernel sources, concatenated."""
    import hashlib
    h = hashlib.sha256()
    for fn in files:
        with open(fn, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = [os.path.join(ROOT, "kv_cache_computation_gb300", "csrc", f)
                  for f in ("mac_attention.cu", "mac_plan.cuh", "mac_device.cuh", "mac_internal.cuh")]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attention_kernel_128k.json")


def profiled_traffic(kernel_files, path=TRAFFIC_FILE):
    """DRAM bytes per launch of the attention kernel (ncu dram__bytes_read.sum
    + dram__bytes_write.sum) as recorded in the committed capture file, if
    that capture was taken on the current kernel sources; else None."""
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("kernel_source_sha256_16") != kernel_source_sha(kernel_files):
            return None
        return float(rec["traffic_bytes_per_launch"])
    except (OSError, ValueError, KeyError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = str(device_index)
        try:   # nvidia-smi ignores CUDA_VISIBLE_DEVICES: address the GPU by UUID
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            self.idx = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        self.proc = None
        self.path = os.path.join("/tmp", f"mac_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def host_inputs(inp, t, keys=("q_pre", "q_post", "k_new", "v_new")):
    from kv_cache_computation_gb300 import workloads as W
    return [W.bf16_bits(inp[k][t]) for k in keys]


def run_oracle(cfg, K_dev, V_dev, inp, budget_s, max_steps, fixed_steps=None, warm=0):
    """Time the fp64 oracle on the host cores on this workload.

    Calibrates on one whole step, then times either ``fixed_steps`` steps
    (each a sample of query heads sized so the run fits ``budget_s``) or as
    many whole steps as fit ``budget_s`` (2 .. max_steps).  Then one
    full-attention step on all cores and one MAC step on a single core (a
    head sample, scaled).  Returns (us per whole step, OpenMP threads,
    description of the sample, dict of the extra timings and the CPU model)."""
    import oracle
    from kv_cache_computation_gb300 import workloads as W
    B, H = cfg.batch, cfg.heads
    n_need = warm + 3 + (fixed_steps if fixed_steps else max_steps)   # + the full-attention and one-core steps
    t_max = cfg.context + n_need + 1
    Ko = np.zeros((B, t_max, cfg.kv_heads, cfg.head_dim), np.uint16)
    Vo = np.zeros_like(Ko)
    Ko[:, :cfg.context] = W.bf16_bits(K_dev)
    Vo[:, :cfg.context] = W.bf16_bits(V_dev)
    st = oracle.MacState(Ko, Vo, H, cfg.ring_len, cfg.band_r, cfg.tau)
    for b in range(B):
        st.reset(b, cfg.context)
    t = 0
    for _ in range(warm):
        st.step(*host_inputs(inp, t))
        t += 1
    t0 = time.perf_counter()
    st.step(*host_inputs(inp, t))
    full_s = time.perf_counter() - t0
    t += 1
    heads = H
    if fixed_steps:
        n = fixed_steps
        while heads > 1 and n * full_s * heads / H > budget_s:
            heads //= 2
    else:
        n = int(min(max_steps, max(2, budget_s // max(full_s, 1e-9))))
        while heads > 1 and n * full_s * heads / H > budget_s:
            heads //= 2
    t0 = time.perf_counter()
    for _ in range(n):
        st.step(*host_inputs(inp, t), heads=(0, heads))
        t += 1
    el = time.perf_counter() - t0
    us = el / n * 1e6 * (H / heads)
    sample = (f"{n} decode steps of this workload on the fp64 oracle"
              + ("" if heads == H else f", query heads 0..{heads - 1} of {H} per step, scaled x{H // heads} "
                                       "to a whole step")
              + f"; {el:.1f} s of CPU time")
    threads = oracle.num_threads()
    extra = {"cpu_model": cpu_model()}
    # full attention (every head over the whole context), one step on all cores
    t0 = time.perf_counter()
    st.full_step(*host_inputs(inp, t)[1:])
    extra["full_attention_us_per_step"] = round((time.perf_counter() - t0) * 1e6, 1)
    t += 1
    # one core: one MAC step over a sample of heads, scaled
    h1 = max(1, H // 16)
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        st.step(*host_inputs(inp, t), heads=(0, h1))
        extra["single_core_us_per_step"] = round((time.perf_counter() - t0) * 1e6 * H / h1, 1)
        extra["single_core_sample"] = f"one decode step, query heads 0..{h1 - 1} of {H}, scaled x{H // h1}"
    finally:
        oracle.set_num_threads(threads)
    return us, threads, sample, extra


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def graph_time(fn, t0, n, stream, eager=False):
    """us per call of fn(t0..t0+n-1): captured once into a CUDA graph and
    replayed (per-call launches when eager), device events on ``stream``."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    g = None
    if not eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for t in range(t0, t0 + n):
                    fn(t)
        torch.cuda.synchronize()
    e0.record(stream)
    if g is not None:
        g.replay()
    else:
        for t in range(t0, t0 + n):
            fn(t)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / n


def attention_bytes(st, B, H, G):
    """Algorithmic bytes of the attention launches counted in ``st``: 512 B
    per streamed (KV head, token), 256 B of query per head and step, 520 B
    of partial summary per work item and head."""
    return st["kv_tokens_read"] * BYTES_PER_KV_TOKEN + st["steps"] * B * H * 256 + st["work_items"] * G * (128 * 4 + 8)


def method_points(dev, peak, specs, steps=48, warm=4, prof_steps=16, eager=False, on_point=None, plan_mode=0):
    """The MAC step against the in-build full split-KV step (mac_full_step)
    on forced-hit workloads (one handle per (kv_heads, batch, context), the
    same prefill and inputs for both): us/step, KV bytes read vs full, head
    hit rate, and the HBM fraction of the step (KV bytes read / step time)
    and of its attention kernel (algorithmic bytes / event-timed launch,
    from a second pass with events between the kernels)."""
    from kv_cache_computation_gb300 import MacAttention
    from kv_cache_computation_gb300 import workloads as W
    stream = torch.cuda.current_stream()
    res = []
    for kv, B, ctx, rates in specs:
        n_all = warm + steps + prof_steps
        base = W.sweep_point(ctx, B, 0.0, kv, steps=n_all)
        H, G = base.heads, base.group
        max_ctx = ctx + n_all + 2
        mac = MacAttention(H, kv, 128, base.ring_len, base.band_r, base.tau, max_batch=B, max_ctx=max_ctx,
                           page_size=16, plan_mode=plan_mode)
        pt = W.page_tables(B, (max_ctx + 15) // 16, seed=base.seed).to(dev)
        for b in range(B):
            mac.set_page_table(b, pt[b].contiguous())
        Kp, Vp = W.prefill_kv(base, device=dev)
        out = torch.empty((B, H, 128), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)

        def restart():
            mac.sync()
            for b in range(B):
                mac.reset_request(b)
                mac.append_kv(b, Kp[b], Vp[b])
            torch.cuda.synchronize()

        def measure(step, t_warm):
            for t in range(t_warm):
                step(t)
            mac.sync()
            mac.reset_stats()
            us = graph_time(step, t_warm, steps, stream, eager=eager)
            mac.join()
            st = mac.stats()
            mac.reset_stats()
            mac.set_profiling(True)
            for t in range(t_warm + steps, t_warm + steps + prof_steps):
                step(t)
            mac.join()
            torch.cuda.synchronize()
            pr = mac.profile()
            st_p = mac.stats()
            mac.set_profiling(False)
            n_p = max(1, pr["steps"])
            attn_us = pr["attention_ms"] * 1e3 / n_p
            attn_gbs = attention_bytes(st_p, B, H, G) / n_p / (attn_us * 1e-6) / 1e9
            kv_read, kv_full = _kv_bytes(st)
            phases = {k.replace("_ms", ""): round(pr[k] * 1e3 / n_p, 2)
                      for k in ("match_plan_ms", "attention_ms", "combine_ms")}
            phases["work_items"] = round(st_p["work_items"] / n_p, 1)
            # the attention kernel the step ran on (the library picks it per step)
            phases["kernel"] = "tcgen05" if st_p.get("tcgen05_steps", 0) > 0 else "mma.sync"
            return us, st, kv_read, kv_full, attn_us, attn_gbs, phases

        for rate in rates:
            cfg = W.sweep_point(ctx, B, rate, kv, steps=n_all)
            inp = W.decode_inputs(cfg, device=dev)
            restart()
            us, st, kv_read, kv_full, attn_us, attn_gbs, ph = measure(
                lambda t: mac.decode_step(inp["q_pre"][t], inp["q_post"][t], inp["k_new"][t], inp["v_new"][t],
                                          out=out, lse=lse), warm)
            restart()
            f_us, _, f_read, _, f_attn_us, f_attn_gbs, f_ph = measure(
                lambda t: mac.full_step(inp["q_post"][t], inp["k_new"][t], inp["v_new"][t], out=out, lse=lse), warm)
            step_gbs = kv_read / steps / (us * 1e-6) / 1e9
            f_step_gbs = f_read / steps / (f_us * 1e-6) / 1e9
            res.append({"kind": "mqa" if kv == 1 else "gqa", "heads": H, "kv_heads": kv, "batch": B, "context": ctx,
                        "forced_hit": rate, "mac_us_per_step": round(us, 2), "full_us_per_step": round(f_us, 2),
                        "ratio_full_over_mac": round(f_us / us, 3),
                        "kv_bytes_read_vs_full": round(kv_read / max(1, kv_full), 4),
                        "hit_rate": round(st["hits"] / max(1, st["head_decisions"]), 4),
                        "mac_step_hbm_frac": round(step_gbs / peak, 4),
                        "full_step_hbm_frac": round(f_step_gbs / peak, 4),
                        "mac_attention_us": round(attn_us, 2), "mac_attention_frac": round(attn_gbs / peak, 4),
                        "full_attention_us": round(f_attn_us, 2), "full_attention_frac": round(f_attn_gbs / peak, 4),
                        "mac_phase_us": ph, "full_phase_us": f_ph})
            if on_point is not None:
                on_point(res[-1])
        del Kp, Vp
        mac.close()
        torch.cuda.empty_cache()
    return res


def bench_ours(args, ws, rank, local):
    from kv_cache_computation_gb300 import MacAttention
    from kv_cache_computation_gb300 import workloads as W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K_steps, W_steps = args.steps, args.warmup
    total_steps = W_steps + 6 * K_steps + 2
    cfg = workload(args.workload, args.band_r, total_steps)
    B, H, Hkv, G = cfg.batch, cfg.heads, cfg.kv_heads, cfg.group

    Kp, Vp = W.prefill_kv(cfg, device=dev)
    inp = W.decode_inputs(cfg, device=dev)
    max_ctx = cfg.context + total_steps
    page = 16 if cfg.paged else 0
    mac = MacAttention(H, Hkv, cfg.head_dim, cfg.ring_len, cfg.band_r, cfg.tau, max_batch=B, max_ctx=max_ctx,
                       page_size=page, plan_mode=args.plan_mode, amend_band=args.amend_band)
    if page:
        ppr = (max_ctx + 15) // 16
        pt = W.page_tables(B, ppr, seed=cfg.seed).to(dev)
        for b in range(B):
            mac.set_page_table(b, pt[b].contiguous())
    for b in range(B):
        mac.append_kv(b, Kp[b].contiguous(), Vp[b].contiguous())
    out = torch.empty((B, H, cfg.head_dim), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    step_args = lambda t: (inp["q_pre"][t], inp["q_post"][t], inp["k_new"][t], inp["v_new"][t])
    stream = torch.cuda.current_stream()

    # warm-up
    for t in range(W_steps):
        mac.decode_step(*step_args(t), out=out, lse=lse)
    mac.sync()
    torch.cuda.synchronize()
    mac.reset_stats()

    # Timed region: the K-step decode loop, captured once into a CUDA graph
    # (as a serving loop runs it; capture itself is untimed) and replayed;
    # device events on the launching stream.  --eager times per-call launches.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph = None
    if not args.eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for t in range(W_steps, W_steps + K_steps):
                    mac.decode_step(*step_args(t), out=out, lse=lse)
                mac.join()
        torch.cuda.synchronize()
        mac.reset_stats()
    with ClockSampler(local) as clocks:
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for t in range(W_steps, W_steps + K_steps):
                mac.decode_step(*step_args(t), out=out, lse=lse)
            mac.join()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    ms = e0.elapsed_time(e1)
    st = mac.stats()
    clk = clocks.summary()
    ms_max = max_over_ranks(ms, ws, dev)
    us_step = ms_max * 1e3 / K_steps
    del graph

    # the same K steps launched call by call from Python (host-bound when a
    # step's GPU work is shorter than the launch path)
    t_eager = W_steps + K_steps
    torch.cuda.synchronize()
    e0.record(stream)
    for t in range(t_eager, t_eager + K_steps):
        mac.decode_step(*step_args(t), out=out, lse=lse)
    mac.join()
    e1.record(stream)
    torch.cuda.synchronize()
    eager_us = max_over_ranks(e0.elapsed_time(e1), ws, dev) * 1e3 / K_steps

    # per-kernel durations: the next K steps again with CUDA events around
    # every launch (on the stream each kernel runs on); these events sit
    # between the kernels, so this pass is kept out of the headline time
    mac.reset_stats()
    mac.set_profiling(True)
    for t in range(W_steps + 2 * K_steps, W_steps + 3 * K_steps):
        mac.decode_step(*step_args(t), out=out, lse=lse)
    mac.join()
    torch.cuda.synchronize()
    prof = mac.profile()
    mac.set_profiling(False)
    st_p = mac.stats()

    # end to end through the C ABI with host (pinned) buffers: every step one
    # host-to-device copy of its packed inputs and one device-to-host copy of
    # its packed result (out, then lse).  The copies run on a second stream,
    # double-buffered: step i + 1's inputs travel while step i computes, and
    # step i's result returns while step i + 1 computes.
    keys = ("q_pre", "q_post", "k_new", "v_new")
    e2e_first = W_steps + 3 * K_steps
    sizes = [inp[k][0].numel() for k in keys]
    offs = [sum(sizes[:i]) for i in range(len(keys))]
    h_pack = torch.empty((K_steps, sum(sizes)), dtype=torch.bfloat16).pin_memory()
    for i in range(K_steps):
        for k, o, n in zip(keys, offs, sizes):
            h_pack[i, o:o + n] = inp[k][e2e_first + i].reshape(-1).cpu()
    n_out, n_lse = B * H * cfg.head_dim * 2, B * H * 4
    d_pack = [torch.empty(sum(sizes), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    d_in = [[p[o:o + n].view(inp[k][0].shape) for k, o, n in zip(keys, offs, sizes)] for p in d_pack]
    d_res = [torch.empty(n_out + n_lse, dtype=torch.uint8, device=dev) for _ in range(2)]
    out_e = [r[:n_out].view(torch.bfloat16).view(B, H, cfg.head_dim) for r in d_res]
    lse_e = [r[n_out:].view(torch.float32).view(B, H) for r in d_res]
    h_res = torch.empty((K_steps, n_out + n_lse), dtype=torch.uint8).pin_memory()
    cs = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of the buffer's next step have arrived
    ev_done = [torch.cuda.Event() for _ in range(2)]   # the buffer's step has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # the buffer's result has been read back

    def e2e_loop(main):
        cs.wait_stream(main)
        with torch.cuda.stream(cs):
            d_pack[0].copy_(h_pack[0], non_blocking=True)
            ev_in[0].record(cs)
        for i in range(K_steps):
            j = i & 1
            if i + 1 < K_steps:
                with torch.cuda.stream(cs):
                    if i >= 1:
                        cs.wait_event(ev_done[j ^ 1])   # step i - 1 has consumed that buffer
                    d_pack[j ^ 1].copy_(h_pack[i + 1], non_blocking=True)
                    ev_in[j ^ 1].record(cs)
            main.wait_event(ev_in[j])
            if i >= 2:
                main.wait_event(ev_out[j])   # step i - 2's result has left that buffer
            mac.decode_step(*d_in[j], out=out_e[j], lse=lse_e[j], stream=main)
            ev_done[j].record(main)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_done[j])
                h_res[i].copy_(d_res[j], non_blocking=True)
                ev_out[j].record(cs)
        mac.join(stream=main)
        main.wait_stream(cs)

    # like the headline: the loop captured once into a CUDA graph (copies
    # included) and replayed; --eager issues it call by call
    graph = None
    if not args.eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                e2e_loop(cap)
        torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    if graph is not None:
        graph.replay()
    else:
        e2e_loop(stream)
    e3.record(stream)
    torch.cuda.synchronize()
    del graph
    e2e_staged_us = max_over_ranks(e2.elapsed_time(e3), ws, dev) * 1e3 / K_steps
    h2d = sum(sizes) * 2
    d2h = n_out + n_lse

    # end to end through the host-buffer entry point (the call a user with
    # host tensors makes): each step's inputs and results live in their own
    # pinned host buffers, which the step's kernels read and write in place
    # over the host link; captured and replayed like the loops above
    h_first = e2e_first + K_steps
    h_in = [[inp[k][h_first + i].cpu().contiguous().pin_memory() for k in keys] for i in range(K_steps)]
    h_out = [torch.empty((B, H, cfg.head_dim), dtype=torch.bfloat16).pin_memory() for _ in range(K_steps)]
    h_lse = [torch.empty((B, H), dtype=torch.float32).pin_memory() for _ in range(K_steps)]

    def host_loop(main):
        for i in range(K_steps):
            mac.decode_step_host(*h_in[i], out=h_out[i], lse=h_lse[i], stream=main)
        mac.join(stream=main)

    graph = None
    if not args.eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                host_loop(cap)
        torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    e2.record(stream)
    if graph is not None:
        graph.replay()
    else:
        host_loop(stream)
    e3.record(stream)
    torch.cuda.synchronize()
    del graph
    e2e_us = max_over_ranks(e2.elapsed_time(e3), ws, dev) * 1e3 / K_steps
    if not all(torch.isfinite(x.float()).all() for x in (h_out[-1], h_lse[-1])):
        raise RuntimeError("host-buffer decode step left non-finite results")

    # the build's own full split-KV decode (every head a miss, no ring) on
    # the same handle and inputs, timed like the headline
    f_first = h_first + K_steps
    mac.sync()
    full_us = max_over_ranks(graph_time(lambda t: mac.full_step(inp["q_post"][t], inp["k_new"][t], inp["v_new"][t],
                                                                 out=out, lse=lse),
                                        f_first, K_steps, stream, eager=args.eager), ws, dev)

    # bytes
    kv_read = st["kv_tokens_read"] * BYTES_PER_KV_TOKEN
    kv_full = st["kv_tokens_full"] * BYTES_PER_KV_TOKEN
    steps = st["steps"]
    items = st["work_items"]
    partial = items * G * (128 * 4 + 8)
    # the attention kernel's bytes over the profiled pass
    attn_bytes = (st_p["kv_tokens_read"] * BYTES_PER_KV_TOKEN + st_p["steps"] * B * H * 256
                  + st_p["work_items"] * G * (128 * 4 + 8))
    L = cfg.ring_len
    ring = steps * B * H * L * 256 + st["hits"] * (128 * 4 + 4)
    io = steps * (B * H * 256 * 2 + B * Hkv * 512 + B * H * 256 + B * H * 4) + 2 * partial
    amend_w = steps * B * H * (256 + 128 * 4 + 4)
    step_bytes = kv_read + ring + io + amend_w
    hbm_gbs = step_bytes / (ms * 1e-3) / 1e9
    attn_s = prof["attention_ms"] * 1e-3
    peak, peak_kind = measured_peaks()
    achieved = attn_bytes / attn_s / 1e9 if attn_s > 0 else None
    traffic = profiled_traffic(KERNEL_SOURCES)
    launches = prof["steps"] or st_p["steps"]

    result = {
        "metric": METRIC, "value": round(us_step, 3), "unit": "us/step", "n_gpus": ws, "steps": K_steps,
        "warmup": W_steps, "ms_per_step": round(us_step / 1e3, 6), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "batch": B, "context": cfg.context, "heads": H, "kv_heads": Hkv,
                   "head_dim": cfg.head_dim, "ring_len": L, "band_r": cfg.band_r, "tau": cfg.tau,
                   "page_size": page, "plan_mode": args.plan_mode, "amend_band": args.amend_band,
                   "accumulate": "fp32",
                   "l2": f"inputs larger than L2 (KV {B * Hkv * cfg.context * BYTES_PER_KV_TOKEN / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "timing": ("CUDA-graph replay of the K-step decode loop" if not args.eager else
                   "per-call launches from Python"),
        "eager_us_per_step": round(eager_us, 3),
        "tokens_per_s": round(sum_over_ranks(B, ws, dev) / (us_step * 1e-6), 1),
        "hbm_gbs_step": round(hbm_gbs, 1),
        "hbm_frac_of_8tbs": round(hbm_gbs / NOMINAL_HBM_GBS, 4),
        "kv_bytes_read_vs_full": round(kv_read / kv_full, 5) if kv_full else None,
        "hit_rate": round(st["hits"] / max(1, st["head_decisions"]), 5),
        "phase_us_per_step": {k.replace("_ms", ""): round(v * 1e3 / launches, 3) for k, v in prof.items()
                              if k.endswith("_ms") and (k != "amend_ms" or args.amend_band == 1)},
        "full_us_per_step": round(full_us, 3),
        "ratio_full_over_mac": round(full_us / us_step, 4),
        "roofline": {"kernel": "attention_kernel", "bound": "hbm",
                     "achieved": round(achieved, 1) if achieved else None, "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4) if achieved else None,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": round(attn_bytes / launches),
                     "avg_launch_us": round(attn_s / launches * 1e6, 3),
                     "timing": "CUDA events around each attention launch over a second pass of K steps "
                               "(events between kernels disable launch overlap, so that pass is not the headline)",
                     "traffic": traffic,
                     "traffic_source": ("quoted from profiles/attention_kernel_128k.json: one ncu capture of this "
                                        "kernel source on this workload (hash-checked)") if traffic else
                                       "no ncu capture of the current kernel source"},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/step", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "api": "mac_decode_step_host: pinned host inputs read and results written in place by the "
                       "step's kernels",
                "staged_us_per_step": round(e2e_staged_us, 3),
                "staged": "mac_decode_step on device buffers with explicit pinned-host copies on a second "
                          "stream, double-buffered"},
        # per step: match_plan, attention, combine (+ the side-stream Amend when it recomputes the band)
        "gpu_launches": int(launches_per_step(cfg, args.amend_band) * K_steps),
        "clocks": clk,
        "stats": {"removal_direct": st["removal_direct"], "device_error": st["device_error"],
                  "work_items_per_step": round(items / max(1, steps), 1)},
    }
    mac.sync()
    if not args.no_method_points:
        # the method against full attention where hits skip KV: GQA 1 x 128K
        # at 90 % forced hits, MQA 1 x 128K and 32 x 128K at 0 and 90 %
        specs = [(8, 1, 131072, (0.9,)), (1, 1, 131072, (0.0, 0.9)), (1, 32, 131072, (0.0, 0.9))]
        result["method_points"] = {
            "workload": "forced-hit streams (per request, KV group and step), paged 16, ring 16, r 64, tau 0.3; "
                        "us/step from CUDA-graph replays of 48 steps; fractions of the measured HBM peak",
            "points": method_points(dev, peak, specs)}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        us, cores, sample, extra = run_oracle(cfg, Kp, Vp, inp, args.cpu_budget, max_steps=min(K_steps, 256))
        result["cpu_baseline"] = {"value": round(us, 1), "unit": "us/step", "cores": cores, "kind": "oracle",
                                  "sample": sample, **extra}
    mac.close()
    return result


def _kv_bytes(stats):
    return stats["kv_tokens_read"] * BYTES_PER_KV_TOKEN, stats["kv_tokens_full"] * BYTES_PER_KV_TOKEN


def bench_stack(args, ws, rank, local):
    """Qwen3-30B-A3B-shaped attention stack: one handle per layer, a step is
    one decode step of every layer (Amend of layer l overlaps layers l+1..
    when it runs on the side stream)."""
    from kv_cache_computation_gb300 import MacAttention
    from kv_cache_computation_gb300 import workloads as W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K_steps, W_steps = args.steps, args.warmup
    prof_steps = min(K_steps, 16)
    total = W_steps + K_steps + prof_steps + 1
    cfg = W.qwen_moe_stack_120k_b4(steps=total, tau=args.tau if args.tau is not None else 0.3, layers=args.layers)
    B, H, Hkv, G = cfg.batch, cfg.heads, cfg.kv_heads, cfg.group
    max_ctx = cfg.context + total
    ppr = (max_ctx + 15) // 16
    pt = W.page_tables(B, ppr, seed=cfg.seed).to(dev)
    macs, inps = [], []
    for layer in range(cfg.layers):
        mac = MacAttention(H, Hkv, cfg.head_dim, cfg.ring_len, cfg.band_r, cfg.tau, max_batch=B, max_ctx=max_ctx,
                           page_size=16, plan_mode=args.plan_mode, amend_band=args.amend_band)
        for b in range(B):
            mac.set_page_table(b, pt[b].contiguous())
        Kp, Vp = W.prefill_kv(cfg, layer=layer, device=dev)
        for b in range(B):
            mac.append_kv(b, Kp[b].contiguous(), Vp[b].contiguous())
        del Kp, Vp
        macs.append(mac)
        inps.append(W.decode_inputs(cfg, layer=layer, device=dev))
    out = torch.empty((B, H, cfg.head_dim), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)

    def run(t0, n):
        for t in range(t0, t0 + n):
            for mac, inp in zip(macs, inps):
                mac.decode_step(inp["q_pre"][t], inp["q_post"][t], inp["k_new"][t], inp["v_new"][t], out=out, lse=lse)

    run(0, W_steps)
    for m in macs:
        m.sync()
    torch.cuda.synchronize()
    for m in macs:
        m.reset_stats()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(stream)
        run(W_steps, K_steps)
        for m in macs:
            m.join()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    clk = clocks.summary()
    sts = [m.stats() for m in macs]
    kv_read = sum(_kv_bytes(st)[0] for st in sts)
    kv_full = sum(_kv_bytes(st)[1] for st in sts)
    hits = sum(st["hits"] for st in sts)
    dec = sum(st["head_decisions"] for st in sts)
    # per-kernel durations on a second pass with events around every launch
    for m in macs:
        m.reset_stats()
        m.set_profiling(True)
    run(W_steps + K_steps, prof_steps)
    for m in macs:
        m.join()
    torch.cuda.synchronize()
    profs = [m.profile() for m in macs]
    sts_p = [m.stats() for m in macs]
    for m in macs:
        m.set_profiling(False)
    attn_ms = sum(p_["attention_ms"] for p_ in profs)
    launches = sum(p_["steps"] for p_ in profs)
    attn_bytes = sum(st["kv_tokens_read"] * BYTES_PER_KV_TOKEN + st["steps"] * B * H * 256
                     + st["work_items"] * G * (128 * 4 + 8) for st in sts_p)
    peak, peak_kind = measured_peaks()
    achieved = attn_bytes / (attn_ms * 1e-3) / 1e9
    us = ms * 1e3 / K_steps
    res = {
        "metric": METRIC, "value": round(us, 2), "unit": "us/step", "n_gpus": ws, "steps": K_steps,
        "warmup": W_steps, "ms_per_step": round(us / 1e3, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "layers": cfg.layers, "batch": B, "context": cfg.context, "heads": H,
                   "kv_heads": Hkv, "head_dim": cfg.head_dim, "ring_len": cfg.ring_len, "band_r": cfg.band_r,
                   "tau": cfg.tau, "page_size": 16, "amend_band": args.amend_band,
                   "l2": "inputs larger than L2", "step": "one decode step of every layer"},
        "tokens_per_s": round(sum_over_ranks(B, ws, dev) / (us * 1e-6), 1),
        "hbm_gbs_step": round(kv_read / K_steps / (us * 1e-6) / 1e9, 1),
        "kv_bytes_read_vs_full": round(kv_read / kv_full, 5),
        "hit_rate": round(hits / max(1, dec), 5),
        "phase_us_per_layer_step": {k.replace("_ms", ""): round(sum(p_[k] for p_ in profs) * 1e3 / launches, 3)
                                    for k in ("match_plan_ms", "attention_ms", "combine_ms", "amend_ms")},
        "roofline": {"kernel": "attention_kernel", "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "avg_launch_us": round(attn_ms * 1e3 / launches, 3), "traffic": None},
        "gpu_launches": int(launches_per_step(cfg, args.amend_band) * K_steps * cfg.layers),
        "clocks": clk,
    }
    for m in macs:
        m.close()
    return res


def bench_sweep(args, ws, rank, local):
    """Context x batch x forced hit rate, MQA and GQA: the MAC path against the
    build's own full split-KV decode (mac_full_step) on the same handle.
    Prints one JSON line per point (rank 0)."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ctxs = [int(x) for x in args.sweep_contexts.split(",")]
    batches = [int(x) for x in args.sweep_batches.split(",")]
    rates = tuple(float(x) for x in args.sweep_rates.split(","))
    kvs = [int(x) for x in args.sweep_kv_heads.split(",")]
    peak, _ = measured_peaks()
    specs = [(kv, B, ctx, rates) for kv in kvs for ctx in ctxs for B in batches]

    def emit(pt):
        if rank == 0:
            print(json.dumps({"workload": "forced_hit_sweep", "plan_mode": args.plan_mode, **pt}), flush=True)

    method_points(dev, peak, specs, steps=args.steps, warm=args.warmup, prof_steps=min(16, args.steps),
                  eager=args.eager, on_point=emit, plan_mode=args.plan_mode)
    return None


def bench_match_windows(args, ws, rank, local):
    """Match-stage latency against the window length L and the GQA setting
    (analogue of the paper's Figure 8(a)): rings filled to L entries by
    seeding, then K decode steps with per-phase events.  One JSON line per
    point."""
    from kv_cache_computation_gb300 import MacAttention
    from kv_cache_computation_gb300 import workloads as W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ctx, steps, warm = 32768, args.steps, args.warmup
    for kv in [int(x) for x in args.match_kv_heads.split(",")]:
        for L in [int(x) for x in args.match_windows.split(",")]:
            cfg = W.DecodeConfig(f"match_window_gqa32x{kv}_ctx{ctx}_L{L}", 1, 32, kv, 128, ctx, warm + steps + 1, L, 64,
                                 0.3, rho=0.95, paged=True, seed=20260331 + 6)
            mac = MacAttention(32, kv, 128, L, 64, 0.3, max_batch=1, max_ctx=ctx + warm + steps + 8, page_size=16)
            pt = W.page_tables(1, (ctx + warm + steps + 8 + 15) // 16, seed=cfg.seed).to(dev)
            mac.set_page_table(0, pt[0].contiguous())
            Kp, Vp = W.prefill_kv(cfg, device=dev)
            mac.append_kv(0, Kp[0], Vp[0])
            del Kp, Vp
            # L prefill entries (query values only matter for the scan cost)
            g = torch.Generator(device=dev)
            g.manual_seed(L)
            qs = torch.randn((L, 32, 128), generator=g, device=dev).to(torch.bfloat16)
            o = torch.zeros((L, 32, 128), dtype=torch.float32, device=dev)
            lse = torch.full((L, 32), -float("inf"), dtype=torch.float32, device=dev)
            mac.seed_ring(0, qs, o, lse, list(range(ctx - L + 1, ctx + 1)))
            inp = W.decode_inputs(cfg, device=dev)
            step = lambda t: mac.decode_step(inp["q_pre"][t], inp["q_post"][t], inp["k_new"][t], inp["v_new"][t])
            for t in range(warm):
                step(t)
            mac.sync()
            mac.set_profiling(True)
            for t in range(warm, warm + steps):
                step(t)
            mac.sync()
            pr = mac.profile()
            mac.set_profiling(False)
            if rank == 0:
                print(json.dumps({"workload": "match_window_sweep", "kind": "mqa" if kv == 1 else "gqa",
                                  "heads": 32, "kv_heads": kv, "window": L, "context": ctx,
                                  "match_us": round(pr["match_plan_ms"] * 1e3 / pr["steps"], 2),
                                  "attention_us": round(pr["attention_ms"] * 1e3 / pr["steps"], 2)}), flush=True)
            mac.close()
    return None


def _prefix_summaries(Kp, Vp, q_post, pos, band_r, G, scale):
    """AS_{1:pos-r} of prefill queries (what the caller's prefill attention
    yields for the ring entries it seeds), in fp64 on the GPU: Kp, Vp bf16
    [T, Hkv, d] of one request; q_post bf16 [n, H, d]; pos 1-based [n].
    Returns o fp32 [n, H, d], lse fp32 [n, H] (AS_empty = (0, -inf))."""
    n, H, d = q_post.shape
    K = Kp.double().repeat_interleave(G, dim=1).transpose(0, 1)          # [H, T, d]
    V = Vp.double().repeat_interleave(G, dim=1).transpose(0, 1)
    q = q_post.double().transpose(0, 1)                                  # [H, n, d]
    z = torch.matmul(q, K.transpose(1, 2)) * scale                      # [H, n, T]
    T = K.shape[1]
    lim = torch.as_tensor(pos, device=z.device) - band_r                # tokens [0, pos - r)
    mask = torch.arange(T, device=z.device)[None, :] < lim[:, None]
    z = torch.where(mask[None], z, torch.full_like(z, -math.inf))
    lse = torch.logsumexp(z, dim=-1)                                     # [H, n]
    w = torch.exp(z - torch.where(torch.isfinite(lse), lse, torch.zeros_like(lse))[..., None])
    o = torch.matmul(w, V)                                               # [H, n, d]
    return o.transpose(0, 1).float().contiguous(), lse.transpose(0, 1).float().contiguous()


def bench_rectification(args, ws, rank, local):
    """Synthetic analogue of the paper's Figures 4 and 5: the MAC output
    against full attention (both on this GPU, same inputs).  Three studies,
    one JSON line per point:
      tau_band -- AR(1) streams: hit rate, skipped prefix and error by reuse
                  gap over threshold x window x band;
      gap      -- streams that recur at a chosen gap (q~_t = q~_{t-gap} +
                  0.1 eps): error by reuse gap x band (Figure 4);
      window   -- topic-revisiting streams with the ring seeded from prefill
                  queries: acceptance, skipped prefix and KV read vs window
                  at a fixed threshold (Figure 5, bottom row)."""
    from kv_cache_computation_gb300 import MacAttention
    from kv_cache_computation_gb300 import workloads as W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ctx, steps = 8192, args.steps
    studies = args.rect_studies.split(",")

    def run(cfg, seed_n=0):
        L, r, tau = cfg.ring_len, cfg.band_r, cfg.tau
        mk = lambda: MacAttention(cfg.heads, cfg.kv_heads, 128, L, r, tau, max_batch=1,
                                  max_ctx=ctx + cfg.steps + 1, page_size=0)
        mac, full = mk(), mk()
        Kp, Vp = W.prefill_kv(cfg, device=dev)
        mac.append_kv(0, Kp[0], Vp[0])
        full.append_kv(0, Kp[0], Vp[0])
        if seed_n:
            q_pre, q_post = W.prefill_queries(cfg, device=dev)
            pos = list(range(ctx - seed_n + 1, ctx + 1))
            o, lse = _prefix_summaries(Kp[0], Vp[0], q_post[:, 0], pos, r, cfg.group, 1 / math.sqrt(128))
            mac.seed_ring(0, q_pre[:, 0].contiguous(), o, lse, pos)
        inp = W.decode_inputs(cfg, device=dev)
        errs, hits, skipped, total = {}, 0, 0.0, 0
        mac.reset_stats()
        for t in range(cfg.steps):
            a = [inp[k][t] for k in ("q_pre", "q_post", "k_new", "v_new")]
            pos = mac.read_ring(0)["pos"]      # before the step: its insert may overwrite the matched entry
            o_mac, _ = mac.decode_step(*a)
            o_full, _ = full.full_step(*a[1:])
            dec = mac.decisions(1)
            e = ((o_mac.float() - o_full.float()).abs().amax(-1) / o_full.float().abs().amax(-1)).cpu().numpy()[0]
            m = ctx + t + 1
            for h in range(cfg.heads):
                total += 1
                if dec["hit"][0, h]:
                    hits += 1
                    p = int(pos[dec["slot"][0, h]])
                    skipped += max(0, p - r) / m
                    errs.setdefault(m - p, []).append(float(e[h]))
        st = mac.stats()
        mac.close()
        full.close()
        return {"hit_rate": round(hits / total, 4), "skipped_prefix_fraction": round(skipped / total, 4),
                "kv_bytes_read_vs_full": round(st["kv_tokens_read"] / max(1, st["kv_tokens_full"]), 4),
                "mean_error_on_hits": round(float(np.mean([x for v in errs.values() for x in v])), 6) if hits else None,
                "error_by_gap": {str(k): [round(float(np.mean(v)), 6), len(v)] for k, v in sorted(errs.items())}}

    def emit(line):
        if rank == 0:
            print(json.dumps(line), flush=True)

    if "tau_band" in studies:
        for rho in (0.95, 0.99):
            for tau in (0.2, 0.3, 0.4, 0.5):
                for L in (4, 16, 64):
                    for r in (16, 64, 256):
                        cfg = W.DecodeConfig(f"rect_rho{rho}_tau{tau}_L{L}_r{r}", 1, 32, 8, 128, ctx, steps, L, r, tau,
                                             rho=rho, paged=False, seed=20260331 + 7)
                        emit({"workload": "rectification_study", "study": "tau_band", "rho": rho, "tau": tau,
                              "window": L, "band_r": r, "context": ctx, "steps": steps, **run(cfg)})
    if "gap" in studies:
        for gap in (1, 2, 4, 8, 16, 32):
            for r in (16, 64, 256):
                cfg = W.DecodeConfig(f"rect_gap{gap}_r{r}", 1, 32, 8, 128, ctx, steps, 32, r, 0.3, gap=gap,
                                     gap_noise=0.1, paged=False, seed=20260331 + 8)
                emit({"workload": "rectification_study", "study": "gap", "gap": gap, "gap_noise": 0.1, "tau": 0.3,
                      "window": 32, "band_r": r, "context": ctx, "steps": steps, **run(cfg)})
    if "window" in studies:
        for L in (16, 64, 256, 1024):
            cfg = W.DecodeConfig(f"rect_topics_L{L}", 1, 32, 8, 128, ctx, steps, L, 64, 0.3, topics=32,
                                 topic_stay=0.9, topic_noise=0.1, lead=L, paged=False, seed=20260331 + 9)
            emit({"workload": "rectification_study", "study": "window", "window": L, "tau": 0.3, "band_r": 64,
                  "topics": 32, "topic_stay": 0.9, "seeded_entries": L, "context": ctx, "steps": steps,
                  **run(cfg, seed_n=L)})
    return None


def bench_reference(args, ws, rank, local):
    """The fp64 oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    import oracle
    from kv_cache_computation_gb300 import workloads as W
    K_steps, W_steps = args.steps, args.warmup
    cfg = workload(args.workload, args.band_r, W_steps + K_steps + 4)
    Kp, Vp = W.prefill_kv(cfg)
    inp = W.decode_inputs(cfg)
    us, cores, sample, extra = run_oracle(cfg, Kp, Vp, inp, args.ref_budget, max_steps=K_steps,
                                          fixed_steps=K_steps, warm=W_steps)
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/step", "n_gpus": ws,
            "steps": K_steps, "warmup": W_steps, "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "batch": cfg.batch, "context": cfg.context, "heads": cfg.heads,
                       "kv_heads": cfg.kv_heads, "head_dim": cfg.head_dim, "ring_len": cfg.ring_len,
                       "band_r": cfg.band_r, "tau": cfg.tau},
            "cpu_baseline": {"value": round(us, 1), "unit": "us/step", "cores": cores, "kind": "oracle",
                             "sample": sample, **extra},
            "e2e": {"value": round(us, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_128k_b1_hetero")
    ap.add_argument("--band-r", type=int, default=64)
    ap.add_argument("--plan-mode", type=int, default=0, help="0 span-proportional, 1 equal split per group")
    ap.add_argument("--amend-band", type=int, default=0,
                    help="0 reuse Complete's band summary, 1 recompute the band in Amend")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds of oracle work for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-method-points", action="store_true",
                    help="skip the MAC-vs-full forced-hit points of the default run")
    ap.add_argument("--eager", action="store_true", help="time per-call launches instead of a CUDA-graph replay")
    ap.add_argument("--tau", type=float, default=None, help="threshold for the layer-stack workload (0.3 or 0.45)")
    ap.add_argument("--layers", type=int, default=48, help="layers of the stack workload")
    ap.add_argument("--sweep-contexts", default="4096,16384,65536,131072")
    ap.add_argument("--sweep-batches", default="1,8,32")
    ap.add_argument("--sweep-rates", default="0,0.5,0.9,1.0")
    ap.add_argument("--sweep-kv-heads", default="1,8")
    ap.add_argument("--match-windows", default="16,64,256,512,1024,2048", help="ring lengths of match_windows")
    ap.add_argument("--rect-studies", default="tau_band,gap,window", help="studies of the rectification workload")
    ap.add_argument("--match-kv-heads", default="1,8", help="KV heads (32 q heads) of match_windows")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    ws, rank, local = dist_init()
    if args.impl == "reference":
        res = bench_reference(args, ws, rank, local)
    elif args.workload == "qwen_stack_120k_b4":
        res = bench_stack(args, ws, rank, local)
    elif args.workload == "sweep":
        res = bench_sweep(args, ws, rank, local)
    elif args.workload == "match_windows":
        res = bench_match_windows(args, ws, rank, local)
    elif args.workload == "rectification":
        res = bench_rectification(args, ws, rank, local)
    else:
        res = bench_ours(args, ws, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
