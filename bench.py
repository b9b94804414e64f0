"""Benchmark of the PolyKV hot path: encode the shared pool, then run
multi-agent decode attention over it, on synthetic inputs of the
Llama-3-8B shape (32 layers, 8 kv heads, 32 q heads, head_dim 128, bf16,
4096-token shared context, 15 agents).

A step = one encode of the whole context (keys -> q8_0, values -> FWHT +
3-bit codes) + one decode attention of every agent's query over the pool.
Prints one JSON line (rank 0). `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "pool decode-attention HBM GB/s (% of peak) & encode tokens/s, Llama-3-8B shape"
DEFAULT_WORKLOAD = "llama3_8b_4096_a15"


def algorithmic_bytes(w: synth.Workload, n_ctx: int, n_agents: int):
    """(encode bytes, attend bytes) per call, from the pool format (plus the private suffixes)."""
    L, H, Hq, d = w.n_layers, w.n_kv_heads, w.n_q_heads, w.head_dim
    per_tok_pool = d + 2 * (d // 32) + 3 * d // 8 + 2
    pool = L * H * n_ctx * per_tok_pool
    enc = L * H * n_ctx * d * 2 * 2 + pool          # read K, V (16-bit), write the pool
    att = pool + L * n_agents * Hq * d * 2 + L * n_agents * Hq * d * 4   # pool + q + fp32 out
    att += L * n_agents * H * w.suffix_len * d * 2 * 2                   # private suffix K, V
    return enc, att


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor peak (TFLOP/s, burst) from MEASURED_PEAKS.json, else the fallback figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f).get("bf16_tflops", 1900.0))
    return 1900.0


ATTEND_SOURCES = ["attend_tc.cu", "attend_warp.cu", "attend_simt.cu", "attend_suffix.cu", "merge_row.cuh"]


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "serving_q8_encode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str, workload: str, src_hash: str):
    """Per-launch DRAM bytes recorded from an ncu capture, if the kernel's source
    has not changed since (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    e = j.get(kernel, {}).get(workload)
    if not e or e.get("src_hash") != src_hash:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        # 20 ms sampling; if this nvidia-smi refuses that interval, the recipe's 200 ms
        for period in ("20", "200"):
            try:
                fd, self.path = tempfile.mkstemp(suffix=".csv")
                os.close(fd)
                self.f = open(self.path, "w")
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                              "--format=csv,noheader,nounits", "-lms", period], stdout=self.f,
                                             stderr=subprocess.DEVNULL)
            except Exception:
                self.proc = None
                return
            # the timed region starts only once the sampler is live (its first row is written), so
            # that its samples fall inside the region rather than after it
            t_end = time.time() + 3.0
            while time.time() < t_end and self.proc.poll() is None:
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.01)
            if self.proc.poll() is None or os.path.getsize(self.path) > 0:
                return
            self.f.close()
            os.unlink(self.path)
        self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- multi-rank helpers
class L2Flush:
    """Evicts the L2 between timed launches: writes a buffer twice the L2's size, then reads another
    one of the same size, so that the L2 holds clean lines of neither the inputs nor the written
    buffer and the timed kernel pays for no write-back of the flush's own dirty lines."""

    def __init__(self, torch, dev):
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = 2 * l2 // 4 + 1024
        self.torch = torch
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self, i: int):
        self.w.fill_(float(i))
        self.torch.sum(self.r, dim=0, keepdim=True, out=self.sink)

    describe = "flushed between launches (2x L2 written, then 2x L2 of another buffer read)"


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's time: every rank gets the maximum of x over the process group."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank: float, ms: float) -> float:
    """Whole-job throughput: every rank moves bytes_per_rank per step (weak scaling), and the step
    takes the slowest rank's time."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, w: synth.Workload):
    """The CPU oracle, timed as it stands, on a bounded sample per step: one layer and two kv heads
    (all their tokens, agents and query heads, and the private suffix when the workload has one),
    scaled to the whole workload's algorithmic bytes."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    c32, b32 = oracle.codebook.codebook_f32()
    heads = min(2, w.n_kv_heads)
    G = w.n_q_heads // w.n_kv_heads
    kb, vb = synth.gen_kv(1, w.n_kv_heads, w.n_ctx, w.head_dim, w.dtype, 0)
    qb = synth.gen_q(1, w.n_agents, w.n_q_heads, w.head_dim, w.dtype, 0)
    kb, vb = kb[:, :heads], vb[:, :heads]
    qb = np.ascontiguousarray(qb[:, :, :heads * G])
    sfx = {}
    if w.suffix_len:
        skb, svb = synth.gen_suffix(1, w.n_agents, w.n_kv_heads, w.suffix_len, w.head_dim, w.dtype, 0)
        sfx = dict(suffix_k_bits=np.ascontiguousarray(skb[:, :, :heads]),
                   suffix_v_bits=np.ascontiguousarray(svb[:, :, :heads]))
    enc_b, att_b = algorithmic_bytes(w, w.n_ctx, w.n_agents)
    frac = heads / (w.n_layers * w.n_kv_heads)
    sample_bytes = (enc_b + att_b) * frac

    def step():
        pool = oracle.attention.encode_pool(kb, vb, w.dtype, b32)
        oracle.attention.attend_pool(qb, w.dtype, pool, w.n_ctx, c32, **sfx)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = sample_bytes / dt / 1e9
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(w.describe(), sample=f"1 of {w.n_layers} layers x {heads} of {w.n_kv_heads} kv heads per step"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"encode + attend of 1 layer x {heads} kv heads x {w.n_ctx} tokens x "
                                   f"{w.n_agents} agents per step; numpy (BLAS may thread)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _oracle_layer(job):
    """One layer of the workload through the CPU oracle, encode and attend timed separately. Runs in a
    spawned worker process with one BLAS thread (the parent sets the thread counts before spawning)."""
    name, layer_seed, n_layers_override = job
    import oracle
    w = synth.WORKLOADS[name]
    c32, b32 = oracle.codebook.codebook_f32()
    kb, vb = synth.gen_kv(1, w.n_kv_heads, w.n_ctx, w.head_dim, w.dtype, layer_seed)
    qb = synth.gen_q(1, w.n_agents, w.n_q_heads, w.head_dim, w.dtype, layer_seed)
    sfx = {}
    if w.suffix_len:
        skb, svb = synth.gen_suffix(1, w.n_agents, w.n_kv_heads, w.suffix_len, w.head_dim, w.dtype, layer_seed)
        sfx = dict(suffix_k_bits=skb, suffix_v_bits=svb)
    t0 = time.perf_counter()
    pool = oracle.attention.encode_pool(kb, vb, w.dtype, b32)
    t1 = time.perf_counter()
    oracle.attention.attend_pool(qb, w.dtype, pool, w.n_ctx, c32, **sfx)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


class _one_thread_env:
    """Sets the BLAS/OpenMP thread counts to 1 while worker processes are spawned: a spawned child reads
    them when it first imports numpy, which happens before any pool initializer runs."""
    names = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")

    def __enter__(self):
        self.old = {v: os.environ.get(v) for v in self.names}
        os.environ.update({v: "1" for v in self.names})

    def __exit__(self, *exc):
        for v, old in self.old.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old


def cpu_baseline(w: synth.Workload, budget_s: float = 20.0):
    """The CPU oracle, as it stands, on a bounded sample of the workload (whole layers), in two variants:
    one process with one thread, and one single-threaded process per host core working on different
    layers at once. Encode and attend are timed separately; throughputs are scaled to the full workload's
    algorithmic bytes (GB/s) and tokens/s. Processes are spawned, so this is safe after GPU work."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    enc_b, att_b = algorithmic_bytes(w, w.n_ctx, w.n_agents)
    enc_l, att_l = enc_b / w.n_layers, att_b / w.n_layers          # bytes per layer
    ctx = mp.get_context("spawn")
    t_start = time.perf_counter()
    with _one_thread_env(), ctx.Pool(processes=1) as pool:
        single = pool.map(_oracle_layer, [(w.name, 0, None)])
    se, sa = single[0]
    # all cores: as many one-layer jobs as fit in the budget, one per core per round
    rounds = max(1, min(4, int(budget_s / max(se + sa, 1e-3) / 2)))
    with _one_thread_env(), ctx.Pool(processes=cores) as pool:
        pool.map(abs, range(cores))                                    # workers up before the clock starts
        t0 = time.perf_counter()
        res = pool.map(_oracle_layer, [(w.name, 100 + i, None) for i in range(cores * rounds)], chunksize=1)
        wall = time.perf_counter() - t0
    enc_sum = sum(r[0] for r in res)
    att_sum = sum(r[1] for r in res)
    n_lay = len(res)
    # the all-core wall time covers encode + attend of n_lay layers; split it in proportion to CPU time
    enc_wall = wall * enc_sum / (enc_sum + att_sum)
    att_wall = wall - enc_wall
    all_gbs = n_lay * (enc_l + att_l) / wall / 1e9
    return {"value": all_gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_lay} layers of {w.n_layers} (encode + attend, all kv heads and agents), one "
                      f"single-threaded spawned process per core; single-thread variant: 1 layer",
            "all_cores": {"gbs": all_gbs, "encode_tokens_per_s": n_lay * w.n_ctx / w.n_layers / enc_wall,
                          "encode_gbs": n_lay * enc_l / enc_wall / 1e9,
                          "attend_gbs": n_lay * att_l / att_wall / 1e9, "processes": cores, "layers": n_lay},
            "single_thread": {"gbs": (enc_l + att_l) / (se + sa) / 1e9,
                              "encode_tokens_per_s": w.n_ctx / w.n_layers / se, "encode_gbs": enc_l / se / 1e9,
                              "attend_gbs": att_l / sa / 1e9, "encode_s_per_layer": se, "attend_s_per_layer": sa},
            "seconds": time.perf_counter() - t_start}


# ----------------------------------------------------------------------------- polykv arm
def run_polykv(args, w: synth.Workload):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import serving_q8_encode_gb300 as pk

    L, H, Hq, d, T, A = w.n_layers, w.n_kv_heads, w.n_q_heads, w.head_dim, w.n_ctx, w.n_agents
    kb, vb = synth.gen_kv(L, H, T, d, w.dtype, seed=rank)
    qb = synth.gen_q(L, A, Hq, d, w.dtype, seed=rank)
    k = torch.from_numpy(kb.view(np.int16)).to(dev)
    v = torch.from_numpy(vb.view(np.int16)).to(dev)
    q = torch.from_numpy(qb.view(np.int16)).to(dev)
    pool = pk.Pool(L, H, d, T, w.dtype, device=dev)
    out = torch.empty((L, A, Hq, d), dtype=torch.float32, device=dev)
    pool.encode(k, v)  # so the prefix is valid for the workspace query
    ext = None
    if w.suffix_len:
        skb, svb = synth.gen_suffix(L, A, H, w.suffix_len, d, w.dtype, seed=rank)
        sk = torch.from_numpy(skb.view(np.int16)).to(dev)
        sv = torch.from_numpy(svb.view(np.int16)).to(dev)
        ext = pk.AttendExt(sk.data_ptr(), sv.data_ptr(), w.suffix_len)
    ws = torch.empty(max(16, pk.polykv_attend_ex_workspace_size(pool.handle, A, Hq, T, ext)), dtype=torch.uint8,
                     device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)

    def attend():
        pk.polykv_attend_ex(pool.handle, q.data_ptr(), out.data_ptr(), A, Hq, T, 0.0, ext, ws.data_ptr(), ws.numel(),
                            stream.cuda_stream)

    def step():
        pool.encode(k, v, stream=stream)
        attend()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush(i)  # L2 flush between steps (outside the events)
        ev[i][0].record(stream)
        pool.encode(k, v, stream=stream)
        ev[i][1].record(stream)
        attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    enc_ms = [e[0].elapsed_time(e[1]) for e in ev]
    att_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_ms = float(np.mean([a + b for a, b in zip(enc_ms, att_ms)]))        # the K timed steps' average
    enc_ms_m, att_ms_m = float(np.median(enc_ms)), float(np.median(att_ms))  # per-kernel medians

    # attention alone, L2 flushed before each launch (the pool is read from HBM)
    att_alone = []
    for i in range(args.steps):
        flush(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        attend()
        e1.record(stream)
        e1.synchronize()
        att_alone.append(e0.elapsed_time(e1))
    att_alone_ms = float(np.median(att_alone))

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    hk = torch.from_numpy(kb.view(np.int16)).pin_memory()
    hv = torch.from_numpy(vb.view(np.int16)).pin_memory()
    hq = torch.from_numpy(qb.view(np.int16)).pin_memory()
    hout = torch.empty((L, A, Hq, d), dtype=torch.float32).pin_memory()
    e2e_ms = []
    for i in range(0 if args.no_e2e else max(2, args.steps // 2) + 1):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        q.copy_(hq, non_blocking=True)
        pool.encode(k, v, stream=stream)
        attend()
        hout.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        if i > 0:
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_ms_m = float(np.median(e2e_ms)) if e2e_ms else float("nan")

    def allmax(x):
        return max_over_ranks(x, world, dev)

    step_ms = allmax(step_ms)
    enc_ms_m = allmax(enc_ms_m)
    att_ms_m = allmax(att_ms_m)
    att_alone_ms = allmax(att_alone_ms)
    e2e_ms_m = allmax(e2e_ms_m)

    enc_b, att_b = algorithmic_bytes(w, T, A)
    peak, peak_src = measured_peaks()
    value = whole_job_gbs(world, enc_b + att_b, step_ms)
    att_gbs = att_b / (att_alone_ms * 1e-3) / 1e9
    enc_gbs = enc_b / (enc_ms_m * 1e-3) / 1e9
    enc_tok_s = world * T / (enc_ms_m * 1e-3)
    dominant = "encode" if enc_ms_m >= att_ms_m else "attend"
    if dominant == "encode":
        kname, kbytes, kms, files = "encode_kernel", enc_b, enc_ms_m, ["encode.cu"]
    else:
        kname, kbytes, kms, files = "attend", att_b, att_ms_m, ATTEND_SOURCES
    achieved = kbytes / (kms * 1e-3) / 1e9
    traffic = traffic_from_profiles(kname, w.name, kernel_source_hash(files))
    att_traffic = traffic_from_profiles("attend", w.name, kernel_source_hash(ATTEND_SOURCES))
    h2d = kb.nbytes + vb.nbytes + qb.nbytes
    d2h = L * A * Hq * d * 4
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16->u8/i8 codes, f32 accumulate", "data": "synthetic",
        "config": dict(w.describe(), l2=L2Flush.describe,
                       step="encode whole context + attend all agents", parallelism=f"replicas x{world}"),
        "attend": {"gbs": att_gbs, "frac_of_peak": att_gbs / peak, "us": att_alone_ms * 1e3,
                   "us_in_step": att_ms_m * 1e3, "bytes": att_b, "traffic": att_traffic},
        "encode": {"tokens_per_s": enc_tok_s, "gbs": enc_gbs, "frac_of_peak": enc_gbs / peak,
                   "us": enc_ms_m * 1e3, "bytes": enc_b},
        "roofline": {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": {"value": whole_job_gbs(world, enc_b + att_b, e2e_ms_m), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_m},
        "gpu_launches": args.steps * (3 + (1 if w.suffix_len else 0)),
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_sweep(args):
    """Encode-only and attend-only throughput at the Llama-3-8B shape over the pages' context lengths
    and agent counts; one JSON object with the grid (instead of the single bench line)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import serving_q8_encode_gb300 as pk

    base = synth.WORKLOADS[DEFAULT_WORKLOAD]
    L, H, Hq, d = args.layers or base.n_layers, base.n_kv_heads, base.n_q_heads, base.head_dim
    dev = torch.device("cuda", 0)
    peak, peak_src = measured_peaks()
    bf16_peak = measured_bf16_tflops()
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    rows = []
    for T in args.sweep_ctx:
        kb, vb = synth.gen_kv(L, H, T, d, base.dtype, seed=0)
        k = torch.from_numpy(kb.view(np.int16)).to(dev)
        v = torch.from_numpy(vb.view(np.int16)).to(dev)
        del kb, vb
        pool = pk.Pool(L, H, d, T, base.dtype, device=dev)
        pool.encode(k, v)

        def timed(fn, reps):
            ts = []
            for i in range(reps + 2):
                flush(i)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                if i >= 2:
                    ts.append(e0.elapsed_time(e1) * 1e3)
            return float(np.median(ts))

        w = synth.Workload("sweep", L, H, Hq, d, T, 1, base.dtype)
        enc_b, _ = algorithmic_bytes(w, T, 1)
        enc_us = timed(lambda: pool.encode(k, v, stream=stream), args.steps)
        rows.append({"mode": "encode", "n_ctx": T, "us": enc_us, "tokens_per_s": T / (enc_us * 1e-6),
                     "gbs": enc_b / (enc_us * 1e-6) / 1e9})
        for A in args.sweep_agents:
            qb = synth.gen_q(L, A, Hq, d, base.dtype, seed=0)
            q = torch.from_numpy(qb.view(np.int16)).to(dev)
            out = torch.empty((L, A, Hq, d), dtype=torch.float32, device=dev)
            ws = torch.empty(max(16, pool.workspace_size(A, Hq, T)), dtype=torch.uint8, device=dev)
            _, att_b = algorithmic_bytes(w, T, A)
            att_us = timed(lambda: pool.attend(q, T, out=out, workspace=ws, stream=stream), args.steps)
            rows.append({"mode": "attend", "n_ctx": T, "n_agents": A, "us": att_us,
                         "gbs": att_b / (att_us * 1e-6) / 1e9, "frac_of_peak": att_b / (att_us * 1e-6) / 1e9 / peak,
                         "pool_bytes": att_b - L * A * Hq * d * 6})
            del out, ws
            if args.chunk > 0:
                # query-chunk mode: C query tokens per agent with their own K/V, causal inside the chunk;
                # the pool part is a dense contraction (R = A*C*G rows per kv head), so report tensor use
                C = args.chunk
                qcb = synth.gen_q(L, A * C, Hq, d, base.dtype, seed=1).reshape(L, A, C, Hq, d)
                ckb, cvb = synth.gen_suffix(L, A, H, C, d, base.dtype, seed=1)
                qc = torch.from_numpy(qcb.view(np.int16)).to(dev)
                ck = torch.from_numpy(ckb.view(np.int16)).to(dev)
                cv = torch.from_numpy(cvb.view(np.int16)).to(dev)
                del qcb, ckb, cvb
                outc = torch.empty((L, A, C, Hq, d), dtype=torch.float32, device=dev)
                ext = pk.AttendExt(chunk_k=ck.data_ptr(), chunk_v=cv.data_ptr(), chunk_len=C)
                wsc = torch.empty(max(16, pk.polykv_attend_ex_workspace_size(pool.handle, A, Hq, T, ext)),
                                  dtype=torch.uint8, device=dev)
                ch_us = timed(lambda: pool.attend_chunk(qc, T, ck, cv, out=outc, workspace=wsc, stream=stream),
                              max(2, args.steps // 4))
                R = A * C * (Hq // H)
                flops = 4.0 * R * T * d * L * H + 4.0 * (C * (C + 1) / 2) * (Hq // H) * d * L * A * H
                # tensor-core MMAs issued (M=128, N=64, K=16): 8 for the keys (4 q8_0 blocks x 2 K-steps)
                # and 8 for the values per 128-token tile and row group of up to 64 query rows
                mma_flops = 2.0 * 128 * 64 * 16 * (8 + 8) * ((R + 63) // 64) * ((T + 127) // 128) * L * H
                rows.append({"mode": "attend_chunk", "n_ctx": T, "n_agents": A, "chunk": C, "us": ch_us,
                             "query_tokens_per_s": A * C / (ch_us * 1e-6),
                             "tflops": flops / (ch_us * 1e-6) / 1e12,
                             "tensor_issued_tflops": mma_flops / (ch_us * 1e-6) / 1e12,
                             "tensor_frac_of_bf16_peak": mma_flops / (ch_us * 1e-6) / 1e12 / bf16_peak})
                del qc, ck, cv, outc, wsc
                torch.cuda.empty_cache()
        del pool, k, v
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": f"llama3_8b shape ({L} layers), encode-only and attend-only", "peak_gbs": peak,
                      "peak_source": peak_src, "bf16_tflops_peak": bf16_peak, "l2": L2Flush.describe,
                      "rows": rows}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="polykv", choices=["polykv", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--sweep", action="store_true",
                    help="encode-only / attend-only grid over context {600,1851,4096,7194} x agents {1,2,4,8,15}")
    ap.add_argument("--chunk", type=int, default=0,
                    help="with --sweep: also time query-chunk mode with this many query tokens per agent")
    ap.add_argument("--sweep-ctx", type=lambda x: [int(v) for v in x.split(",")], default=[600, 1851, 4096, 7194],
                    help="with --sweep: comma-separated context lengths")
    ap.add_argument("--sweep-agents", type=lambda x: [int(v) for v in x.split(",")], default=[1, 2, 4, 8, 15],
                    help="with --sweep: comma-separated agent counts")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the layer count (smaller cases for profiler captures)")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.layers is not None:
        import dataclasses
        w = dataclasses.replace(w, n_layers=args.layers, name=f"{w.name}_L{args.layers}")
    if args.sweep:
        return run_sweep(args)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_polykv(args, w)


if __name__ == "__main__":
    sys.exit(main())
