"""Benchmark of the rotated INT2 KV-cache decode step on GB300.

One step = the whole hot path for one batch, one kvq_append_decode call:
quantise-and-append one new K/V token per sequence (centre, rotate, clip, INT2
pack into its page) and split-K INT2 decode attention over the paged cache
(query rotation, scores, online softmax, P.V, log-sum-exp combine, inverse value
rotation).  The same step as two calls (kvq_append, kvq_decode) is reported too.

Workload (default): Qwen3-8B-shaped layer, batch 16, 32 query / 8 KV heads,
head_dim 128, context 32768 per sequence in 16-token pages over a shuffled pool.
The cache is built once before timing; each step appends the token at position
32767 (rewriting that slot) and decodes over all 32768 positions.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead.
Under torchrun (N > 1) every rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rotated_int2_kv_kvq_gb300 import workloads as W  # noqa: E402

METRIC = "INT2 decode-attn cache GB/s (% of HBM peak) & decode steps/s at 32K ctx"
UNIT = "GB/s"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_int2_qwen3_8b_32k.md")
DECODE_SRC = os.path.join(ROOT, "rotated_int2_kv_kvq_gb300", "csrc", "kvq_decode.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_32k")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller profiling cases)")
    ap.add_argument("--no-bf16", action="store_true", help="skip the BF16 comparison kernel")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (tiny_1k, long_128k, ragged_64, full_stack_36l)")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the decode kernel from the committed ncu summary,
    or None if the summary is missing or was taken on a different kernel source."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    text = open(PROFILE_SUMMARY).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kvq_decode\.cu`?\s*sha256\[:16\]:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != source_hash(DECODE_SRC):
        return None
    return float(m.group(1))


def max_over_ranks(value, dist=None):
    """Max of a float over all ranks of the default process group (the value
    itself without one).  NCCL groups reduce a CUDA tensor, others a CPU one."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return float(value)
    import torch

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, max_ms, world):
    """Weak scaling: every rank processes units_per_rank; the job takes the
    slowest rank's time."""
    return units_per_rank * world / (max_ms * 1e-3)


def l2_bytes(torch):
    """L2 cache size of the current device (cudaDevAttrL2CacheSize)."""
    prop = torch.cuda.get_device_properties(torch.cuda.current_device())
    v = getattr(prop, "L2_cache_size", 0)
    if v:
        return int(v)
    import ctypes

    rt = ctypes.CDLL("libcudart.so")
    out = ctypes.c_int(0)
    rt.cudaDeviceGetAttribute(ctypes.byref(out), 89, torch.cuda.current_device())
    return int(out.value)


def replicas_for(bytes_per_step, l2):
    """Copies of a cache that one timed loop cycles through so that successive
    steps never find their cache in L2: enough for at least twice the L2 size."""
    if bytes_per_step >= 2 * l2:
        return 1
    return int(min(4096, -(-2 * l2 // max(1, bytes_per_step))))


def l2_note(bytes_per_step, replicas, l2):
    mb = bytes_per_step / 1e6
    if replicas > 1:
        return (f"cache {mb:.2f} MB per step is smaller than twice L2 ({l2 / 1e6:.1f} MB): "
                f"steps cycle through {replicas} replicas ({replicas * mb:.0f} MB), no flush")
    if bytes_per_step >= 2 * l2:
        return f"inputs larger than L2: {mb:.0f} MB of cache per step vs L2 {l2 / 1e6:.1f} MB, no flush"
    return f"cache {mb:.0f} MB per step vs L2 {l2 / 1e6:.1f} MB (between 1x and 2x L2), no flush"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.mark = 0
        self.path = os.path.join("/tmp", f"kvq_clocks_{os.getpid()}.csv")

    def _lines(self):
        try:
            with open(self.path) as f:
                return f.read().splitlines()
        except OSError:
            return []

    def start(self):
        """Start sampling every 100 ms; returns once the sampler has written its
        first (idle) line, so that every later line falls in the measured window."""
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 10.0 and not self._lines() and self.proc.poll() is None:
            time.sleep(0.05)
        self.mark = len(self._lines())

    def samples(self):
        return max(0, len(self._lines()) - self.mark) if self.proc is not None else 0

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for i, line in enumerate(f):
                if i < self.mark:
                    continue
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------

def oracle_sample_setup(wl, seq=0, kv=0):
    """One (sequence, KV head) of the workload, built by the oracle alone."""
    import oracle

    ctx = int(W.seq_lens(wl)[seq])
    pages = ctx // 16
    pt = np.arange(pages, dtype=np.int32)[None, :]
    pool = np.zeros(pages * 1152, np.uint8)
    R = W.rotations(wl)[:, kv:kv + 1].copy()
    mu = W.key_mean(wl)[kv:kv + 1].copy()
    Kt = W.tokens(wl, 0, seq, 0, 0, ctx)[:, kv:kv + 1].copy()
    Vt = W.tokens(wl, 0, seq, 1, 0, ctx)[:, kv:kv + 1].copy()
    oracle.append_int2(pool, pages, 1, Kt, Vt, np.zeros(ctx), np.arange(ctx), pt, R, mu,
                       wl.clip_k, wl.clip_v)
    G = wl.num_heads // wl.num_kv_heads
    q = W.queries(wl)[seq:seq + 1, kv * G:(kv + 1) * G].copy()
    return dict(pool=pool, pages=pages, pt=pt, R=R, mu=mu, K=Kt[-1:], V=Vt[-1:], q=q, G=G, ctx=ctx,
                Kall=Kt, Vall=Vt, seq=seq, kv=kv)


def oracle_step(wl, s):
    """Append the last token again and decode the G query heads of the sample."""
    import oracle

    ctx = s["ctx"]
    oracle.append_int2(s["pool"], s["pages"], 1, s["K"], s["V"], [0], [ctx - 1], s["pt"], s["R"],
                       s["mu"], wl.clip_k, wl.clip_v)
    oracle.decode_pairs("int2", s["pool"], s["pages"], s["G"], 1, s["q"], s["pt"], [ctx],
                        [[0, h] for h in range(s["G"])], R=s["R"])


def cpu_oracle_rate(wl, min_seconds=10.0, max_steps=None, warmup=0, max_seconds=None, sample=None):
    """Cache GB/s of the oracle on (sequence 0, KV head 0): each step reads that
    head's whole context once for its G query heads.  Stops after max_steps
    steps, or after max_seconds if that comes first."""
    s = sample if sample is not None else oracle_sample_setup(wl)
    for _ in range(warmup):
        oracle_step(wl, s)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(wl, s)
        n += 1
        el = time.perf_counter() - t0
        if (max_steps is not None and n >= max_steps) or (max_steps is None and el >= min_seconds):
            break
        if max_seconds is not None and el >= max_seconds:
            break
    bytes_per_step = s["ctx"] * W.cache_bytes_per_token_head("int2")
    return bytes_per_step * n / el / 1e9, n, el


def _oracle_proc(wl_name, seq, kv, seconds, barrier, q):
    """One process of the all-cores oracle baseline: build the (seq, kv) sample,
    wait for the others, then run oracle steps for `seconds`."""
    wl = W.WORKLOADS[wl_name]
    s = oracle_sample_setup(wl, seq, kv)
    oracle_step(wl, s)
    barrier.wait(timeout=600)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle_step(wl, s)
        n += 1
    q.put((n, time.perf_counter() - t0))


def cpu_oracle_rate_all_cores(wl, seconds=10.0):
    """The same oracle step on every core this process may run on, one process
    per core, each on its own (sequence, KV head) sample, started together
    (spawned processes: CUDA is already initialised here).  Returns (cache GB/s
    over all processes, processes, steps, seconds) or None if a process failed."""
    import multiprocessing as mp

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    ctx = mp.get_context("spawn")
    barrier, q = ctx.Barrier(cores), ctx.Queue()
    units = [(u % wl.batch, (u // wl.batch) % wl.num_kv_heads) for u in range(cores)]
    procs = [ctx.Process(target=_oracle_proc, args=(wl.name, sq, kv, seconds, barrier, q))
             for sq, kv in units]
    for p in procs:
        p.start()
    try:
        res = [q.get(timeout=900) for _ in procs]
    except Exception:
        res = None
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    if not res or any(p.exitcode != 0 for p in procs):
        return None
    steps = sum(n for n, _ in res)
    wall = max(el for _, el in res)
    bytes_per_step = wl.ctx * W.cache_bytes_per_token_head("int2")
    return bytes_per_step * steps / wall / 1e9, cores, steps, wall


def parity_sample(pool_np, pt_np, s, wl):
    """Codes, scales and zeros of the library's pool against the oracle's own
    append of the cpu_baseline sample (one sequence, one KV head, the whole
    context): differing codes are split into those whose pre-rounding value
    lies within 1 ulp of a rounding boundary (allowed, counted) and others."""
    import oracle

    rec = 1152
    Hkv = wl.num_kv_heads
    gpu = pool_np.reshape(-1, Hkv, rec)
    ref = s["pool"].reshape(-1, rec)
    ctx, seq, kv = s["ctx"], s["seq"], s["kv"]
    near = other = 0
    for j in range((ctx + 15) // 16):
        g, o = gpu[pt_np[seq, j], kv], ref[j]
        if np.array_equal(g, o):
            continue
        for tau in range(min(16, ctx - 16 * j)):
            p = 16 * j + tau
            for which in (0, 1):
                c1, s1, z1 = oracle.int2_load(g, which, tau)
                c2, s2, z2 = oracle.int2_load(o, which, tau)
                if (s1, z1) != (s2, z2):
                    other += 1
                bad = np.nonzero(np.asarray(c1) != np.asarray(c2))[0]
                if len(bad) == 0:
                    continue
                x = (s["Kall"] if which == 0 else s["Vall"])[p, 0]
                mu = s["mu"][0] if which == 0 else None
                clip = wl.clip_k if which == 0 else wl.clip_v
                t = oracle.quantize(x, s["R"][which, 0], clip, mu=mu)[4]
                for i in bad:
                    frac = abs(float(t[i]) - np.floor(float(t[i])) - 0.5)
                    if frac <= np.spacing(np.float32(t[i])):
                        near += 1
                    else:
                        other += 1
    return {"boundary_code_mismatches": near, "other_mismatches": other,
            "codes_compared": 2 * 128 * ctx, "token_heads": ctx,
            "sample": f"sequence {seq} / KV head {kv}, all {ctx} positions, against the "
                      f"oracle's append of the same tokens (the cpu_baseline sample)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload]
    # at most about four minutes of oracle work: the line reports the steps timed
    gbs, n, el = cpu_oracle_rate(wl, max_steps=max(1, args.steps), warmup=min(max(0, args.warmup), 3),
                                 max_seconds=240.0)
    sample = (f"float64 oracle, sequence 0 / KV head 0 of {wl.name}: per step re-quantise one "
              f"token and decode {wl.num_heads // wl.num_kv_heads} query heads over "
              f"{int(W.seq_lens(wl)[0])} "
              f"tokens ({n} steps, {el:.1f} s)")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": args.gpus,
        "steps": n, "warmup": args.warmup, "ms_per_step": el / n * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "ctx": wl.ctx,
                   "heads": wl.num_heads, "kv_heads": wl.num_kv_heads, "head_dim": 128,
                   "page": 16},
        "cpu_baseline": {"value": gbs, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def measure_prefill_append(K, torch, h, pool, npool, kd, vd, sid, pos, pt, Hkv, reps=5):
    """Quantise-on-append of one sequence's prefill (the last sequence of the
    cache build, appended again: the same bytes are rewritten), `reps` calls
    back to back on the device.  The kernel is bound by its fixed-order fp32
    rotation (fmaf chains): 2 x 128 x 128 flop per token, KV head and K|V,
    against the fp32 FMA rate of the SMs at the maximum SM clock."""
    n = int(kd.shape[0])
    for _ in range(2):
        K.kvq_append(h, pool, npool, kd, vd, sid, pos, pt)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        K.kvq_append(h, pool, npool, kd, vd, sid, pos, pt)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    flop = n * Hkv * 2 * 2 * 128 * 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    peak = sms * 128 * 2 * 2.07e9 / 1e12      # fp32 FMA lanes x 2 flop x 2070 MHz
    achieved = flop / (us * 1e-6) / 1e12
    return {"tokens": n, "kv_heads": Hkv, "us_per_call": us, "tokens_per_s": n / (us * 1e-6),
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "kernel": "append_int2_kernel",
                         "peak_kind": f"nominal fp32 FMA rate: {sms} SMs x 128 lanes x 2 flop x "
                                      f"2070 MHz (no measured fp32 peak on this pool)"},
            "calls": reps}


def measure_workload(K, torch, wl, splits_list, steps, warmup, l2, peak, cpu_seconds=0.0):
    """The decode step (kvq_append_decode: append each sequence's token at
    position len-1, decode over len tokens) on one of the other workloads.
    A cache smaller than twice L2 is replicated and the steps cycle through the
    replicas (one pool, one page table per replica).  Returns one dict per split
    count, with the oracle's rate on the workload's first (sequence, KV head)
    when cpu_seconds > 0."""
    B, H, Hkv = wl.batch, wl.num_heads, wl.num_kv_heads
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    lens = W.seq_lens(wl)
    pt_np, npool = W.page_table(wl)
    cache_bytes = int(lens.sum()) * Hkv * W.cache_bytes_per_token_head("int2")
    R = replicas_for(cache_bytes, l2)
    h = K.kvq_create(K.make_layout(H, Hkv, wl.clip_k, wl.clip_v))
    K.kvq_set_rotation(h, torch.from_numpy(W.rotations(wl)).cuda(),
                       torch.from_numpy(W.key_mean(wl)).cuda())
    rec = K.kvq_page_bytes(h)
    pool = torch.zeros(R * npool * rec, dtype=torch.uint8, device="cuda")
    pt0 = i32(pt_np)
    t_build = time.perf_counter()
    for g0 in range(0, B, 4):
        seqs = list(range(g0, min(B, g0 + 4)))
        n = [int(lens[b]) - 1 for b in seqs]
        Ks = W.tokens_many(wl, 0, seqs, 0, 0, n)
        Vs = W.tokens_many(wl, 0, seqs, 1, 0, n)
        for b, k, v, m in zip(seqs, Ks, Vs, n):
            if m > 0:
                K.kvq_append(h, pool, R * npool, dev(k), dev(v), i32(np.full(m, b)),
                             i32(np.arange(m)), pt0)
    for r in range(1, R):
        pool[r * npool * rec:(r + 1) * npool * rec].copy_(pool[:npool * rec])
    pts = i32(np.stack([np.where(pt_np >= 0, pt_np + r * npool, -1) for r in range(R)]))
    torch.cuda.synchronize()
    t_build = time.perf_counter() - t_build
    k_new = np.stack([W.token_at(wl, 0, b, 0, int(lens[b]) - 1) for b in range(B)])
    v_new = np.stack([W.token_at(wl, 0, b, 1, int(lens[b]) - 1) for b in range(B)])
    kd, vd, qd, seq_lens = dev(k_new), dev(v_new), dev(W.queries(wl)), i32(lens)
    out = torch.empty((B, H, 128), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    res = []
    for sp in splits_list:
        splits = sp or K.kvq_auto_splits(h, B, pt_np.shape[1])
        ws = torch.empty(K.kvq_workspace_bytes(h, B, splits), dtype=torch.uint8, device="cuda")

        def run(n, first):
            for i in range(first, first + n):
                K.kvq_append_decode(h, pool, R * npool, kd, vd, qd, pts[i % R], seq_lens, out, ws,
                                    splits)

        run(warmup, 0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(steps, warmup)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        K.kvq_profile_enable(h, True)
        run(steps, warmup + steps)
        kms, kn = K.kvq_profile_read(h)
        K.kvq_profile_enable(h, False)
        kern_ms = kms / max(1, kn)
        kgbs = cache_bytes / (kern_ms * 1e-3) / 1e9
        res.append({"splits": splits, "us_per_step": ms * 1e3, "steps_per_s": 1e3 / ms,
                    "cache_bytes_per_step": cache_bytes,
                    "cache_gbs": cache_bytes / (ms * 1e-3) / 1e9,
                    "kernel_us": kern_ms * 1e3, "kernel_gbs": kgbs, "kernel_frac_of_peak": kgbs / peak,
                    "l2": l2_note(cache_bytes, R, l2), "replicas": R, "steps": steps})
    assert K.kvq_get_status(h) == 0, f"device status bits set on {wl.name}"
    cpu = None
    if cpu_seconds > 0:
        gbs_cpu, n_cpu, el_cpu = cpu_oracle_rate(wl, min_seconds=cpu_seconds)
        cpu = {"value": gbs_cpu, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"float64 oracle on sequence 0 / KV head 0 ({int(lens[0])} tokens), "
                         f"{n_cpu} steps in {el_cpu:.1f} s"}
    out_d = {"workload": wl.name, "batch": B, "heads": H, "kv_heads": Hkv,
             "ctx": int(lens.max()) if wl.ragged else int(wl.ctx),
             "cache_build_s": round(t_build, 1), "cpu_baseline": cpu}
    if wl.ragged:
        out_d["ctx_min"] = int(lens.min())
        out_d["tokens"] = int(lens.sum())
    if len(res) == 1:
        out_d.update(res[0])
    else:
        out_d["by_splits"] = res
    del pool
    return out_d



def run_ours(args):
    import torch

    from rotated_int2_kv_kvq_gb300 import kvq as K

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    K.load_library()
    wl = W.WORKLOADS[args.workload]
    if args.batch:
        import dataclasses

        wl = dataclasses.replace(wl, batch=args.batch)
    B, H, Hkv, ctx = wl.batch, wl.num_heads, wl.num_kv_heads, wl.ctx
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    lens = W.seq_lens(wl)
    pt_np, npool = W.page_table(wl)
    pt = i32(pt_np)
    max_pages = pt_np.shape[1]
    layout = K.make_layout(H, Hkv, wl.clip_k, wl.clip_v)
    h = K.kvq_create(layout)
    K.kvq_set_rotation(h, torch.from_numpy(W.rotations(wl)).cuda(),
                       torch.from_numpy(W.key_mean(wl)).cuda())
    pool = torch.zeros(npool * K.kvq_page_bytes(h), dtype=torch.uint8, device="cuda")
    bf16_pool = None
    if not args.no_bf16:
        bf16_pool = torch.zeros(npool * K.kvq_bf16_page_bytes(h), dtype=torch.uint8,
                                device="cuda")
    # build the cache: positions [0, len-1) of every sequence
    t_build = time.perf_counter()
    for g0 in range(0, B, 4):
        seqs = list(range(g0, min(B, g0 + 4)))
        n = [int(lens[s]) - 1 for s in seqs]
        Ks = W.tokens_many(wl, 0, seqs, 0, 0, n)
        Vs = W.tokens_many(wl, 0, seqs, 1, 0, n)
        for s, k, v, m in zip(seqs, Ks, Vs, n):
            sid, pos = i32(np.full(m, s)), i32(np.arange(m))
            kd, vd = dev(k), dev(v)
            K.kvq_append(h, pool, npool, kd, vd, sid, pos, pt)
            if bf16_pool is not None:
                K.kvq_bf16_append(h, bf16_pool, npool, kd, vd, sid, pos, pt)
    torch.cuda.synchronize()
    t_build = time.perf_counter() - t_build
    prefill = measure_prefill_append(K, torch, h, pool, npool, kd, vd, sid, pos, pt, Hkv)
    # step inputs: the token at position len-1 of every sequence, and the queries
    k_new = np.stack([W.token_at(wl, 0, b, 0, int(lens[b]) - 1) for b in range(B)])
    v_new = np.stack([W.token_at(wl, 0, b, 1, int(lens[b]) - 1) for b in range(B)])
    q_np = W.queries(wl)
    kd_new, vd_new, qd = dev(k_new), dev(v_new), dev(q_np)
    sid, pos = i32(np.arange(B)), i32(lens - 1)
    seq_lens = i32(lens)
    splits = args.splits or K.kvq_auto_splits(h, B, max_pages)
    ws = torch.empty(K.kvq_workspace_bytes(h, B, splits), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, H, 128), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    # One decode step through the library's one-call form: append each
    # sequence's token at position len-1, then decode (3 kernel launches).
    def step():
        K.kvq_append_decode(h, pool, npool, kd_new, vd_new, qd, pt, seq_lens, out, ws, splits)

    # The same step as two calls (append, then decode: 4 launches).
    def step_two_calls():
        K.kvq_append(h, pool, npool, kd_new, vd_new, sid, pos, pt)
        K.kvq_decode(h, pool, npool, qd, pt, seq_lens, out, ws, splits)

    def timed(fn, steps, warmup, profile=False):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        if profile:
            K.kvq_profile_enable(h, True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        kern = K.kvq_profile_read(h) if profile else None
        if profile:
            K.kvq_profile_enable(h, False)
        ms = max_over_ranks(ms, dist)
        return ms, kern

    # Headline region: plain steps.  The kernel timing below records CUDA events
    # between the chained kernels, which stops them overlapping, so it runs as a
    # separate timed region of the same steps.
    clocks = Clocks(local)
    clocks.start()
    ms, _ = timed(step, args.steps, args.warmup)
    # A short timed region may end before the sampler's next line: keep the GPU
    # on the same (untimed) step until three samples under load exist.
    extra, t_extra = 0, time.time()
    while clocks.proc is not None and clocks.samples() < 3 and time.time() - t_extra < 10.0:
        for _ in range(100):
            step()
        torch.cuda.synchronize()
        extra += 100
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = "warm-up + timed steps" + (f" + {extra} untimed steps" if extra else "")
    pms, kern = timed(step, args.steps, max(3, args.warmup // 4), profile=True)
    assert K.kvq_get_status(h) == 0, "device status bits set during the benchmark"
    ms_step = ms / args.steps
    cache_bytes = int(lens.sum()) * Hkv * W.cache_bytes_per_token_head("int2")
    gbs_rank = cache_bytes / (ms_step * 1e-3) / 1e9
    value = whole_job_rate(cache_bytes, ms_step, world) / 1e9
    peak, peak_kind = measured_peaks()
    kern_ms = kern[0] / max(1, kern[1]) if kern else None
    achieved = cache_bytes / (kern_ms * 1e-3) / 1e9 if kern_ms else None
    traffic = profiled_traffic()

    # e2e: the same step through the public API with pinned host buffers: copy this
    # step's inputs (q and the new K/V token) in and the attention output out.
    # The step's inputs (q, new K, new V) sit in one pinned host buffer and
    # arrive with one copy into one device buffer; the calls take views of it.
    # A serving loop overlaps the copies with the neighbouring steps' compute:
    # step i's inputs are copied in on an input-copy stream into one of two
    # buffers while step i-1 computes, and step i's output is copied out on an
    # output-copy stream while step i+1 computes (two copy streams, so an input
    # copy never queues behind the previous step's output copy).  Every step
    # still moves its bytes through the public API inside the timed region; the
    # cache and the step order are the same as above.
    nq, nk = q_np.size, k_new.size
    in_h = torch.from_numpy(np.concatenate([q_np.reshape(-1), k_new.reshape(-1),
                                            v_new.reshape(-1)]).view(np.int16)).pin_memory()
    in_d = [torch.empty_like(in_h, device="cuda") for _ in range(2)]
    views = [(d[:nq].view(qd.shape), d[nq:nq + nk].view(kd_new.shape),
              d[nq + nk:].view(vd_new.shape)) for d in in_d]
    out_d = [torch.empty((B, H, 128), dtype=torch.float32, device="cuda") for _ in range(2)]
    out_h = [torch.empty((B, H, 128), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_done:
        e.record(stream)
    for e in ev_out:
        e.record(stream)

    def e2e_steps(n):
        for i in range(n):
            sl = i % 2
            with torch.cuda.stream(h2d_stream):
                h2d_stream.wait_event(ev_done[sl])            # buffer free (step i - 2 done)
                in_d[sl].copy_(in_h, non_blocking=True)
                ev_in[sl].record(h2d_stream)
            stream.wait_event(ev_in[sl])
            stream.wait_event(ev_out[sl])                     # out_d[sl] read out (step i - 2)
            q2, k2, v2 = views[sl]
            K.kvq_append_decode(h, pool, npool, k2, v2, q2, pt, seq_lens, out_d[sl], ws, splits)
            ev_done[sl].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_done[sl])
                out_h[sl].copy_(out_d[sl], non_blocking=True)
                ev_out[sl].record(d2h_stream)
        stream.wait_stream(h2d_stream)
        stream.wait_stream(d2h_stream)                      # the last output is on the host

    e2e_steps(max(3, args.warmup // 2))
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist)
    e2e_gbs = cache_bytes / (e2e_ms / args.steps * 1e-3) / 1e9 * world
    h2d = in_h.numel() * 2
    d2h = out_h[0].numel() * 4

    # BF16 comparison kernel: same step on the BF16 cache
    bf16 = None
    if bf16_pool is not None:
        ws16 = torch.empty(K.kvq_bf16_workspace_bytes(h, B, 0), dtype=torch.uint8, device="cuda")

        def bf16_step():
            K.kvq_bf16_append(h, bf16_pool, npool, kd_new, vd_new, sid, pos, pt)
            K.kvq_bf16_decode(h, bf16_pool, npool, qd, pt, seq_lens, out, ws16, 0)

        bsteps = max(3, args.steps // 4)
        bms, bkern = timed(bf16_step, bsteps, max(3, args.warmup // 4), profile=True)
        bbytes = int(lens.sum()) * Hkv * W.cache_bytes_per_token_head("bf16")
        bkern_ms = bkern[0] / max(1, bkern[1])
        bf16 = {"steps_per_s": bsteps / (bms * 1e-3), "ms_per_step": bms / bsteps,
                "cache_bytes_per_step": bbytes,
                "kernel_gbs": bbytes / (bkern_ms * 1e-3) / 1e9,
                "kernel_frac_of_peak": bbytes / (bkern_ms * 1e-3) / 1e9 / peak,
                "int2_speedup_steps": (args.steps / (ms * 1e-3)) / (bsteps / (bms * 1e-3))}

    # Folded rotations: with R_K folded into the query projection (q R_K passed in,
    # KVQ_Q_ROTATED) and R_V into W_V / W_O (rotated-basis output,
    # KVQ_OUT_ROTATED) a step does no rotation work at all.  The time saved is the
    # rotations' overhead (the OptR page states about 2 % or less).
    hf = K.kvq_create(K.make_layout(H, Hkv, wl.clip_k, wl.clip_v, out_rotated=True,
                                    q_rotated=True))
    Rb = W.rotations(wl)
    K.kvq_set_rotation(hf, torch.from_numpy(Rb).cuda(), torch.from_numpy(W.key_mean(wl)).cuda())
    qf64 = W.bf16_bits_to_float(q_np).astype(np.float64)
    qrot_np = np.stack([qf64[:, hh] @ Rb[0, hh // (H // Hkv)].astype(np.float64)
                        for hh in range(H)], axis=1)
    qrd = dev(W.to_bf16_bits(qrot_np.astype(np.float32)))

    def folded_step():
        K.kvq_append_decode(hf, pool, npool, kd_new, vd_new, qrd, pt, seq_lens, out, ws, splits)

    fms, _ = timed(folded_step, args.steps, args.warmup)
    tms, _ = timed(step_two_calls, args.steps, args.warmup)
    ums, _ = timed(step, args.steps, args.warmup)      # the default step again, back to back
    folded = {"ms_per_step": fms / args.steps, "default_ms_per_step": ums / args.steps,
              "rotation_overhead_pct": 100.0 * (ums - fms) / fms,
              "flags": "KVQ_Q_ROTATED | KVQ_OUT_ROTATED"}
    two_calls = {"ms_per_step": tms / args.steps, "launches_per_step": 4,
                 "calls": "kvq_append + kvq_decode"}
    assert K.kvq_get_status(hf) == 0, "device status bits set during the folded benchmark"

    # The OptR setting: 64 sink + 256 recent tokens kept in BF16 beside the INT2
    # cache.  A step appends the new token to both caches (the INT2 copy is there
    # for when the token leaves the window) and decodes with the window: one
    # kvq_append_decode_window call (3 launches); the same step as three separate
    # calls (5 launches) is timed beside it.
    window = None
    if bf16_pool is not None:
        sink, recent = 64, 256

        def window_step():
            K.kvq_append_decode_window(h, pool, npool, bf16_pool, npool, pt, kd_new, vd_new, qd, pt,
                                       seq_lens, sink, recent, out, ws, splits)

        def window_step_separate():
            K.kvq_append(h, pool, npool, kd_new, vd_new, sid, pos, pt)
            K.kvq_bf16_append(h, bf16_pool, npool, kd_new, vd_new, sid, pos, pt)
            K.kvq_decode_window(h, pool, npool, bf16_pool, npool, pt, qd, pt, seq_lens, sink,
                                recent, out, ws, splits)

        wms, _ = timed(window_step, args.steps, args.warmup)
        _, wkern = timed(window_step, args.steps, max(3, args.warmup // 4), profile=True)
        wsep, _ = timed(window_step_separate, args.steps, args.warmup)
        n_win = [min(int(L), sink + recent) for L in lens]
        wbytes = Hkv * sum((int(L) - n) * W.cache_bytes_per_token_head("int2") +
                           n * W.cache_bytes_per_token_head("bf16") for L, n in zip(lens, n_win))
        window = {"sink": sink, "recent": recent, "ms_per_step": wms / args.steps,
                  "steps_per_s": args.steps / (wms * 1e-3),
                  "cache_bytes_per_step": wbytes,
                  "cache_gbs": wbytes / (wms / args.steps * 1e-3) / 1e9,
                  "int2_kernel_ms": wkern[0] / max(1, wkern[1]),
                  "effective_bits": W.effective_bits_window(ctx, sink, recent),
                  "effective_bits_64k": W.effective_bits_window(65536, sink, recent),
                  "launches_per_step": 3,
                  "separate_calls_ms_per_step": wsep / args.steps,
                  "separate_calls": "kvq_append + kvq_bf16_append + kvq_decode_window"}
        assert K.kvq_get_status(h) == 0, "device status bits set during the window benchmark"

    # the other workloads of the same path (sub-objects of this line)
    l2 = l2_bytes(torch)
    configs = None
    if not args.no_configs and world == 1 and not args.batch:
        cs, cw = max(50, min(args.steps, 200)), min(max(3, args.warmup), 20)
        cpu_s = 0.0 if args.no_cpu else 3.0
        configs = {
            "tiny_1k": measure_workload(K, torch, W.WORKLOADS["tiny_1k"], [0], cs, cw, l2, peak,
                                        cpu_s),
            "long_128k": measure_workload(K, torch, W.WORKLOADS["long_128k"], [64, 128, 256], cs,
                                          cw, l2, peak, cpu_s),
            "ragged_64": measure_workload(K, torch, W.WORKLOADS["ragged_64"], [0], cs, cw, l2,
                                          peak, cpu_s),
        }
        fs, _ = measure_full_stack(K, torch, max(20, min(args.steps, 100)), min(max(3, args.warmup), 10),
                                   local, None, clocks_on=False)
        configs["full_stack_36l"] = fs
        torch.cuda.empty_cache()

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu:
        sample = oracle_sample_setup(wl)
        parity = parity_sample(pool.cpu().numpy(), pt_np, sample, wl)
        gbs_cpu, n_cpu, el_cpu = cpu_oracle_rate(wl, min_seconds=10.0, sample=sample)
        cpu = {"value": gbs_cpu, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"float64 oracle on sequence 0 / KV head 0: re-quantise one token and "
                         f"decode {H // Hkv} query heads over {ctx} tokens per step, "
                         f"{n_cpu} steps in {el_cpu:.1f} s"}
        allc = cpu_oracle_rate_all_cores(wl, seconds=10.0)
        if allc is not None:
            cpu["all_cores"] = {"value": allc[0], "unit": UNIT, "cores": allc[1], "kind": "oracle",
                                "sample": f"the same step, one process per core on its own "
                                          f"(sequence, KV head): {allc[2]} steps in "
                                          f"{allc[3]:.1f} s"}

    launches = 3 * args.steps       # append + q-rotation, split-K attention, split merge
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int2 codes, fp16 mma, fp32 accumulate",
        "data": "synthetic",
        "config": {"workload": wl.name, "batch": B, "ctx": ctx, "heads": H, "kv_heads": Hkv,
                   "head_dim": 128, "page": 16, "splits": splits,
                   "l2": l2_note(cache_bytes, 1, l2),
                   "cache_build_s": round(t_build, 1)},
        "steps_per_s": world * args.steps / (ms * 1e-3),
        "pct_of_hbm_peak": 100.0 * gbs_rank / peak,
        "effective_bits": W.effective_bits(128),
        "cache_bytes_per_step": cache_bytes,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                     "kernel": "decode_int2_kernel", "peak_kind": peak_kind,
                     "kernel_ms": kern_ms, "kernel_launches": kern[1] if kern else None,
                     "profiled_region_ms_per_step": pms / args.steps},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_gbs, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "bf16_comparison": bf16,
        "prefill_append": prefill,
        "bf16_window": window,
        "folded_rotations": folded,
        "two_call_step": two_calls,
        "clocks": clk,
        "gpu_launches": launches,
        "parity": parity,
        "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# The 36-layer stack: one decode step = every layer appends one token per
# sequence and decodes, captured as one CUDA graph
# ---------------------------------------------------------------------------

FULL_STACK_METRIC = "decode steps/s of a 36-layer stack (append + INT2 decode per layer)"


def measure_full_stack(K, torch, steps, warmup, local=0, dist=None, clocks_on=True):
    """Build the 36 layers' caches (8192-token prefill per sequence), capture
    one decode step (every layer appends one token per sequence and decodes)
    as a CUDA graph and time `steps` replays; also the same step run eagerly
    and as an unfused graph (append and decode as separate calls)."""
    from rotated_int2_kv_kvq_gb300.pipeline import DecodeStepGraph, LayerCache

    wl = W.WORKLOADS["full_stack_36l"]
    B, H, Hkv, L, P, S = (wl.batch, wl.num_heads, wl.num_kv_heads, wl.layers, wl.prefill,
                          wl.decode_steps)
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    t_build = time.perf_counter()
    layers = []
    K_tab = torch.empty((S, L, B, Hkv, 128), dtype=torch.int16, device="cuda")
    V_tab = torch.empty_like(K_tab)
    q_tab = torch.empty((S, L, B, H, 128), dtype=torch.int16, device="cuda")
    for l in range(L):
        h = K.kvq_create(K.make_layout(H, Hkv, wl.clip_k, wl.clip_v))
        K.kvq_set_rotation(h, torch.from_numpy(W.rotations(wl, l)).cuda(),
                           torch.from_numpy(W.key_mean(wl, l)).cuda())
        pt_np, npool = W.page_table(wl, l)
        pool = torch.zeros(npool * K.kvq_page_bytes(h), dtype=torch.uint8, device="cuda")
        pt = i32(pt_np)
        Ks = W.tokens_many(wl, l, range(B), 0, 0, P + S)
        Vs = W.tokens_many(wl, l, range(B), 1, 0, P + S)
        for b in range(B):
            K.kvq_append(h, pool, npool, dev16(Ks[b][:P]), dev16(Vs[b][:P]), i32(np.full(P, b)),
                         i32(np.arange(P)), pt)
        K_tab[:, l] = dev16(np.stack([Ks[b][P:] for b in range(B)], axis=1))
        V_tab[:, l] = dev16(np.stack([Vs[b][P:] for b in range(B)], axis=1))
        q_tab[:, l] = dev16(np.stack([W.queries(wl, l, st) for st in range(S)]))
        layers.append(LayerCache(h, pool, npool, pt))
    lens_tab = i32(np.stack([np.full(B, P + st + 1) for st in range(S)]))
    pos_tab = i32(np.stack([np.full(B, P + st) for st in range(S)]))
    torch.cuda.synchronize()
    t_build = time.perf_counter() - t_build

    def make(fused):
        g = DecodeStepGraph(layers, B, H, Hkv, fused=fused)
        g.load(K_tab[0], V_tab[0], q_tab[0], lens_tab[0], pos_tab[0])
        return g

    stream = torch.cuda.current_stream()

    def timed(g, n, warm, graph=True):
        """Step i uses the inputs of decode step i mod S (positions P + i mod S)."""
        def one(i):
            s = i % S
            g.load(K_tab[s], V_tab[s], q_tab[s], lens_tab[s], pos_tab[s])
            if graph:
                g.replay()
            else:
                g.run()

        for i in range(warm):
            one(i)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            one(warm + i)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), dist)

    fused_g = make(True)
    fused_g.capture()
    clocks = Clocks(local) if clocks_on else None
    if clocks:
        clocks.start()
    ms = timed(fused_g, steps, warmup)
    clk = None
    if clocks:
        extra, t_extra = 0, time.time()
        while clocks.proc is not None and clocks.samples() < 3 and time.time() - t_extra < 10.0:
            for _ in range(20):
                fused_g.replay()
            torch.cuda.synchronize()
            extra += 20
        clk = clocks.stop()
        if clk is not None:
            clk["window"] = "warm-up + timed steps" + (f" + {extra} untimed steps" if extra else "")
    n_eager = max(3, steps // 4)
    eager_ms = timed(fused_g, n_eager, 3, graph=False) / n_eager
    unfused_g = make(False)
    unfused_g.capture()
    unfused_ms = timed(unfused_g, steps, warmup) / steps
    status = [K.kvq_get_status(c.h) for c in layers]
    assert not any(status), f"device status bits set: {status}"
    ms_step = ms / steps
    # algorithmic INT2 cache bytes per step at the mean context of the S steps
    mean_ctx = P + (S + 1) / 2.0
    cache_bytes = L * B * Hkv * mean_ctx * W.cache_bytes_per_token_head("int2")
    peak, peak_kind = measured_peaks()
    l2 = l2_bytes(torch)
    res = {
        "workload": wl.name, "layers": L, "batch": B, "heads": H, "kv_heads": Hkv, "prefill": P,
        "ctx": f"{P + 1}..{P + S}", "splits": fused_g.splits, "steps": steps,
        "steps_per_s": 1e3 / ms_step, "ms_per_step": ms_step, "per_layer_us": ms_step * 1e3 / L,
        "cache_bytes_per_step": cache_bytes,
        "cache_gbs": cache_bytes / (ms_step * 1e-3) / 1e9,
        "pct_of_hbm_peak": 100.0 * cache_bytes / (ms_step * 1e-3) / 1e9 / peak,
        "peak_kind": peak_kind, "launches_per_step": 3 * L, "graph": True,
        "eager_ms_per_step": eager_ms, "unfused_graph_ms_per_step": unfused_ms,
        "l2": l2_note(cache_bytes, 1, l2) + f" (over {L} pools)",
        "cache_build_s": round(t_build, 1),
    }
    del layers, K_tab, V_tab, q_tab
    return res, clk


def run_workload(args):
    """One of the other workloads alone (the sub-objects of the default line's
    `configs`), on one GPU: `--splits` fixes the split count (default: the
    automatic one; long_128k: 64, 128 and 256)."""
    import torch

    from rotated_int2_kv_kvq_gb300 import kvq as K

    K.load_library()
    wl = W.WORKLOADS[args.workload]
    splits = [args.splits] if args.splits else ([64, 128, 256] if wl.name == "long_128k" else [0])
    peak, peak_kind = measured_peaks()
    r = measure_workload(K, torch, wl, splits, max(20, args.steps), max(3, args.warmup),
                         l2_bytes(torch), peak, 0.0 if args.no_cpu else 3.0)
    first = r["by_splits"][0] if "by_splits" in r else r
    line = {
        "metric": f"{wl.name}: INT2 decode step, cache GB/s", "value": first["cache_gbs"],
        "unit": UNIT, "n_gpus": 1, "steps": max(20, args.steps), "warmup": max(3, args.warmup),
        "ms_per_step": first["us_per_step"] * 1e-3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int2 codes, fp16 mma, fp32 accumulate",
        "data": "synthetic", "config": {"workload": wl.name}, "peak_kind": peak_kind,
        "result": r,
    }
    print(json.dumps(line), flush=True)


def run_full_stack(args):
    import torch

    from rotated_int2_kv_kvq_gb300 import kvq as K

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    K.load_library()
    steps = min(args.steps, 1000)
    r, clk = measure_full_stack(K, torch, steps, args.warmup, local, dist)
    line = {
        "metric": FULL_STACK_METRIC, "value": world * r["steps_per_s"], "unit": "steps/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int2 codes, fp16 mma, fp32 accumulate", "data": "synthetic",
        "config": {k: r[k] for k in ("workload", "layers", "batch", "heads", "kv_heads",
                                     "prefill", "ctx", "splits", "l2", "cache_build_s")},
        "per_layer_us": r["per_layer_us"], "cache_gbs": r["cache_gbs"],
        "pct_of_hbm_peak": r["pct_of_hbm_peak"], "peak_kind": r["peak_kind"],
        "launches_per_step": r["launches_per_step"], "graph": True,
        "eager_ms_per_step": r["eager_ms_per_step"],
        "unfused_graph_ms_per_step": r["unfused_graph_ms_per_step"],
        "clocks": clk,
        "gpu_launches": r["launches_per_step"] * steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# OptR rotation calibration of one layer (off the decode path)
# ---------------------------------------------------------------------------

OPTR_METRIC = "OptR calibration of one layer (8 KV heads, 80 + 80 Adam steps): seconds"


def optr_flops_per_step(T, Nq, G, Dm, D=128):
    """Algorithmic fp32 flops of one key step plus one value step of one KV
    head with gradient: the objective's contractions (rotations, logits,
    attention products, post-W_O error and their transposes), not counting the
    matrix exponentials."""
    QG = Nq * G
    key = (2 * T * D * D) * 5 + (2 * QG * T * D) * 4 + (2 * Nq * G * D * Dm) * 2
    value = (2 * T * D * D) * 5 + (2 * QG * T * D) * 3 + (2 * Nq * G * D * Dm) * 2
    return key + value


def run_optr(args):
    import torch

    from rotated_int2_kv_kvq_gb300 import kvq as K

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    K.load_library()
    wl = W.WORKLOADS["qwen3_8b_32k"]
    T, Nq, Dm, steps = 4096, 64, 4096, 80
    H, G = wl.num_kv_heads, wl.num_heads // wl.num_kv_heads
    Kb, Vb, Qb, Wo = W.calibration_traces(wl, 0, T, Nq, Dm)
    d16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    inputs = (d16(Kb), d16(Vb), d16(Qb), torch.from_numpy(Wo).cuda(),
              torch.from_numpy(W.rotations(wl)).cuda(), torch.from_numpy(W.key_mean(wl)).cuda(),
              wl.clip_k, wl.clip_v)
    ws = torch.empty(K.kvq_optr_workspace_bytes(H, T, Nq, G, Dm), dtype=torch.uint8, device="cuda")
    for _ in range(max(1, args.warmup)):
        K.kvq_optr_calibrate(*inputs, steps=2, workspace=ws)
    torch.cuda.synchronize()
    reps = max(1, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        R, hist = K.kvq_optr_calibrate(*inputs, steps=steps, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / reps
    h = hist.cpu().numpy()
    flops = optr_flops_per_step(T, Nq, G, Dm) * steps * H
    nominal = 152 * 128 * 2 * 2.07e9 / 1e12       # fp32 FMA, TFLOP/s
    cpu = None
    if not args.no_cpu:
        from oracle import optr

        f = lambda b: W.bf16_bits_to_float(b).astype(np.float64)
        Wh = Wo.reshape(H, Dm, G, 128).transpose(0, 2, 1, 3)
        R0 = W.rotations(wl).astype(np.float64)
        mu = W.key_mean(wl).astype(np.float64)
        n_cpu = 2
        t0 = time.perf_counter()
        optr.calibrate(R0[0, 0], R0[1, 0], f(Kb[0]), f(Vb[0]), f(Qb[0]), Wh[0], mu[0], wl.clip_k,
                       wl.clip_v, steps=n_cpu)
        el = time.perf_counter() - t0
        cpu_layer_s = el / n_cpu * steps * H
        cpu = {"value": cpu_layer_s, "unit": "s per layer (extrapolated)", "cores": 1,
               "kind": "oracle",
               "sample": f"float64 oracle, KV head 0: {n_cpu} key + {n_cpu} value steps in "
                         f"{el:.1f} s, scaled to {steps} + {steps} steps x {H} heads"}
    line = {
        "metric": OPTR_METRIC, "value": sec, "unit": "s", "n_gpus": 1, "steps": reps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3 / (2 * steps), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "optr_calib", "kv_heads": H, "group": G, "calib_tokens": T,
                   "query_positions": Nq, "d_model": Dm, "adam_steps": steps, "lr": 1e-3},
        "roofline": {"bound": "alu", "achieved": flops / sec / 1e12, "peak": nominal,
                     "unit": "TFLOP/s", "frac": flops / sec / 1e12 / nominal, "traffic": None,
                     "peak_kind": "fp32 FMA nominal: 152 SMs x 128 lanes x 2 x 2.07 GHz",
                     "note": "products with 64-multiple M and N (except those by a 128 x 128 "
                             "matrix) run on mma.sync tensor cores with each fp32 operand split into three bf16 parts (six products), the rest in "
                             "fp32; achieved counts the algorithmic fp32 flops once"},
        "losses": {"key": [float(h[0, 0].mean()), float(h[0, -1].mean())],
                   "value": [float(h[1, 0].mean()), float(h[1, -1].mean())]},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "full_stack_36l":
        run_full_stack(args)
    elif args.workload == "optr_calib":
        run_optr(args)
    elif args.workload in ("tiny_1k", "long_128k", "ragged_64"):
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
