"""Benchmark of one decode step over a paged, quantized KV cache.

A step is the whole hot path for every layer of a 32-layer model: quantize and
append one new K/V token per sequence into the layer's pool, then run paged
decode attention of the step's Q over each sequence's cached K/V.  The default
workload is 64 sequences x 2048 tokens, 32 Q / 8 KV heads, head_dim 128, block
16, INT8 per-group-128 KV; every layer has its own pool (32 pools, 9.8 GB), so
no layer's reads can be served from L2.

Prints one JSON line.  `value` is the effective HBM bandwidth of the step:
algorithmic bytes (KV codes + scales + Q + block tables + context lengths read
by decode, plus the append's fp16 input and code/scale output) over the
device-timed step.  Also reported: decode tokens/s, the decode launch's
roofline fraction, an end-to-end number through the Python API with host
buffers, and the CPU oracle timed on a bounded sample on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Paged quantized-KV decode: effective HBM GB/s (% of peak) and decode tok/s"
FORMAT_NAME = {0: "fp16", 1: "int8 per-token", 2: "int8 per-channel", 3: "int8 per-group",
               4: "fp8 e4m3 per-token", 5: "int4 per-group", 6: "fp8 e5m2 (no scale)"}
ESIZE = {0: 2, 1: 1, 2: 1, 3: 1, 4: 1, 5: 0.5, 6: 1}  # bytes per code
GROUPED = (3, 5)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "decode_traffic.json")
KERNEL_SOURCES = ["paged_quantized_kv_kvq_gb300/csrc/kvq_decode_impl.cuh",
                  "paged_quantized_kv_kvq_gb300/csrc/kvq_common.cuh",
                  "paged_quantized_kv_kvq_gb300/csrc/kvq_decode.cu"]


# ----------------------------------------------------------------- byte model
def layer_bytes(w, fmt, group, seqs=None):
    """Algorithmic bytes of one layer's append + decode for the given sequences."""
    seqs = np.arange(w.S) if seqs is None else np.asarray(seqs)
    L = w.context_lens[seqs].astype(np.int64)
    n = len(seqs)
    es = ESIZE[fmt]
    tok = int(L.sum())
    codes = int(tok * w.Hkv * w.D * 2 * es)
    if fmt in GROUPED:
        scales = tok * w.Hkv * 2 * (w.D // group) * 4
    elif fmt in (1, 4):
        scales = tok * 2 * 4
    elif fmt == 2:
        scales = 2 * w.Hkv * w.D * 4
    else:
        scales = 0
    q = n * w.Hq * w.D * 2
    tables = int(((L + w.bs - 1) // w.bs).sum()) * 4 + n * 4
    decode = codes + scales + q + tables
    app_scales = (n * w.Hkv * 2 * (w.D // max(group, 1)) * 4 if fmt in GROUPED else
                  {1: n * 2 * 4, 4: n * 2 * 4}.get(fmt, 0))
    append = n * w.Hkv * w.D * 2 * 2 + n * 8 + int(n * w.Hkv * w.D * 2 * es) + app_scales
    unique_codes = codes
    unique_decode = decode
    if w.shared_prefix_tokens and n > 1:
        # the shared prefix blocks exist once in HBM
        dup = (n - 1) * w.shared_prefix_tokens
        unique_codes -= int(dup * w.Hkv * w.D * 2 * es)
        unique_decode -= int(dup * w.Hkv * w.D * 2 * es)
        if fmt in GROUPED:
            unique_decode -= dup * w.Hkv * 2 * (w.D // group) * 4
        elif fmt in (1, 4):
            unique_decode -= dup * 2 * 4
    return {"decode": decode, "append": append, "codes": codes, "scales": scales,
            "unique_codes": unique_codes, "unique_decode": unique_decode,
            "output": n * w.Hq * w.D * 4}


def step_bytes(w):
    tot = {"decode": 0, "append": 0, "codes": 0, "scales": 0, "unique_codes": 0,
           "unique_decode": 0, "output": 0}
    for fmt, group in w.layer_formats:
        for k, v in layer_bytes(w, fmt, group).items():
            tot[k] += v
    return tot


def kernel_sha():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()


def read_traffic(workload):
    try:
        rec = json.load(open(PROFILE_TRAFFIC))
    except (OSError, ValueError):
        return None
    if rec.get("kernel_sha256") != kernel_sha() or rec.get("workload") != workload:
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- ranks
def max_over_ranks(x, dist, device):
    """The slowest rank's time: the job ends when its last rank does (every
    rank reaches this call; no-op for a single process)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step, world, ms_per_step):
    """Whole-job GB/s: every rank processes its own replica of the step (weak
    scaling), all within the slowest rank's step time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0}, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        busy = [x for x in sm if mx and x > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def gpu_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        parts = [p for p in vis.split(",") if p.strip()]
        if local_rank < len(parts) and parts[local_rank].strip().isdigit():
            return int(parts[local_rank])
    return local_rank


# ----------------------------------------------------------------- kernel breakdown
LAUNCH_RECORDS = {"decode": os.path.join(ROOT, "profiles", "decode_launches.json"),
                  "prefill": os.path.join(ROOT, "profiles", "prefill_launches.json")}


def library_sha():
    """Hash of every library source (kernels, launchers, the C ABI)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "paged_quantized_kv_kvq_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            h.update(open(os.path.join(d, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "kvq.h"), "rb").read())
    return h.hexdigest()


def kernel_breakdown(kind, workload, layers, ms_step):
    """Per-kernel device times of one layer's launches, from the committed ncu
    launch list of this very library build (profiles/<kind>_launches.json,
    `gpu__time_duration.sum`, launches serialised and cold), with each
    kernel's share of the layer apportioned to this run's live step time
    (live, a layer's launches overlap through programmatic dependent launch,
    so the serialised sum exceeds the live time per layer).  Unavailable when
    the record was taken on other sources or another workload."""
    try:
        rec = json.load(open(LAUNCH_RECORDS[kind]))
    except (OSError, ValueError) as e:
        return {"unavailable": "no launch record: %s" % str(e)[:80]}
    if rec.get("library_sha256") != library_sha() or rec.get("workload") != workload:
        return {"unavailable": "the launch record was taken on other library sources or another "
                               "workload (%s)" % rec.get("workload")}
    ks = rec["kernels"]
    tot = sum(k["avg_us"] * k["per_layer"] for k in ks.values())
    live = 1e3 * ms_step / layers
    out = {name: {"ncu_avg_us": k["avg_us"], "launches_per_layer": k["per_layer"],
                  "share": round(k["avg_us"] * k["per_layer"] / tot, 4),
                  "apportioned_live_us_per_layer": round(live * k["avg_us"] * k["per_layer"] / tot, 3)}
           for name, k in ks.items()}
    return {"kernels": out, "ncu_sum_per_layer_us": round(tot, 3),
            "live_step_per_layer_us": round(live, 3), "source": rec.get("source", "")}


# ----------------------------------------------------------------- oracle leg
def oracle_sample(w, fmt, group, seqs, oracle_mod, synth, kv_heads=None):
    """Set up the oracle's cache for `seqs` of layer 0 (untimed); returns a
    callable that runs the step (append the new tokens, decode) on it.  With
    kv_heads = n, only the first n KV heads (and their Q heads) take part."""
    hk = w.Hkv if kv_heads is None else kv_heads
    hq = hk * w.G
    table = w.block_table[seqs]
    nblk = [(int(w.context_lens[s]) + w.bs - 1) // w.bs for s in seqs]
    used = np.unique(np.concatenate([table[i, :nblk[i]] for i in range(len(seqs))]))
    remap = np.full(w.num_blocks, -1, np.int64)
    remap[used] = np.arange(len(used))
    ctable = np.where(table >= 0, remap[np.clip(table, 0, None)], 0).astype(np.int32)
    cache = oracle_mod.OracleCache(fmt, len(used), w.bs, hk, w.D, group)
    idx = w.fill_token_index()
    keep = np.isin(idx[:, 0], seqs)
    if w.shared_prefix_tokens and 0 not in seqs:
        keep |= (idx[:, 0] == 0) & (idx[:, 1] < w.shared_prefix_tokens)
    slots = w.fill_slots()[keep]
    k, v = synth.kv_tokens(w, 0, idx[keep])
    k, v = np.ascontiguousarray(k[:, :hk]), np.ascontiguousarray(v[:, :hk])
    cs = remap[slots // w.bs] * w.bs + slots % w.bs
    if fmt == 2:
        cache.calibrate(k, v)
    cache.append(k, v, cs)
    ks, vs = synth.step_kv(w, 0)
    st = w.step_slots()[seqs]
    st = remap[st // w.bs] * w.bs + st % w.bs
    q = np.ascontiguousarray(synth.queries(w, 0)[seqs][:, :hq])
    lens = w.context_lens[seqs]
    ks, vs = np.ascontiguousarray(ks[seqs][:, :hk]), np.ascontiguousarray(vs[seqs][:, :hk])

    def run():
        cache.append(ks, vs, st)
        return cache.decode(q, ctable, lens)

    return run


def cpu_baseline(w, budget_s=12.0):
    """Time the oracle (as it stands) on host cores on a bounded sample of the
    workload: layer 0, the first n sequences, n sized to ~budget_s of work."""
    import oracle
    from paged_quantized_kv_kvq_gb300 import synth

    oracle.build()
    fmt, group = w.layer_formats[0]
    run1 = oracle_sample(w, fmt, group, [0], oracle, synth)
    t0 = time.perf_counter()
    run1()
    t1 = time.perf_counter() - t0
    n = int(max(1, min(w.S, round(budget_s / max(t1, 1e-3)))))
    seqs = list(range(n))
    run = oracle_sample(w, fmt, group, seqs, oracle, synth)
    t0 = time.perf_counter()
    run()
    once = time.perf_counter() - t0
    # repeat the same step (append rewrites the same slots) to ~budget_s of work
    reps = int(max(1, min(50, round(budget_s / max(once, 1e-3)))))
    t0 = time.perf_counter()
    for _ in range(reps):
        run()
    dt = (time.perf_counter() - t0) / reps
    b = layer_bytes(w, fmt, group, seqs)
    nbytes = b["decode"] + b["append"]
    return {"value": nbytes / dt / 1e9, "unit": "GB/s",
            "cores": min(oracle.num_threads(), n * w.Hq),
            "kind": "oracle",
            "sample": "layer 0 of %d, sequences 0..%d of %d (append of the step token + float64 "
                      "paged decode) run %d times, %.2f s of CPU work, %d algorithmic bytes per run"
                      % (w.layers, n - 1, w.S, reps, dt * reps, nbytes),
            "seconds": dt, "bytes": nbytes}


def cpu_baseline_prefill(w, budget_s=12.0):
    """Time the oracle (as it stands) on host cores on a bounded sample of the
    prefill workload: layer 0, sequence 0's whole prompt appended, then the
    causal attention of its last n query tokens (every Q head), n sized to
    ~budget_s of work; TFLOP/s on the same algorithmic count as the GPU leg."""
    import oracle
    from paged_quantized_kv_kvq_gb300 import synth

    oracle.build()
    fmt, group = w.layer_formats[0]
    Ls = int(w.context_lens[0])
    nb = (Ls + w.bs - 1) // w.bs
    cache = oracle.OracleCache(fmt, nb, w.bs, w.Hkv, w.D, group)
    idx = np.stack([np.zeros(Ls, np.int64), np.arange(Ls, dtype=np.int64)], axis=1)
    k, v = synth.kv_tokens(w, 0, idx)
    if fmt == oracle.INT8_PER_CHANNEL:
        cache.calibrate(k, v)
    cache.append(k, v, np.arange(Ls, dtype=np.int64))
    row = np.arange(nb, dtype=np.int32)
    q_all = np.random.default_rng(11).standard_normal((Ls, w.Hq, w.D)).astype(np.float16)

    def run(n):
        lens = np.arange(Ls - n + 1, Ls + 1, dtype=np.int32)
        cache.decode(q_all[Ls - n:], np.repeat(row[None], n, axis=0), lens)
        return 4 * w.Hq * w.D * int(lens.astype(np.int64).sum())

    t0 = time.perf_counter()
    run(1)
    t1 = time.perf_counter() - t0
    n = int(max(1, min(Ls, round(budget_s / max(t1, 1e-4)))))
    t0 = time.perf_counter()
    flop = run(n)
    dt = time.perf_counter() - t0
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": min(oracle.num_threads(), n * w.Hq),
            "kind": "oracle",
            "sample": "layer 0 of %d, sequence 0 (%d-token prompt appended), causal float64 attention "
                      "of its last %d query tokens x %d heads: %.2f s of CPU work, %d algorithmic FLOP"
                      % (w.layers, Ls, n, w.Hq, dt, flop),
            "seconds": dt, "flop": flop}


def workload_config(w):
    return {"workload": w.name, "layers": w.layers, "seqs": w.S,
            "context_lens": "%d..%d (mean %.0f)" % (w.context_lens.min(), w.context_lens.max(),
                                                   w.context_lens.mean()),
            "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D, "block_size": w.bs,
            "kv_format": sorted({"%s%s" % (FORMAT_NAME[f], (" %d" % g) if f in GROUPED else "")
                                 for f, g in w.layer_formats}),
            "pool_blocks_per_layer": w.num_blocks}


# ----------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch

    import paged_quantized_kv_kvq_gb300 as kvq
    from paged_quantized_kv_kvq_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    kvq.lib()
    w = synth.workload(args.workload, layers=args.layers, bs=args.block_size)
    stream = torch.cuda.current_stream()

    # -- per-layer pools, filled with the cached tokens (untimed set-up)
    pools = []
    fill_slots = torch.from_numpy(w.fill_slots()).to(dev)
    fill_idx = w.fill_token_index()
    for layer, (fmt, group) in enumerate(w.layer_formats):
        pool = kvq.KVPool(w.num_blocks, w.bs, w.Hkv, w.D, fmt, group, device=dev)
        if w.drift_sigma > 0 or fmt == kvq.KVQ_INT8_PER_CHANNEL:
            ks_, vs_ = [], []
            for s in range(w.S):
                t0 = w.shared_prefix_tokens if (s > 0 and w.shared_prefix_tokens) else 0
                k, v = synth.device_kv(w, layer, s, 0, int(w.context_lens[s]) - 1, dev)
                ks_.append(k[t0:]); vs_.append(v[t0:])
            k_all, v_all = torch.cat(ks_), torch.cat(vs_)
            if fmt == kvq.KVQ_INT8_PER_CHANNEL:
                kvq.kvq_calibrate_channel_scales(pool.handle, k_all, v_all)
            for a in range(0, k_all.shape[0], 1 << 16):
                b = min(k_all.shape[0], a + (1 << 16))
                pool.append(k_all[a:b], v_all[a:b], fill_slots[a:b])
            del k_all, v_all, ks_, vs_
        else:
            n = fill_slots.numel()
            for a in range(0, n, 1 << 16):
                b = min(n, a + (1 << 16))
                k, v = synth.device_kv(w, layer, -1, a, b, dev)
                pool.append(k, v, fill_slots[a:b])
        pools.append(pool)
    torch.cuda.synchronize()
    for p in pools:
        assert p.error() == kvq.KVQ_OK

    # -- step inputs, resident in HBM
    L = w.layers
    q = torch.stack([synth.device_queries(w, l, dev) for l in range(L)])
    kn = torch.empty((L, w.S, w.Hkv, w.D), dtype=torch.float16, device=dev)
    vn = torch.empty_like(kn)
    for l in range(L):
        for s in range(w.S):
            pos = int(w.context_lens[s]) - 1
            if w.drift_sigma > 0:
                k, v = synth.device_kv(w, l, s, 0, pos + 1, dev)
                kn[l, s], vn[l, s] = k[pos], v[pos]
            else:
                k, v = synth.device_kv(w, l, 10 ** 6 + s, pos, pos + 1, dev)
                kn[l, s], vn[l, s] = k[0], v[0]
    slots = torch.from_numpy(w.step_slots()).to(dev)
    table = torch.from_numpy(w.block_table).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    max_ctx = int(w.context_lens.max())
    out = torch.empty((L, w.S, w.Hq, w.D), dtype=torch.float32, device=dev)
    # The shared-prefix cascade reads the prefix once per kv head for all
    # sequences.  The repeated prefix reads of the plain decode hit the 129 MB
    # L2 and overlap the HBM-bound rest, so the cascade pays only when the
    # prefix is at least as long as the average suffix ("auto").
    P = 0
    if w.shared_prefix_tokens:
        mean_suffix = float(np.mean(w.context_lens)) - w.shared_prefix_tokens
        use = {"on": True, "off": False}.get(args.cascade, w.shared_prefix_tokens >= mean_suffix)
        use = use and w.bs != 8  # the cascade takes blocks of 16 tokens or more
        P = w.shared_prefix_tokens // w.bs if use else 0
    if P:
        ws_need = max(kvq.kvq_cascade_workspace_bytes(p.handle, w.S, w.Hq, max_ctx) for p in pools)
    else:
        ws_need = max(kvq.kvq_decode_workspace_bytes(p.handle, w.S, w.Hq, max_ctx) for p in pools)
    ws = torch.empty(max(ws_need, 256), dtype=torch.uint8, device=dev)
    sm_scale = w.D ** -0.5

    fused = args.step_api == "fused"

    def decode_call(l, qq, ln, oo, st=None):
        st = stream if st is None else st
        if P:
            kvq.kvq_cascade_decode(pools[l].handle, qq[l], table, ln, max_ctx, P, sm_scale, oo[l],
                                   ws, st)
        else:
            kvq.kvq_paged_decode(pools[l].handle, qq[l], table, ln, max_ctx, sm_scale, oo[l], ws,
                                 0, st)

    def layer_step(l, qq, kk, vv, sl, ln, oo, st=None):
        st = stream if st is None else st
        if fused and P:
            kvq.kvq_cascade_decode_step(pools[l].handle, kk[l], vv[l], qq[l], table, ln,
                                        max_ctx, P, sm_scale, oo[l], ws, st)
        elif fused:
            # one call: append at position L-1 (slot from the block table),
            # then the decode as a programmatic dependent of the append
            kvq.kvq_decode_step(pools[l].handle, kk[l], vv[l], qq[l], table, ln, max_ctx,
                                sm_scale, oo[l], ws, st)
        else:
            pools[l].append(kk[l], vv[l], sl, st)
            decode_call(l, qq, ln, oo, st)

    # No events between layers inside a step: an event record between two
    # kernels ends the programmatic-dependent overlap of the launches.
    def step(qq, kk, vv, sl, ln, oo, st=None):
        for l in range(L):
            layer_step(l, qq, kk, vv, sl, ln, oo, st)

    for _ in range(args.warmup):
        step(q, kn, vn, slots, lens, out)
    torch.cuda.synchronize()
    for p in pools:
        assert p.error() == kvq.KVQ_OK

    # The step as one CUDA graph (the same calls captured once, every kernel
    # and programmatic edge kept), replayed each timed step, as a serving loop
    # replays its decode graph; plain stream launches if capture is refused.
    launch = "stream"
    graph = None
    if not args.no_graph:
        try:
            cap = torch.cuda.Stream(device=dev)
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                step(q, kn, vn, slots, lens, out, cap)
            cap.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                step(q, kn, vn, slots, lens, out, cap)
            torch.cuda.synchronize()
            for _ in range(args.warmup):
                graph.replay()
            torch.cuda.synchronize()
            launch = "graph"
        except Exception as e:  # noqa: BLE001 -- reported in the JSON line
            graph = None
            launch = "stream (graph capture refused: %s)" % str(e).splitlines()[0][:120]
            torch.cuda.synchronize()
    for p in pools:
        assert p.error() == kvq.KVQ_OK

    def timed_step():
        if graph is not None:
            graph.replay()
        else:
            step(q, kn, vn, slots, lens, out)

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    # -- device-timed region
    K = args.steps
    sampler = ClockSampler(gpu_index(local_rank))
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        timed_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    # -- the dominant kernel alone: each layer's decode call (decode kernel and
    # its dependent split merge) bracketed by events on the launching stream,
    # over the same pools and inputs, right after the step region
    KR = max(1, min(K, 50))
    evs = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
           for _ in range(KR * L)]
    for i in range(KR):
        for l in range(L):
            ev = evs[i * L + l]
            ev[0].record(stream)
            decode_call(l, q, lens, out)
            ev[1].record(stream)
    torch.cuda.synchronize()
    # -- the same calls once more with an event after each of the call's
    # kernels (kvq_set_phase_events): the decode kernel's own device time,
    # then the merge's (with the cascade, the prefix kernel's first)
    names = (["kvq_rows_kernel"] if P else []) + ["kvq_decode_kernel", "kvq_merge_kernel"]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(KR * L)]
    for e in kev:  # torch creates its CUDA events at their first record
        for x in e:
            x.record(stream)
    for i in range(KR):
        for l in range(L):
            ev = kev[i * L + l]
            kvq.kvq_set_phase_events(ev[1:])
            ev[0].record(stream)
            decode_call(l, q, lens, out)
    kvq.kvq_set_phase_events([])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / K
    dec_ms = [a.elapsed_time(b) for a, b in evs]
    seg_ms = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(len(names))] for e in kev])
    kern_ms = {n: float(seg_ms[:, j].mean()) for j, n in enumerate(names)}
    ms = max_over_ranks(ms, dist, dev)

    # -- end to end through the Python API with host buffers
    pin = lambda x: x.cpu().pin_memory()
    q_h, kn_h, vn_h, sl_h, ln_h = pin(q), pin(kn), pin(vn), pin(slots), pin(lens)
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    q_d, kn_d, vn_d = torch.empty_like(q), torch.empty_like(kn), torch.empty_like(vn)
    sl_d, ln_d = torch.empty_like(slots), torch.empty_like(lens)
    # the fused step derives the slots on the device; the separate one copies them
    h2d_in = (q_h, kn_h, vn_h, ln_h) if fused else (q_h, kn_h, vn_h, sl_h, ln_h)
    h2d = sum(x.numel() * x.element_size() for x in h2d_in)
    d2h = out_h.numel() * out_h.element_size()

    # The copies overlap the layers, as a serving loop would run them: the
    # inputs go up on one copy stream in two chunks (the first IN0 layers, then
    # the rest, which lands while those run), the outputs come back on another
    # in chunks of OUT_CH layers as they complete.  Few chunks, because each
    # event between two launches ends their programmatic-dependent overlap.
    # Everything lies between the step's first and last event on the compute
    # stream: the copy streams start after the first, the compute stream waits
    # for the last read-back.
    cp_in, cp_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    IN0, OUT_CH = min(4, L), 8
    in_chunks = [(0, IN0)] + ([(IN0, L)] if L > IN0 else [])

    def e2e_step(st=None):
        st = stream if st is None else st
        go = torch.cuda.Event()
        go.record(st)
        cp_in.wait_event(go)
        cp_out.wait_event(go)
        in_ev = []
        with torch.cuda.stream(cp_in):
            ln_d.copy_(ln_h, non_blocking=True)
            if not fused:
                sl_d.copy_(sl_h, non_blocking=True)
            for a, b_ in in_chunks:
                q_d[a:b_].copy_(q_h[a:b_], non_blocking=True)
                kn_d[a:b_].copy_(kn_h[a:b_], non_blocking=True)
                vn_d[a:b_].copy_(vn_h[a:b_], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cp_in)
                in_ev.append(ev)
        o0 = 0
        for l in range(L):
            for c, (a, _) in enumerate(in_chunks):
                if l == a:
                    st.wait_event(in_ev[c])
            layer_step(l, q_d, kn_d, vn_d, sl_d, ln_d, out, st)
            if (l + 1) % OUT_CH == 0 or l == L - 1:
                ev = torch.cuda.Event()
                ev.record(st)
                cp_out.wait_event(ev)
                with torch.cuda.stream(cp_out):
                    out_h[o0:l + 1].copy_(out[o0:l + 1], non_blocking=True)
                o0 = l + 1
        done = torch.cuda.Event()
        done.record(cp_out)
        st.wait_event(done)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    # the whole end-to-end step (copies on their streams included) as one
    # graph too, when the step itself was captured
    e2e_launch = "stream"
    e2e_graph = None
    if graph is not None:
        try:
            cap2 = torch.cuda.Stream(device=dev)
            cap2.wait_stream(stream)
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph, stream=cap2):
                e2e_step(cap2)
            torch.cuda.synchronize()
            for _ in range(max(1, args.warmup)):
                e2e_graph.replay()
            torch.cuda.synchronize()
            e2e_launch = "graph"
        except Exception as e:  # noqa: BLE001 -- reported in the JSON line
            e2e_graph = None
            e2e_launch = "stream (graph capture refused: %s)" % str(e).splitlines()[0][:120]
            torch.cuda.synchronize()
            # fresh copy streams, in case the failed capture left its mark on them
            cp_in, cp_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_timed():
        if e2e_graph is not None:
            e2e_graph.replay()
        else:
            e2e_step()

    K2 = max(1, min(K, 50))
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(K2):
        e2e_timed()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / K2, dist, dev)
    for p in pools:
        assert p.error() == kvq.KVQ_OK

    # -- per-kernel device times of a few steps (a CUPTI trace, outside the
    # timed regions): explains the step time by its kernels
    kernel_times = kernel_breakdown("decode", w.name if w.bs == 16 else "%s bs%d" % (w.name, w.bs), L, ms)

    b = step_bytes(w)
    step_total = b["decode"] + b["append"]
    value = job_gbs(step_total, world, ms)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    dec_avg_ms = float(np.mean(dec_ms))
    # algorithmic HBM bytes of each layer's call (formats may differ by layer;
    # with the cascade the shared prefix is read once)
    lbytes = [layer_bytes(w, f, g)["unique_decode" if P else "decode"] for f, g in w.layer_formats]
    per_launch = float(np.mean(lbytes))
    call_achieved = per_launch / (dec_avg_ms * 1e-3) / 1e9
    # the roofline's kernel: the decode kernel, which moves every algorithmic
    # byte of the plain call; with the cascade the bytes are split between
    # the prefix kernel and the decode, so the call stands for them
    rk_ms = dec_avg_ms if P else kern_ms["kvq_decode_kernel"]
    achieved = per_launch / (rk_ms * 1e-3) / 1e9
    # launches per layer: append, decode and split merge, plus the prefix
    # kernel with the cascade
    launches_per_layer = 3 + (1 if P else 0)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "i8/e4m3 codes x f16 mma -> f32 acc",
        "data": "synthetic (seeded on-device normal draws with the workload's outlier/drift structure)",
        "config": workload_config(w),
        "run": {
            "l2": "inputs larger than L2: %d per-layer pools, %.1f GB"
                  % (L, sum(p.buffer.numel() for p in pools) / 1e9),
            "step": ("per layer: kvq_%sdecode_step (append 1 token/seq at L-1, then decode)"
                     % ("cascade_" if P else "") if fused else
                     "per layer: kvq_append (1 token/seq) then kvq_%s"
                     % ("cascade_decode" if P else "paged_decode")),
            "shared_prefix_blocks_read_once": P,
        },
        "kernel_times": kernel_times,
        "pct_of_peak": round(100 * value / world / peak, 2),
        "decode_tok_per_s": round(world * w.S / (ms * 1e-3), 1),
        "bytes_per_step": b,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": read_traffic(w.name) if w.bs == 16 else None,
                     "kernel": ("kvq_cascade_decode call (prefix kernel, decode kernel and split "
                                "merge, each a programmatic dependent of the one before; bytes "
                                "count the shared prefix once), every layer's, %d calls timed one "
                                "by one after the step region" % (KR * L) if P else
                                "kvq_decode_kernel, every layer's, %d launches after the step "
                                "region, each timed from an event just before its kvq_paged_decode "
                                "call to one the library records right after the kernel "
                                "(kvq_set_phase_events)" % (KR * L)),
                     "bytes_per_launch": round(per_launch), "avg_launch_ms": round(rk_ms, 5),
                     "peak_source": "%s hbm_gbs" % peak_kind,
                     "call": {"what": "the whole %s call (%s), calls timed one by one, no events "
                                      "between its kernels"
                                      % ("kvq_cascade_decode" if P else "kvq_paged_decode",
                                         " + ".join(names)),
                              "avg_ms": round(dec_avg_ms, 5), "achieved": round(call_achieved, 1),
                              "frac": round(call_achieved / peak, 4)},
                     "kernels_live_ms": {n: round(v, 5) for n, v in kern_ms.items()}},
        "e2e": {"value": round(job_gbs(step_total, world, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": K2,
                "overlap": "inputs in two chunks (first %d layers, then the rest) and outputs in "
                           "chunks of %d layers on two copy streams, overlapping the layers"
                           % (IN0, OUT_CH), "launch": e2e_launch},
        "gpu_launches": K * L * launches_per_layer,
        "launch": launch,
        "clocks": clocks,
    }
    del pools
    return res


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the workload (layer 0, one sequence), timed on the host cores."""
    from paged_quantized_kv_kvq_gb300 import synth
    import oracle

    w = synth.workload(args.workload, bs=args.block_size)
    fmt, group = w.layer_formats[0]
    oracle.build()
    # one step = sequence 0 of layer 0, all its heads
    run = oracle_sample(w, fmt, group, [0], oracle, synth)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    b = layer_bytes(w, fmt, group, [0])
    nbytes = b["decode"] + b["append"]
    v = nbytes / dt / 1e9
    sample = ("layer 0 of %d, sequence 0 of %d with its %d KV / %d Q heads (append of the step "
              "token + float64 paged decode over %d tokens) per step"
              % (w.layers, w.S, w.Hkv, w.Hq, int(w.context_lens[0])))
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (numpy seeded)",
            "config": workload_config(w),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s",
                             "cores": min(oracle.num_threads(), w.Hq),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_prefill(args, rank, world, local_rank):
    """Prefill of fresh prompts: per layer, append every prompt token's K/V
    (quantized) and run causal attention of all prompt tokens over the cache.
    Metric: algorithmic attention FLOP/s (4 * Hq * D per (query, key) pair
    with key <= query: Q.K and P.V, 2 FLOP per multiply-add)."""
    import torch

    import paged_quantized_kv_kvq_gb300 as kvq
    from paged_quantized_kv_kvq_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    kvq.lib()
    w = synth.workload(args.workload, S=args.prefill_seqs, layers=args.layers)
    stream = torch.cuda.current_stream()
    L = w.layers
    lens = w.context_lens.astype(np.int64)
    T = int(lens.sum())
    slots = torch.from_numpy(np.concatenate([w.slots_for(s, 0, int(lens[s]))
                                             for s in range(w.S)])).to(dev)
    qs = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(dev)
    table = torch.from_numpy(w.block_table).to(dev)
    ln = torch.from_numpy(w.context_lens).to(dev)
    pools = [kvq.KVPool(w.num_blocks, w.bs, w.Hkv, w.D, f, g, device=dev) for f, g in w.layer_formats]
    kin, vin, qin = [], [], []
    for l in range(L):
        ks, vs = zip(*[synth.device_kv(w, l, s, 0, int(lens[s]), dev) for s in range(w.S)])
        kin.append(torch.cat(ks))
        vin.append(torch.cat(vs))
        g = torch.Generator(device=dev)
        g.manual_seed(7919 * (l + 1))
        qin.append(torch.randn((T, w.Hq, w.D), generator=g, device=dev).half())
    out = torch.empty((T, w.Hq, w.D), dtype=torch.float32, device=dev)
    mq = int(lens.max())
    sm_scale = w.D ** -0.5
    # --prefill-api ex: two passes (the key steps staged once as fp16 tiles
    # in a workspace, then attention); plain: kvq_prefill, one pass
    ex = args.prefill_api == "ex"
    ws_n = max(kvq.kvq_prefill_workspace_bytes(p.handle, w.S, mq) for p in pools) if ex else 0
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev) if ws_n else None

    def attend(l):
        if ex:
            kvq.kvq_prefill_ex(pools[l].handle, qin[l], qs, mq, table, ln, mq, sm_scale, out, ws,
                               stream)
        else:
            kvq.kvq_prefill(pools[l].handle, qin[l], qs, mq, table, ln, mq, sm_scale, out, stream)

    def step():
        for l in range(L):
            kvq.kvq_append(pools[l].handle, kin[l], vin[l], slots, stream)
            attend(l)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for p in pools:
        assert p.error() == kvq.KVQ_OK
    K = args.steps
    dist = None
    if world > 1:
        import torch.distributed as dist
    sampler = ClockSampler(gpu_index(local_rank))
    sampler.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    # the attention kernel alone, per layer, for the roofline
    KR = max(1, min(K, 10))
    evs = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
           for _ in range(KR * L)]
    for i in range(KR):
        for l in range(L):
            evs[i * L + l][0].record(stream)
            attend(l)
            evs[i * L + l][1].record(stream)
    torch.cuda.synchronize()
    # the same calls with an event after each of their kernels
    # (kvq_set_phase_events): the attention kernel's own device time
    names = (["kvq_prefill_stage_kernel", "attention"] if ex else ["attention"])
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(KR * L)]
    for e in kev:  # torch creates its CUDA events at their first record
        for x in e:
            x.record(stream)
    for i in range(KR):
        for l in range(L):
            ev = kev[i * L + l]
            kvq.kvq_set_phase_events(ev[1:])
            ev[0].record(stream)
            attend(l)
    kvq.kvq_set_phase_events([])
    torch.cuda.synchronize()
    seg_ms = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(len(names))] for e in kev])
    kern_ms = {n: float(seg_ms[:, j].mean()) for j, n in enumerate(names)}
    # -- end to end: every step copies each layer's prompt K/V and Q in from
    # pinned host memory and each layer's output back, on two copy streams
    # that overlap the layers (layer l+1's inputs arrive while layer l runs;
    # outputs alternate between two device buffers); one host copy of a
    # layer's inputs stands for every layer's (the same bytes move)
    k_h = kin[0].cpu().pin_memory()
    v_h = vin[0].cpu().pin_memory()
    q_h = qin[0].cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    outs = [out, torch.empty_like(out)]
    cp_in, cp_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d = (k_h.numel() * k_h.element_size() + v_h.numel() * v_h.element_size() +
           q_h.numel() * q_h.element_size()) * L
    d2h = out_h.numel() * out_h.element_size() * L

    def e2e_step():
        in_ev, out_ev = [], []
        cp_in.wait_stream(stream)
        for l in range(L):
            with torch.cuda.stream(cp_in):
                kin[l].copy_(k_h, non_blocking=True)
                vin[l].copy_(v_h, non_blocking=True)
                qin[l].copy_(q_h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cp_in)
                in_ev.append(ev)
        for l in range(L):
            stream.wait_event(in_ev[l])
            if l >= 2:
                stream.wait_event(out_ev[l - 2])  # its output buffer has been read back
            kvq.kvq_append(pools[l].handle, kin[l], vin[l], slots, stream)
            o = outs[l % 2]
            if ex:
                kvq.kvq_prefill_ex(pools[l].handle, qin[l], qs, mq, table, ln, mq, sm_scale, o,
                                   ws, stream)
            else:
                kvq.kvq_prefill(pools[l].handle, qin[l], qs, mq, table, ln, mq, sm_scale, o,
                                stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            cp_out.wait_event(ev)
            with torch.cuda.stream(cp_out):
                out_h.copy_(o, non_blocking=True)
                ev2 = torch.cuda.Event()
                ev2.record(cp_out)
                out_ev.append(ev2)
        stream.wait_stream(cp_out)

    e2e_step()
    torch.cuda.synchronize()
    K2 = max(1, min(K, 5))
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(K2):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / K2, dist, dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / K, dist, dev)
    att_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    pairs = int((lens * (lens + 1) // 2).sum())
    flop_layer = 4 * pairs * w.Hq * w.D
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0)))
    call_achieved = flop_layer / (att_ms * 1e-3) / 1e12
    ak_ms = kern_ms["attention"]
    achieved = flop_layer / (ak_ms * 1e-3) / 1e12
    value = world * flop_layer * L / (ms * 1e-3) / 1e12
    return {
        "metric": "Paged quantized-KV prefill: causal attention TFLOP/s (algorithmic)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "i8 codes x f16 mma -> f32 acc",
        "data": "synthetic (seeded on-device normal draws)",
        "config": {"workload": "%s prefill" % w.name, "layers": L, "prompts": w.S,
                   "prompt_len": int(lens.max()), "q_heads": w.Hq, "kv_heads": w.Hkv,
                   "head_dim": w.D, "block_size": w.bs,
                   "kv_format": sorted({"%s%s" % (FORMAT_NAME[f], (" %d" % g) if f in GROUPED else "")
                                        for f, g in w.layer_formats}),
                   "step": "per layer: kvq_append (every prompt token) then kvq_prefill%s"
                           % ("_ex" if ex else "")},
        "prompt_tok_per_s": round(world * T / (ms * 1e-3), 1),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": ("the attention kernel of kvq_prefill_ex (kvq_prefill_ws_kernel: "
                                "tcgen05.mma kind::f16 over the staged fp16 key steps" if ex else
                                "the attention kernel of kvq_prefill (tcgen05.mma kind::f16, codes "
                                "converted in the kernel") + ", fp32 accumulators in TMEM), every "
                               "layer's, %d launches after the step region, each timed from the "
                               "event the library records after the call's previous kernel (or "
                               "one just before the call) to the one it records right after this "
                               "kernel (kvq_set_phase_events)" % (KR * L),
                     "flop_per_launch": flop_layer, "avg_launch_ms": round(ak_ms, 4),
                     "peak_source": "%s bf16_tflops_sustained (f16 has the bf16 rate)" % peak_kind,
                     "call": {"what": "the whole kvq_prefill%s call, calls timed one by one, no "
                                      "events between its kernels" % ("_ex" if ex else ""),
                              "avg_ms": round(att_ms, 4), "achieved": round(call_achieved, 2),
                              "frac": round(call_achieved / peak, 4)},
                     "kernels_live_ms": {n: round(v, 5) for n, v in kern_ms.items()}},
        "e2e": {"value": round(world * flop_layer * L / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": K2,
                "overlap": "each layer's inputs on one copy stream ahead of the layers, each "
                           "layer's output read back on another as it completes"},
        "kernel_times": (kernel_breakdown("prefill", "%s prefill" % w.name, L, att_ms * L)
                         if ex else {"unavailable": "launch record taken for kvq_prefill_ex"}),
        "gpu_launches": K * L * (3 if ex else 2),  # append, (staging,) attention
        "clocks": clocks,
    }


def launch_replicas(n, check_gpus=True):
    """Start n ranks of this script, one per GPU (RANK, LOCAL_RANK, WORLD_SIZE,
    MASTER_ADDR/PORT set as torchrun would); returns the worst exit code.
    Rank 0 prints the job's JSON line."""
    import socket

    if check_gpus:
        import torch

        have = torch.cuda.device_count()
        if have < n:
            print("bench.py: --gpus %d but only %d GPU(s) visible" % (n, have), file=sys.stderr)
            return 2
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + sys.argv[1:],
                                      env=env))
    rcs = [p.wait() for p in procs]
    return max(rcs, key=abs)


def launcher_selftest(rank, world):
    """Every rank joins a gloo group and reports a step time of rank + 1 ms;
    rank 0 prints the slowest and how many ranks took part."""
    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("gloo")
    d = dist if world > 1 else None
    ms = max_over_ranks(1.0 + rank, d, torch.device("cpu"))
    joined = torch.ones(1)
    if d is not None:
        d.all_reduce(joined)
    if rank == 0:
        print(json.dumps({"launcher_selftest": True, "n_gpus": world,
                          "ranks_joined": int(joined.item()), "ms_per_step": ms,
                          "job_gbs_for_1GB_per_rank": job_gbs(1e9, world, ms)}), flush=True)
    if d is not None:
        d.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 1000 decode steps, 10 prefill steps)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gqa_64x2048")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cascade", default="auto", choices=["auto", "on", "off"],
                    help="shared-prefix workloads: attend the prefix once for all sequences "
                         "(auto: when the prefix is at least the mean suffix length)")
    ap.add_argument("--step-api", default="fused", choices=["fused", "separate"],
                    help="fused: one kvq_decode_step call per layer; separate: kvq_append "
                         "then kvq_paged_decode")
    ap.add_argument("--op", default="decode", choices=["decode", "prefill"],
                    help="decode: the decode step (default); prefill: prompt prefill")
    ap.add_argument("--prefill-seqs", type=int, default=8,
                    help="prompts in the prefill batch (--op prefill)")
    ap.add_argument("--prefill-api", default="ex", choices=["plain", "ex"],
                    help="--op prefill: kvq_prefill (one pass) or kvq_prefill_ex (key steps "
                         "staged once in a workspace, then attention)")
    ap.add_argument("--block-size", type=int, default=None,
                    help="tokens per block (default: the workload's; 8, 16, 32 or 64)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step as plain stream launches instead of a CUDA graph")
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer layers (profiling runs only; the bench line uses all)")
    ap.add_argument("--launcher-selftest", action="store_true",
                    help="CPU check of the replica launcher: every rank joins a gloo group, "
                         "rank 0 prints the max-over-ranks arithmetic; no GPU work")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.steps is None:
        args.steps = 10 if args.op == "prefill" else 1000
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # the oracle on the host cores: rank 0 alone runs and prints
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not started by torchrun: start the N replica ranks here
        sys.exit(launch_replicas(args.gpus, check_gpus=not args.launcher_selftest))
    if args.gpus != world:
        sys.exit("bench.py: --gpus %d but WORLD_SIZE=%d; launch one rank per GPU"
                 % (args.gpus, world))
    if args.launcher_selftest:
        launcher_selftest(rank, world)
        return

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.op == "prefill":
        res = run_prefill(args, rank, world, local_rank)
        if rank == 0:
            if world == 1 and not args.no_cpu_baseline:
                from paged_quantized_kv_kvq_gb300 import synth

                res["cpu_baseline"] = cpu_baseline_prefill(
                    synth.workload(args.workload, S=args.prefill_seqs, layers=args.layers))
            print(json.dumps(res), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            from paged_quantized_kv_kvq_gb300 import synth

            res["cpu_baseline"] = cpu_baseline(synth.workload(args.workload, bs=args.block_size))
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
