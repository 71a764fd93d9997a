"""Benchmark of the routed-expert FFN step on one GB300 (one JSON line).

Workload (N=1): one MoE layer at the pages' scale, single-stream decode:
d=2048, f=768, 512 routed experts + 1 shared, top-10, 3-bit g32 experts
(2,064,384 B each), all 512 experts resident in the VRAM cache, 10,000
sequential calls of one fresh token each.  A step is one pass over the
10,000-call stream: router + top-k, cache lookup/stamp, dequant SwiGLU of the
11 experts and the combine, per call, as the CUDA library runs them (the
10,000 calls are captured once into a CUDA graph of moe_forward calls and
replayed per step).

value: tokens/s per MoE layer (= calls/s at T=1) with inputs resident in
HBM.  e2e: the same through the C ABI with the step's 10,000 tokens copied
from pinned host memory before and the 10,000 outputs copied back after, in
the timed region.  roofline: algorithmic bytes of one call, the distinct
experts it runs (11 at T=1, counted from the cache statistics) x 2,064,384 B
= 22,708,224 B at T=1 (router weights, 2 MiB, reported separately), over the
average per-call duration (one kernel launch per call), against the
measured HBM copy bandwidth.  --tokens T runs verify batches of T tokens
per call instead (value then counts all T tokens).
cpu_baseline: the fp64 CPU oracle on a bounded sample of calls, on every
host core (one process per core) and on one thread.
prefill (by default at T=1 with the default call count; --no-prefill drops
it): the 12,288-token chunk and the chunk-size sweep, expert FLOP rate
against the measured bf16 tensor peak.

stack (by default at T=1 with the default call count; --no-stack drops it):
the two 48-layer stacks with the 8,445-slot cache starting empty, misses
pulled by the GPU from the host pool -- the verify stack (T=5, Zipf s=1.1)
and the concurrent stack (T=16, Zipf s=0.8) -- 3 warm-up passes over 2,000
calls, then the timed pass; tokens/s of the whole 48-layer stack against
max(distinct-expert bytes / HBM, miss bytes / measured H2D).

--impl reference times the CPU oracle itself (the pages publish no code and
no number for this step; the oracle is the only reference implementation).
--stack-sweep adds the verify-width x cache-capacity sweep.
"""

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np

CALLS = 10_000
DEFAULT_CALLS = CALLS
EXPERT_BYTES = 2_064_384
ROUTER_BYTES = 512 * 2048 * 2
L2_BYTES = 129 * 1024 * 1024
METRIC = "MoE expert-stack tokens/s (decode & 12,288-chunk prefill); HBM GB/s vs roofline"
WORKLOAD = ("decode-layer: d=2048 f=768 E=512 top-10 + 1 shared expert, 3-bit g32 fp16-scale experts, "
            "T=1 token per call, 10,000 sequential calls, all 512 experts resident")


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# the sources the decode kernel is compiled from
DECODE_SOURCES = ("decode_ffn.cu", "select.cuh", "common.cuh", "internal.h", "repack.cuh", "fetch.cuh")


def source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "expert_cached_decode_gb300", "csrc")
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "decode_ffn_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("source_hash") != source_hash():
        return None
    return d.get("dram_bytes_per_call")


class ClockSampler:
    def __init__(self, out):
        self.out = out
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self, dev_index=0):
        if self.proc is None or not os.path.exists(self.out):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for ln in open(self.out):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9 or not parts[0].isdigit() or int(parts[0]) != dev_index:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        mx = float(rows[0][2])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [v for v in sm if v > 0.5 * mx] or sm
        return {"sm_mhz": float(np.median(loaded)), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


def workload_name(calls, T):
    name = WORKLOAD if T == 1 else WORKLOAD.replace("T=1 token per call", f"T={T} tokens per call (verify batch)")
    return name if calls == CALLS else name + f" (profiling run: {calls} calls)"


def build_decode_layer(calls, seed_cfg=2, T=1):
    import torch
    from moe_inputs import synth
    from expert_cached_decode_gb300.layer import MoELayer
    s = synth(seed_cfg)
    wl = s.wl
    wr, _, b = s.router(0)
    shared = np.stack([s.shared_packed(0)])
    pool = torch.empty((wl.keys, s.B), dtype=torch.uint8, pin_memory=True)
    pv = pool.numpy()
    for e in range(wl.keys):
        s.expert_packed(e, out=pv[e])
    layer = MoELayer(wl.d, wl.f, wl.n_experts, wl.top_k, 1, wr.reshape(1, wl.n_experts, wl.d), b.reshape(1, -1),
                     shared, pool)
    layer._pool = pool
    layer.moe_cache_configure(wl.capacity, np.arange(wl.keys))
    xs = s.tokens_many(0, list(range(calls)), T=T).reshape(calls, T, wl.d)
    return s, layer, xs


PREFILL_FLOPS_PER_TOKEN = 11 * 3 * 2 * 2048 * 768          # (k+1) experts x 3 matrices x 2 d f
ROUTER_FLOPS_PER_TOKEN = 2 * 2048 * 512


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured (bf16 burst; fp16 dense rate is the same)"
    return 1900.0, "fallback"


def run_prefill(steps, warmup, sweep=(4096, 6144, 8192, 12288, 16384)):
    """12,288-token prefill chunk at one layer (all 512 experts resident) and
    the chunk-size sweep: tokens/s and tensor-core FLOP rate of the whole call."""
    import torch
    from moe_inputs import synth
    from expert_cached_decode_gb300.layer import MoELayer
    s = synth(5)
    wl = s.wl
    wr, _, b = s.router(0)
    shared = np.stack([s.shared_packed(0)])
    pool = torch.empty((wl.keys, s.B), dtype=torch.uint8, pin_memory=True)
    pv = pool.numpy()
    for e in range(wl.keys):
        s.expert_packed(e, out=pv[e])
    layer = MoELayer(wl.d, wl.f, wl.n_experts, wl.top_k, 1, wr.reshape(1, wl.n_experts, wl.d),
                     b.reshape(1, -1), shared, pool)
    layer.moe_cache_configure(wl.capacity, np.arange(wl.keys))
    peak, src = tensor_peak()
    out = {"workload": "prefill-chunk: one layer, T tokens bf16 N(0,1), top-10/512 + shared, all experts resident",
           "flops_per_token": PREFILL_FLOPS_PER_TOKEN, "router_flops_per_token": ROUTER_FLOPS_PER_TOKEN,
           "peak_tflops": peak, "peak_source": src, "sweep": []}
    stream = torch.cuda.Stream()
    for T in sweep:
        xb = s.tokens_many(0, [T], T=T)[0]
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        y = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                layer.moe_forward(0, x, y)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(steps):
                layer.moe_forward(0, x, y)
        e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1) / steps
        tflops = PREFILL_FLOPS_PER_TOKEN * T / (ms / 1e3) / 1e12
        out["sweep"].append({"T": T, "ms": ms, "tokens_per_s": T / (ms / 1e3), "tflops": tflops,
                             "frac": tflops / peak})
    layer.moe_sync()
    layer.close()
    main = [r for r in out["sweep"] if r["T"] == 12288]
    if main:
        out["tokens_per_s"] = main[0]["tokens_per_s"]
        out["roofline"] = {"bound": "tensor", "achieved": main[0]["tflops"], "peak": peak, "unit": "TFLOP/s",
                           "frac": main[0]["frac"],
                           "note": "whole prefill call (router GEMM, top-k, sort, gather, gate/up and down "
                                   "grouped GEMMs) against the expert FLOPs T*103,809,024"}
    return out


# -------------------------------------------------------- KV-streaming window --
def run_kv_window(steps=20, warmup=3, n_layers=2):
    """KV-streaming window (NEXT-4): per layer 131,072 cells of 1,056 B, the
    first 32,768 in VRAM and the rest in page-locked host memory.  A step
    reads every block of every layer once (a dense attention read; the pages
    do not give which blocks their sparse attention reads), resident blocks
    from HBM, the others straight from host memory.  Bound: the host part at
    the measured host->device rate, the HBM part (window read + all blocks
    written) at the measured HBM rate, whichever is longer."""
    import torch
    from moe_inputs.kv import KV_BLOCK_CELLS, KV_CELL_BYTES, KV_CONTEXT_CELLS, KV_RESIDENT_CELLS, kv_cells
    from expert_cached_decode_gb300.layer import KVWindow
    n, R, cb, bc = KV_CONTEXT_CELLS, KV_RESIDENT_CELLS, KV_CELL_BYTES, KV_BLOCK_CELLS
    host = torch.empty(n_layers * (n - R) * cb, dtype=torch.uint8, pin_memory=True)
    kv = KVWindow(n_layers, n, R, cb, bc, host)
    try:
        for l in range(n_layers):
            src = torch.from_numpy(kv_cells(0, l, n, cb)).cuda()
            kv.moe_kv_write(l, 0, src)
            torch.cuda.synchronize()
            del src
        nb = n // bc
        ids = torch.arange(nb, dtype=torch.int32, device="cuda")
        dst = torch.empty((nb, bc * cb), dtype=torch.uint8, device="cuda")
        stream = torch.cuda.current_stream()
        def step():
            for l in range(n_layers):
                kv.moe_kv_read_blocks(l, ids, dst, stream)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        r0, h0 = kv.moe_kv_stats()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        r1, h1 = kv.moe_kv_stats()
        host_bytes = n_layers * (n - R) * cb
        hbm_bytes = n_layers * (R * cb + n * cb)   # window read + every block written
        h2d = measure_h2d_gbs()
        hbm, kind = peaks()
        t_bound = max(host_bytes / (h2d * 1e9), hbm_bytes / (hbm * 1e9))
        return {"workload": f"kv-window: {n_layers} layers x {n:,} cells x {cb} B, first {R:,} cells of each in "
                            f"VRAM, blocks of {bc} cells, every block read once per step",
                "ms_per_step": ms, "blocks_per_step": n_layers * nb,
                "block_hit_rate": (h1 - h0) / max(1, r1 - r0),
                "host_gbs": host_bytes / (ms / 1e3) / 1e9, "total_gbs": n_layers * n * cb / (ms / 1e3) / 1e9,
                "h2d_gbs_measured": h2d,
                "roofline": {"bound": "h2d" if host_bytes / h2d >= hbm_bytes / hbm else "hbm",
                             "bound_ms": t_bound * 1e3, "frac": t_bound * 1e3 / ms,
                             "note": "host part at the measured cudaMemcpy H2D rate (expert-sized copies from "
                                     "pinned memory), HBM part (window read + blocks written) at "
                                     f"MEASURED_PEAKS.json hbm_gbs ({kind})"},
                "gpu_launches_per_step": n_layers}
    finally:
        kv.close()


# ------------------------------------------------------------ 48-layer stack --
def _draw_layer_tokens(args):
    cfg_id, lam, layer, calls, T = args
    sys.path.insert(0, ROOT)
    from moe_inputs import Synth, WORKLOADS
    s = Synth(WORKLOADS[cfg_id], bias_lambda=lam)
    return layer, s.tokens_many(layer, list(range(calls)), T=T)


def draw_stack_tokens(cfg_id, calls, n_layers, workers=16, T=None):
    """Seeded activations [L, calls, T, d] (bf16 bits) of a stack workload,
    one spawn-pool job per layer (T defaults to the workload's)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    from moe_inputs import BIAS_LAMBDA
    out = [None] * n_layers
    with cf.ProcessPoolExecutor(max_workers=min(workers, n_layers), mp_context=mp.get_context("spawn")) as ex:
        for layer, xs in ex.map(_draw_layer_tokens, [(cfg_id, BIAS_LAMBDA, l, calls, T) for l in range(n_layers)]):
            out[layer] = xs
    return np.stack(out)


def _fill_pool_range(args):
    shm_name, B, cfg_id, lam, lo, hi = args
    sys.path.insert(0, ROOT)
    from multiprocessing import shared_memory
    from moe_inputs import Synth, WORKLOADS
    shm = shared_memory.SharedMemory(name=shm_name)
    try:
        view = np.ndarray((hi - lo, B), dtype=np.uint8, buffer=shm.buf, offset=lo * B)
        s = Synth(WORKLOADS[cfg_id], bias_lambda=lam)
        for p in range(lo, hi):
            s.expert_packed(p, out=view[p - lo])
        del view
    finally:
        shm.close()
    return hi - lo


def make_host_pool(cfg_id, entries, workers=16):
    """Canonical packed experts of host-pool entries [0, entries) in a shared
    memory block filled by a spawn pool (the library registers it)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    from multiprocessing import shared_memory
    from moe_inputs import WORKLOADS, BIAS_LAMBDA, expert_nbytes
    wl = WORKLOADS[cfg_id]
    B = expert_nbytes(wl.d, wl.f)
    shm = shared_memory.SharedMemory(create=True, size=entries * B)
    step = max(1, (entries + workers * 4 - 1) // (workers * 4))
    jobs = [(shm.name, B, cfg_id, BIAS_LAMBDA, lo, min(entries, lo + step)) for lo in range(0, entries, step)]
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        assert sum(ex.map(_fill_pool_range, jobs)) == entries
    return shm, np.ndarray((entries, B), dtype=np.uint8, buffer=shm.buf)


def pack_pool_in_place(pool, d, f, chunk=256):
    """Re-lay the canonical experts of `pool` (numpy [P][B_x]) into the
    device block layout, chunk by chunk through device memory, on the GPU."""
    import torch
    from expert_cached_decode_gb300.layer import moe_pack_experts
    n, B = pool.shape
    src = torch.empty((chunk, B), dtype=torch.uint8, device="cuda")
    dst = torch.empty((chunk, B), dtype=torch.uint8, device="cuda")
    for i0 in range(0, n, chunk):
        m = min(chunk, n - i0)
        src[:m].copy_(torch.from_numpy(pool[i0:i0 + m]))
        moe_pack_experts(src[:m], dst[:m], m, d, f)
        torch.from_numpy(pool[i0:i0 + m]).copy_(dst[:m].cpu())
    torch.cuda.synchronize()


def measure_h2d_gbs(chunk=EXPERT_BYTES, total=1 << 30, reps=5):
    """Host -> device bandwidth of back-to-back expert-sized copies from pinned memory."""
    import torch
    n = total // chunk
    src = torch.empty((n, chunk), dtype=torch.uint8, pin_memory=True)
    dst = torch.empty((n, chunk), dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    out = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        with torch.cuda.stream(st):
            for i in range(n):
                dst[i].copy_(src[i], non_blocking=True)
        e1.record(st)
        st.synchronize()
        out.append(n * chunk / (e0.elapsed_time(e1) / 1e3) / 1e9)
    return float(np.median(out))


def run_stack(cfg_id, pool_entries=0, calls=0, miss_mode=1, pool_layout=1, aheads=(False,)):
    """48-layer stack with the 8,445-slot cache that starts empty (miss path):
    the warm-up passes over the call stream, then the measured pass.
    miss_mode 1: the GPU reads missing experts from the host pool itself;
    0: the host issues the copies after reading the routing plan.
    pool_layout 1: the host pool holds the device block layout (converted
    once at setup), so a missing expert is computed straight from it while
    it is written to its slot; 0: canonical, fetched and re-laid out first.
    aheads: one result per entry, on the same layer and host pool (the cache
    reconfigured, so it starts empty each time).  ahead True: every
    layer-call made with moe_forward_ahead naming the next
    layer-call of its pass (cross-layer lookahead; the stack's layers take
    independent tokens), so its routing, cache step and misses run one
    launch early; the first call of a pass prepares itself."""
    import time
    import torch
    from moe_inputs import Synth, WORKLOADS, BIAS_LAMBDA, expert_nbytes
    from expert_cached_decode_gb300.layer import MoELayer
    wl = WORKLOADS[cfg_id]
    calls = calls or wl.calls
    P = pool_entries or wl.keys
    t0 = time.time()
    xs = draw_stack_tokens(cfg_id, calls, wl.n_layers)
    shm, pool = make_host_pool(cfg_id, P)
    if pool_layout == 1:
        pack_pool_in_place(pool, wl.d, wl.f)
    s = Synth(wl, bias_lambda=BIAS_LAMBDA)
    wr = np.stack([s.router(l)[0] for l in range(wl.n_layers)])
    b = np.stack([s.router(l)[2] for l in range(wl.n_layers)])
    shared = np.stack([s.shared_packed(l) for l in range(wl.n_layers)])
    layer = MoELayer(wl.d, wl.f, wl.n_experts, wl.top_k, wl.n_layers, wr, b, shared, pool,
                     host_pool_entries=0 if P == wl.keys else P, host_pool_layout=pool_layout)
    layer.moe_set_miss_mode(miss_mode)
    setup_s = time.time() - t0
    xdev = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty((wl.tokens, wl.d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    steps = [(c, l) for c in range(calls) for l in range(wl.n_layers)]
    runs = []

    for ahead in aheads:
        layer.moe_cache_configure(wl.capacity)
        def one_pass():
            for i, (c, l) in enumerate(steps):
                if ahead:
                    nc, nl = steps[i + 1] if i + 1 < len(steps) else (0, 0)
                    layer.moe_forward_ahead(l, xdev[l, c], y, next_layer=nl,
                                            next_x=xdev[nl, nc] if i + 1 < len(steps) else None)
                else:
                    layer.moe_forward(l, xdev[l, c], y)

        with torch.cuda.stream(stream):
            for _ in range(wl.warm_passes):
                one_pass()
        stream.synchronize()
        before = layer.moe_cache_stats()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            one_pass()
        e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1)
        after = layer.moe_cache_stats()
        dlt = {k: after[k] - before[k] for k in after}
        runs.append((ahead, ms, dlt))
    layer.close()
    del pool
    shm.close()
    shm.unlink()
    h2d = measure_h2d_gbs()
    hbm, _ = peaks()
    B = expert_nbytes(wl.d, wl.f)
    out = []
    for ahead, ms, dlt in runs:
        distinct_bytes = (dlt["distinct_hits"] + dlt["distinct_misses"] + dlt["layer_calls"]) * B  # + shared
        t_bound = max(distinct_bytes / (hbm * 1e9), dlt["miss_bytes"] / (h2d * 1e9))
        tokens = calls * wl.tokens
        out.append({"workload": f"{wl.name}: 48 layers, T={wl.tokens} per call, Zipf s={wl.zipf_s} (lambda "
                            f"{BIAS_LAMBDA}), {wl.capacity} slots starting empty, {wl.warm_passes} warm-up passes "
                            f"then the measured pass of {calls} calls",
                "miss_copies": ("host-issued cudaMemcpyAsync" if miss_mode == 0 else
                                "GPU computes each missing expert straight from the host pool (device block layout) "
                                "and writes it to its victim slot" if pool_layout == 1 else
                                "GPU fetches each missing expert from the host pool (canonical) into its slot, then "
                                "computes"),
                "host_pool_layout": "device block layout" if pool_layout == 1 else "canonical",
                "lookahead": ("each layer-call routes the next one and copies its misses (moe_forward_ahead)"
                              if ahead else "none"),
                "host_pool_entries": P,
                "host_pool_note": "expert (l, e) is read from entry (512 l + e) mod P; copy sizes, counts and "
                                  "the cache's behaviour do not depend on P",
                "tokens_per_s": tokens / (ms / 1e3), "ms_measured_pass": ms,
                "token_hit_rate": dlt["token_hits"] / max(1, dlt["token_hits"] + dlt["token_misses"]),
                "distinct_expert_bytes": distinct_bytes, "miss_bytes": dlt["miss_bytes"],
                "h2d_gbs_measured": h2d, "hbm_gbs": hbm,
                "roofline": {"bound_ms": 1e3 * t_bound, "frac": 1e3 * t_bound / ms,
                             "note": "max(distinct-expert bytes / HBM, miss bytes / measured H2D)",
                             "serialised_bound_ms": 1e3 * (distinct_bytes / (hbm * 1e9) + dlt["miss_bytes"] / (h2d * 1e9)),
                             "serialised_note": "distinct-expert bytes / HBM + miss bytes / H2D: copies and expert "
                                                "reads never overlapping"},
                "setup_s": setup_s})
    return out


def run_stack_sweep(pool_entries=2048, calls=500, tokens=(1, 4, 7), capacities=(9057, 8445, 6144)):
    """Draft width x cache capacity sweep on the verify stack (48 layers,
    Zipf s=1.1): for each verify width T (1 + draft tokens) and capacity C
    the cache starts empty, 3 warm-up passes over `calls` calls, then the
    timed pass; misses pulled by the GPU.  Tokens of width T are the first T
    rows of the widest draw (the generator is prefix-consistent)."""
    import time
    import torch
    from moe_inputs import Synth, WORKLOADS, BIAS_LAMBDA
    from expert_cached_decode_gb300.layer import MoELayer
    cfg_id = 3
    wl = WORKLOADS[cfg_id]
    t0 = time.time()
    xs = draw_stack_tokens(cfg_id, calls, wl.n_layers, T=max(tokens))
    shm, pool = make_host_pool(cfg_id, pool_entries)
    pack_pool_in_place(pool, wl.d, wl.f)
    s = Synth(wl, bias_lambda=BIAS_LAMBDA)
    wr = np.stack([s.router(l)[0] for l in range(wl.n_layers)])
    b = np.stack([s.router(l)[2] for l in range(wl.n_layers)])
    shared = np.stack([s.shared_packed(l) for l in range(wl.n_layers)])
    layer = MoELayer(wl.d, wl.f, wl.n_experts, wl.top_k, wl.n_layers, wr, b, shared, pool,
                     host_pool_entries=pool_entries, host_pool_layout=1)
    layer.moe_set_miss_mode(1)
    setup_s = time.time() - t0
    xdev = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).cuda()
    stream = torch.cuda.Stream()
    rows = []
    for T in tokens:
        y = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
        for C in capacities:
            layer.moe_cache_configure(C)
            with torch.cuda.stream(stream):
                for _ in range(wl.warm_passes):
                    for c in range(calls):
                        for l in range(wl.n_layers):
                            layer.moe_forward(l, xdev[l, c, :T], y)
            stream.synchronize()
            before = layer.moe_cache_stats()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                for c in range(calls):
                    for l in range(wl.n_layers):
                        layer.moe_forward(l, xdev[l, c, :T], y)
            e1.record(stream)
            stream.synchronize()
            ms = e0.elapsed_time(e1)
            after = layer.moe_cache_stats()
            dl = {k: after[k] - before[k] for k in after}
            lc = max(1, dl["layer_calls"])
            rows.append({"T": T, "capacity": C, "tokens_per_s": calls * T / (ms / 1e3),
                         "token_hit_rate": dl["token_hits"] / max(1, dl["token_hits"] + dl["token_misses"]),
                         "distinct_experts_per_layer_call": (dl["distinct_hits"] + dl["distinct_misses"]) / lc,
                         "misses_per_layer_call": dl["distinct_misses"] / lc,
                         "us_per_layer_call": 1e3 * ms / lc})
    layer.close()
    del pool
    shm.close()
    shm.unlink()
    return {"workload": f"verify stack (48 layers, Zipf s={wl.zipf_s}, lambda {BIAS_LAMBDA}), cache starting empty, "
                        f"{wl.warm_passes} warm-up passes then the timed pass over {calls} calls; GPU pulls misses; "
                        f"host pool {pool_entries} entries", "setup_s": setup_s, "rows": rows}


def _oracle_child(n_calls, threads=1, first=0):
    """Command and environment of a child process that times the fp64 oracle
    on calls [first, first + n_calls) of the decode stream with BLAS limited
    to `threads`; it prints {"seconds", "calls"}."""
    env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    code = f"""
import sys, time, json
sys.path.insert(0, {ROOT!r})
import numpy as np
from moe_inputs import synth, bf16_bits_to_f64
from oracle.routing import route
from oracle.packed import unpack_expert
from oracle.ffn import layer_forward
s = synth(2); wl = s.wl
_, wr64, b = s.router(0)
xs = s.tokens_many(0, list(range({first}, {first} + {n_calls})), T=1)
# inputs (packed experts) drawn before timing; the oracle's own work is timed
need = set()
for i in range({n_calls}):
    need |= set(route(bf16_bits_to_f64(xs[i]), wr64, b, wl.top_k)[0].ravel().tolist())
packed = {{e: s.expert_packed(e) for e in sorted(need)}}
shared_p = s.shared_packed(0)
t0 = time.perf_counter()
for i in range({n_calls}):
    x64 = bf16_bits_to_f64(xs[i])
    idx, w, _ = route(x64, wr64, b, wl.top_k)
    shared = unpack_expert(shared_p, wl.d, wl.f)
    y = layer_forward(x64, idx, w, lambda e: unpack_expert(packed[e], wl.d, wl.f), shared)
dt = time.perf_counter() - t0
print(json.dumps({{"seconds": dt, "calls": {n_calls}}}))
"""
    return [sys.executable, "-c", code], env


def cpu_oracle_sample(n_calls, threads=1):
    """Time the fp64 oracle on the first n_calls of the decode stream in a
    child process with BLAS limited to `threads`."""
    cmd, env = _oracle_child(n_calls, threads)
    r = subprocess.run(cmd, capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_oracle_all_cores(n_per_core):
    """The same oracle on every host core: one child process per core (1 BLAS
    thread each) on disjoint call ranges, started together; rate = all calls /
    the longest child's timed loop."""
    cores = len(os.sched_getaffinity(0))
    procs = []
    for w in range(cores):
        cmd, env = _oracle_child(n_per_core, 1, first=w * n_per_core)
        procs.append(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env))
    secs = []
    for p in procs:
        out, err = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(err[-2000:])
        secs.append(json.loads(out.strip().splitlines()[-1])["seconds"])
    return {"calls": cores * n_per_core, "seconds": max(secs), "cores": cores}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    n = args.ref_calls
    times = []
    calls = 0
    cores = 1
    for _ in range(args.warmup):
        cpu_oracle_sample(max(1, n // 4))
    for _ in range(args.steps):
        r = cpu_oracle_all_cores(n)
        times.append(r["seconds"])
        calls += r["calls"]
        cores = r["cores"]
    tot = sum(times)
    value = calls / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": f"{n} calls per host core per step ({cores} cores)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} calls of the decode stream per core and step, one process per "
                                       "core, 1 BLAS thread each, fp64 numpy"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu(args):
    import torch
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    CALLS = args.calls
    T = args.tokens
    s, layer, xs = build_decode_layer(CALLS, T=T)
    wl = s.wl
    d = wl.d
    x_host = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).pin_memory()
    x_dev = x_host.cuda()
    y_dev = torch.empty((CALLS, T, d), dtype=torch.float32, device="cuda")
    y_host = torch.empty((CALLS, T, d), dtype=torch.float32).pin_memory()

    stream = torch.cuda.Stream()
    # warm the kernels (function attributes, first launches) outside capture
    with torch.cuda.stream(stream):
        for i in range(8):
            layer.moe_forward(0, x_dev[i], y_dev[i])
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(CALLS):
            layer.moe_forward(0, x_dev[i], y_dev[i])
    torch.cuda.synchronize()
    layer.moe_sync()

    def step():
        graph.replay()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st0 = layer.moe_cache_stats()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(os.path.join(os.environ.get("BENCH_LOG_DIR", "."), f"clocks_rank{rank}.csv"))
    torch.cuda.synchronize()
    with clk:
        time.sleep(0.3)
        e0.record(cur)
        for _ in range(args.steps):
            step()
        e1.record(cur)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    layer.moe_sync()
    st1 = layer.moe_cache_stats()
    # distinct routed experts per call in the timed steps (+ the shared one)
    exp_per_call = 1.0 + (st1["distinct_hits"] - st0["distinct_hits"]) / max(1, st1["layer_calls"] - st0["layer_calls"])
    alg_bytes = exp_per_call * EXPERT_BYTES
    value = CALLS * T * args.steps / (ms / 1e3)
    per_call_s = (ms / 1e3) / (CALLS * args.steps)

    # end to end: H2D of the step's inputs, the calls, D2H of the outputs
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        x_dev.copy_(x_host, non_blocking=True)
        graph.replay()
        y_host.copy_(y_dev, non_blocking=True)
    torch.cuda.synchronize()
    e2.record(cur)
    for _ in range(args.steps):
        x_dev.copy_(x_host, non_blocking=True)
        graph.replay()
        y_host.copy_(y_dev, non_blocking=True)
    e3.record(cur)
    torch.cuda.synchronize()
    ms_e2e = e2.elapsed_time(e3)
    e2e_value = CALLS * T * args.steps / (ms_e2e / 1e3)
    stats = layer.moe_cache_stats()

    if rank == 0:
        hbm, peak_kind = peaks()
        achieved = alg_bytes / per_call_s / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 mma operands, f32 accumulate (3-bit weights)",
            "data": "synthetic",
            "config": {"workload": workload_name(CALLS, T),
                       "calls_per_step": CALLS, "us_per_call": 1e6 * per_call_s, "tokens_per_call": T, "layers": 1,
                       "experts_per_call": exp_per_call,
                       "l2": "inputs larger than L2: 512 resident experts = 1.06 GB > 129 MB L2 "
                             "(the shared expert and the router stay L2-resident across calls)",
                       "graph": "10,000 moe_forward calls captured once, replayed per step",
                       "parallelism": "single GPU"},
            "gpu_launches": CALLS * args.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": recorded_traffic(),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                         "kernel": "decode_ffn_kernel with fused routing: one launch per call (average launch "
                                   "duration = call duration, launch gaps included; back to back, CUDA graph)",
                         "alg_bytes_per_launch": alg_bytes, "router_bytes": ROUTER_BYTES},
            "e2e": {"value": e2e_value, "unit": "tokens/s",
                    "h2d_bytes_per_step": int(x_host.numel() * 2), "d2h_bytes_per_step": int(y_host.numel() * 4)},
            "clocks": clk.summary(local),
            "cache": {"token_hits": stats["token_hits"], "token_misses": stats["token_misses"]},
        }
        if args.prefill and T == 1 and CALLS == DEFAULT_CALLS:
            try:
                line["prefill"] = run_prefill(args.prefill_steps, 3)
            except Exception as ex:   # reported, not hidden
                line["prefill"] = {"error": str(ex)[:300]}
        if args.stack_sweep:
            try:
                line["stack_sweep"] = run_stack_sweep(calls=args.stack_sweep)
            except Exception as ex:   # reported, not hidden
                line["stack_sweep"] = {"error": str(ex)[:300]}
        if args.stack and T == 1 and CALLS == DEFAULT_CALLS:
            try:
                cfgs = (3, 4) if args.stack_config == 0 else (args.stack_config,)
                modes = (1, 0) if args.stack_mode < 0 else (args.stack_mode,)
                line["stack"] = [r for c in cfgs for m in modes
                                 for r in run_stack(c, args.stack_pool, miss_mode=m, pool_layout=args.stack_pool_layout,
                                                    aheads=(False, True) if m == 1 and args.stack_pool_layout == 1
                                                    else (False,))]
            except Exception as ex:   # reported, not hidden
                line["stack"] = {"error": str(ex)[:300]}
        if args.kv and T == 1 and CALLS == DEFAULT_CALLS:
            try:
                line["kv_window"] = run_kv_window()
            except Exception as ex:   # reported, not hidden
                line["kv_window"] = {"error": str(ex)[:300]}
        if not args.no_cpu_baseline and T == 1:
            n = args.cpu_calls
            ra = cpu_oracle_all_cores(n)
            r1 = cpu_oracle_sample(n)
            line["cpu_baseline"] = {"value": ra["calls"] / ra["seconds"], "unit": "tokens/s", "cores": ra["cores"],
                                    "kind": "oracle",
                                    "sample": f"{ra['calls']} calls of the decode stream ({n} per core, one "
                                              f"process per core, 1 BLAS thread each), fp64 numpy oracle",
                                    "one_thread": {"value": n / r1["seconds"], "cores": 1,
                                                   "sample": f"first {n} calls, 1 BLAS thread"}}
        print(json.dumps(line), flush=True)
    layer.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--cpu-calls", type=int, default=12)
    ap.add_argument("--ref-calls", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", action="store_true", default=True,
                    help="also time the 12,288-token prefill chunk and sweep (the default at T=1)")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false")
    ap.add_argument("--prefill-steps", type=int, default=5)
    ap.add_argument("--stack", action="store_true", default=True,
                    help="also run the 48-layer stacks (T=5 Zipf 1.1, T=16 Zipf 0.8) with the 8,445-slot cache "
                         "(the default at T=1)")
    ap.add_argument("--no-stack", dest="stack", action="store_false")
    ap.add_argument("--stack-pool", type=int, default=2048,
                    help="host-pool entries for --stack: expert (l, e) reads entry (512 l + e) mod P; "
                         "0 = one per (layer, expert), 50.7 GB, slow to fill (default 2048, 4.2 GB)")
    ap.add_argument("--stack-config", type=int, default=0, choices=(0, 3, 4),
                    help="--stack: 3 = verify stack only, 4 = concurrent stack only (default both)")
    ap.add_argument("--stack-pool-layout", type=int, default=1, choices=(0, 1),
                    help="host pool of the stacks: 1 device block layout (default), 0 canonical")
    ap.add_argument("--stack-mode", type=int, default=1, choices=(-1, 0, 1),
                    help="--stack: 1 = GPU pulls misses (default), 0 = host-issued copies, -1 = both")
    ap.add_argument("--stack-sweep", type=int, default=0, metavar="CALLS",
                    help="verify width (T = 1, 4, 7) x cache capacity (9,057 / 8,445 / 6,144) sweep on the "
                         "verify stack, CALLS calls per pass")
    ap.add_argument("--kv", action="store_true", default=True,
                    help="also time the KV-streaming window (dense block reads of two 131,072-cell layers)")
    ap.add_argument("--no-kv", dest="kv", action="store_false")
    ap.add_argument("--kv-only", action="store_true", help="time only the KV-streaming window")
    ap.add_argument("--prefill-only", type=int, default=0, metavar="T",
                    help="time only the prefill path at T tokens (profiling runs)")
    ap.add_argument("--tokens", type=int, default=1, choices=range(1, 17), metavar="T",
                    help="tokens per decode call (1 + draft tokens verified together; the workload is T=1)")
    ap.add_argument("--calls", type=int, default=CALLS,
                    help="calls per step (the workload is 10,000; smaller only for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.gpus != 1 or _dist()[0] != 1:
        # the step runs on one GPU by scope; there is no multi-GPU arm
        print(f"bench.py: single GPU only (got --gpus {args.gpus}, WORLD_SIZE {_dist()[0]})", file=sys.stderr)
        sys.exit(2)
    elif args.kv_only:
        import torch
        torch.cuda.set_device(_dist()[2])
        print(json.dumps({"kv_window": run_kv_window(args.steps, args.warmup)}), flush=True)
    elif args.prefill_only:
        import torch
        torch.cuda.set_device(_dist()[2])
        print(json.dumps({"prefill": run_prefill(args.steps, args.warmup, sweep=(args.prefill_only,))}), flush=True)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
