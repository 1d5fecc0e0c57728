#!/usr/bin/env python3
"""Benchmark of the paged decode hot path on GB300: prints ONE JSON line.

A step is one decode step of one attention layer for the whole batch: the
append of every sequence's new K/V row (kvc_append) followed by paged decode
attention over the whole cache (kvc_decode_attention, whose split-K merge runs
inside the same call). Inputs are resident in HBM; the L2 is flushed (a
256 MiB write) between timed steps, outside the timed events.

Default workload: a Llama-3-8B-shaped layer, 32 query / 8 kv heads, head dim
128, bf16, batch 32, context lengths uniform in [512, 4096] (seed 43),
block size 16, physical blocks randomly permuted in a pool with 10% spare.
``value`` is decode-attention GB/s over the algorithmic bytes of a step (K/V
rows actually attended, q, out, the table entries read, lengths, plus the
append's reads and writes). The other shapes (all-4096 contexts, the shared-
prefix MHA batch, the long-context split-K batch, MLA, the tiny fp32 model)
are measured too and reported under ``variants``.

--impl reference times the CPU oracle instead (bounded samples of the same
workload on the host cores), for the driver's ratio.
"""

from __future__ import annotations

import os

# The oracle legs run NumPy single-threaded (their core count is reported as 1).
for _v in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "OMP_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention HBM GB/s (% of 8 TB/s roofline) and seq·layer steps/s on 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20

MAIN = dict(name="gqa_llama3_8b_layer", batch=32, hq=32, hkv=8, d=128, bs=16, lens=(512, 4096), dtype="bf16",
            seed=43)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            return float(j["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="kvc_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ workloads

def step_bytes(case_lens, hq, hkv, d, bs, elt, out_elt, unique_kv_rows=None):
    """Algorithmic bytes of one step (append + decode)."""
    B = len(case_lens)
    rows = sum(case_lens) if unique_kv_rows is None else unique_kv_rows
    kv = rows * hkv * d * elt * 2
    q = B * hq * d * elt
    out = B * hq * d * out_elt
    tables = sum(-(-n // bs) for n in case_lens) * 4
    lens = B * 4
    decode = kv + q + out + tables + lens
    append = B * hkv * d * elt * 2 * 2 + B * 8
    return decode, append


class GqaStep:
    """Device-resident inputs of one decode step plus the calls that run it."""

    def __init__(self, kvc, case, out_dtype, window=None):
        import torch
        self.kvc = kvc
        self.case = case
        self.window = window
        self.dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
        lens = case["context_lens"].tolist()
        self.lens = lens
        self.B, self.hq, self.d = case["q"].shape
        _, self.hkv, self.bs, _ = case["k_cache"].shape
        self.slots = kvc.slots_from_tables(case["block_tables"], self.bs, list(range(self.B)),
                                           [n - 1 for n in lens]).cuda()
        self.out = torch.empty((self.B, self.hq, self.d), dtype=out_dtype, device="cuda")
        self.ws = kvc.new_decode_workspace(self.B, self.hq, self.hkv, self.d, self.bs,
                                           case["block_tables"].shape[1])
        self.scale = 1.0 / math.sqrt(self.d)

    def append(self):
        d = self.dev
        self.kvc.append(d["k_new"], d["v_new"], self.slots, d["k_cache"], d["v_cache"])

    def decode(self):
        d = self.dev
        self.kvc.decode_attention(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                  self.scale, self.out, self.ws, window=self.window)


class L2Flush:
    """Evicts the inputs from L2 between timed steps: writes a buffer larger than
    L2, then reads a second one, so that the dirty lines of the write are
    written back to HBM before the timed region instead of during it."""

    def __init__(self):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")

    def run(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def flush_buffer():
    return L2Flush()


def time_steps(step, steps, warmup, flush, sampler=None):
    """Per-step CUDA-event times (ms) of append and decode, L2 flushed between steps."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.run()
        step.append()
        step.decode()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if sampler:
        sampler.start()
        time.sleep(0.2)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    # whole steps: nothing between the append and the decode, so the decode
    # may start its prologue while the append runs (programmatic launch)
    for i in range(steps):
        flush.run()
        ev[i][0].record(stream)
        step.append()
        step.decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks = sampler.stop() if sampler else None
    step_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(steps)]
    # the decode alone (the event before it also keeps it from overlapping the append)
    for i in range(steps):
        flush.run()
        step.append()
        ev[i][1].record(stream)
        step.decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]
    return step_ms, dec_ms, wall, clocks


def time_e2e(kvc, step, steps, warmup, flush):
    """Same step through the public API from pinned host memory: one H2D copy of the step's inputs (q, new
    k/v, tables, lengths, slots, packed at 256-byte offsets in one pinned staging buffer; the library calls
    take device views into its device copy), kvc_append, kvc_decode_attention, and a D2H copy of the output.
    The four operations are captured once in a CUDA graph and replayed every step (the host waits for each
    step's result before the next). Returns (ms per step, H2D bytes, D2H bytes, whether a graph was used)."""
    import torch
    c = step.case
    parts = [("q", c["q"]), ("k_new", c["k_new"]), ("v_new", c["v_new"]), ("block_tables", c["block_tables"]),
             ("context_lens", c["context_lens"]), ("slots", step.slots.cpu())]
    offs, total = {}, 0
    for name, t in parts:
        offs[name] = total
        total += -(-t.numel() * t.element_size() // 256) * 256
    host = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device="cuda")
    v = {}
    for name, t in parts:
        t = t.detach().to("cpu").contiguous()
        nb = t.numel() * t.element_size()
        host[offs[name]:offs[name] + nb].copy_(t.view(-1).view(torch.uint8))
        v[name] = dev_buf[offs[name]:offs[name] + nb].view(t.dtype).view(t.shape)
    dev = step.dev
    out = torch.empty_like(step.out)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h = out_h.numel() * out_h.element_size()

    def one():
        dev_buf.copy_(host, non_blocking=True)
        kvc.append(v["k_new"], v["v_new"], v["slots"], dev["k_cache"], dev["v_cache"])
        kvc.decode_attention(v["q"], dev["k_cache"], dev["v_cache"], v["block_tables"], v["context_lens"],
                             step.scale, out, step.ws)
        out_h.copy_(out, non_blocking=True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(max(3, warmup)):
            one()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one()
        graph = g
    except Exception as e:  # report it; the same calls then run eagerly
        print(f"e2e: CUDA graph capture failed ({type(e).__name__}: {e}); timing eager calls", file=sys.stderr)
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else one
    for _ in range(warmup):
        flush.run()
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(steps):
        flush.run()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()  # the host needs the result before the next step
        ts.append(a.elapsed_time(b))
    ok = bool(torch.equal(out_h, out.cpu()))
    if not ok:
        print("e2e: the host copy of the output differs from the device output", file=sys.stderr)
    return statistics.mean(ts), total, d2h, graph is not None


# --------------------------------------------------------------- oracle

def oracle_sample_seconds(case, seqs, units=None):
    """Times the oracle (append + decode) on the given sequences of a case.

    Returns (seconds, algorithmic bytes of that sample).
    """
    import numpy as np
    import torch
    from oracle import paged as OP

    def f64(t):
        return t.detach().cpu().to(torch.float64).numpy()

    bs = case["block_size"]
    tab = case["block_tables"]
    hkv = case["k_cache"].shape[1]
    hq, d = case["q"].shape[1], case["q"].shape[2]
    lens = [int(case["context_lens"][i]) for i in seqs]
    used = []
    rows = []
    for i, n in zip(seqs, lens):
        nb = -(-n // bs)
        rows.append(list(range(len(used), len(used) + nb)))
        used.extend(int(x) for x in tab[i, :nb])
    maxb = max(len(r) for r in rows)
    table = np.zeros((len(seqs), maxb), dtype=np.int64)
    for r, row in enumerate(rows):
        table[r, :len(row)] = row
    idx = torch.as_tensor(used, dtype=torch.long, device=case["k_cache"].device)
    kc = f64(case["k_cache"][idx])
    vc = f64(case["v_cache"][idx])
    q = f64(case["q"][list(seqs)])
    kn = f64(case["k_new"][list(seqs)])
    vn = f64(case["v_new"][list(seqs)])
    slots = np.array([table[r, (n - 1) // bs] * bs + (n - 1) % bs for r, n in enumerate(lens)], dtype=np.int64)
    t0 = time.perf_counter()
    kc2, vc2 = OP.append_to_paged(kn, vn, slots, kc, vc)
    OP.paged_decode(q, kc2, vc2, table, lens, 1.0 / math.sqrt(d))
    dt = time.perf_counter() - t0
    elt = case["q"].element_size()
    dec, app = step_bytes(lens, hq, hkv, d, bs, elt, elt)
    return dt, dec + app


def cpu_baseline(case, budget_s=10.0):
    """Oracle GB/s on whole sequences of the workload, cycling over the batch until about budget_s of CPU work."""
    B = case["q"].shape[0]
    n_done, tot_t, tot_b = 0, 0.0, 0
    while tot_t < budget_s and n_done < 50 * B:
        dt, by = oracle_sample_seconds(case, [n_done % B])
        tot_t += dt
        tot_b += by
        n_done += 1
    return {"value": round(tot_b / tot_t / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"append + decode of {n_done} whole sequences (all heads) of the same workload, cycling "
                      f"over its {B} sequences, float64 NumPy, single thread; {tot_t:.1f} s"}


_POOL_CASE = None


def _pool_init(args):
    """Pool worker start: rebuild the seeded workload on the CPU (not timed)."""
    global _POOL_CASE
    from paged_kv_cache_157_gb300 import workloads as W
    _POOL_CASE = W.gqa_case(*args)


def _pool_ready(_):
    time.sleep(0.2)  # spreads these tasks over the workers, each past its start-up
    return os.getpid()


def _pool_task(i):
    return oracle_sample_seconds(_POOL_CASE, [i])


def cpu_baseline_pool(tasks_per_core=48):
    """The same oracle on all host cores: a process pool (spawn start) over the sequences of the workload, each
    worker with its own copy of it; value = algorithmic bytes of all tasks / wall time of the pool run."""
    import multiprocessing as mp
    m = MAIN
    cores = len(os.sched_getaffinity(0))
    args = (m["batch"], m["hq"], m["hkv"], m["d"], m["bs"], m["lens"], m["dtype"], m["seed"])
    with mp.get_context("spawn").Pool(cores, initializer=_pool_init, initargs=(args,)) as pool:
        pool.map(_pool_ready, range(2 * cores), chunksize=1)
        n = cores * tasks_per_core
        t0 = time.perf_counter()
        res = pool.map(_pool_task, [i % m["batch"] for i in range(n)], chunksize=1)
        wall = time.perf_counter() - t0
    by = sum(b for _, b in res)
    return {"value": round(by / wall / 1e9, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"append + decode of {n} whole sequences (all heads), cycling over the {m['batch']} "
                      f"sequences, float64 NumPy, a spawn process pool of {cores} workers over sequences; "
                      f"{wall:.1f} s wall"}


# --------------------------------------------------------------- variants

def measure_gqa_case(kvc, case, steps, warmup, flush, unique_rows=None, window=None):
    import torch
    st = GqaStep(kvc, case, torch.bfloat16, window)
    step_ms, dec_ms, _, _ = time_steps(st, steps, warmup, flush)
    lens = st.lens if window is None else [min(n, window) for n in st.lens]  # rows actually read
    dec_b, app_b = step_bytes(lens, st.hq, st.hkv, st.d, st.bs, case["q"].element_size(), 2, unique_rows)
    ms = statistics.mean(step_ms)
    dms = statistics.mean(dec_ms)
    res = {"ms_per_step": round(ms, 5), "gbps": round((dec_b + app_b) / ms / 1e6, 1),
           "decode_ms": round(dms, 5), "decode_gbps": round(dec_b / dms / 1e6, 1),
           "frac_of_8tbs": round(dec_b / dms / 1e6 / NOMINAL_HBM_GBS, 4),
           "seq_layer_steps_per_s": round(len(lens) / (ms / 1e3), 1), "bytes_per_step": dec_b + app_b}
    del st
    torch.cuda.empty_cache()
    return res


def run_variant(kvc, name, flush, steps):
    import torch
    from paged_kv_cache_157_gb300 import workloads as W
    if name == "gqa_b32_ctx4096":
        c = W.gqa_case(32, 32, 8, 128, 16, [4096] * 32, "bf16", 43, device="cuda")
        return measure_gqa_case(kvc, c, steps, 5, flush)
    if name == "mha_shared_prefix_8x8":
        c = W.shared_case(8, 8, 2048, 256, 32, 128, 16, "f16", 44, device="cuda")
        unique = 8 * 2048 + 64 * 256
        r = measure_gqa_case(kvc, c, steps, 5, flush, unique_rows=unique)
        logical, _ = step_bytes(c["context_lens"].tolist(), 32, 32, 128, 16, 2, 2)
        r["logical_decode_bytes"] = logical
        r["note"] = "gbps counts each shared prompt block once (unique physical bytes)"
        return r
    if name == "gqa_long_splitk":
        c = W.gqa_case(4, 64, 8, 128, 16, [32768, 65536, 131072, 131072], "bf16", 45, device="cuda")
        return measure_gqa_case(kvc, c, max(5, steps // 4), 3, flush)
    if name == "gqa_window_b32_ctx4096_w1024":
        c = W.gqa_case(32, 32, 8, 128, 16, [4096] * 32, "bf16", 43, device="cuda")
        r = measure_gqa_case(kvc, c, steps, 5, flush, window=1024)
        r["note"] = "sliding window of 1024 rows: bytes count the visible rows only"
        return r
    if name == "gqa_fp8_b32_ctx4096":
        return measure_fp8(kvc, flush, steps)
    if name == "gqa_int8_b32_ctx4096":
        return measure_fp8(kvc, flush, steps, int8=True)
    if name == "mha_shared_prefix_8x8_cascade":
        return measure_shared_prefix(kvc, flush, steps)
    if name == "gqa_spec4_b32_ctx4096":
        return measure_multi(kvc, flush, steps, 4)
    if name == "cow_copy_blocks_2048":
        return measure_copy_blocks(kvc, flush, steps)
    if name == "gqa_ragged_17_31_32":
        c = W.gqa_case(3, 64, 8, 128, 16, [17, 31, 32], "bf16", 45, device="cuda")
        return measure_gqa_case(kvc, c, steps, 5, flush)
    if name == "tiny_mha_fp32":
        return measure_tiny(kvc, flush, steps)
    if name == "host_pool_shared_8x8":
        return measure_host_pool(kvc, steps)
    if name == "mla_deepseek_v2":
        return measure_mla(kvc, flush, steps)
    raise ValueError(f"unknown workload {name}")


TARGET = "gqa_b32_ctx4096"
VARIANTS = ("mha_shared_prefix_8x8", "gqa_long_splitk", "gqa_ragged_17_31_32", "tiny_mha_fp32",
            "mla_deepseek_v2", "gqa_window_b32_ctx4096_w1024", "cow_copy_blocks_2048", "gqa_fp8_b32_ctx4096",
            "gqa_int8_b32_ctx4096", "gqa_spec4_b32_ctx4096", "mha_shared_prefix_8x8_cascade",
            "host_pool_shared_8x8")


def with_measured_fraction(r):
    """Adds the decode's fraction of the measured (or fallback) HBM copy peak to a variant's record."""
    peak, kind = peaks()
    g = r.get("decode_gbps", r.get("gbps")) if isinstance(r, dict) else None
    if g is not None and "error" not in r:
        r[f"frac_of_{kind}_hbm"] = round(g / peak, 4)
    return r


def variants(kvc, flush, steps):
    import torch
    out = {}
    for name in VARIANTS:
        try:
            out[name] = with_measured_fraction(run_variant(kvc, name, flush, steps))
        except Exception as e:  # report, do not hide, a failing variant
            out[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return out


def measure_host_pool(kvc, steps):
    """The host step of the sharing workload: 8 prompts of 2048 tokens, each forked 8 ways (64 sequences,
    prompt blocks at refcount 8) with 256 private tokens; per step every sequence reserves one slot
    (kvc_seq_reserve, one call per sequence, or kvc_seq_reserve_batch, one call for all) and the 64 table rows
    are rebuilt (kvc_build_block_tables). Timed on the host through ctypes with preallocated buffers, so the
    figures include the per-call binding overhead."""
    import ctypes
    lib = kvc.raw()
    bs, max_blocks = 16, 160
    pool = kvc.BlockPool(4096, bs)
    seqs = []
    for _ in range(8):
        p = pool.add()
        pool.reserve(p, 2048)
        seqs.extend(pool.fork(p) for _ in range(8))
        pool.free(p)
    for sq in seqs:
        pool.reserve(sq, 256)
    n = len(seqs)
    ids = (ctypes.c_int64 * n)(*seqs)
    tab = (ctypes.c_int32 * (n * max_blocks))()
    lens = (ctypes.c_int32 * n)()
    slot = (ctypes.c_int64 * n)()
    h = pool._h
    steps = min(steps, (max_blocks * bs - 2304) // 4)  # two loops, each adds `steps` tokens per sequence
    t_res = t_batch = t_tab = 0.0
    for _ in range(steps):
        t0 = time.perf_counter()
        for sq in seqs:
            if lib.kvc_seq_reserve(h, sq, 1, slot) != 0:
                raise RuntimeError("kvc_seq_reserve failed")
        t1 = time.perf_counter()
        if lib.kvc_build_block_tables(h, ids, n, tab, max_blocks, lens) != 0:
            raise RuntimeError("kvc_build_block_tables failed")
        t_tab += time.perf_counter() - t1
        t_res += t1 - t0
    for _ in range(steps):
        t0 = time.perf_counter()
        if lib.kvc_seq_reserve_batch(h, ids, n, 1, slot) != 0:
            raise RuntimeError("kvc_seq_reserve_batch failed")
        t_batch += time.perf_counter() - t0
    st = pool.stats()
    pool.close()
    return {"us_per_step": round((t_batch + t_tab) / steps * 1e6, 2),
            "reserve_batch_64_us": round(t_batch / steps * 1e6, 2),
            "reserve_64_calls_us": round(t_res / steps * 1e6, 2),
            "build_tables_64x160_us": round(t_tab / steps * 1e6, 2), "steps": steps, "final_stats": st,
            "note": "host CPU only, through ctypes; us_per_step = one batch reserve + one table build"}


def measure_tiny(kvc, flush, steps):
    """1 sequence, 2 layers, 4 heads x 32, fp32: seq*layer decode steps per second (append + decode). Eager
    calls, and the same four calls (append and decode of both layers) captured once as a CUDA graph and
    replayed per step, as a latency-bound serving loop would run them (L2 flushed between steps either way)."""
    import torch
    from paged_kv_cache_157_gb300 import workloads as W
    res, sts = [], []
    for L in range(2):
        c = W.gqa_case(1, 4, 4, 32, 16, [69], "f32", 42 + L, device="cuda")
        st = GqaStep(kvc, c, torch.float32)
        step_ms, _, _, _ = time_steps(st, steps, 5, flush)
        res.append(statistics.mean(step_ms))
        sts.append(st)
    ms = sum(res)
    out = {"ms_per_step_2_layers": round(ms, 5), "seq_layer_steps_per_s": round(2 / (ms / 1e3), 1),
           "note": "latency-bound: one sequence of 69 tokens"}
    try:
        cur = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            for st in sts:
                st.append()
                st.decode()
        cur.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for st in sts:
                st.append()
                st.decode()
        for _ in range(5):
            flush.run()
            g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            flush.run()
            a.record(cur)
            g.replay()
            b.record(cur)
        torch.cuda.synchronize()
        gms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        out["graph_ms_per_step_2_layers"] = round(gms, 5)
        out["graph_seq_layer_steps_per_s"] = round(2 / (gms / 1e3), 1)
    except RuntimeError as e:  # report, do not hide, a failed capture
        out["graph_error"] = str(e)[:200]
    return out


def measure_fp8(kvc, flush, steps, int8=False):
    """Llama-3-8B-shaped layer over a one-byte cache, FP8 e4m3 or INT8 (batch 32, lengths 4096): the quantising
    append of the new tokens + the one-byte decode (bf16 queries and output). Bytes: 1 per cached K/V element + 4
    per (row, kv head) of V scales, plus q, out, tables, lengths."""
    import torch
    from paged_kv_cache_157_gb300 import workloads as W
    c = (W.int8_case if int8 else W.fp8_case)(32, 32, 8, 128, 16, [4096] * 32, 94, device="cuda")
    append_fn = kvc.append_int8 if int8 else kvc.append_fp8
    decode_fn = kvc.decode_attention_int8 if int8 else kvc.decode_attention_fp8
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    lens = c["context_lens"].tolist()
    B, hq, hkv, D, bs = 32, 32, 8, 128, 16
    slots = kvc.slots_from_tables(c["block_tables"], bs, list(range(B)), [n - 1 for n in lens]).cuda()
    out = torch.empty((B, hq, D), dtype=torch.bfloat16, device="cuda")
    ws = kvc.new_decode_workspace(B, hq, hkv, D, bs, c["block_tables"].shape[1])
    scale = 1.0 / math.sqrt(D)

    class S:
        def append(self):
            append_fn(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"], d["v_scale"], d["k_scale"])

        def decode(self):
            decode_fn(d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"], d["block_tables"],
                      d["context_lens"], scale, out, ws)

    step_ms, dec_ms, _, _ = time_steps(S(), steps, 5, flush)
    rows = sum(lens)
    dec_b = rows * hkv * (2 * D + 4) + 2 * B * hq * D * 2 + sum(-(-n // bs) for n in lens) * 4 + B * 4
    dms = statistics.mean(dec_ms)
    bf16_equiv = rows * hkv * D * 2 * 2
    return {"decode_ms": round(dms, 5), "decode_gbps": round(dec_b / dms / 1e6, 1),
            "frac_of_8tbs": round(dec_b / dms / 1e6 / NOMINAL_HBM_GBS, 4),
            "bf16_equivalent_gbps": round(bf16_equiv / dms / 1e6, 1),
            "ms_per_step": round(statistics.mean(step_ms), 5), "bytes_per_step": dec_b,
            "note": "bf16_equivalent_gbps counts the bytes the same rows take in bf16"}


def measure_multi(kvc, flush, steps, T=4):
    """Llama-3-8B-shaped layer verifying T speculated tokens per sequence (batch 32, lengths 4096 after the
    append): kvc_append of the B*T new rows + kvc_decode_attention_multi (bf16). Bytes: every cached K/V row
    once (all T tokens share each page), plus q, out, tables, lengths."""
    import torch
    from paged_kv_cache_157_gb300 import workloads as W
    B, hq, hkv, D, bs = 32, 32, 8, 128, 16
    c = W.multi_case(B, T, hq, hkv, D, bs, [4096] * B, "bf16", 95, device="cuda")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    lens = c["context_lens"].tolist()
    slots = kvc.slots_from_tables(c["block_tables"], bs, [i for i in range(B) for _ in range(T)],
                                  [n - T + t for n in lens for t in range(T)]).cuda()
    out = torch.empty((B, T, hq, D), dtype=torch.bfloat16, device="cuda")
    ws = kvc.new_multi_workspace(B, T, hq, hkv, D, bs, c["block_tables"].shape[1])
    scale = 1.0 / math.sqrt(D)
    kn, vn = d["k_new"].reshape(B * T, hkv, D), d["v_new"].reshape(B * T, hkv, D)

    class S:
        def append(self):
            kvc.append(kn, vn, slots, d["k_cache"], d["v_cache"])

        def decode(self):
            kvc.decode_attention_multi(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                       scale, out, ws)

    step_ms, dec_ms, _, _ = time_steps(S(), steps, 5, flush)
    dec_b = sum(lens) * hkv * D * 2 * 2 + 2 * B * T * hq * D * 2 + sum(-(-n // bs) for n in lens) * 4 + B * 4
    dms = statistics.mean(dec_ms)
    return {"decode_ms": round(dms, 5), "decode_gbps": round(dec_b / dms / 1e6, 1),
            "frac_of_8tbs": round(dec_b / dms / 1e6 / NOMINAL_HBM_GBS, 4),
            "query_tokens_per_s": round(B * T / (dms / 1e3), 1),
            "ms_per_step": round(statistics.mean(step_ms), 5), "bytes_per_step": dec_b,
            "note": f"{T} new tokens per sequence attend causally in one pass over the pages"}


def measure_shared_prefix(kvc, flush, steps):
    """Config 3 through kvc_decode_attention_shared_prefix: 8 prompts x 2048 tokens forked 8 ways + 256 private
    tokens each, 32 heads x 128, fp16; the step appends the 64 new tokens (private blocks) and decodes; bytes
    count each shared block once (unique physical bytes)."""
    import torch
    from paged_kv_cache_157_gb300 import workloads as W
    c = W.shared_case(8, 8, 2048, 256, 32, 128, 16, "f16", 44, device="cuda")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    lens = c["context_lens"].tolist()
    B = 64
    slots = kvc.slots_from_tables(c["block_tables"], 16, list(range(B)), [n - 1 for n in lens]).cuda()
    out = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = kvc.shared_prefix_workspace(B, 8, 32, 32, 128, 16, c["block_tables"].shape[1])
    prefix = torch.full((8,), 2048, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(128)

    class S:
        def append(self):
            kvc.append(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"])

        def decode(self):
            kvc.decode_attention_shared_prefix(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                               d["context_lens"], 8, prefix, scale, out, ws)

    step_ms, dec_ms, _, _ = time_steps(S(), steps, 5, flush)
    unique = 8 * 2048 + 64 * 256
    dec_b, _ = step_bytes(lens, 32, 32, 128, 16, 2, 2, unique)
    dms = statistics.mean(dec_ms)
    return {"decode_ms": round(dms, 5), "decode_gbps": round(dec_b / dms / 1e6, 1),
            "frac_of_8tbs": round(dec_b / dms / 1e6 / NOMINAL_HBM_GBS, 4),
            "ms_per_step": round(statistics.mean(step_ms), 5), "bytes_per_step": dec_b,
            "note": "kvc_decode_attention_shared_prefix (shared prompt rows read once per group); unique bytes"}


def measure_copy_blocks(kvc, flush, steps):
    """Copy-on-write: 2048 (shared, fresh) block pairs copied in the K and the V pool of the Llama-3-8B layer
    (8 kv heads x 16 rows x 128 dims bf16 = 32 KB per block and pool); bytes = read + write."""
    import torch
    from paged_kv_cache_157_gb300 import workloads as W
    nblk, n_pairs = 16384, 2048
    g = torch.Generator(device="cuda")
    g.manual_seed(71)
    kc = W.normal((nblk, 8, 16, 128), "bf16", g)
    vc = W.normal((nblk, 8, 16, 128), "bf16", g)
    perm = torch.randperm(nblk, generator=torch.Generator().manual_seed(72))[:2 * n_pairs]
    pairs = perm.view(n_pairs, 2).to(torch.int64).cuda()

    class S:
        def append(self):
            pass

        def decode(self):
            kvc.copy_blocks(kc, pairs)
            kvc.copy_blocks(vc, pairs)

    _, dec_ms, _, _ = time_steps(S(), steps, 5, flush)
    moved = 2 * 2 * n_pairs * kc[0].numel() * kc.element_size()
    dms = statistics.mean(dec_ms)
    return {"ms": round(dms, 5), "gbps": round(moved / dms / 1e6, 1), "bytes_per_step": moved,
            "note": "read + write bytes of two kvc_copy_blocks calls (K and V pools)"}


def measure_mla(kvc, flush, steps):
    import torch
    from paged_kv_cache_157_gb300 import workloads as W
    try:
        kvc.decode_mla_workspace_size(64, 128, 512, 64, 64, 128)
    except kvc.KvcError as e:
        return {"unavailable": str(e)}
    c = W.mla_case(64, 128, 512, 64, 64, (1024, 8192), "bf16", 46, device="cuda")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
    lens = c["context_lens"].tolist()
    B = 64
    slots = kvc.slots_from_tables(c["block_tables"], 64, list(range(B)), [n - 1 for n in lens]).cuda()
    out = torch.empty((B, 128, 512), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(1, kvc.decode_mla_workspace_size(B, 128, 512, 64, 64, c["block_tables"].shape[1])),
                     dtype=torch.uint8, device="cuda")
    scale = 1.0 / 24.0

    class S:
        def append(self):
            kvc.append_latent(d["c_new"], slots, d["latent_cache"], 512)

        def decode(self):
            kvc.decode_attention_mla(d["q"], d["latent_cache"], d["block_tables"], d["context_lens"], scale, 512,
                                     out, ws)

    step_ms, dec_ms, _, _ = time_steps(S(), steps, 5, flush)
    rows = sum(lens)
    dec_b = rows * 576 * 2 + B * 128 * 576 * 2 + B * 128 * 512 * 2 + sum(-(-n // 64) for n in lens) * 4 + B * 4
    flops = rows * 128 * 2 * (576 + 512)
    dms = statistics.mean(dec_ms)
    return {"decode_ms": round(dms, 5), "decode_gbps": round(dec_b / dms / 1e6, 1),
            "tflops": round(flops / dms / 1e9, 1), "frac_of_8tbs": round(dec_b / dms / 1e6 / NOMINAL_HBM_GBS, 4),
            "ms_per_step": round(statistics.mean(step_ms), 5), "bytes_per_step": dec_b, "flops_per_step": flops}


# ------------------------------------------------------------------- main

def traffic_from_profile():
    """DRAM bytes per launch of the decode kernel from the committed ncu summary, if the
    kernel source has not changed since it was taken; else None."""
    p = os.path.join(ROOT, "profiles", "gqa_decode_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        j = json.load(open(p))
        if j.get("source_sha256") != kernel_source_sha():
            return None
        return j.get("dram_bytes_per_launch")
    except Exception:
        return None


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("decode_gqa_mma.cuh", "decode_gqa_impl.cuh", "decode_gqa.h", "kvc_device.cuh", "decode_gqa_api.cu",
              "decode_gqa_mma_launch.cuh"):
        h.update(open(os.path.join(ROOT, "paged_kv_cache_157_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def max_over_ranks(values, world, device):
    """Each value's maximum over the ranks (the slowest replica sets the time); one rank returns them as is."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def replica_gbps(world, bytes_per_step, ms_per_step):
    """Whole-job GB/s of `world` replicas that each move bytes_per_step per step in ms_per_step."""
    return world * bytes_per_step / (ms_per_step / 1e3) / 1e9


def run_kvc(args):
    import torch
    import torch.distributed as dist
    import paged_kv_cache_157_gb300 as kvc
    from paged_kv_cache_157_gb300 import build_lib
    from paged_kv_cache_157_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if rank == 0:
        build_lib.build()
    if world > 1:
        dist.barrier()
    kvc.raw()

    m = MAIN
    case = W.gqa_case(m["batch"], m["hq"], m["hkv"], m["d"], m["bs"], m["lens"], m["dtype"], m["seed"],
                      device="cuda")
    step = GqaStep(kvc, case, torch.bfloat16)
    flush = flush_buffer()
    sampler = ClockSampler(local) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms, dec_ms, wall, clocks = time_steps(step, args.steps, args.warmup, flush, sampler)
    if world > 1:
        dist.barrier()
    total_ms, dec_avg = max_over_ranks([sum(step_ms), statistics.mean(dec_ms)], world, "cuda")
    ms = total_ms / args.steps
    dec_b, app_b = step_bytes(step.lens, step.hq, step.hkv, step.d, step.bs, 2, 2)
    per_step = dec_b + app_b
    value = replica_gbps(world, per_step, ms)
    if rank != 0:
        dist.destroy_process_group()
        return
    peak, peak_kind = peaks()
    achieved = dec_b / (dec_avg / 1e3) / 1e9
    e2e_ms, h2d, d2h, e2e_graph = time_e2e(kvc, step, min(args.steps, 500), min(args.warmup, 10), flush)
    e2e_value = per_step / (e2e_ms / 1e3) / 1e9
    # The batch the bandwidth target is stated on (batch 32, every context 4096), measured on every run and
    # reported inside `roofline` and as the last key of the line.
    tgt_full = with_measured_fraction(run_variant(kvc, TARGET, flush, max(10, min(args.steps, 200))))
    target = {k: tgt_full[k] for k in ("decode_ms", "decode_gbps", "frac_of_8tbs", f"frac_of_{peak_kind}_hbm",
                                       "ms_per_step", "gbps") if k in tgt_full}
    target["target"] = "decode >= 0.75 of 8 TB/s (<= 0.0895 ms for 536.9 MB of K/V + q/out)"
    var = {} if args.no_variants else variants(kvc, flush, max(10, min(args.steps, 200)))
    cpu = None if args.no_cpu_baseline else cpu_baseline(case)
    cpu_pool = None if args.no_cpu_baseline else cpu_baseline_pool()
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/K/V, uniform lengths, permuted block pool)",
        "config": {
            "workload": "GQA decode, Llama-3-8B-shaped layer: batch 32, 32 q / 8 kv heads, head_dim 128, bf16, "
                        "context lengths U[512,4096] (seed 43), block_size 16, permuted pool (+10% spare); "
                        "step = kvc_append of 32 new tokens + kvc_decode_attention (bf16 out)",
            "batch": m["batch"], "n_q_heads": m["hq"], "n_kv_heads": m["hkv"], "head_dim": m["d"],
            "block_size": m["bs"], "context_lens": "U[512,4096]", "mean_context_len": statistics.mean(step.lens),
            "l2": "flushed between timed steps (256 MiB write, then a 256 MiB read that drains the dirty lines; "
                  "outside the timed events)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "frac_of_8tbs": round(value / NOMINAL_HBM_GBS, 4),
        "seq_layer_steps_per_s": round(world * m["batch"] / (ms / 1e3), 1),
        "bytes_per_step": per_step,
        "roofline": {"bound": "hbm", "kernel": "kvc_decode_attention (gqa_mma_kernel + gqa_mma_merge_kernel, timed together)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "traffic": traffic_from_profile(), "algorithmic_bytes_per_launch": dec_b,
                     "target_b32_ctx4096": target},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5),
                "how": ("one packed H2D copy + kvc_append + kvc_decode_attention + D2H of the output, "
                        + ("replayed as one CUDA graph" if e2e_graph else "eager calls (graph capture failed)"))},
        "gpu_launches": 2 * args.steps,  # kvc_append + kvc_decode_attention per step
        "clocks": clocks,
        "timed_wall_s": round(wall, 4),
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_pool,
        "variants": var,
        "target_b32_ctx4096": target,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle on the host cores: each step a bounded sample (one whole sequence) of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from paged_kv_cache_157_gb300 import workloads as W
    m = MAIN
    case = W.gqa_case(m["batch"], m["hq"], m["hkv"], m["d"], m["bs"], m["lens"], m["dtype"], m["seed"])
    for i in range(args.warmup):
        oracle_sample_seconds(case, [i % m["batch"]])
    budget = 150.0
    tot_t, tot_b, n = 0.0, 0, 0
    t_start = time.perf_counter()
    for i in range(args.steps):
        dt, by = oracle_sample_seconds(case, [i % m["batch"]])
        tot_t += dt
        tot_b += by
        n += 1
        if time.perf_counter() - t_start > budget:
            break
    value = tot_b / tot_t / 1e9
    ms = tot_t / n * 1e3
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": 1, "steps": n, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (same seeded workload)",
        "config": {"workload": "same as the kvc arm; each step is one whole sequence (all heads) of it",
                   "requested_steps": args.steps},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "append + decode of one sequence (all heads) per step, float64 NumPy, "
                                   "single thread"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["kvc", "reference"], default="kvc")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=("main", TARGET) + VARIANTS, default="main",
                    help="time one other workload alone (prints its measurement, not the contract line)")
    ap.add_argument("--gqa-engine", choices=("auto", "cuda-core", "tensor-core", "warp-mma"), default="auto",
                    help="with --workload: 'cuda-core' forces the CUDA-core kernel, 'tensor-core' puts wide query "
                         "groups on the tcgen05 kernel at any size, 'warp-mma' keeps them on the warp-MMA kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload != "main":
        import paged_kv_cache_157_gb300 as kvc
        from paged_kv_cache_157_gb300 import build_lib
        build_lib.build()
        kvc.set_option(kvc.OPT_GQA_ENGINE, {"auto": 0, "cuda-core": 1, "tensor-core": 2, "warp-mma": 3}[args.gqa_engine])
        print(json.dumps({"workload": args.workload, "gqa_engine": args.gqa_engine,
                          **with_measured_fraction(run_variant(kvc, args.workload, flush_buffer(), args.steps))}),
              flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kvc(args)


if __name__ == "__main__":
    main()
