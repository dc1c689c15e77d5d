#!/usr/bin/env python
"""Benchmark of the OSCAR decode step (INT2 rotated KV append + mixed-precision
paged decode) on one GB300, printing one JSON line.

A step is one decode step of a batch: oscar_append_decode, which appends each
sequence's current token (INT2 pool and its BF16 window row, as
oscar_append_mixed) and decodes over the whole cache (as oscar_decode).  The default workload is the
batch-1 long decode (32 query / 8 KV heads, head_dim 128, context 32768, sink
64 + window 128 in BF16, group 64, shuffled pages).  Its cache (21.7 MB) fits
in L2, so the benchmark builds enough independent cache replicas (disjoint
pages of one pool) that the replicas together exceed 3x the L2 size and
cycles through them, one replica per step.

The K timed steps are captured in CUDA graphs and timed with CUDA events on
the launching stream; W warm-up steps run first.  Also reported: the decode
alone (roofline of the dominant kernel), the in-repo BF16 paged decode over
the same tokens (speedup reference), an end-to-end figure through the public
API with host buffers, and the fp64 CPU oracle on a bounded sample.

--impl reference times that oracle instead (the slow CPU restatement of the
same computation), on the same workload and metric.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "oscar_decode HBM GB/s (% of peak) & tokens/s; INT2 vs BF16 decode speedup"
E2E_IN_FLIGHT = 4  # steps of independent batches in flight in the end-to-end loop


# --------------------------------------------------------------------------- helpers

def algorithmic_bytes_decode(w, batch_lens, n_q_heads=None, n_kv_heads=None):
    """Bytes a decode step must move: INT2 codes + scale/zero of bulk tokens, BF16
    sink/window tokens, q in and fp32 out (rotations and page tables not counted).
    ``w`` is anything with num_q_heads, num_kv_heads, head_dim, group_size,
    sink_len and window_len attributes."""
    H = w.num_kv_heads if n_kv_heads is None else n_kv_heads
    Hq = w.num_q_heads if n_q_heads is None else n_q_heads
    D, G, S, W = w.head_dim, w.group_size, w.sink_len, w.window_len
    per_bulk = 2 * (D // 4) + 2 * (D // G) * 2 * 2
    per_bf16 = 2 * D * 2
    total = 0
    for L in batch_lens:
        n_bf16 = min(S, L) + max(0, L - max(S, L - W))
        n_bulk = L - n_bf16
        total += H * (n_bulk * per_bulk + n_bf16 * per_bf16)
    total += len(batch_lens) * Hq * D * (2 + 4)
    return total


def algorithmic_bytes_append(w, n_tokens, bf16_rows=False):
    """Bytes of an append: read K, V (bf16) and the slot; write the INT2 rows (codes
    and fp16 scale/zero); with bf16_rows also the K and V rows of the sink/window."""
    D, G, H = w.head_dim, w.group_size, w.num_kv_heads
    rows = H * 2 * D * 2 + 12 if bf16_rows else 0  # + sequence id and position
    return n_tokens * (H * 2 * D * 2 + 8 + H * (2 * (D // 4) + 2 * (D // G) * 2 * 2) + rows)


def algorithmic_bytes_bf16(w, batch_lens):
    return sum(w.num_kv_heads * L * 2 * w.head_dim * 2 for L in batch_lens) + \
        len(batch_lens) * w.num_q_heads * w.head_dim * (2 + 4)


class ClockSampler:
    """Background nvidia-smi sampler of SM clocks and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.interval = interval_ms
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        used = inside
        where = "timed_region"
        if not inside:  # region shorter than the sampling interval: nearest samples
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            used = [p for (_, p) in near]
            where = "adjacent_to_timed_region"
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in used if num(p[1]) is not None]
        mx = [num(p[2]) for p in used if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in used for i in range(4) if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(used), "where": where}


_T0 = time.perf_counter()


def cuda_runtime():
    """The CUDA runtime library the OSCAR library links (already loaded in this
    process), for the end-to-end loop's graph launches and events."""
    ok = sys.modules["int2_rotated_kv_append_gb300"]
    ok.load_library()
    rt = None
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if rt is None:
        raise RuntimeError("libcudart not found")
    P = ctypes.c_void_p
    rt.cudaGraphLaunch.argtypes = [P, P]
    rt.cudaGraphUpload.argtypes = [P, P]
    rt.cudaEventRecord.argtypes = [P, P]
    rt.cudaEventSynchronize.argtypes = [P]
    rt.cudaEventDestroy.argtypes = [P]
    rt.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(P), ctypes.c_uint]
    return rt


def log(msg: str):
    """Progress line on stderr (the JSON result goes to stdout)."""
    print(f"[bench {time.perf_counter() - _T0:8.2f}s] {msg}", file=sys.stderr, flush=True)


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_peak_bf16():
    """Dense bf16 tensor TFLOP/s as a burst (a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def workload_config(args, w, batch, seq_len, pps, l2_policy):
    """The config object of the JSON line (the same for both arms)."""
    from int2_rotated_kv_append_gb300 import synth
    return {"workload": synth.CONFIG_NAMES[args.config] + ": decode step = append current token (INT2 + BF16 window) + "
                        "mixed-precision paged decode",
            "batch": batch, "seq_len": seq_len, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "sink": w.sink_len, "window": w.window_len, "group": w.group_size,
            "page_size": 16, "pages_per_split": "auto" if pps == 0 else pps, "l2_policy": l2_policy}


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one oscar_decode
# launch (q-rotation + split + merge kernels) on the batch-1 32K, batch-64 and
# batch-4 131K workloads, from one ncu capture of the three kernels each (cold caches: the
# split partials are re-read from DRAM there, from L2 in the timed loop).
MEASURED_DECODE_TRAFFIC = {1: 556288 + 22832896 + 324864,
                           2: 1072640 + 428843264 + 4089088 + 8044544,
                           3: 613888 + 341584384 + 5817856 + 18014464}


def cpu_model() -> str:
    """The host CPU's model name as /proc/cpuinfo or the platform reports it ("unknown" if neither does)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "hardware", "cpu model"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine() or "unknown"


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (the slowest rank's time is the job's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_rank_step per step (weak scaling)."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    """The fp64 CPU oracle timed on the host cores, one rank only."""
    if rank != 0:
        return
    import concurrent.futures
    import numpy as np
    import torch

    from int2_rotated_kv_append_gb300 import synth
    from int2_rotated_kv_append_gb300.synth import bits16
    from oracle import oracle as O

    O.build_oracle()
    w = synth.make_config(args.config)
    # The oracle's own append builds the cache it then decodes (host memory).
    codes = np.zeros(w.num_pages * w.num_kv_heads * 2 * 16 * w.head_dim // 4, np.uint8)
    sz = np.zeros(w.num_pages * w.num_kv_heads * 2 * 16 * (w.head_dim // w.group_size) * 2, np.uint16)
    kb, vb = bits16(w.k), bits16(w.v)
    Rk, Rv, ck, cv = (t.cpu().numpy() for t in (w.R_k, w.R_v, w.clip_k, w.clip_v))
    slots = w.slot_mapping.numpy()
    threads = min(os.cpu_count() or 1, 32)
    chunks = np.array_split(np.arange(w.num_tokens), threads)

    def app(ix):
        O.append(w.dims, kb[ix], vb[ix], Rk, Rv, ck, cv, slots[ix], codes, sz)
    with concurrent.futures.ThreadPoolExecutor(threads) as ex:
        list(ex.map(app, chunks))
    sink, win = w.sink_window()
    sinkb, winb, qb = bits16(sink), bits16(win), bits16(w.q)
    pt, lens = w.page_table.numpy(), w.seq_lens.numpy()
    gqa = w.num_q_heads // w.num_kv_heads

    def sample_step(i, L):
        # one KV head's query group over the first L tokens of sequence 0, GQA heads in parallel threads
        h = i % w.num_kv_heads
        lens_s = lens.copy()
        lens_s[0] = L
        pairs = [[(0, h * gqa + j)] for j in range(gqa)]
        with concurrent.futures.ThreadPoolExecutor(gqa) as ex:
            list(ex.map(lambda pr: O.decode(w.dims, w.batch, qb, Rk, Rv, codes, sz, sinkb, winb, pt, lens_s,
                                            w.sink_len, w.window_len, 0.0, pairs=pr), pairs))
    # Calibrate the sample length so the whole run stays within ~2 minutes.
    L_full = int(lens[0])
    t = time.perf_counter()
    sample_step(0, L_full)
    t_full = time.perf_counter() - t
    budget = 120.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, budget / max(t_full, 1e-6))
    L = max(w.sink_len + w.window_len + 16, int(L_full * frac))
    for i in range(args.warmup):
        sample_step(i, L)
    t = time.perf_counter()
    for i in range(args.steps):
        sample_step(i, L)
    el = time.perf_counter() - t
    step_bytes = algorithmic_bytes_decode(w, [L], n_q_heads=gqa, n_kv_heads=1)
    value = step_bytes * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, w, w.batch, int(lens.max()), 0, "host memory (fp64 CPU oracle)"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": gqa, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"per step: the {gqa} query heads of one KV head of sequence 0 over its first "
                                   f"{L} of {L_full} tokens (fp64 oracle, one thread per query head)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- our arm

def capture_graph(fn, n, dev):
    """CUDA graph of a chunk of calls fn(0..per-1), replayed n // per times (per | n, per <= 1000)."""
    import torch
    per = n if n <= 1000 else next(d for d in range(1000, 0, -1) if n % d == 0)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(min(3, n)):
            fn(i)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per):
            fn(i)
    return g, n // per


def upload_graph(g):
    """cudaGraphUpload of a captured torch CUDA graph on the current stream."""
    import torch
    rt = cuda_runtime()
    rc = rt.cudaGraphUpload(ctypes.c_void_p(g.raw_cuda_graph_exec()),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise RuntimeError(f"cudaGraphUpload failed ({rc})")


def timed_graph(fn, n, warm, dev, world, barrier):
    """n calls of fn captured in CUDA graphs, after `warm` untimed calls; CUDA events
    on the replaying stream, a synchronize and a barrier on both sides; the slowest
    rank's milliseconds and the host clock around the timed region."""
    import torch
    g, reps = capture_graph(fn, n, dev)
    if warm > 0:
        gw, rw = capture_graph(fn, warm, dev)
        for _ in range(rw):
            gw.replay()
    # The timed graph is uploaded to the device before the timed region (no work runs):
    # a graph's first launch otherwise uploads its nodes as it goes, about 1 us per
    # step at B=1 over 20 or 200 steps.
    upload_graph(g)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    e1.synchronize()
    t1 = time.perf_counter()
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    return ms, (t0, t1)


class DecodeSetup:
    """One decode workload on the device: enough cache replicas (disjoint pages of
    one pool) that they exceed 3x L2, the INT2 and BF16 caches built by the
    library's appends, per-replica inputs in one staging block (q, k, v, slots of
    the current token), and the calls of a step (append, decode, BF16 decode)."""

    def __init__(self, cfg, dev, l2, replicas=0, pps=-1, in_flight=1):
        import numpy as np
        import torch

        import int2_rotated_kv_append_gb300 as ok
        from int2_rotated_kv_append_gb300 import synth
        from int2_rotated_kv_append_gb300.cache import Bf16Cache, Int2Cache

        self.cfg = cfg
        base_lens = synth.config_seq_lens(cfg)
        B = len(base_lens)
        one = types.SimpleNamespace(num_q_heads=64 if cfg == 3 else 32, num_kv_heads=8, head_dim=128,
                                    group_size=64, sink_len=64, window_len=256 if cfg == 3 else 128)
        w0_bytes = algorithmic_bytes_decode(one, base_lens)
        NR = max(1, math.ceil(3 * l2 / w0_bytes)) if replicas <= 0 else replicas
        log(f"generating workload: config {cfg}, {NR} replicas")
        w = synth.make_config(cfg, device=dev, replicas=NR)
        log("building INT2 and BF16 caches")
        cache = Int2Cache(w, device=dev, pages_per_split=None if pps < 0 else pps)
        cache.prefill()
        bf = Bf16Cache(w, device=dev, pages_per_split=None if pps < 0 else pps)
        bf.prefill()
        torch.cuda.synchronize()
        self.w, self.cache, self.bf, self.NR, self.B, self.l2 = w, cache, bf, NR, B, l2
        H, Hq, D = w.num_kv_heads, w.num_q_heads, w.head_dim
        lens_all = w.seq_lens.tolist()
        self.lens_all = lens_all
        # Current token (position L-1) of every sequence: the K/V appended by each step.
        starts = np.cumsum([0] + lens_all)[:-1]
        cur = torch.as_tensor(starts + np.array(lens_all) - 1, dtype=torch.long)
        k_cur = w.k[cur.to(dev)].contiguous()
        v_cur = w.v[cur.to(dev)].contiguous()
        s_cur = w.slot_mapping[cur].to(dev).contiguous()
        p_cur = w.tok_pos[cur].to(dev).contiguous()                  # position L - 1 of the current token
        i_cur = torch.arange(B, dtype=torch.int32, device=dev)      # sequence index inside a replica
        q = w.q.contiguous()
        out = torch.empty((w.batch, Hq, D), dtype=torch.float32, device=dev)
        out_bf = torch.empty_like(out)
        ws = cache.workspace(max(lens_all))
        ws_bf = bf.workspace()
        # A step's inputs (q, k, v, slots) sit in one staging block per replica, so the
        # end-to-end loop moves them host -> device with a single copy.
        in_sizes = [B * Hq * D * 2, B * H * D * 2, B * H * D * 2, B * 8]
        in_offs = [0]
        for sz_ in in_sizes[:-1]:
            in_offs.append((in_offs[-1] + sz_ + 255) // 256 * 256)
        per_stage = (in_offs[-1] + in_sizes[-1] + 255) // 256 * 256
        stage = torch.empty(NR * per_stage, dtype=torch.uint8, device=dev)

        def stage_view(r, idx, dtype, shape):
            base = r * per_stage + in_offs[idx]
            return stage[base:base + in_sizes[idx]].view(dtype).view(shape)

        def views(r):
            sl = slice(r * B, (r + 1) * B)
            x = dict(q=stage_view(r, 0, torch.bfloat16, (B, Hq, D)), k=stage_view(r, 1, torch.bfloat16, (B, H, D)),
                     v=stage_view(r, 2, torch.bfloat16, (B, H, D)), slots=stage_view(r, 3, torch.int64, (B,)))
            x["q"].copy_(q[sl])
            x["k"].copy_(k_cur[sl])
            x["v"].copy_(v_cur[sl])
            x["slots"].copy_(s_cur[sl])
            x.update(pos=p_cur[sl], pt=cache.page_table[sl], lens=cache.seq_lens[sl], sink=cache.sink[sl],
                     win=cache.window[sl], out=out[sl], out_bf=out_bf[sl], bpt=bf.page_table[sl],
                     blens=bf.seq_lens[sl])
            return x
        V = [views(r) for r in range(NR)]
        msl_r = [max(lens_all[r * B:(r + 1) * B]) for r in range(NR)]
        self.V, self.stage, self.per_stage, self.out = V, stage, per_stage, out

        def append_r(r):
            # the current token into the INT2 pool and its BF16 row into the window ring
            x = V[r]
            ok.oscar_append_mixed(w.dims, x["k"], x["v"], cache.R_k, cache.R_v, cache.clip_k, cache.clip_v,
                                  x["pt"], x["slots"], i_cur, x["pos"], x["lens"], w.sink_len, w.window_len,
                                  cache.int2_pages, cache.scale_zero, x["sink"], x["win"])

        def decode_r(r):
            x = V[r]
            ok.oscar_decode(w.dims, B, msl_r[r], cache.pps, x["q"], cache.R_k, cache.R_v, cache.int2_pages,
                            cache.scale_zero, x["sink"], x["win"], x["pt"], x["lens"], w.sink_len, w.window_len,
                            0.0, x["out"], ws)

        def bf16_r(r):
            x = V[r]
            ok.oscar_bf16_decode(w.dims, B, msl_r[r], bf.pps, x["q"], bf.pages, x["bpt"], x["blens"], 0.0,
                                 x["out_bf"], ws_bf)

        # one workspace per step in flight (the end-to-end loop runs up to in_flight
        # steps of different replicas at once, on as many streams)
        wss = [ws] + [cache.workspace(max(lens_all)).clone() for _ in range(min(in_flight, NR) - 1)]

        def step_r(r, slot=0):
            # one call: the current tokens appended (INT2 pool, BF16 window rows), then the decode
            x = V[r]
            ok.oscar_append_decode(w.dims, B, msl_r[r], cache.pps, x["q"], x["k"], x["v"], cache.R_k, cache.R_v,
                                   cache.clip_k, cache.clip_v, x["slots"], cache.int2_pages, cache.scale_zero,
                                   x["sink"], x["win"], x["pt"], x["lens"], w.sink_len, w.window_len, 0.0, x["out"],
                                   wss[slot])

        def step(i):
            step_r(i % NR)

        self.append_r, self.decode_r, self.bf16_r, self.step = append_r, decode_r, bf16_r, step
        self.step_r = step_r

    def bytes_decode(self):
        return algorithmic_bytes_decode(self.w, self.lens_all[:self.B])

    def bytes_step(self):
        return self.bytes_decode() + algorithmic_bytes_append(self.w, self.B, bf16_rows=True)


def extra_config_line(cfg, dev, l2, K, Wm, world, barrier) -> dict:
    """The decode step, the decode alone and the BF16 reference decode of another
    workload, timed as the main one (CUDA graphs over cache replicas larger than
    L2, CUDA events, W warm-up calls), with its own roofline."""
    import torch

    from int2_rotated_kv_append_gb300 import synth
    S = DecodeSetup(cfg, dev, l2)
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.1)
    ms_step, (t0, t1) = timed_graph(S.step, K, Wm, dev, world, barrier)
    clocks = sampler.summary(t0, t1)
    sampler.stop()
    ms_dec, _ = timed_graph(lambda i: S.decode_r(i % S.NR), K, Wm, dev, world, barrier)
    ms_bf, _ = timed_graph(lambda i: S.bf16_r(i % S.NR), K, Wm, dev, world, barrier)
    w, B = S.w, S.B
    dec_us, bf_us, step_us = ms_dec / K * 1e3, ms_bf / K * 1e3, ms_step / K * 1e3
    peak, peak_kind = measured_peak_hbm()
    nbytes = S.bytes_decode()
    achieved = nbytes / (dec_us * 1e-6) / 1e9
    lens = S.lens_all[:B]
    line = {"workload": synth.CONFIG_NAMES[cfg], "batch": B, "seq_len_min": min(lens), "seq_len_max": max(lens),
            "seq_len_mean": sum(lens) / B, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "sink": w.sink_len, "window": w.window_len, "group": w.group_size,
            "pages_per_split": "auto" if S.cache.pps == 0 else S.cache.pps,
            "l2_policy": f"inputs larger than L2: {S.NR} cache replica(s) in disjoint pages, "
                         f"{S.NR * nbytes / 1e6:.0f} MB cycled (L2 {l2 / 1e6:.0f} MB)",
            "us_per_step": step_us, "value": whole_job_gbps(world, S.bytes_step(), ms_step / K), "unit": "GB/s",
            "tokens_per_s": world * B / (step_us * 1e-6),
            "decode_us": dec_us, "bf16_decode_us": bf_us, "speedup_vs_bf16": bf_us / dec_us,
            "bf16_decode_GBps": algorithmic_bytes_bf16(w, lens) / (bf_us * 1e-6) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": MEASURED_DECODE_TRAFFIC.get(cfg), "kernel": "oscar_decode per launch",
                         "peak_source": f"{peak_kind} hbm_gbs", "bytes_per_launch": nbytes},
            "clocks": clocks}
    log(f"config {cfg}: step {step_us:.2f} us, decode {dec_us:.2f} us ({achieved / peak:.3f} of HBM), "
        f"bf16 {bf_us:.2f} us ({bf_us / dec_us:.2f}x)")
    del S
    torch.cuda.empty_cache()
    return line


def run_ours(args, world, rank, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    import int2_rotated_kv_append_gb300 as ok
    from int2_rotated_kv_append_gb300 import build as okbuild

    okbuild.build()
    ok.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    S = DecodeSetup(args.config, dev, l2, args.replicas, args.pps, in_flight=args.e2e_in_flight)
    w, cache, bf, NR, B, V = S.w, S.cache, S.bf, S.NR, S.B, S.V
    H, Hq, D = w.num_kv_heads, w.num_q_heads, w.head_dim
    lens_all = S.lens_all
    msl = max(lens_all)
    stage, per_stage, out = S.stage, S.per_stage, S.out
    append_r, decode_r, bf16_r, step, step_r = S.append_r, S.decode_r, S.bf16_r, S.step, S.step_r

    def timed(fn, n, warm):
        return timed_graph(fn, n, warm, dev, world, barrier)

    log("caches built; timing")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.1)
    K, Wm = args.steps, args.warmup
    ms, (t0, t1) = timed(step, K, Wm)
    clocks = sampler.summary(t0, t1)
    log(f"step: {ms / K * 1e3:.2f} us")
    # Decode alone and the BF16 reference decode over the same tokens.
    ms_dec, _ = timed(lambda i: decode_r(i % NR), K, Wm)
    log(f"decode: {ms_dec / K * 1e3:.2f} us")
    ms_bf, _ = timed(lambda i: bf16_r(i % NR), K, Wm)
    log(f"bf16 decode: {ms_bf / K * 1e3:.2f} us")
    ms_app, _ = timed(lambda i: append_r(i % NR), K, Wm)
    log(f"append: {ms_app / K * 1e3:.2f} us")
    # Warm L2: replica 0 decoded again and again (its cache stays in L2 when it fits).
    Kw = min(K, 2000)
    ms_warm, _ = timed(lambda i: decode_r(0), Kw, Wm)
    # Single launch: one decode issued on its own (no graph), L2 flushed before it.
    flush_buf = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    single = []
    for j in range(25):
        flush_buf.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        decode_r(j % NR)
        e1.record()
        e1.synchronize()
        single.append(e0.elapsed_time(e1) * 1e3)
    del flush_buf
    single_us = statistics.median(single[5:])
    log(f"decode warm L2: {ms_warm / Kw * 1e3:.2f} us, single launch: {single_us:.2f} us")
    sampler.stop()

    step_bytes_dec = algorithmic_bytes_decode(w, lens_all[:B])
    step_bytes_app = algorithmic_bytes_append(w, B, bf16_rows=True)
    step_bytes = step_bytes_dec + step_bytes_app
    ms_step = ms / K
    value = whole_job_gbps(world, step_bytes, ms_step)
    dec_us = ms_dec / K * 1e3
    achieved = step_bytes_dec / (dec_us * 1e-6) / 1e9
    peak, peak_kind = measured_peak_hbm()
    bf_us = ms_bf / K * 1e3

    # kernels of one oscar_append_decode: q-rotation, decode, merge; with a window the
    # decode's sink/window CTA appends the current token (the tensor-core kernels),
    # without one the append kernel runs first
    step_kernels = 3 if w.window_len >= 1 and w.head_dim == 128 else 4

    # End to end through the public API with pinned host buffers.
    # the end-to-end loop is timed by the host clock: at least 1000 steps (about 13 ms
    # at B=1) whatever K is, so that a short run still times it to within a few percent
    E = max(min(K, 2000), 1000)
    log("end-to-end loop")
    stage_h = stage.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    stream = torch.cuda.current_stream()

    # One CUDA graph per cache replica holds a whole step: the host->device copy of
    # its inputs, the oscar_append_decode call and the device->host copy of its
    # output.  NF steps are in flight, as in a serving loop with NF independent
    # batches: replica r's graph runs on stream r % NF with its own workspace, so the
    # copies, launches and kernel ramps of one step overlap the others' kernels, and
    # before launching step i the host waits until the output of step i - NF has
    # landed in host memory.  The loop launches the graphs and records and waits on
    # the events through the CUDA runtime (about 4 us of host time per launch,
    # against 12 us through torch's graph replay with a stream switch).
    NF = min(args.e2e_in_flight, NR)

    def e2e_body(r):
        sl = slice(r * B, (r + 1) * B)
        x = V[r]
        stage[r * per_stage:(r + 1) * per_stage].copy_(stage_h[r * per_stage:(r + 1) * per_stage], non_blocking=True)
        step_r(r, slot=r % NF)
        out_h[sl].copy_(x["out"], non_blocking=True)

    streams = [torch.cuda.Stream() for _ in range(NF)]
    for s_ in streams:
        s_.wait_stream(stream)
    for r in range(NR):
        with torch.cuda.stream(streams[r % NF]):
            e2e_body(r)
    for s_ in streams:
        stream.wait_stream(s_)
    torch.cuda.synchronize()
    graphs = []
    for r in range(NR):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=streams[r % NF]):
            e2e_body(r)
        graphs.append(g)
    rt = cuda_runtime()
    gexec = [ctypes.c_void_p(g.raw_cuda_graph_exec()) for g in graphs]
    sptr = [ctypes.c_void_p(s_.cuda_stream) for s_ in streams]
    done = []
    for _ in range(NF):
        ev = ctypes.c_void_p()
        if rt.cudaEventCreateWithFlags(ctypes.byref(ev), 2) != 0:  # cudaEventDisableTiming
            raise RuntimeError("cudaEventCreateWithFlags failed")
        done.append(ev)

    def e2e_run(n):
        for i in range(n):
            k = i % NF
            if i >= NF and rt.cudaEventSynchronize(done[k]) != 0:  # step i - NF's output is in host memory
                raise RuntimeError("cudaEventSynchronize failed")
            r = i % NR
            if rt.cudaGraphLaunch(gexec[r], sptr[r % NF]) != 0 or rt.cudaEventRecord(done[k], sptr[r % NF]) != 0:
                raise RuntimeError("cudaGraphLaunch / cudaEventRecord failed")
        torch.cuda.synchronize()

    e2e_run(min(50, E))
    barrier()
    te = time.perf_counter()
    e2e_run(E)
    te = time.perf_counter() - te
    e2e_ms = max_over_ranks(te / E * 1e3, world, dev)
    h2d = per_stage  # q, k, v and slots of the step in one copy (256-byte aligned parts)
    d2h = B * Hq * D * 4

    for ev in done:
        rt.cudaEventDestroy(ev)
    log(f"e2e: {e2e_ms * 1e3:.2f} us/step ({NF} steps in flight)")
    extra = {}
    for cfg in args.extra_configs:
        if cfg != args.config:
            extra[f"config{cfg}"] = extra_config_line(cfg, dev, l2, K, Wm, world, barrier)
    append_line = append_workload(dev) if rank == 0 and not args.no_append else None
    extend_line = extend_workload(dev) if rank == 0 and not args.no_extend else None
    calib_line = calibrate_workload(dev) if rank == 0 and not args.no_calibrate else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        log("cpu baseline (oracle)")
        cpu = cpu_baseline(w, cache, B, step_bytes)
        if calib_line is not None:
            calib_line["cpu_oracle"] = cpu_calibration_baseline()
            calib_line["gpu_vs_cpu_oracle"] = calib_line["cpu_oracle"]["us_per_matrix"] * 16 / calib_line["us"]

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": workload_config(args, w, B, msl, cache.pps,
                                      f"inputs larger than L2: {NR} cache replicas in disjoint pages, "
                                      f"{NR * step_bytes_dec / 1e6:.0f} MB cycled (L2 {l2 / 1e6:.0f} MB)"),
            "tokens_per_s": world * B / (ms_step * 1e-3),
            "us_per_step": ms_step * 1e3,
            "decode_us": dec_us, "append_us": ms_app / K * 1e3, "bf16_decode_us": bf_us,
            "decode_warm_l2_us": ms_warm / Kw * 1e3,
            "decode_warm_l2_note": "one replica decoded repeatedly in a CUDA graph: its cache "
                                   + ("fits" if step_bytes_dec <= l2 else "does not fit") + " in L2",
            "decode_single_launch_us": single_us,
            "decode_single_launch_note": "one decode call (three kernels) launched on its own, L2 flushed "
                                         "before it, CUDA events around it; median of 20",
            "speedup_vs_bf16": bf_us / dec_us,
            "bf16_decode_GBps": algorithmic_bytes_bf16(w, lens_all[:B]) / (bf_us * 1e-6) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": MEASURED_DECODE_TRAFFIC.get(args.config),
                         "kernel": "oscar_decode (q-rotate + split + merge) per launch",
                         "peak_source": f"{peak_kind} hbm_gbs", "bytes_per_launch": step_bytes_dec},
            "cpu_baseline": cpu,
            "e2e": {"value": whole_job_gbps(world, step_bytes, e2e_ms), "unit": "GB/s", "steps": E,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "in_flight": NF,
                    "mode": f"one CUDA graph per step (H2D inputs, oscar_append_decode, D2H output) launched by "
                            f"cudaGraphLaunch; {NF} steps in flight on {NF} streams (independent cache replicas, one "
                            f"workspace each), the host waits for step i-{NF}'s output (cudaEventSynchronize) before "
                            f"launching step i"},
            "gpu_launches": K * step_kernels,
            **extra,
            "append_workload": append_line,
            "extend_workload": extend_line,
            "calibrate_workload": calib_line,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def extend_workload(dev):
    """The extend (chunked prefill) workload: 32 sequences of 8192 cached tokens
    (the last 16 of each are the new chunk), 32 query / 8 KV heads, head_dim 128,
    group 64, sink 64, window 128; one oscar_extend_varlen over the 512 query rows.  Its
    algorithmic bytes count each sequence's cache once (rows of a sequence share
    its pages through L2) plus q in and fp32 out; the cache (168 MB) exceeds L2."""
    import torch

    from int2_rotated_kv_append_gb300 import synth
    from int2_rotated_kv_append_gb300.cache import Int2Cache

    B, L, chunk = 32, 8192, 16
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=64,
                            window_len=128, seq_lens=[L] * B, seed=11, device=dev)
    cache = Int2Cache(w, device=dev)
    cache.prefill()
    q_start = torch.arange(0, B * chunk + 1, chunk, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(3)
    q = torch.randn((B * chunk, w.num_q_heads, w.head_dim), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty((B * chunk, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)

    def run():
        cache.extend_varlen(q, q_start, chunk, out=out)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    ts = []
    for _ in range(10):
        flush.zero_()  # evict the cache from L2 between runs
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    ts.sort()
    us = ts[len(ts) // 2]
    nbytes = algorithmic_bytes_decode(w, [L] * B) - B * w.num_q_heads * w.head_dim * 6 + \
        B * chunk * w.num_q_heads * w.head_dim * 6
    peak, peak_kind = measured_peak_hbm()
    achieved = nbytes / (us * 1e-6) / 1e9
    return {"workload": f"extend: {B} sequences x {L} cached tokens, last {chunk} are new (causal query rows), "
                        "Hq 32 / Hkv 8, D 128, G 64, sink 64, window 128; L2 flushed between runs",
            "us": us, "query_tokens_per_s": B * chunk / (us * 1e-6),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "bytes_per_launch": nbytes,
                         "peak_source": f"{peak_kind} hbm_gbs"},
            "note": "oscar_extend_varlen: the INT2 pages and the BF16 sink/window rows are read once per tile of "
                    "16 query rows (GQA 4) of a sequence, on tcgen05"}


def calibrate_workload(dev):
    """The offline calibration workload: 16384 calibration vectors x 8 KV heads of
    head_dim 128 for keys (the workloads' K distribution) and values (N(0, 1)); one
    oscar_calibrate call (covariance, Jacobi eigenvectors, |x.R|, 0.999 quantile) per
    run, L2 flushed between runs.  Its bytes: the samples read twice (moments and
    rotation), |x.R| written and read once (fp32)."""
    import torch

    import int2_rotated_kv_append_gb300 as ok
    from int2_rotated_kv_append_gb300 import synth

    N, H, D = 16384, 8, 128
    k = synth.calibration_samples(N, H, D, 4, "qwen", device=dev)
    v = synth.calibration_samples(N, H, D, 5, "normal", device=dev)
    dims = ok.make_dims(H, H, D, 16, D, 1, 1)
    ws = torch.empty(ok.oscar_calibrate_workspace_bytes(dims, N), dtype=torch.uint8, device=dev)

    def outputs():
        return {"R": torch.empty(H, D, D, device=dev), "clip": torch.empty(H, D, device=dev),
                "eigenvalues": torch.empty(H, D, device=dev), "sweeps": torch.empty(H, dtype=torch.int32, device=dev)}

    out_k, out_v = outputs(), outputs()

    def run():
        ok.oscar_calibrate(dims, N, k, v, 1, 0.999, out_k, out_v, ws)

    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    ts = []
    for _ in range(10):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    ts.sort()
    us = ts[len(ts) // 2]
    nbytes = 2 * (2 * N * H * D * 2) + 2 * (2 * N * H * D * 4)
    sweeps = out_k["sweeps"].tolist() + out_v["sweeps"].tolist()
    return {"workload": f"calibration: {N} samples x {H} KV heads x D {D}, keys and values, centred covariance, "
                        "clip at the 0.999 quantile; L2 flushed between runs",
            "us": us, "matrices_per_s": 2 * H / (us * 1e-6), "samples_per_s": N / (us * 1e-6),
            "GBps_samples_and_rotated": nbytes / (us * 1e-6) / 1e9, "jacobi_sweeps": sweeps,
            "note": "one oscar_calibrate call (5 kernels) per run; the Jacobi eigensolver (about 9 sweeps x "
                    "127 rounds, 2 barriers each, 8 CTAs per matrix) takes most of it"}


def append_workload(dev):
    """The append throughput workload: a prefill append of 16384 tokens x 8 KV
    heads (K and V) into the paged INT2 cache, and a decode append of 256 tokens
    at random slots.  The prefill's dominant work is the rotation (2 * 2 * D^2 flop
    per token and head, K and V) on tensor cores: its roofline is the measured
    dense bf16 tensor rate.  The kernel executes three bf16 products per rotation
    (R split into hi + mid + lo), reported beside it."""
    import torch

    import int2_rotated_kv_append_gb300 as ok
    from int2_rotated_kv_append_gb300 import synth
    from int2_rotated_kv_append_gb300.cache import Int2Cache

    w = synth.make_config(4, device=dev)
    cache = Int2Cache(w, device=dev)
    # two copies of the prefill's K/V (134 MB together, more than L2), used in turn
    kv_sets = [(w.k.contiguous(), w.v.contiguous()), (w.k.clone(), w.v.clone())]
    k, v = kv_sets[0]
    slots = w.slot_mapping.to(dev).contiguous()
    kd, vd, sd = synth.decode_append_batch(w, 256, device=dev)
    sd = sd.to(dev)
    turn = [0]

    def prefill():
        kk, vv = kv_sets[turn[0] % 2]
        turn[0] += 1
        ok.oscar_append(w.dims, kk, vv, cache.R_k, cache.R_v, cache.clip_k, cache.clip_v, cache.page_table, slots,
                        cache.int2_pages, cache.scale_zero)

    def dec_append():
        ok.oscar_append(w.dims, kd, vd, cache.R_k, cache.R_v, cache.clip_k, cache.clip_v, cache.page_table, sd,
                        cache.int2_pages, cache.scale_zero)

    # the same appends with a key offset (per-channel key means, fp32 [Hkv][D])
    off = w.k.to(torch.float32).mean(dim=0).contiguous()

    def prefill_off():
        kk, vv = kv_sets[turn[0] % 2]
        turn[0] += 1
        ok.oscar_append(w.dims, kk, vv, cache.R_k, cache.R_v, cache.clip_k, cache.clip_v, cache.page_table, slots,
                        cache.int2_pages, cache.scale_zero, offset_k=off)

    def dec_append_off():
        ok.oscar_append(w.dims, kd, vd, cache.R_k, cache.R_v, cache.clip_k, cache.clip_v, cache.page_table, sd,
                        cache.int2_pages, cache.scale_zero, offset_k=off)

    def time_it(fn, n):
        # n calls captured in one CUDA graph (the host's launch cost is not timed, as
        # in the decode measurements), CUDA events around a replay
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) / n * 1e3

    pre_us = time_it(prefill, 20)
    dec_us = time_it(dec_append, 200)
    pre_off_us = time_it(prefill_off, 20)
    dec_off_us = time_it(dec_append_off, 200)
    T, H, D = w.num_tokens, w.num_kv_heads, w.head_dim
    flops = 2 * T * H * 2 * D * D  # K and V: 2 D^2 flop each per token and head
    bf16_peak, bf16_src = measured_peak_bf16()
    achieved = flops / (pre_us * 1e-6) / 1e12
    return {"workload": "prefill append 16384 tokens x 8 KV heads (K and V), head_dim 128, group 64; "
                        "decode append of 256 tokens at random slots",
            "prefill_us": pre_us, "prefill_tokens_per_s": T / (pre_us * 1e-6),
            "prefill_GBps": algorithmic_bytes_append(w, T) / (pre_us * 1e-6) / 1e9,
            "prefill_roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                                 "frac": achieved / bf16_peak, "peak_source": bf16_src + " bf16_tflops (burst)",
                                 "executed_tflops": 3 * achieved,
                                 "note": "tcgen05 bf16 MMAs with R as three bf16 terms: 3x the algorithmic flops"},
            "decode_append_256_us": dec_us,
            "key_offset": {"prefill_us": pre_off_us, "decode_append_256_us": dec_off_us,
                           "note": "the same appends with a per-(KV head, channel) key offset subtracted"},
            "note": "calls captured in a CUDA graph; the prefill alternates between two copies of its K/V "
                    "(134 MB, more than L2); the decode append's 256 tokens stay in L2"}


def cpu_baseline(w, cache, B, step_bytes):
    """The oracle, as it stands, on one full step of replica 0 (append + decode),
    repeated up to ~10 s; one thread per (sequence, query head)."""
    import concurrent.futures

    import numpy as np
    import torch

    from int2_rotated_kv_append_gb300.synth import bits16
    from oracle import oracle as O

    O.build_oracle()
    codes = cache.int2_pages.cpu().numpy()
    sz = cache.scale_zero.view(torch.int16).cpu().numpy().view(np.uint16)
    sinkb, winb = bits16(cache.sink), bits16(cache.window)
    qb = bits16(w.q)
    Rk, Rv, ck, cv = (t.cpu().numpy() for t in (w.R_k, w.R_v, w.clip_k, w.clip_v))
    pt, lens = w.page_table.numpy(), w.seq_lens.numpy()
    lens_all = lens.tolist()
    starts = np.cumsum([0] + lens_all)[:-1]
    cur = starts[:B] + np.array(lens_all[:B]) - 1
    kb, vb = bits16(w.k[torch.as_tensor(cur, device=w.k.device)]), bits16(w.v[torch.as_tensor(cur, device=w.k.device)])
    slots = w.slot_mapping.numpy()[cur]
    pairs = [(b, h) for b in range(B) for h in range(w.num_q_heads)]
    threads = max(1, min(os.cpu_count() or 1, len(pairs)))

    def one_step():
        O.append(w.dims, kb, vb, Rk, Rv, ck, cv, slots, codes, sz)
        with concurrent.futures.ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda pr: O.decode(w.dims, w.batch, qb, Rk, Rv, codes, sz, sinkb, winb, pt, lens,
                                            w.sink_len, w.window_len, 0.0, pairs=[pr]), pairs))
    n, t = 0, time.perf_counter()
    while True:
        one_step()
        n += 1
        el = time.perf_counter() - t
        if el > 10.0 or n >= 20:
            break
    return {"value": step_bytes * n / el / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(), "host_cores": os.cpu_count(),
            "sample": f"{n} full step(s) of one replica (append of {B} token(s) + decode of {len(pairs)} "
                      f"(sequence, query head) pairs), fp64 oracle, {threads} threads",
            "s_per_step": el / n}


def cpu_calibration_baseline():
    """The calibration oracle, as it stands (fp64 numpy), on one matrix of the
    calibration workload (16384 key samples of one KV head, D 128), repeated up to ~5 s."""
    import numpy as np

    from int2_rotated_kv_append_gb300 import synth
    from int2_rotated_kv_append_gb300.synth import bits16
    from oracle import calibration as CAL

    x = bits16(synth.calibration_samples(16384, 8, 128, 4, "qwen", device="cpu"))[:, :1, :]
    x = np.ascontiguousarray(x)
    n, t = 0, time.perf_counter()
    while True:
        CAL.calibrate(x, centered=True, q=0.999)
        n += 1
        el = time.perf_counter() - t
        if el > 5.0 or n >= 20:
            break
    return {"us_per_matrix": el / n * 1e6, "kind": "oracle", "cores": os.cpu_count(),
            "sample": f"{n} run(s) of one matrix (16384 samples x D 128), numpy fp64 (BLAS threads as installed)"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, choices=[1, 2, 3],
                    help="workload: 1 batch-1 32K (default), 2 batch-64 mixed lengths, 3 batch-4 131K")
    ap.add_argument("--replicas", type=int, default=0, help="cache replicas (0: enough to exceed 3x L2)")
    ap.add_argument("--pps", type=int, default=-1, help="pages per split for both decodes (-1: the workload's, 0: auto)")
    ap.add_argument("--extra-configs", default="2,3",
                    help="comma-separated workloads (2, 3) measured after the main one and reported under "
                         "config2 / config3 of the same line ('' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-append", action="store_true", help="skip the append throughput workload")
    ap.add_argument("--no-extend", action="store_true", help="skip the extend (chunked prefill) workload")
    ap.add_argument("--no-calibrate", action="store_true", help="skip the offline calibration workload")
    ap.add_argument("--e2e-in-flight", type=int, default=E2E_IN_FLIGHT,
                    help="independent steps in flight in the end-to-end loop (one stream and workspace each)")
    args = ap.parse_args()
    args.extra_configs = [int(c) for c in args.extra_configs.split(",") if c.strip()]
    if any(c not in (1, 2, 3) for c in args.extra_configs):
        ap.error("--extra-configs takes workloads 1, 2, 3")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.e2e_in_flight < 1:
        ap.error("--e2e-in-flight must be >= 1")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
