"""R-SWA benchmark on one GB300 (replicas on N GPUs under torchrun).

Headline workload (single page, bf16): B 1, H 10, d 128, prefix m 288 (256
visual tokens + 32 prompt), window n 128, T 6000 output tokens.  One step is
the whole hot path over that input: the prefix prefill (cache write +
attention over the 288 prefix rows) followed by 6000 fused append+decode
steps through the ring cache.  Value: output tokens/s.

The JSON line also carries one roofline entry per bound kernel and workload
(the metric's decode GB/s and prefill TFLOP/s):
  decode_sweep     B 32, m 2600, T in 256 .. 100000: flat per-step latency
  batched_decode   B 64, m_b ~ U{256..2048}, ring full (T 4096), one step
  prefill          B 1, m 10272, T 22496 (32K rows), 12 independent layers
  long_prefix      B 1, m 10272 (40 pages), one step through 12 layers
  batched GQA      B 64, 32 query heads over 8 KV heads
and the per-step latency of the single-page decode loop at every t, for
R-SWA and for the standard full cache (n = T).  Everything else measured
goes to the file named by --extras-out.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W]
                       [--impl ours|reference] [--no-extras]
                       [--extras-out PATH]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("R-SWA decode HBM GB/s & tokens/s vs T; prefill TFLOP/s "
          "(fraction of GB300 peak)")
L2_FLUSH_BYTES = 256 << 20          # > 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "decode_kernel": ["decode.cu", "attend.cuh", "rswa_device.cuh", "tc_ptx.cuh"],
    "decode_cluster_kernel": ["decode.cu", "attend.cuh", "rswa_device.cuh",
                              "tc_ptx.cuh"],
    "decode_gqa_tc_kernel": ["decode_gqa_tc.cu", "tc_ptx.cuh", "rswa_device.cuh"],
    "decode_gqa_sk_kernel": ["decode_gqa_sk.cu", "tc_ptx.cuh", "rswa_device.cuh"],
    "decode_stream_kernel": ["decode_stream.cu", "attend.cuh", "rswa_device.cuh",
                             "tc_ptx.cuh"],
    "block_tc_kernel": ["block_tc.cu", "tc_ptx.cuh", "rswa_device.cuh"],
    "prefill_tc_kernel": ["prefill_tc.cu", "tc_ptx.cuh", "rswa_device.cuh"],
}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p.get(k, FALLBACK_PEAKS[k])) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha(name):
    """Hash of the sources a kernel is built from ("kernel@workload" keys
    hash the kernel's)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sliding_window_attention_02_gb300", "csrc")
    for f in KERNEL_SOURCES.get(name.split("@")[0], []):
        p = os.path.join(csrc, f)
        if os.path.exists(p):
            with open(p, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's
    sources are unchanged since it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(name)
    if not rec or rec.get("source_sha") != kernel_sha(name):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle sampling during a timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[3:7]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads (setup shared with the full-size GPU tests)
# ---------------------------------------------------------------------------

def setup_single_page(dev, seed=0, n=None):
    """Cache and inputs of the single-page workload, plus CUDA graphs for the
    prefix prefill and the 6000-step fused decode loop.  `n` overrides the
    window (n >= T gives the standard full-cache MHA baseline)."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    w = workloads.WORKLOADS["single_page_bf16"]
    B, H, d, m, T = w.batch, w.heads, w.head_dim, w.m, w.T
    n = w.n if n is None else n
    Q, K, V = workloads.qkv(m + T, H, d, seed, w.std, torch.bfloat16, device=dev)
    cache = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16, device=dev)
    Op = torch.empty(m, H, d, dtype=torch.bfloat16, device=dev)
    Od = torch.empty(T, B, H, d, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(device=dev)
    st = {"w": w, "n": n, "Q": Q, "K": K, "V": V, "cache": cache, "Op": Op,
          "Od": Od, "stream": s}

    def prefill():
        cache.prefill(Q[:m], K[:m], V[:m], Op, [m], 0, stream=s)

    def decode_loop():
        for t in range(T):
            cache.decode_step_fused(Q[m + t][None], K[m + t][None],
                                    V[m + t][None], Od[t], stream=s)

    st["prefill"], st["decode_loop"] = prefill, decode_loop
    with torch.cuda.stream(s):
        prefill()
        decode_loop()          # eager run before capture
    torch.cuda.synchronize(dev)
    g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=s):
        prefill()
    with torch.cuda.graph(g2, stream=s):
        decode_loop()
    st["g_prefill"], st["g_decode"] = g1, g2
    return st


def single_page_bytes_per_decode(w):
    """Algorithmic bytes of one fused decode launch, averaged over the loop:
    K and V of the m + min(n, t + 1) attended keys for every head, plus q, k,
    v read and o written."""
    B, H, d, m, n, T = w.batch, w.heads, w.head_dim, w.m, w.n, w.T
    keys = sum(m + min(n, t + 1) for t in range(T)) / T
    return B * H * d * 2 * (2 * keys + 4)


def setup_batched(dev, seed=0):
    """64 sequences with ragged prefixes and a full ring (T = 4096)."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    w = workloads.WORKLOADS["batched_decode_bf16"]
    B, H, d, n, T = w.batch, w.heads, w.head_dim, w.n, w.T
    m_list = workloads.prefix_lengths(B, *w.m_range, seed=seed)
    rows = sum(m + T for m in m_list)
    _, K, V = workloads.qkv(rows, H, d, seed, 1.0, torch.bfloat16, device=dev)
    cache = rswa.RswaCache(w.m_range[1], n, H, d, B, rswa.RSWA_BF16, device=dev)
    cache.prefill(None, K, V, None, m_list, T)
    steps = workloads.qkv(64 * B, H, d, seed + 1000, 1.0, torch.bfloat16,
                          device=dev)
    return {"w": w, "cache": cache, "m_list": m_list, "K": K, "V": V,
            "steps": steps}


def setup_batched_gqa(dev, seed=0):
    """The batched-decode shape with 32 query heads over 8 KV heads."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    w = workloads.WORKLOADS["batched_decode_bf16"]
    B, d, n, T = w.batch, w.head_dim, w.n, w.T
    H, Hkv = 32, 8
    m_list = workloads.prefix_lengths(B, *w.m_range, seed=seed)
    rows = sum(m + T for m in m_list)
    K = workloads.normal((rows, Hkv, d), 3 * seed + 1, 1.0, torch.bfloat16, dev)
    V = workloads.normal((rows, Hkv, d), 3 * seed + 2, 1.0, torch.bfloat16, dev)
    cache = rswa.RswaCache(w.m_range[1], n, H, d, B, rswa.RSWA_BF16, device=dev,
                           kv_heads=Hkv)
    cache.prefill(None, K, V, None, m_list, T)
    q = workloads.normal((16 * B, H, d), 5000, 1.0, torch.bfloat16, dev)
    k = workloads.normal((16 * B, Hkv, d), 5001, 1.0, torch.bfloat16, dev)
    v = workloads.normal((16 * B, Hkv, d), 5002, 1.0, torch.bfloat16, dev)
    return {"w": w, "H": H, "Hkv": Hkv, "cache": cache, "m_list": m_list,
            "K": K, "V": V, "steps": (q, k, v)}


def batched_step_bytes(m_list, w):
    B, H, d, n = w.batch, w.heads, w.head_dim, w.n
    keys = sum(m + n for m in m_list)
    return H * d * 2 * (2 * keys + 4 * B)


def setup_sweep(dev, seed=0):
    """32 sequences, m 2600; ring filled by a prefill of n outputs; t_b is
    then restored to each swept T (rswa_cache_set_t)."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    w = workloads.WORKLOADS["decode_sweep_bf16"]
    B, H, d, m, n = w.batch, w.heads, w.head_dim, w.m, w.n
    _, K, V = workloads.qkv(B * (m + n), H, d, seed, 1.0, torch.bfloat16,
                            device=dev)
    cache = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16, device=dev)
    cache.prefill(None, K, V, None, [m] * B, n)
    steps = workloads.qkv(64 * B, H, d, seed + 2000, 1.0, torch.bfloat16,
                          device=dev)
    return {"w": w, "cache": cache, "K": K, "V": V, "steps": steps}


def setup_prefill(dev, layers=None, seed0=0):
    """Multi-page prefill: 12 layers with independent seeded Q/K/V."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    w = workloads.WORKLOADS["multipage_prefill_bf16"]
    B, H, d, m, n, T = w.batch, w.heads, w.head_dim, w.m, w.n, w.T
    layers = w.layers if layers is None else layers
    L = m + T
    qkv = [workloads.qkv(L, H, d, seed0 + i, 1.0, torch.bfloat16, device=dev)
           for i in range(layers)]
    caches = [rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16, device=dev)
              for _ in range(layers)]
    outs = [torch.empty(L, H, d, dtype=torch.bfloat16, device=dev)
            for _ in range(layers)]
    return {"w": w, "qkv": qkv, "caches": caches, "outs": outs}


def prefill_flops(w):
    """4 * d * |visible pairs| * H: QK^T and PV over the R-SWA mask only."""
    m, n, T, H, d = w.m, w.n, w.T, w.heads, w.head_dim
    pairs = m * (m + 1) // 2 + T * m + sum(min(n, t + 1) for t in range(T))
    return 4 * d * pairs * H * w.batch


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------

def events_time(fn, stream, iters, flush=None):
    """Mean ms of fn() over iters, CUDA events on `stream`, optional L2 flush
    between iterations (outside the timed events)."""
    import torch
    times = []
    for _ in range(iters):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            fn()
            e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return times


GRAPH_STEPS = 16


def run_long_prefix_decode(dev, peaks, layers=12):
    """B 1, H 10, d 128, n 128: one fused decode step through every layer's
    cache (12 layers, as a multi-page model decodes after its prefill) for
    prefixes of 4, 16 and 40 pages.  The 12 caches (up to 0.64 GB) do not
    stay in L2, so each step reads them from HBM."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    H, d, n = 10, 128, 128
    s = torch.cuda.Stream(device=dev)
    steps = workloads.qkv(16, H, d, 5, 1.0, torch.bfloat16, device=dev)
    o = torch.empty(1, H, d, dtype=torch.bfloat16, device=dev)
    rows = []
    for m in (1056, 4128, 10272):
        caches = []
        for layer in range(layers):
            _, K, V = workloads.qkv(m + n, H, d, layer, 1.0, torch.bfloat16,
                                    device=dev)
            c = rswa.RswaCache(m, n, H, d, 1, rswa.RSWA_BF16, device=dev)
            c.prefill(None, K, V, None, [m], n, stream=s)
            caches.append(c)
            del K, V
        idx = [0]

        def step():
            i = idx[0] % 16
            idx[0] += 1
            for c in caches:
                c.decode_step_fused(steps[0][i][None], steps[1][i][None],
                                    steps[2][i][None], o, stream=s)
        ms = graph_step_ms(step, s, 16, 5)
        per_layer = H * d * 2 * (2 * (m + n) + 4)
        nbytes = layers * per_layer
        gbs = nbytes / (ms * 1e-3) / 1e9
        rows.append({"m": m, "us_per_layer": round(ms * 1e3 / layers, 3),
                     "bytes_per_layer": per_layer, "GB_per_s": round(gbs, 1),
                     "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)})
        del caches
        torch.cuda.empty_cache()
    return {"kernel": "decode_stream_kernel",
            "workload": "B1 H10 d128 n128 bf16 fused decode through %d layers' "
                        "caches, prefix of 4/16/40 pages (%.2f GB per step at "
                        "40 pages, from HBM)" % (
                            layers, layers * 10 * 128 * 2 * 2 * (10272 + 128) / 1e9),
            "points": rows}


def run_block_decode(dev, peaks, blocks=(1, 4, 16, 64, 256, 1024), reps=16):
    """Multi-query decode (rswa_decode_block) on the single-page cache: one
    call decodes and appends `block` consecutive tokens per sequence (the
    shape of verifying drafted tokens; past n = 128, chunked prefill of
    output text into the cache).  Per call latency and tokens/s."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    w = workloads.WORKLOADS["single_page_bf16"]
    B, H, d, m, n = w.batch, w.heads, w.head_dim, w.m, w.n
    s = torch.cuda.Stream(device=dev)
    rows = []
    for k in blocks:
        Q, K, V = workloads.qkv(m + reps * k, H, d, 0, w.std, torch.bfloat16,
                                device=dev)
        c = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16, device=dev)
        c.prefill(None, K[:m], V[:m], None, [m], 0, stream=s)
        o = torch.empty(B, k, H, d, dtype=torch.bfloat16, device=dev)
        blk = [tuple(x[m + i * k:m + (i + 1) * k][None].contiguous()
                     for x in (Q, K, V)) for i in range(reps)]
        idx = [0]

        def step():
            q, kk, vv = blk[idx[0] % reps]
            idx[0] += 1
            c.decode_block(q, kk, vv, o, stream=s)
        ms = graph_step_ms(step, s, reps, 5)
        rows.append({"block": k, "us_per_call": round(ms * 1e3, 2),
                     "tokens_per_s": round(B * k / (ms * 1e-3), 1)})
        del c, Q, K, V
    return {"workload": "B1 H10 d128 m288 n128 bf16 (single-page cache), "
                        "rswa_decode_block with blocks of %s tokens"
                        % "/".join(str(b) for b in blocks),
            "points": rows}


def run_vanilla_swa(dev, peaks, layers=3):
    """Vanilla SWA (m = 0: the window slides over every token): a 32K-row
    prefill (band tiles only) and a batched fused decode step with a full
    ring, through the same kernels."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    H, d, n, L = 10, 128, 128, 32768
    s = torch.cuda.Stream(device=dev)
    pairs = sum(min(n, i + 1) for i in range(L))
    qkv = [workloads.qkv(L, H, d, 100 + l, 1.0, torch.bfloat16, device=dev)
           for l in range(layers)]
    caches = [rswa.RswaCache(0, n, H, d, 1, rswa.RSWA_BF16, device=dev)
              for _ in range(layers)]
    outs = [torch.empty(L, H, d, dtype=torch.bfloat16, device=dev)
            for _ in range(layers)]

    def pstep():
        for (Q, K, V), c, O in zip(qkv, caches, outs):
            c.prefill(Q, K, V, O, [0], L, stream=s)
    with torch.cuda.stream(s):
        pstep()
    ms = statistics.mean(events_time(pstep, s, 3)) / layers
    tf = 4 * d * pairs * H / (ms * 1e-3) / 1e12
    pre = {"rows": L, "ms_per_layer": round(ms, 4), "visible_pairs_per_head": pairs,
           "TFLOP_per_s": round(tf, 1),
           "frac_bf16_sustained": round(tf / peaks["bf16_tflops_sustained"], 4)}
    del qkv, caches, outs
    torch.cuda.empty_cache()
    # 256 sequences: 170 MB of window per step, more than L2 holds.  The
    # ring is filled by a prefill of n outputs, then t_b is set to 4096.
    B, T = 256, 4096
    _, K, V = workloads.qkv(B * n, H, d, 7, 1.0, torch.bfloat16, device=dev)
    c = rswa.RswaCache(0, n, H, d, B, rswa.RSWA_BF16, device=dev)
    c.prefill(None, K, V, None, [0] * B, n, stream=s)
    torch.cuda.synchronize()
    c.set_t([T] * B)
    steps = workloads.qkv(16 * B, H, d, 8, 1.0, torch.bfloat16, device=dev)
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    idx = [0]

    def dstep():
        i = idx[0] % 16
        idx[0] += 1
        c.decode_step_fused(steps[0][i * B:(i + 1) * B], steps[1][i * B:(i + 1) * B],
                            steps[2][i * B:(i + 1) * B], o, stream=s)
    ms = graph_step_ms(dstep, s, 16, 5)
    nbytes = B * H * d * 2 * (2 * n + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    dec = {"batch": B, "us_per_step": round(ms * 1e3, 2), "GB_per_s": round(gbs, 1),
           "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    return {"workload": "vanilla SWA, m = 0, n = 128, H10 d128 bf16: prefill of "
                        "32768 rows (%d layers) and a B256 fused decode step "
                        "with a full ring (t_b 4096)" % layers,
            "prefill": pre, "decode": dec}


def run_mha_baseline(dev, quick=False):
    """R-SWA (n = 128) against the standard full cache (n = T = 6000, i.e.
    every output stays visible: plain causal attention) on the single-page
    shape, through the same kernels.  Per-step decode latency at several t,
    the live cache size at each t, and the whole 6000-step decode loop."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    w = workloads.WORKLOADS["single_page_bf16"]
    B, H, d, m, T = w.batch, w.heads, w.head_dim, w.m, w.T
    s = torch.cuda.Stream(device=dev)
    Q, K, V = workloads.qkv(m + T, H, d, 0, w.std, torch.bfloat16, device=dev)
    steps = workloads.qkv(16, H, d, 77, w.std, torch.bfloat16, device=dev)
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    points = []
    caches = {}
    for name, n in (("rswa", w.n), ("mha", T)):
        c = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16, device=dev)
        c.prefill(None, K, V, None, [m], T, stream=s)   # all 6000 outputs
        caches[name] = c
    for t in ((512, 2048, 5984) if quick else (128, 512, 1024, 2048, 4096, 5984)):
        row = {"t": t}
        for name, c in caches.items():
            c.set_t([t], stream=s)
            idx = [0]

            def step():
                i = idx[0] % 16
                idx[0] += 1
                c.decode_step_fused(steps[0][i][None], steps[1][i][None],
                                    steps[2][i][None], o, stream=s)
            row[name + "_us"] = round(1e3 * graph_step_ms(step, s, 16, 3), 3)
            c.set_t([t], stream=s)
            row[name + "_cache_bytes"] = c.cache_bytes(0)
        points.append(row)
    del caches
    loops = {}
    for name, n in (("rswa", w.n), ("mha", T)):
        sp = setup_single_page(dev, n=n)
        with torch.cuda.stream(sp["stream"]):
            sp["g_prefill"].replay()
        ts = events_time(lambda: sp["g_decode"].replay(), sp["stream"],
                         1 if quick else 3)
        loops[name] = T / (statistics.mean(ts) * 1e-3)
        del sp
    return {"workload": "B1 H10 d128 m288 bf16 decode: R-SWA n=128 vs full "
                        "cache n=6000 (standard MHA), same kernels",
            "points": points,
            "loop_tokens_per_s": {k: round(v, 1) for k, v in loops.items()},
            "loop_speedup": round(loops["rswa"] / loops["mha"], 3)}


def graph_step_ms(step, stream, nsteps, iters):
    """Mean ms per step: `nsteps` steps captured in one CUDA graph, replayed
    `iters` times (after 2 warm-up replays), timed with events on `stream`.
    Inputs of these workloads exceed L2, so no flush is needed."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(nsteps):
            step()
    with torch.cuda.stream(stream):
        for _ in range(2):
            g.replay()
    ts = events_time(lambda: g.replay(), stream, iters)
    return statistics.mean(ts) / nsteps


def per_step_profile(dev, n=None):
    """Device time of every decode step of the single-page loop: a CUDA
    graph of the prefix prefill and the T fused steps with a timing event
    recorded between consecutive steps (event nodes in the graph).  The
    event between two steps keeps the next step from starting before the
    previous one ends, so each figure is the step's whole latency, without
    the overlap of the back-to-back loop.  Returns per-step microseconds."""
    import torch
    import sliding_window_attention_02_gb300 as rswa
    import workloads
    w = workloads.WORKLOADS["single_page_bf16"]
    B, H, d, m, T = w.batch, w.heads, w.head_dim, w.m, w.T
    n = w.n if n is None else n
    Q, K, V = workloads.qkv(m + T, H, d, 0, w.std, torch.bfloat16, device=dev)
    cache = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16, device=dev)
    Op = torch.empty(m, H, d, dtype=torch.bfloat16, device=dev)
    Od = torch.empty(T, B, H, d, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(device=dev)
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(T + 1)]

    def body(record):
        cache.prefill(Q[:m], K[:m], V[:m], Op, [m], 0, stream=s)
        for t in range(T):
            if record:
                ev[t].record(s)
            cache.decode_step_fused(Q[m + t][None], K[m + t][None],
                                    V[m + t][None], Od[t], stream=s)
        if record:
            ev[T].record(s)
    with torch.cuda.stream(s):
        body(False)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        body(True)
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    torch.cuda.synchronize(dev)
    us = [1e3 * ev[t].elapsed_time(ev[t + 1]) for t in range(T)]
    del g, cache
    return us


def step_stats(us):
    """p50 / p99 / max / min / mean of a list of per-step microseconds."""
    xs = sorted(us)
    q = lambda f: xs[min(len(xs) - 1, int(round(f * (len(xs) - 1))))]
    return {"p50": round(q(0.5), 3), "p99": round(q(0.99), 3),
            "max": round(xs[-1], 3), "min": round(xs[0], 3),
            "mean": round(statistics.mean(xs), 3)}


def step_growth(us, warm=128):
    """Least-squares slope (ns per output token) of per-step latency over
    t >= warm, and the latency ratio of the last 512 steps to steps
    warm .. warm + 511."""
    ts = list(range(warm, len(us)))
    ys = us[warm:]
    mt, my = statistics.mean(ts), statistics.mean(ys)
    var = sum((t - mt) ** 2 for t in ts)
    slope = sum((t - mt) * (y - my) for t, y in zip(ts, ys)) / var
    ratio = statistics.mean(us[-512:]) / statistics.mean(us[warm:warm + 512])
    return {"slope_ns_per_token": round(1e3 * slope, 4),
            "late_to_early": round(ratio, 4)}


def boundary_jumps(us, periods=(64, 128, 256), span=8, skip=128):
    """Latency step at t = multiples of each period (mean of the `span`
    steps from t minus the mean of the `span` steps before t), against the
    same statistic at every other t: shows whether per-step latency jumps
    when the number of cached keys crosses an alignment boundary."""
    def jump(t):
        return statistics.mean(us[t:t + span]) - statistics.mean(us[t - span:t])
    ts = range(max(skip, span), len(us) - span)
    every = [jump(t) for t in ts]
    out = {"all_t_mean_us": round(statistics.mean(every), 4),
           "all_t_p99_us": round(sorted(every)[int(0.99 * (len(every) - 1))], 4)}
    for p in periods:
        at = [jump(t) for t in ts if t % p == 0]
        out[f"at_{p}_mean_us"] = round(statistics.mean(at), 4)
        out[f"at_{p}_max_us"] = round(max(at), 4)
    return out


def run_extras(dev, peaks, quick=False):
    import torch
    out = {}
    s = torch.cuda.Stream(device=dev)
    # batched decode --------------------------------------------------------
    bt = setup_batched(dev)
    w = bt["w"]
    B, H, d = w.batch, w.heads, w.head_dim
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    q, k, v = bt["steps"]
    idx = [0]

    def bstep():
        i = idx[0] % 64
        idx[0] += 1
        bt["cache"].decode_step_fused(q[i * B:(i + 1) * B], k[i * B:(i + 1) * B],
                                      v[i * B:(i + 1) * B], o, stream=s)
    ms = graph_step_ms(bstep, s, GRAPH_STEPS, 3 if quick else 10)
    nbytes = batched_step_bytes(bt["m_list"], w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["batched_decode"] = {
        "workload": "B64 H10 d128 m~U{256..2048} n128 T4096 bf16, one fused step",
        "us_per_step": round(ms * 1e3, 2), "tokens_per_s": round(B / (ms * 1e-3), 1),
        "algorithmic_bytes": nbytes, "GB_per_s": round(gbs, 1),
        "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
        "l2": "inputs (%.2f GB) larger than L2" % (nbytes / 1e9),
        "timing": "%d fused steps per CUDA graph, events around replays" % GRAPH_STEPS}
    del bt
    # batched decode with grouped heads (32 query / 8 KV heads) ------------
    gq = setup_batched_gqa(dev)
    H, Hkv = gq["H"], gq["Hkv"]
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    q, k, v = gq["steps"]
    idx = [0]

    def gstep():
        i = idx[0] % 16
        idx[0] += 1
        gq["cache"].decode_step_fused(q[i * B:(i + 1) * B], k[i * B:(i + 1) * B],
                                      v[i * B:(i + 1) * B], o, stream=s)
    ms = graph_step_ms(gstep, s, GRAPH_STEPS, 3 if quick else 10)
    # each KV head is read once per step; q, o per query head
    nbytes = d * 2 * (2 * Hkv * sum(m + w.n for m in gq["m_list"]) +
                      2 * B * H + 2 * B * Hkv)
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["batched_decode_gqa"] = {
        "workload": "B64 H32 (8 KV heads) d128 m~U{256..2048} n128 T4096 bf16, "
                    "one fused step",
        "us_per_step": round(ms * 1e3, 2), "algorithmic_bytes": nbytes,
        "GB_per_s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    del gq
    # decode sweep ----------------------------------------------------------
    sw = setup_sweep(dev)
    w = sw["w"]
    B, H, d, m, n = w.batch, w.heads, w.head_dim, w.m, w.n
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    q, k, v = sw["steps"]
    rows = []
    nbytes = H * d * 2 * (2 * B * (m + n) + 4 * B)
    for T in w.T_sweep:
        sw["cache"].set_t([T] * B)
        idx = [0]

        def sstep():
            i = idx[0] % 64
            idx[0] += 1
            sw["cache"].decode_step_fused(q[i * B:(i + 1) * B], k[i * B:(i + 1) * B],
                                          v[i * B:(i + 1) * B], o, stream=s)
        ms = graph_step_ms(sstep, s, GRAPH_STEPS, 3 if quick else 6)
        gbs = nbytes / (ms * 1e-3) / 1e9
        rows.append({"T": T, "us_per_step": round(ms * 1e3, 2),
                     "GB_per_s": round(gbs, 1),
                     "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)})
    us = [r["us_per_step"] for r in rows]
    out["decode_sweep"] = {
        "workload": "B32 H10 d128 m2600 n128 bf16, T set by rswa_cache_set_t",
        "algorithmic_bytes": nbytes, "points": rows,
        "latency_spread": round((max(us) - min(us)) / statistics.mean(us), 4)}
    del sw
    # one sequence decoding over a long prefix (after a multi-page prefill) --
    out["long_prefix_decode"] = run_long_prefix_decode(dev, peaks)
    torch.cuda.empty_cache()
    out["block_decode"] = run_block_decode(dev, peaks)
    torch.cuda.empty_cache()
    out["vanilla_swa"] = run_vanilla_swa(dev, peaks)
    torch.cuda.empty_cache()
    # standard-MHA baseline (the pages' comparison) -------------------------
    out["mha_baseline"] = run_mha_baseline(dev, quick)
    torch.cuda.empty_cache()
    # multi-page prefill ----------------------------------------------------
    pf = setup_prefill(dev, layers=2 if quick else None)
    w = pf["w"]
    layers = len(pf["caches"])

    def pstep():
        for (Q, K, V), c, O in zip(pf["qkv"], pf["caches"], pf["outs"]):
            c.prefill(Q, K, V, O, [w.m], w.T, stream=s)
    with torch.cuda.stream(s):
        pstep()
    ts = events_time(pstep, s, 2 if quick else 3)
    ms = statistics.mean(ts)
    flops = prefill_flops(w) * layers
    tf = flops / (ms * 1e-3) / 1e12
    out["prefill"] = {
        "workload": "B1 H10 d128 m10272 T22496 (32K) n128 bf16, %d layers" % layers,
        "ms_per_step": round(ms, 3), "layers": layers, "algorithmic_flops": flops,
        "TFLOP_per_s": round(tf, 1),
        "frac_bf16_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
        "frac_bf16_burst": round(tf / peaks["bf16_tflops"], 4)}
    return out


# ---------------------------------------------------------------------------
# CPU oracle timing (runs in a subprocess pinned to one thread)
# ---------------------------------------------------------------------------

def oracle_single_page_sample(budget_s, max_steps=None):
    """Oracle time of the single-page workload: the 288-row prefix prefill,
    then the decode steps in order (t = 0, 1, ...) until all T are done or
    `budget_s` seconds (or max_steps) have passed.  When the budget ends the
    loop early, the remaining steps are costed at the mean of the steady
    steps timed (t >= n: every step attends m + n keys, as all later steps
    do)."""
    import numpy as np
    import torch
    import oracle
    import workloads
    w = workloads.WORKLOADS["single_page_bf16"]
    H, d, m, n, T = w.heads, w.head_dim, w.m, w.n, w.T
    Q, K, V = workloads.qkv(m + T, H, d, 0, w.std, torch.bfloat16)
    Q, K, V = (x.double().numpy() for x in (Q, K, V))
    t0 = time.perf_counter()
    oracle.prefill_attention(Q[:m], K[:m], V[:m], m, n)
    state = oracle.prefill_cache(K[:m], V[:m], m, n, 0)
    t1 = time.perf_counter()
    steps, steady, t_steady = 0, 0, 0.0
    while True:
        a = time.perf_counter()
        state, _, _ = oracle.decode_step_fused(state, Q[m + steps], K[m + steps],
                                               V[m + steps], n)
        b = time.perf_counter()
        if steps >= n:
            steady += 1
            t_steady += b - a
        steps += 1
        el = b - t1
        if el >= budget_s or steps >= T or (max_steps and steps >= max_steps):
            break
    t_pre = t1 - t0
    if steps >= T or steady == 0:
        est = t_pre + el * T / steps
    else:
        est = t_pre + el + (T - steps) * t_steady / steady
    return {"tokens_per_s": T / est, "prefill_s": t_pre, "decode_steps": steps,
            "decode_s_per_step": el / steps, "whole": steps >= T}


def oracle_steady_sampler(n_steps, t_start):
    """The reference arm's step: `n_steps` fused decode steps of the
    single-page workload at t = t_start .. t_start + n_steps - 1, after the
    ring is full (each attends m + n keys per head, as every step past the
    first n of the workload does).  The cache state at t_start is built once,
    untimed, by the oracle's own prefill_cache; the oracle's state
    transitions return new states, so every call starts from it.  Returns a
    function that runs the sample and returns its seconds."""
    import torch
    import oracle
    import workloads
    w = workloads.WORKLOADS["single_page_bf16"]
    H, d, m, n = w.heads, w.head_dim, w.m, w.n
    Q, K, V = workloads.qkv(m + t_start + n_steps, H, d, 0, w.std, torch.bfloat16)
    Q, K, V = (x.double().numpy() for x in (Q, K, V))
    state0 = oracle.prefill_cache(K[:m + t_start], V[:m + t_start], m, n, t_start)

    def run():
        state = state0
        t0 = time.perf_counter()
        for t in range(t_start, t_start + n_steps):
            state, _, _ = oracle.decode_step_fused(state, Q[m + t], K[m + t],
                                                   V[m + t], n)
        return time.perf_counter() - t0
    return run


def host_cores():
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_config_samples(rows_prefill=128):
    """Oracle (one thread) on the other workloads, each a bounded sample:
    one fused decode step of the batched and of the sweep workload (every
    sequence; cache contents are constant arrays of the right shapes, as the
    time does not depend on the values), and `rows_prefill` seeded rows of
    one multi-page prefill layer, extrapolated to 12 layers by the number of
    visible (query, key) pairs."""
    import numpy as np
    import torch
    import oracle
    import workloads
    rng = np.random.default_rng(0)
    out = {}

    def decode_all(B, H, d, m_list, n, T):
        states = []
        for m in m_list:
            states.append({"Kp": np.full((m, H, d), 0.01),
                           "Vp": np.full((m, H, d), 0.02),
                           "Kr": np.full((n, H, d), 0.01),
                           "Vr": np.full((n, H, d), 0.02), "t": T})
        q = np.full((B, H, d), 0.03)
        t0 = time.perf_counter()
        for b, st in enumerate(states):
            oracle.decode_step_fused(st, q[b], q[b, :], q[b, :], n)
        return time.perf_counter() - t0

    w = workloads.WORKLOADS["batched_decode_bf16"]
    m_list = workloads.prefix_lengths(w.batch, *w.m_range, seed=0)
    out["batched_decode"] = {"s_per_step": round(
        decode_all(w.batch, w.heads, w.head_dim, m_list, w.n, w.T), 4)}
    w = workloads.WORKLOADS["decode_sweep_bf16"]
    out["decode_sweep"] = {"s_per_step": round(
        decode_all(w.batch, w.heads, w.head_dim, [w.m] * w.batch, w.n, 4096), 4)}
    w = workloads.WORKLOADS["multipage_prefill_bf16"]
    L = w.m + w.T
    Q, K, V = workloads.qkv(L, w.heads, w.head_dim, 0, 1.0, torch.bfloat16)
    Q, K, V = (x.double().numpy() for x in (Q, K, V))
    rows = sorted(rng.choice(L, size=rows_prefill, replace=False).tolist())
    t0 = time.perf_counter()
    oracle.prefill_attention(Q, K, V, w.m, w.n, rows=rows)
    el = time.perf_counter() - t0
    def pairs(i):   # |N(i)|: i + 1 in the prefix, m + min(n, i - m + 1) after
        return i + 1 if i < w.m else w.m + min(w.n, i - w.m + 1)
    sample_pairs = sum(pairs(i) for i in rows)
    total_pairs = sum(pairs(i) for i in range(L))
    out["prefill"] = {"sample_rows": rows_prefill, "sample_s": round(el, 3),
                      "s_per_layer": round(el * total_pairs / sample_pairs, 1),
                      "s_12_layers": round(12 * el * total_pairs / sample_pairs, 1)}
    return out


def run_cpu_configs_worker():
    """oracle_config_samples in a one-thread subprocess without the GPU."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
               MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__),
                        "--cpu-configs-worker"], capture_output=True, text=True,
                       env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    out = json.loads(r.stdout.strip().splitlines()[-1])
    out["cores"] = 1
    out["kind"] = "oracle"
    return out


def run_cpu_worker(budget_s, max_steps=None, threads=1):
    """The oracle in a subprocess with `threads` BLAS/OpenMP threads."""
    t = str(int(threads))
    env = dict(os.environ, OMP_NUM_THREADS=t, OPENBLAS_NUM_THREADS=t,
               MKL_NUM_THREADS=t, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker",
           str(budget_s)]
    if max_steps:
        cmd += ["--cpu-max-steps", str(max_steps)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms, dist=None, device=None):
    """Step time of the whole job: the slowest rank's (timing reduction only;
    the data path has no collective)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_throughput(tokens_per_rank, world_size, ms):
    """Whole-job tokens/s: every rank runs its own replica of the workload
    (weak scaling), so the job processes world_size x the tokens of one."""
    return tokens_per_rank * world_size / (ms * 1e-3)


REF_SAMPLE_STEPS = 500        # decode steps per reference-arm step
REF_T_START = 5500            # ring full; the workload's last 500 steps


def main_reference(args):
    """The reference arm: the CPU float64 oracle as it stands, on one host
    thread.  One step of this arm is the sampled region itself - the single
    page workload's decode steps t = 5500 .. 5999 - so ms_per_step is the
    time actually spent per step and value is the tokens of that region per
    second.  (The 288-row prefix prefill and the first n steps, while the
    ring fills, are about 2 % of the oracle's time on the whole workload and
    are not in the sample.)"""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"          # before NumPy loads its BLAS
    import workloads
    w = workloads.WORKLOADS["single_page_bf16"]
    run = oracle_steady_sampler(REF_SAMPLE_STEPS, REF_T_START)
    for _ in range(args.warmup):
        run()
    secs = [run() for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(secs)
    v = REF_SAMPLE_STEPS / (ms * 1e-3)
    sample = ("oracle (CPU float64, one thread) on the single-page workload's "
              "fused decode steps t = %d..%d (ring full, m + n = %d keys per "
              "head); one step of this arm = that region"
              % (REF_T_START, REF_T_START + REF_SAMPLE_STEPS - 1, w.m + w.n))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 2),
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": "single_page_bf16", "batch": 1, "heads": 10,
                   "head_dim": 128, "m": 288, "n": 128, "T": 6000,
                   "sample": "decode steps t=%d..%d per step"
                             % (REF_T_START, REF_T_START + REF_SAMPLE_STEPS - 1)},
        "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": sample,
                         "value": round(v, 2), "unit": "tokens/s"},
        "e2e": {"value": round(v, 2), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def roofline_entry(kernel, workload, bound, work, us, peak, peak_name,
                   peak_src, traffic_key=None):
    """One roofline entry: algorithmic bytes (hbm) or flops (tensor) of one
    launch or step over its device time."""
    if bound == "hbm":
        achieved, unit = work / (us * 1e-6) / 1e9, "GB/s"
    else:
        achieved, unit = work / (us * 1e-6) / 1e12, "TFLOP/s"
    return {"kernel": kernel, "workload": workload, "bound": bound,
            "achieved": round(achieved, 1), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(traffic_key or kernel),
            "work": work, "us": round(us, 3), "peak_of": peak_name}


def extra_rooflines(extras, peaks, peak_src):
    """Roofline entries of the bound kernels measured in run_extras."""
    out = []
    hbm = peaks["hbm_gbs"]
    sw = extras.get("decode_sweep")
    if sw:
        us = statistics.mean(p["us_per_step"] for p in sw["points"])
        e = roofline_entry("decode_kernel", "decode_sweep_bf16 (mean over T)",
                           "hbm", sw["algorithmic_bytes"], us, hbm, "hbm_gbs",
                           peak_src, "decode_kernel@sweep")
        e["latency_spread"] = sw["latency_spread"]
        out.append(e)
    bt = extras.get("batched_decode")
    if bt:
        out.append(roofline_entry("decode_kernel", "batched_decode_bf16", "hbm",
                                  bt["algorithmic_bytes"], bt["us_per_step"], hbm,
                                  "hbm_gbs", peak_src, "decode_kernel@batched"))
    pf = extras.get("prefill")
    if pf:
        # per launch (one layer) of 12 back-to-back layers, 13 ms in all:
        # the burst peak applies
        layers = pf.get("layers", 12)
        out.append(roofline_entry("prefill_tc_kernel", "multipage_prefill_bf16 "
                                  "(per layer)", "tensor",
                                  pf["algorithmic_flops"] // layers,
                                  1e3 * pf["ms_per_step"] / layers,
                                  peaks["bf16_tflops"], "bf16_tflops", peak_src,
                                  "prefill_tc_kernel@multipage"))
    lp = extras.get("long_prefix_decode")
    if lp:
        pt = lp["points"][-1]
        out.append(roofline_entry(lp.get("kernel", "decode_kernel"),
                                  "long_prefix m=%d (per layer)" % pt["m"], "hbm",
                                  pt["bytes_per_layer"], pt["us_per_layer"], hbm,
                                  "hbm_gbs", peak_src,
                                  lp.get("kernel", "decode_kernel") + "@long_prefix"))
    gq = extras.get("batched_decode_gqa")
    if gq:
        out.append(roofline_entry("decode_gqa_sk_kernel", "batched_decode_gqa",
                                  "hbm", gq["algorithmic_bytes"], gq["us_per_step"],
                                  hbm, "hbm_gbs", peak_src,
                                  "decode_gqa_sk_kernel@batched"))
    return out


def main_ours(args):
    import torch
    import sliding_window_attention_02_gb300 as rswa
    ws, rank, local = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    rswa.load()
    peaks, peak_src = load_peaks()

    # CPU baseline first (subprocess; one thread, then every core) on rank 0
    cpu = cpu_all = None
    ncores = host_cores()
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = run_cpu_worker(args.cpu_budget)
        if not args.no_extras:
            cpu_all = run_cpu_worker(args.cpu_budget, threads=ncores)
    cpu_configs = None
    if rank == 0 and ws == 1 and not args.no_cpu and not args.no_extras:
        cpu_configs = run_cpu_configs_worker()

    sp = setup_single_page(dev)
    w = sp["w"]
    s = sp["stream"]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        # CUDAGraph.replay() launches on the current stream
        with torch.cuda.stream(s):
            sp["g_prefill"].replay()
            sp["g_decode"].replay()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # timed region: K steps, events per step, L2 flushed between steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            with torch.cuda.stream(s):
                flush.zero_()
                ev[i][0].record(s)
                sp["g_prefill"].replay()
                ev[i][1].record(s)
                sp["g_decode"].replay()
                ev[i][2].record(s)
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    ms = max_over_ranks(statistics.mean(step_ms), dist, dev)
    clocks = clk.summary()
    cache_bytes = sp["cache"].cache_bytes(0)      # C(T) after the loop
    value = job_throughput(w.batch * w.T, ws, ms)

    # dominant kernel: fused decode (6000 launches per step)
    per_launch_us = 1e3 * statistics.mean(dec_ms) / w.T
    head = roofline_entry("decode_cluster_kernel", "single_page_bf16 (headline)",
                          "hbm", round(single_page_bytes_per_decode(w)),
                          per_launch_us, peaks["hbm_gbs"], "hbm_gbs", peak_src)
    head["note"] = ("launch = decode-graph time / 6000; the 2.1 MB cache stays "
                    "in L2 between steps: latency-bound")

    # end-to-end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(sp, dev, args)
        e2e["eager"] = measure_e2e_eager(sp, dev, args)
    del sp
    torch.cuda.empty_cache()

    extras = {}
    per_step = None
    if not args.no_extras and rank == 0:
        try:
            rs = per_step_profile(dev)
            mh = per_step_profile(dev, n=w.T)
            per_step = {"rswa": dict(step_stats(rs), **step_growth(rs)),
                        "mha": dict(step_stats(mh), **step_growth(mh)),
                        "mha_jumps": boundary_jumps(mh),
                        "how": "event between steps in one graph: whole latency "
                               "of each step, no overlap with its neighbours"}
            extras["per_step_us"] = {"rswa": [round(x, 3) for x in rs],
                                     "mha": [round(x, 3) for x in mh]}
        except Exception as exc:           # events in graphs unsupported
            per_step = {"unavailable": repr(exc)[:200]}
        torch.cuda.empty_cache()
        extras.update(run_extras(dev, peaks, quick=args.quick))
        if cpu_configs is not None:
            extras["cpu_oracle"] = cpu_configs
        if cpu_all is not None:
            extras["cpu_baseline_all_cores"] = {
                "value": round(cpu_all["tokens_per_s"], 2), "unit": "tokens/s",
                "cores": ncores, "kind": "oracle"}
    rooflines = [head] + extra_rooflines(extras, peaks, peak_src)

    if rank == 0:
        sw = extras.get("decode_sweep")
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "single_page_bf16", "batch": 1, "heads": 10,
                       "head_dim": 128, "m": 288, "n": 128, "T": 6000,
                       "parallelism": f"replicas x{ws}",
                       "l2": "flushed (256 MB write) before every timed step",
                       "graphs": "prefix prefill and 6000-step decode loop "
                                 "replayed as two CUDA graphs"},
            "roofline": rooflines,
            "peaks": {"source": peak_src, "hbm_gbs": peaks["hbm_gbs"],
                      "bf16_tflops": peaks["bf16_tflops"],
                      "bf16_tflops_sustained": peaks["bf16_tflops_sustained"]},
            "per_step_us": per_step,
            "sweep_us_vs_T": None if not sw else {
                "T": [p["T"] for p in sw["points"]],
                "us": [p["us_per_step"] for p in sw["points"]]},
            "cpu_baseline": None if cpu is None else {
                "value": round(cpu["tokens_per_s"], 2), "unit": "tokens/s",
                "cores": 1, "kind": "oracle",
                "sample": ("the whole workload: 288-row prefix prefill + %d "
                           "decode steps (%.2f ms/step), float64, one thread"
                           % (cpu["decode_steps"], 1e3 * cpu["decode_s_per_step"]))
                          if cpu["whole"] else
                          ("288-row prefix prefill + the first %d decode steps; "
                           "the rest costed at the mean steady step; float64, "
                           "one thread" % cpu["decode_steps"])},
            "e2e": e2e,
            "gpu_launches": args.steps * (2 + w.T),
            "clocks": clocks,
            "cache_bytes_after_T": cache_bytes,
            "extras_file": args.extras_out,
        }
        if args.extras_out:
            with open(args.extras_out, "w") as f:
                json.dump(extras, f)
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def measure_e2e(sp, dev, args):
    """Same workload through the public API: per step the inputs are copied
    from pinned host memory and the outputs read back, inside the timed
    region; the prefill and the 6000 decode calls replay as CUDA graphs."""
    import torch
    w = sp["w"]
    s = sp["stream"]
    hQ, hK, hV = (x.cpu().pin_memory() for x in (sp["Q"], sp["K"], sp["V"]))
    hOp = torch.empty_like(sp["Op"], device="cpu").pin_memory()
    hOd = torch.empty_like(sp["Od"], device="cpu").pin_memory()

    def step():
        with torch.cuda.stream(s):
            sp["Q"].copy_(hQ, non_blocking=True)
            sp["K"].copy_(hK, non_blocking=True)
            sp["V"].copy_(hV, non_blocking=True)
            sp["g_prefill"].replay()
            sp["g_decode"].replay()
            hOp.copy_(sp["Op"], non_blocking=True)
            hOd.copy_(sp["Od"], non_blocking=True)
    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        step()
        e1.record(s)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = statistics.mean(ts)
    h2d = sum(x.numel() * x.element_size() for x in (hQ, hK, hV))
    d2h = hOp.numel() * hOp.element_size() + hOd.numel() * hOd.element_size()
    return {"value": round(w.batch * w.T / (ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms, 4), "mode": "graph replay"}


def measure_e2e_eager(sp, dev, args, steps=3):
    """The same end-to-end step with no graph: the host copies, one
    rswa_prefill call and 6000 rswa_decode_step_fused calls through the C
    ABI (argument checks, ctypes, launch) per step, timed with events."""
    import torch
    w = sp["w"]
    s = sp["stream"]
    m, T = w.m, w.T
    hQ, hK, hV = (x.cpu().pin_memory() for x in (sp["Q"], sp["K"], sp["V"]))
    hOp = torch.empty_like(sp["Op"], device="cpu").pin_memory()
    hOd = torch.empty_like(sp["Od"], device="cpu").pin_memory()
    Q, K, V, Op, Od, cache = (sp[k] for k in ("Q", "K", "V", "Op", "Od", "cache"))
    q = [Q[m + t][None] for t in range(T)]
    k = [K[m + t][None] for t in range(T)]
    v = [V[m + t][None] for t in range(T)]

    def step():
        with torch.cuda.stream(s):
            Q.copy_(hQ, non_blocking=True)
            K.copy_(hK, non_blocking=True)
            V.copy_(hV, non_blocking=True)
            cache.prefill(Q[:m], K[:m], V[:m], Op, [m], 0, stream=s)
            for t in range(T):
                cache.decode_step_fused(q[t], k[t], v[t], Od[t], stream=s)
            hOp.copy_(Op, non_blocking=True)
            hOd.copy_(Od, non_blocking=True)
    step()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        step()
        e1.record(s)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = statistics.mean(ts)
    return {"value": round(w.batch * T / (ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 3), "steps": steps,
            "us_per_token": round(1e3 * ms / T, 3)}


def main_only(args):
    """One workload, warmup + steps launches of its step, no timing lines
    beyond a mean: the command the ncu summaries are taken from."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(device=dev)
    if args.only == "single_page":
        sp = setup_single_page(dev)
        s = sp["stream"]

        def step():
            sp["g_prefill"].replay()
            sp["g_decode"].replay()
    elif args.only == "gqa":
        gq = setup_batched_gqa(dev)
        w = gq["w"]
        o = torch.empty(w.batch, gq["H"], w.head_dim, dtype=torch.bfloat16,
                        device=dev)
        q, k, v = (x[:w.batch] for x in gq["steps"])

        def step():
            gq["cache"].decode_step_fused(q, k, v, o, stream=s)
    elif args.only in ("batched", "sweep"):
        st = setup_batched(dev) if args.only == "batched" else setup_sweep(dev)
        w = st["w"]
        if args.only == "sweep":
            st["cache"].set_t([100000] * w.batch)
        o = torch.empty(w.batch, w.heads, w.head_dim, dtype=torch.bfloat16,
                        device=dev)
        q, k, v = (x[:w.batch] for x in st["steps"])

        def step():
            st["cache"].decode_step_fused(q, k, v, o, stream=s)
    elif args.only == "long_prefix":
        import sliding_window_attention_02_gb300 as rswa
        import workloads
        H, d, n, m = 10, 128, 128, 10272          # one sequence, 40 pages
        layers = args.layers or 2
        caches = []
        for layer in range(layers):
            _, K, V = workloads.qkv(m + n, H, d, layer, 1.0, torch.bfloat16,
                                    device=dev)
            c = rswa.RswaCache(m, n, H, d, 1, rswa.RSWA_BF16, device=dev)
            c.prefill(None, K, V, None, [m], n, stream=s)
            caches.append(c)
        q, k, v = workloads.qkv(1, H, d, 5, 1.0, torch.bfloat16, device=dev)
        o = torch.empty(1, H, d, dtype=torch.bfloat16, device=dev)

        def step():
            for c in caches:
                c.decode_step_fused(q, k, v, o, stream=s)
    elif args.only == "block":
        import sliding_window_attention_02_gb300 as rswa
        import workloads
        w = workloads.WORKLOADS["single_page_bf16"]
        B, H, d, m, n = w.batch, w.heads, w.head_dim, w.m, w.n
        C = args.block
        Q, K, V = workloads.qkv(m + C, H, d, 0, w.std, torch.bfloat16, device=dev)
        c = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16, device=dev)
        c.prefill(None, K[:m], V[:m], None, [m], 0, stream=s)
        q, k, v = (x[m:m + C][None].contiguous() for x in (Q, K, V))
        o = torch.empty_like(q)

        def step():
            c.decode_block(q, k, v, o, stream=s)
    elif args.only == "vanilla_prefill":
        import sliding_window_attention_02_gb300 as rswa
        import workloads
        H, d, n, L = 10, 128, 128, 32768        # m = 0: band tiles only
        Q, K, V = workloads.qkv(L, H, d, 100, 1.0, torch.bfloat16, device=dev)
        c = rswa.RswaCache(0, n, H, d, 1, rswa.RSWA_BF16, device=dev)
        O = torch.empty(L, H, d, dtype=torch.bfloat16, device=dev)

        def step():
            c.prefill(Q, K, V, O, [0], L, stream=s)
    else:
        pf = setup_prefill(dev, layers=args.layers)
        w = pf["w"]

        def step():
            for (Q, K, V), c, O in zip(pf["qkv"], pf["caches"], pf["outs"]):
                c.prefill(Q, K, V, O, [w.m], w.T, stream=s)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            step()
            e1.record(s)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    print(json.dumps({"only": args.only, "ms_per_step": statistics.mean(ms)}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--extras-out", default=None,
                    help="write every extra measurement to this JSON file")
    ap.add_argument("--cpu-worker", type=float, default=None)
    ap.add_argument("--cpu-configs-worker", action="store_true")
    ap.add_argument("--cpu-max-steps", type=int, default=None)
    ap.add_argument("--only", default=None,
                    choices=["single_page", "batched", "sweep", "gqa", "prefill",
                             "vanilla_prefill", "long_prefix", "block"],
                    help="run one workload warmup+steps times and print its "
                         "mean step time (for profiling)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layers with --only prefill or long_prefix")
    ap.add_argument("--block", type=int, default=1024,
                    help="tokens per call with --only block")
    args = ap.parse_args()
    if args.cpu_configs_worker:
        print(json.dumps(oracle_config_samples()))
        return 0
    if args.cpu_worker is not None:
        print(json.dumps(oracle_single_page_sample(args.cpu_worker,
                                                   args.cpu_max_steps)))
        return 0
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return main_reference(args)
    if args.only:
        return main_only(args)
    return main_ours(args)


if __name__ == "__main__":
    sys.exit(main())
