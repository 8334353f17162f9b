"""Benchmark of the DSA indexer hot path on GB300.

One step = the whole path over one batch: the fused indexer score + top-k
(dsa_indexer_logits_topk) followed by the paged mxfp4 gather of the selected rows
(mxfp4_paged_gather).  Headline workload (`value`, `roofline`, `e2e`): the FP8
long-context chunked prefill, the largest configuration that fits one GPU (8192 E4M3
queries at positions 57344..65535 over 65536 E4M3 keys, causal, top-1024, then the
gather of all 8,388,608 selected rows).  The same JSON line carries one sub-record per
other configuration (tiny, Flash decode, Pro decode MTP, 16K prefill) with its fused
and gather times and its own roofline fraction, each from its own timed loop, and under
"next" the rows beyond the hot path proper (FP8-q x FP4-k score, the query and key
producers, the sparse attention over the selection), each with its own roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
    python bench.py --next NAME      # one of the "next" rows alone (a profiler target)

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a bounded
sample of the same workload.  Under torchrun each rank runs its own batch (weak
scaling, no collective on the data path); timing is the max over ranks.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "indexer query-tokens/s (logits+top-k), gather GB/s; % of roofline, 1×GB300"
UNIT = "query-tokens/s"
L2_BYTES = 129 * 2**20
HEADLINE = "fp8_chunked"

WORKLOADS = {
    "tiny": dict(desc="1 seq, 64 queries at 1984..2047 over 2048 contiguous bf16 keys, causal, top-512, "
                      "mxfp4 gather of 512 rows/query (5% padded)", seed=1, bound="tensor"),
    "flash_decode": dict(desc="64 seq x 1 query, L~U[4096,65536], paged bf16 keys bs=64, top-512, "
                              "mxfp4 gather of 512 rows/query", seed=2, bound="hbm"),
    "pro_mtp": dict(desc="32 seq x 2 queries (causal), L~U[32768,131072], paged bf16 keys bs=64, "
                         "top-1024, mxfp4 gather of 1024 rows/query (2% padded)", seed=3, bound="hbm"),
    "prefill": dict(desc="1 seq, T=K=16384, causal, contiguous bf16 keys, fused top-512 (no gather)",
                    seed=4, bound="tensor"),
    "fp8_chunked": dict(desc="1 seq, 8192 E4M3 queries at 57344..65535 over 65536 E4M3 keys, causal, "
                             "top-1024, mxfp4 gather of every selection", seed=5, bound="tensor"),
}


def make_workload(name: str, seed: int, batch: int = 0):
    """The named workload; `batch` > 0 shrinks it for profiler captures: the sequence
    count of a decode batch, the tokens T = K of the prefill, or the query rows of the
    FP8 chunked prefill (the last `batch` positions before 65536)."""
    from deepseek_v4_sparse_dsa_gb300 import synth
    fn = {"tiny": synth.make_tiny, "flash_decode": synth.make_flash_decode, "pro_mtp": synth.make_pro_mtp,
          "prefill": synth.make_prefill, "fp8_chunked": synth.make_fp8_chunked}[name]
    if batch > 0:
        if name in ("prefill", "fp8_chunked"):
            return fn(seed=seed, T=batch)
        if name in ("flash_decode", "pro_mtp"):
            return fn(seed=seed, B=batch)
        raise SystemExit("--batch does not apply to the tiny workload")
    return fn(seed=seed)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "deepseek_v4_sparse_dsa_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary, if it
    was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("src_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- algorithmic work

def algorithmic_work(wl):
    """Bytes / flops one fused call and one gather must move or do (masked work excluded)."""
    vis = wl.visible_len().astype(np.int64)
    T, k = wl.T, wl.topk
    elt = 1 if wl.dtype == "e4m3" else 2
    L = wl.context_lens.astype(np.int64)
    key_bytes = int(L.sum()) * 128 * elt + (int(L.sum()) * 4 if wl.dtype == "e4m3" else 0)
    q_bytes = T * 64 * 128 * elt + T * 64 * 4 + (T * 64 * 4 if wl.dtype == "e4m3" else 0)
    fused_bytes = key_bytes + q_bytes + T * k * 8 + wl.B * 4
    flops = 2 * 64 * 128 * int(vis.sum())
    gather_rows = T * k
    gather_bytes = gather_rows * (68 + 256) + gather_rows * 4
    return dict(fused_bytes=fused_bytes, flops=flops, gather_bytes=gather_bytes)


def roofline_peak(bound: str, dtype: str, peaks):
    """Peak of the fused call's bound: measured HBM copy bandwidth, or the measured
    sustained bf16 dense rate (times 2 for E4M3, the nominal fp8 : bf16 ratio)."""
    if bound == "hbm":
        return peaks["hbm_gbs"], "GB/s"
    return peaks["bf16_tflops_sustained"] * (2.0 if dtype == "e4m3" else 1.0), "TFLOP/s"


def roofline(bound: str, wl, work, fused_ms: float, peaks):
    peak, unit = roofline_peak(bound, wl.dtype, peaks)
    if bound == "hbm":
        achieved = work["fused_bytes"] / (fused_ms * 1e-3) / 1e9
    else:
        achieved = work["flops"] / (fused_ms * 1e-3) / 1e12
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "peak_source": f"{peaks['source']}: " + ("hbm_gbs" if bound == "hbm" else
                                                     "bf16_tflops_sustained" + (" x 2 (fp8)" if wl.dtype == "e4m3"
                                                                                else ""))}


def l2_note(wl, work) -> str:
    """How the timed steps avoid re-reading the previous step's data from the 129 MB L2."""
    if work["fused_bytes"] - wl.T * wl.topk * 8 > L2_BYTES:     # inputs only, not the selection
        return "inputs larger than L2"
    out = wl.T * wl.topk * 256 if wl.kv_fp4 is not None else 0
    if out > L2_BYTES:
        return f"L2 flushed every step by the gather's {out / 2**30:.1f} GiB output write"
    return "inputs fit in L2, not flushed (latency-bound parity case)"


def config_of(name: str, wl, batch: int, world: int):
    """The `config` object of the JSON line (identical for both arms)."""
    info = WORKLOADS[name]
    work = algorithmic_work(wl)
    return {"workload": name + (f"_b{batch}" if batch else ""), "desc": info["desc"], "B": wl.B,
            "next_n": wl.next_n, "topk": wl.topk, "dtype": wl.dtype, "sum_context": int(wl.context_lens.sum()),
            "seed": info["seed"],
            "l2": l2_note(wl, work),
            "parallelism": f"replicas x{world}"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"dsa_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    rows.append(dict(sm=float(parts[2]), max=float(parts[3]), power=float(parts[4]),
                                     hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}
        load = [r for r in rows if r["power"] > 300] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in load),
                "reasons": sorted(reasons), "samples": len(load)}


# ----------------------------------------------------------------------------- our arm

class Runner:
    """One workload resident on the device and its step (fused call, then the gather)."""

    def __init__(self, wl, dev, stream):
        import torch

        from deepseek_v4_sparse_dsa_gb300 import dsa
        from deepseek_v4_sparse_dsa_gb300.device import DeviceBatch
        self.torch, self.dsa = torch, dsa
        self.wl, self.dev, self.stream = wl, dev, stream
        self.db = DeviceBatch.from_workload(wl, dev)
        T, k = wl.T, wl.topk
        self.has_gather = wl.kv_fp4 is not None
        self.ws = self.db.workspace(dsa.DSA_OP_LOGITS_TOPK, k)
        self.idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.gout = torch.empty((T, k, 128), dtype=torch.int16, device=dev) if self.has_gather else None
        # Configurations with padded slots gather a copy of the selection with their seeded
        # fraction of slots set to -1 (made once from the first fused result, outside any
        # timed region; the selection is the same at every step).
        self.sel = self.idx
        if self.has_gather and wl.gather_pad_frac > 0:
            from deepseek_v4_sparse_dsa_gb300 import synth
            m = synth.pad_sel_pos(np.zeros((T, k), np.int32), wl.gather_pad_frac, wl.seed) < 0
            self.fused()
            torch.cuda.synchronize(dev)
            self.sel = self.idx.clone().masked_fill_(torch.from_numpy(m).to(dev), -1)

    def fused(self):
        self.db.logits_topk(self.wl.topk, ws=self.ws, out_idx=self.idx, with_values=False, stream=self.stream)

    def gather(self):
        if self.has_gather:
            self.db.gather(self.sel, out=self.gout, stream=self.stream)

    def step(self):
        self.fused()
        self.gather()

    def timed(self, steps: int, warm_s: float):
        """Mean device ms of the fused call and of the gather over `steps` steps (CUDA
        events on the launching stream), after a warm loop of about `warm_s` seconds;
        also the whole region's ms per step and the library's launches inside it."""
        torch, dev = self.torch, self.dev
        for _ in range(3):
            self.step()
        t_end = time.time() + warm_s
        while time.time() < t_end:
            self.step()
            torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        launches0 = self.dsa.dsa_launch_count()
        t0.record(self.stream)
        for i in range(steps):
            ev[i][0].record(self.stream)
            self.fused()
            ev[i][1].record(self.stream)
            self.gather()
            ev[i][2].record(self.stream)
        t1.record(self.stream)
        torch.cuda.synchronize(dev)
        launches = self.dsa.dsa_launch_count() - launches0
        assert self.dsa.dsa_device_error(self.stream) == 0
        fused_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
        gather_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) if self.has_gather else 0.0
        return fused_ms, gather_ms, t0.elapsed_time(t1) / steps, launches


def sub_record(name: str, dev, stream, peaks, seconds: float):
    """Fused and gather times of one more configuration, with its roofline fraction."""
    info = WORKLOADS[name]
    wl = make_workload(name, info["seed"])
    r = Runner(wl, dev, stream)
    fused_ms, gather_ms, _, _ = r.timed(3, 0.2)
    steps = int(min(400, max(10, seconds * 1e3 / max(fused_ms + gather_ms, 1e-3))))
    fused_ms, gather_ms, step_ms, launches = r.timed(steps, 0.3)
    work = algorithmic_work(wl)
    rec = {"workload": name, "desc": info["desc"], "T": wl.T, "topk": wl.topk, "dtype": wl.dtype,
           "steps": steps, "ms_per_step": step_ms, "fused_ms": fused_ms, "gather_ms": gather_ms,
           "indexer_qtok_s": wl.T / (fused_ms * 1e-3), "value": wl.T / (step_ms * 1e-3),
           "work": work, "roofline": roofline(info["bound"], wl, work, fused_ms, peaks),
           "gpu_launches": int(launches),
           "l2": config_of(name, wl, 0, 1)["l2"]}
    if r.has_gather:
        gbps = work["gather_bytes"] / (gather_ms * 1e-3) / 1e9
        rec["gather_gbps"] = gbps
        rec["gather_frac_hbm"] = gbps / peaks["hbm_gbs"]
    del r
    import torch
    torch.cuda.empty_cache()
    return rec


# ----------------------------------------------------------------------------- the NEXT rows

def time_calls(fn, dev, stream, seconds: float):
    """Mean device ms of fn() (CUDA events on the launching stream around each call) over
    about `seconds` of calls after a warm-up; also the library's launches per call."""
    import torch

    from deepseek_v4_sparse_dsa_gb300 import dsa
    for _ in range(3):
        fn()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    torch.cuda.synchronize(dev)
    steps = int(min(400, max(10, seconds * 1e3 / max(a.elapsed_time(b), 1e-3))))
    for _ in range(max(3, steps // 4)):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    n0 = dsa.dsa_launch_count()
    for e in ev:
        e[0].record(stream)
        fn()
        e[1].record(stream)
    torch.cuda.synchronize(dev)
    launches = (dsa.dsa_launch_count() - n0) / steps
    assert dsa.dsa_device_error(stream) == 0
    return statistics.mean(e[0].elapsed_time(e[1]) for e in ev), steps, launches


def hbm_record(name, desc, nbytes, ms, peaks, steps, launches, l2):
    gbps = nbytes / (ms * 1e-3) / 1e9
    return {"workload": name, "desc": desc, "ms": ms, "steps": steps, "launches_per_call": launches,
            "l2": l2, "roofline": {"bound": "hbm", "achieved": gbps, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": gbps / peaks["hbm_gbs"], "bytes_per_call": int(nbytes),
                                   "peak_source": f"{peaks['source']}: hbm_gbs"}}


def attn_work(ab):
    """Algorithmic bytes and flops of one sparse-attention call: the selected cache rows
    (68 B each, padded slots none), q, the fp32 output, the selection and the sinks;
    2 x 64 x 128 flops per (row, head, selected slot) for the scores and as many for P.V."""
    live = int((ab.sel >= 0).sum())
    nbytes = live * 68 + ab.T * 64 * 128 * (2 + 4) + ab.sel.size * 4 + 64 * 4
    flops = 4 * 64 * 128 * ab.T * ab.topk
    return nbytes, flops


NEXT_NAMES = ("flash_decode_fp4k", "q_rope_quant", "k_hadamard_mxfp4", "sparse_attn_flash_decode",
              "sparse_attn_pro_mtp", "sparse_attn_fp8_chunked")


def next_record(name: str, dev, stream, peaks, seconds: float):
    """One sub-record of the rows beyond the hot path proper: the FP8-q x FP4-k fused score
    on the Flash decode batch, the two producers, or the sparse attention on one shape."""
    import torch

    from deepseek_v4_sparse_dsa_gb300 import dsa, synth
    from deepseek_v4_sparse_dsa_gb300.device import DeviceBatch
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    if name == "flash_decode_fp4k":
        # FP8 queries x FP4 keys read from the paged mxfp4 cache (fused score + top-k)
        wl = synth.make_flash_decode_fp4k()
        db = DeviceBatch.from_workload(wl, dev)
        ws = db.workspace(dsa.DSA_OP_LOGITS_TOPK, wl.topk)
        idx = torch.empty((wl.T, wl.topk), dtype=torch.int32, device=dev)
        ms, steps, launches = time_calls(lambda: db.logits_topk(wl.topk, ws=ws, out_idx=idx, with_values=False,
                                                                stream=stream), dev, stream, seconds)
        L = int(wl.context_lens.sum())
        nbytes = L * 68 + wl.T * 64 * (128 + 4 + 4) + wl.T * wl.topk * 8 + wl.B * 4
        rec = hbm_record(name, "Flash decode batch, E4M3 queries x keys read from the paged mxfp4 cache "
                         "(68 B per key instead of 256), fused top-512", nbytes, ms, peaks, steps, launches,
                         "inputs larger than L2")
        rec["key_bytes_per_key"] = 68
        rec["indexer_qtok_s"] = wl.T / (ms * 1e-3)
        return rec

    rng = synth.Rng(9)
    if name == "q_rope_quant":
        # indexer-Q RoPE + E4M3 quantisation: the FP8 chunked prefill's 8192 x 64 query rows
        T, R, maxpos = 8192, 64, 65536
        q = d(synth.normal_bf16(rng, (T, 64, 128), "q").view(np.int16))
        pos = d((57344 + np.arange(T)).astype(np.int32))
        ang = (np.arange(maxpos)[:, None] * (10000.0 ** (-np.arange(R // 2) / (R // 2)))[None, :])
        table = d(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))
        codes = torch.empty((T, 64, 128), dtype=torch.uint8, device=dev)
        qs = torch.empty((T, 64), dtype=torch.float32, device=dev)
        ms, steps, launches = time_calls(lambda: dsa.dsa_indexer_q_rope_quant(q, pos, table, maxpos, R, T, 64, 128,
                                                                              codes, qs, stream),
                                         dev, stream, seconds)
        nbytes = T * 64 * 128 * (2 + 1) + T * 64 * 4 + T * (4 + R * 4)
        return hbm_record(name, "8192 tokens x 64 heads x 128 dims bf16 -> E4M3 + per-row scale, RoPE on the "
                          "first 64 dims", nbytes, ms, peaks, steps, launches,
                          "input 128 MiB, about the L2 size; not flushed")

    if name == "k_hadamard_mxfp4":
        # indexer-key Hadamard + mxfp4 write into a paged pool: 1M keys
        N = 1 << 20
        k = d(synth.normal_bf16(rng, (N, 128), "k").view(np.int16))
        slots = d(rng.permutation(N, "slots").astype(np.int64))
        fp4 = torch.empty((N, 64), dtype=torch.uint8, device=dev)
        sc = torch.empty((N, 4), dtype=torch.uint8, device=dev)
        ms, steps, launches = time_calls(lambda: dsa.dsa_indexer_k_hadamard_mxfp4(k, slots, N, 128, fp4, sc, N,
                                                                                  stream), dev, stream, seconds)
        return hbm_record(name, "1,048,576 keys x 128 bf16 -> Hadamard -> mxfp4 rows at permuted pool slots",
                          N * (256 + 8 + 68), ms, peaks, steps, launches, "inputs larger than L2")

    # sparse attention over the selection, straight from the paged mxfp4 cache
    shape = name[len("sparse_attn_"):]
    ab = synth.make_attn_config(shape)
    aq, asel = d(ab.q.view(np.int16)), d(ab.sel)
    afp4, asc, atab, asink = d(ab.kv_fp4), d(ab.kv_scale), d(ab.table), d(ab.sink)
    out = torch.empty((ab.T, 64, 128), dtype=torch.float32, device=dev)
    f = lambda: dsa.dsa_sparse_attn_mxfp4(aq, ab.T, 64, 128, asel, ab.topk, afp4, asc, afp4.shape[0],
                                          ab.block_size, atab, atab.shape[1], ab.next_n, asink, ab.scale, out,
                                          stream)
    ms, steps, launches = time_calls(f, dev, stream, seconds)
    nbytes, flops = attn_work(ab)
    gbps, tflops = nbytes / (ms * 1e-3) / 1e9, flops / (ms * 1e-3) / 1e12
    tpeak = peaks["bf16_tflops"]
    bound = "hbm" if nbytes / peaks["hbm_gbs"] >= flops / (tpeak * 1e3) else "tensor"
    return {"workload": name,
            "desc": f"{ab.T} query rows x 64 heads x 128 dims over top-{ab.topk} rows of the paged mxfp4 cache, "
                    "sink logits, fp32 out", "ms": ms, "steps": steps, "launches_per_call": launches,
            "qtok_s": ab.T / (ms * 1e-3),
            "roofline": {"bound": bound, "achieved": gbps if bound == "hbm" else tflops,
                         "peak": peaks["hbm_gbs"] if bound == "hbm" else tpeak,
                         "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                         "frac": gbps / peaks["hbm_gbs"] if bound == "hbm" else tflops / tpeak,
                         "hbm_frac": gbps / peaks["hbm_gbs"], "tensor_frac": tflops / tpeak,
                         "bytes_per_call": int(nbytes), "flops_per_call": int(flops),
                         "peak_source": f"{peaks['source']}: hbm_gbs / bf16_tflops (burst)"}}


def next_records(dev, stream, peaks, seconds: float):
    import torch
    recs = []
    for name in NEXT_NAMES:
        recs.append(next_record(name, dev, stream, peaks, seconds))
        torch.cuda.empty_cache()
    return recs


def run_one_next(args):
    """--next NAME: time one of the rows beyond the hot path on its own (for profiler
    captures of that kernel) and print its record."""
    import torch

    from deepseek_v4_sparse_dsa_gb300 import dsa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dsa.load()
    rec = next_record(args.next, dev, torch.cuda.current_stream(dev), load_peaks(), args.sub_seconds)
    print(json.dumps(rec), flush=True)


def run_ours(args, rank, world):
    import torch

    from deepseek_v4_sparse_dsa_gb300 import dsa

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dsa.load()
    info = WORKLOADS[args.workload]
    wl = make_workload(args.workload, info["seed"] + rank, args.batch)
    stream = torch.cuda.current_stream(dev)
    T, k = wl.T, wl.topk
    run = Runner(wl, dev, stream)
    db = run.db
    work = algorithmic_work(wl)
    peaks = load_peaks()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(dev.index)
    sampler.start()
    for _ in range(args.warmup):
        run.step()
    barrier()
    fused_ms, gather_ms, ms_local, launches = run.timed(args.steps, 1.0)
    barrier()

    # end to end through the public API: pinned host inputs in, results back to pinned host
    h_q = db.q.cpu().pin_memory()
    h_w = db.weights.cpu().pin_memory()
    h_qs = db.q_scale.cpu().pin_memory() if db.q_scale is not None else None
    h_lens = db.context_lens.cpu().pin_memory()
    h_bt = db.block_table.cpu().pin_memory() if db.block_table is not None else None
    h_idx = torch.empty((T, k), dtype=torch.int32).pin_memory()
    h_out = torch.empty((T, k, 128), dtype=torch.int16).pin_memory() if run.has_gather else None
    h2d = sum(x.numel() * x.element_size() for x in (h_q, h_w, h_qs, h_lens, h_bt) if x is not None)
    d2h = h_idx.numel() * 4 + (h_out.numel() * 2 if run.has_gather else 0)

    def e2e_step():
        db.q.copy_(h_q, non_blocking=True)
        db.weights.copy_(h_w, non_blocking=True)
        if h_qs is not None:
            db.q_scale.copy_(h_qs, non_blocking=True)
        db.context_lens.copy_(h_lens, non_blocking=True)
        if h_bt is not None:
            db.block_table.copy_(h_bt, non_blocking=True)
        run.step()
        h_idx.copy_(run.idx, non_blocking=True)
        if run.has_gather:
            h_out.copy_(run.gout, non_blocking=True)

    # Without padded slots (the headline) the steps are pipelined as a caller would run them:
    # a copy stream brings each step's inputs in once the previous fused call has read them,
    # and takes each step's results out while the next step computes (results double-
    # buffered on the device and on the host).  Every step still copies its own inputs in
    # and its own results out inside the timed region.
    pipelined = run.has_gather and wl.gather_pad_frac == 0
    if pipelined:
        cs = torch.cuda.Stream(dev)
        idxs = [run.idx, torch.empty_like(run.idx)]
        gouts = [run.gout, torch.empty_like(run.gout)]
        h_idxs = [h_idx, torch.empty(h_idx.shape, dtype=h_idx.dtype).pin_memory()]
        h_outs = [h_out, torch.empty(h_out.shape, dtype=h_out.dtype).pin_memory()]
        ev_in, ev_read = torch.cuda.Event(), torch.cuda.Event()
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        ev_copied = [torch.cuda.Event(), torch.cuda.Event()]
        step_no = [0]

        def e2e_step():
            b = step_no[0] % 2
            step_no[0] += 1
            with torch.cuda.stream(cs):
                cs.wait_event(ev_read)                 # the previous fused call has read the inputs
                db.q.copy_(h_q, non_blocking=True)
                db.weights.copy_(h_w, non_blocking=True)
                if h_qs is not None:
                    db.q_scale.copy_(h_qs, non_blocking=True)
                db.context_lens.copy_(h_lens, non_blocking=True)
                if h_bt is not None:
                    db.block_table.copy_(h_bt, non_blocking=True)
                ev_in.record(cs)
            stream.wait_event(ev_in)
            stream.wait_event(ev_copied[b])            # this buffer's previous results are out
            db.logits_topk(k, ws=run.ws, out_idx=idxs[b], with_values=False, stream=stream)
            ev_read.record(stream)
            db.gather(idxs[b], out=gouts[b], stream=stream)
            ev_done[b].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_done[b])
                h_idxs[b].copy_(idxs[b], non_blocking=True)
                h_outs[b].copy_(gouts[b], non_blocking=True)
                ev_copied[b].record(cs)

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(3):
        e2e_step()
    if pipelined:
        stream.wait_stream(cs)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    if pipelined:
        stream.wait_stream(cs)                         # the last results are on the host
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    local = torch.tensor([ms_local, e2e_ms], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(local, op=torch.distributed.ReduceOp.MAX)
    ms_step, e2e_ms = float(local[0]), float(local[1])

    subs, nxt = [], []
    if rank == 0 and world == 1 and not args.batch and args.sub:
        del run, db
        torch.cuda.empty_cache()
        for name in WORKLOADS:
            if name != args.workload:
                subs.append(sub_record(name, dev, stream, peaks, args.sub_seconds))
        nxt = next_records(dev, stream, peaks, args.sub_seconds)
    clocks = sampler.stop()
    if rank != 0:
        return None

    out = {
        "metric": METRIC, "value": T * world / (ms_step * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded SplitMix64 generator; no dataset or weights)",
        "config": config_of(args.workload, wl, args.batch, world),
        "indexer_qtok_s": T / (fused_ms * 1e-3),
        "fused_ms": fused_ms,
        "gather_ms": gather_ms,
        "work": work,
        "gather_gbps": (work["gather_bytes"] / (gather_ms * 1e-3) / 1e9) if run_has_gather(wl) else None,
        "gather_frac_hbm": (work["gather_bytes"] / (gather_ms * 1e-3) / 1e9 / peaks["hbm_gbs"])
        if run_has_gather(wl) else None,
        "roofline": dict(kernel="dsa_indexer_logits_topk (plan_kernel + indexer_kernel + merge_kernel)",
                         **roofline(info["bound"], wl, work, fused_ms, peaks),
                         traffic=recorded_traffic(args.workload)),
        "gpu_launches": int(launches),
        "clocks": clocks,
        "e2e": {"value": T * world / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms, "steps": e2e_steps,
                "copies": "overlapped with the next step's compute on a copy stream" if pipelined
                else "in line with the compute on one stream"},
    }
    if subs:
        out["configs"] = subs
    if nxt:
        out["next"] = nxt
    return out, wl


def run_has_gather(wl) -> bool:
    return wl.kv_fp4 is not None


# ----------------------------------------------------------------------------- oracle arm

def oracle_sample(wl, budget_s: float, min_rows: int = 1):
    """Runs the oracle (score, top-k, gather) on query rows until the time budget is used;
    returns (rows done, seconds)."""
    from oracle import dsa_oracle as orc
    order = np.random.default_rng(0).permutation(wl.T)
    t0 = time.perf_counter()
    done = 0
    for t in order:
        lg = orc.indexer_logits(wl.q, wl.q_scale, wl.dtype, wl.weights, wl.k_data, wl.k_scale,
                                wl.block_table, wl.block_size, wl.B, wl.next_n, wl.context_lens,
                                wl.causal, rows=np.array([t]))
        idx, _ = orc.topk_select(lg, wl.topk)
        if wl.kv_fp4 is not None:
            b = t // wl.next_n
            orc.mxfp4_paged_gather(wl.kv_fp4, wl.kv_scale, wl.gather_block_table[b:b + 1], idx, 1, 1,
                                   wl.block_size)
        done += 1
        if done >= min_rows and time.perf_counter() - t0 >= budget_s:
            break
    return done, time.perf_counter() - t0


def cpu_cores() -> int:
    """Worker threads the C++ oracle runs on (every hardware thread unless
    DSA_ORACLE_THREADS says otherwise)."""
    from oracle import dsa_oracle as orc
    return orc.threads_used()


def run_reference(args, rank, world):
    if rank != 0:
        return None
    info = WORKLOADS[args.workload]
    wl = make_workload(args.workload, info["seed"], args.batch)
    for _ in range(args.warmup):
        oracle_sample(wl, 0.0)
    rows = 0
    secs = 0.0
    per_step = []
    budget = min(2.0, 90.0 / max(args.steps, 1))   # the whole run stays near 90 s of oracle work
    for _ in range(args.steps):
        r, s = oracle_sample(wl, budget)
        rows += r
        secs += s
        per_step.append(s / r)
    value = rows / secs
    sample = f"{rows} query rows over {args.steps} steps (score, top-k and gather per row)"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wl.T * statistics.mean(per_step),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded SplitMix64 generator; no dataset or weights)",
        "config": config_of(args.workload, wl, args.batch, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences of a decode workload, query rows of a prefill (0: the workload's own size)")
    ap.add_argument("--no-sub", dest="sub", action="store_false",
                    help="skip the sub-records of the other configurations")
    ap.add_argument("--sub-seconds", type=float, default=0.5, help="timed seconds per sub-record")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    ap.add_argument("--next", default=None, choices=NEXT_NAMES,
                    help="time only this row beyond the hot path (a profiler target) and print its record")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.next:
        run_one_next(args)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if res is not None:
        out, wl = res
        if world == 1:                                   # the CPU baseline is an N = 1 figure
            rows, secs = oracle_sample(wl, args.cpu_baseline_seconds)
            out["cpu_baseline"] = {"value": rows / secs, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                                   "sample": f"{rows} of {wl.T} query rows (score, top-k, gather), "
                                             f"{secs:.1f} s"}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
