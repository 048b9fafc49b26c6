"""Benchmark of the DSA lightning-indexer hot path on GB300.

A step is one pass of the whole path over one batch: key LayerNorm -> RoPE ->
MXFP8 quantisation (dsa_idx_preprocess) followed by the fused score + top-k
(dsa_idx_score_topk), on the single-sequence workload T = S = 32768, 64
indexer heads, head_dim 128 (64 RoPE + 64 NoPE), top-k 2048, MXFP8 scoring.
Inputs are seeded synthetic data already resident in HBM; L2 is flushed
between timed steps.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

--impl reference times the CPU oracle (oracle/) on a bounded sample of the
same workload's query rows.  Under torchrun each rank runs its own replica
of the workload (weak scaling); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_indexer_dsa_gb300 import workloads as W  # noqa: E402

METRIC = "fused indexer score+top-k queries/sec, TFLOP/s and % of GB300 BF16/FP8 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0   # nominal dense ratio (4.5 / 2.25 PFLOP/s)


def describe(wl, prec=None):
    return (f"{wl.name}: {len(wl.doc_lens)} x {wl.max_seqlen} tokens (T={wl.total_tokens}), {wl.n_heads} heads, "
            f"D={wl.head_dim} ({wl.rope_dim} RoPE + {wl.head_dim - wl.rope_dim} NoPE), top-k {wl.index_topk}, "
            f"{(prec or wl.prec).upper()} scoring" + (", key LayerNorm + RoPE in FP32" if wl.layernorm else ""))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def measure_fp8_peak(device):
    """Dense FP8 tensor throughput of this GPU, measured here: cuBLAS through
    torch._scaled_mm on E4M3 operands, 8192^3, best of 10 (CUDA events), in
    TFLOP/s.  Returns (value, source); falls back to the nominal FP8/BF16
    ratio times the BF16 figure when the call is not available."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        one = torch.tensor(1.0, device=device)
        for _ in range(3):
            torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2.0 * n ** 3 / best / 1e9, "measured in this run: torch._scaled_mm E4M3 8192^3, best of 10"
    except Exception as exc:   # noqa: BLE001
        peaks, kind = load_peaks()
        return (peaks["bf16_tflops"] * FP8_OVER_BF16,
                f"{kind} bf16 burst x {FP8_OVER_BF16} (nominal FP8/BF16; FP8 GEMM unavailable: {exc})")


def reduce_max_over_ranks(value, device):
    """Max of a per-rank float over the process group: the slowest rank sets
    the job's time.  Works with any backend (nccl on the GPUs, gloo on CPU)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, steps, max_ms):
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time."""
    return world * units_per_rank * steps / (max_ms / 1e3)


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.out,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_record():
    """Per-launch DRAM bytes of the fused kernel from the committed ncu
    summary, valid only while the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "score_topk_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    h = hashlib.sha256()
    for name in ("score_topk.cu", "dsa_device.cuh", "score_layout.h"):
        with open(os.path.join(ROOT, "sparse_attention_indexer_dsa_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec


def oracle_sample_rate(wl, x, n_rows, seed=0):
    """Queries/s of the CPU oracle on min(n_rows, T) query rows of the bench
    workload in its own precision; returns (rate, seconds, rows timed)."""
    rate, dt = oracle_rate(wl, x, wl.prec, n_rows, seed)
    return rate, dt, min(n_rows, wl.total_tokens)


def oracle_rate(wl, x, prec, n_rows, seed=0):
    """Queries/s of the CPU oracle on `n_rows` query rows of any workload
    (uniformly spread positions), including the key-side work those rows
    need (LayerNorm/RoPE/quantisation, or KPool compression)."""
    import oracle.dsa_oracle as O
    rng = np.random.default_rng(seed)
    T, H, D = wl.total_tokens, wl.n_heads, wl.head_dim
    rows = np.sort(rng.choice(T, size=min(n_rows, T), replace=False))
    cu = wl.cu_seqlens
    t0 = time.perf_counter()
    pos = O.positions_in_document(cu)
    kk = x["k"].astype(np.float64)
    qr = x["q"][rows].astype(np.float64)
    if wl.layernorm:
        kk = O.key_layernorm(x["k"], x["ln_gamma"], x["ln_beta"], 1e-6)
    if wl.rope_dim:
        kk = O.round_fp32(O.apply_rope(kk, pos, wl.rope_dim, wl.rope_base))
        qr = O.round_fp32(O.apply_rope(qr, pos[rows][:, None], wl.rope_dim, wl.rope_base))
    qq = np.zeros((T, H, D))
    w = x["w"].astype(np.float64)
    if wl.kpool > 1:
        kbar, cpools = O.kpool_compress(x["k"], O.bf16_bits_to_float(x["gate_bits"]), x["slot_bias"], cu, wl.kpool)
        qq[rows] = O.round_bf16(qr)
        O.kpool_topk(qq, O.round_bf16(kbar), w, cu, cpools, wl.index_topk, wl.kpool, True, rows=rows)
    else:
        kq = O.scoring_operand(kk, prec)[0]
        qq[rows] = O.scoring_operand(qr.reshape(-1, D), prec)[0].reshape(len(rows), H, D)
        O.indexer_topk(qq, kq, w, cu, wl.index_topk, rows=rows)
    dt = time.perf_counter() - t0
    return len(rows) / dt, dt


def run_table(args):
    """Every configuration x precision: GPU score + top-k time (CUDA events,
    median of 5 after 2 warm-ups, L2 flushed before each), queries/s,
    TFLOP/s, % of peak, and the oracle's queries/s on a row sample.  Prints
    a markdown table (not the JSON line)."""
    import torch
    import sparse_attention_indexer_dsa_gb300 as dsa

    torch.cuda.set_device(0)
    devn = torch.device("cuda", 0)
    peaks, peak_kind = load_peaks()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=devn)
    cases = [("tiny", "bf16"), ("c2", "bf16"), ("c3", "mxfp8"), ("c3", "bf16"), ("thd", "mxfp8"),
             ("kpool", "bf16"), ("target", "mxfp8"), ("target", "bf16"), ("target", "fp8")]
    print(f"| config | precision | score+top-k ms | queries/s | TFLOP/s | % of {peak_kind} peak | "
          f"top-k overlap with BF16 (mean / min) | oracle queries/s ({os.cpu_count()} cores, rows) |")
    print("|---|---|---:|---:|---:|---:|---:|---:|")
    fp8_peak, _ = measure_fp8_peak(devn)
    for name, prec in cases:
        wl = W.config(name)
        x = W.make_inputs(wl)
        T, H, D, K = wl.total_tokens, wl.n_heads, wl.head_dim, wl.index_topk
        cu = torch.from_numpy(wl.cu_seqlens).to(devn)
        q = torch.from_numpy(x["q"]).to(devn)
        k = torch.from_numpy(x["k"]).to(devn)
        w = torch.from_numpy(x["w"]).to(devn)
        g = torch.from_numpy(x["ln_gamma"]).to(devn) if wl.layernorm else None
        b = torch.from_numpy(x["ln_beta"]).to(devn) if wl.layernorm else None
        qo, qs, ko, ks = dsa.preprocess(q, k, cu, wl.max_seqlen, g, b, 1e-6, wl.rope_dim, wl.rope_base, False,
                                        True, prec)
        pool = {}
        if wl.kpool > 1:
            gate = torch.from_numpy(x["gate_bits"].view(np.int16)).to(devn)
            ko, cpools = dsa.kpool_compress(k, gate, torch.from_numpy(x["slot_bias"]).to(devn), cu, wl.kpool)
            ks = None
            pool = dict(kpool_size=wl.kpool, cu_pools=cpools, tail=True)
        ws = dsa.workspace(T, len(wl.doc_lens), wl.max_seqlen, H, D, K, wl.kpool, prec, devn)

        def run():
            return dsa.score_topk(qo, qs, ko, ks, w, cu, wl.max_seqlen, H, K, prec, ws=ws, **pool)

        for _ in range(2):
            run()
        ts = []
        for r in range(5):
            flush.fill_(r)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        if dsa.read_status(ws) != 0:
            raise RuntimeError(f"{name} {prec}: device status {dsa.read_status(ws)}")
        ms = statistics.median(ts)
        overlap = "—"
        if prec != "bf16":   # the same inputs scored in BF16: how many of the 8-bit picks agree
            ia, _, la = run()
            qb, _, kb, _ = dsa.preprocess(q, k, cu, wl.max_seqlen, g, b, 1e-6, wl.rope_dim, wl.rope_base, False,
                                          True, "bf16")
            wsb = dsa.workspace(T, len(wl.doc_lens), wl.max_seqlen, H, D, K, wl.kpool, "bf16", devn)
            ib, _, lb = dsa.score_topk(qb, None, kb, None, w, cu, wl.max_seqlen, H, K, "bf16", ws=wsb, **pool)
            mean, mn = topk_overlap(ia, la, ib, lb)
            overlap = f"{mean:.4f} / {mn:.4f}"
            del qb, kb, wsb, ib, lb
        tf = wl.flops() / ms / 1e9
        peak = fp8_peak if prec in ("mxfp8", "fp8") else peaks["bf16_tflops"]
        n_rows = min(T, args.ref_rows // 8 if T > 4096 else 64)
        orate, _ = oracle_rate(wl, x, prec, n_rows)
        print(f"| {describe(wl, prec)} | {prec.upper()} | {ms:.3f} | {T / ms * 1e3:,.0f} | {tf:.1f} | "
              f"{100 * tf / peak:.1f} | {overlap} | {orate:,.1f} ({n_rows}) |", flush=True)
    table_extra_rows(dsa, devn, flush, fp8_peak)
    print(f"\nPeaks: BF16 {peaks['bf16_tflops']:.1f} TFLOP/s ({peak_kind}); FP8 {fp8_peak:.1f} TFLOP/s "
          f"(E4M3 GEMM measured in this run) for the MXFP8 and FP8 rows.", flush=True)


def table_extra_rows(dsa, devn, flush, fp8_peak):
    """Rows for the paths beyond the plain causal one, MXFP8 throughout, timed
    like the table's other rows (no oracle column):
      * KPool (P = 4) with MXFP8 scoring of the pooled keys;
      * caller-provided compressed keys, ratio 4, top-2048 compressed keys;
      * queries that are the last 8192 of 32768 key tokens (global causal
        offsets), top-2048.
    TFLOP/s from the algorithmic 2*H*D per visible (query, key) pair."""
    import torch
    H, D, K = 64, 128, 2048

    def timed(run):
        for _ in range(2):
            run()
        ts = []
        for r in range(5):
            flush.fill_(r)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def row(label, T, ms, pairs):
        tf = 2.0 * H * D * pairs / ms / 1e9
        print(f"| {label} | MXFP8 | {ms:.3f} | {T / ms * 1e3:,.0f} | {tf:.1f} | {100 * tf / fp8_peak:.1f} | — | — |",
              flush=True)

    # KPool with MXFP8 scoring: pooled BF16 keys quantised like every other operand
    wl = W.config("kpool")
    x = W.make_inputs(wl)
    T, P = wl.total_tokens, wl.kpool
    cu = torch.from_numpy(wl.cu_seqlens).to(devn)
    qc, qs = dsa.quantize_mxfp8(torch.from_numpy(x["q"].reshape(T * H, D)).to(devn))
    kp, cp = dsa.kpool_compress(torch.from_numpy(x["k"]).to(devn),
                                torch.from_numpy(x["gate_bits"].view(np.int16)).to(devn),
                                torch.from_numpy(x["slot_bias"]).to(devn), cu, P)
    kc, ks = dsa.quantize_mxfp8(kp)
    w = torch.from_numpy(x["w"]).to(devn)
    ws = dsa.workspace(T, 1, wl.max_seqlen, H, D, wl.index_topk, P, "mxfp8", devn)
    ms = timed(lambda: dsa.score_topk(qc, qs, kc, ks, w, cu, wl.max_seqlen, H, wl.index_topk, "mxfp8", ws=ws,
                                      kpool_size=P, cu_pools=cp, tail=True))
    row(f"kpool: 1×{T}, P = {P}, top-{wl.index_topk // P} pools + tail, pooled keys in MXFP8", T, ms,
        wl.causal_pairs())
    del qc, qs, kp, kc, ks, ws

    # compressed keys, ratio 4: query t sees floor((t+1)/4) compressed keys
    T, r = 32768, 4
    rng = np.random.default_rng(2024)
    qc, qs = dsa.quantize_mxfp8(torch.from_numpy(rng.standard_normal((T * H, D), dtype=np.float32)).to(devn))
    kc, ks = dsa.quantize_mxfp8(torch.from_numpy(rng.standard_normal((T // r, D), dtype=np.float32)).to(devn))
    w = torch.from_numpy((rng.standard_normal((T, H)) * 0.125).astype(np.float32)).to(devn)
    cu = torch.tensor([0, T], dtype=torch.int32, device=devn)
    cc = torch.tensor([0, T // r], dtype=torch.int32, device=devn)
    ws = dsa.workspace(T, 1, T, H, D, K, r, "mxfp8", devn)
    ms = timed(lambda: dsa.score_topk(qc, qs, kc, ks, w, cu, T, H, K, "mxfp8", ws=ws, kpool_size=r, cu_pools=cc,
                                      compressed=True))
    row(f"compressed keys: 1×{T} queries, ratio {r} ({T // r} keys), top-{K}", T, ms,
        sum((t + 1) // r for t in range(T)))
    del qc, qs, kc, ks, ws

    # global causal offsets: the last Tq of S key tokens
    S, Tq = 32768, 8192
    qc, qs = dsa.quantize_mxfp8(torch.from_numpy(rng.standard_normal((Tq * H, D), dtype=np.float32)).to(devn))
    kc, ks = dsa.quantize_mxfp8(torch.from_numpy(rng.standard_normal((S, D), dtype=np.float32)).to(devn))
    w = torch.from_numpy((rng.standard_normal((Tq, H)) * 0.125).astype(np.float32)).to(devn)
    cq = torch.tensor([0, Tq], dtype=torch.int32, device=devn)
    ck = torch.tensor([0, S], dtype=torch.int32, device=devn)
    ws = dsa.workspace(S, 1, S, H, D, K, 1, "mxfp8", devn)
    ms = timed(lambda: dsa.score_topk_kv(qc, qs, kc, ks, w, cq, ck, Tq, S, H, K, "mxfp8", ws=ws))
    row(f"key offsets: the last {Tq} of {S} tokens as queries, top-{K}", Tq, ms,
        sum(S - Tq + i + 1 for i in range(Tq)))


def topk_overlap(idx_a, len_a, idx_b, len_b):
    """Per-row overlap |A & B| / max(|A|, 1) of two top-k outputs in index
    order (device tensors [T, W] and lengths [T]); returns (mean, min).  Rows
    are ascending, so each entry of A is looked up in B by binary search."""
    import torch
    big = torch.iinfo(torch.int32).max
    w = idx_a.shape[1]
    col = torch.arange(w, device=idx_a.device)[None, :]
    a = torch.where(col < len_a[:, None], idx_a, big)
    b = torch.where(col < len_b[:, None], idx_b, big).contiguous()
    pos = torch.searchsorted(b, a.contiguous()).clamp(max=w - 1)
    hit = (torch.gather(b, 1, pos) == a) & (a != big)
    ov = hit.sum(1).double() / len_a.clamp(min=1).double()
    return float(ov.mean()), float(ov.min())


def _median_ms(fn, flush, stream, reps=5, warm=2):
    import torch
    for _ in range(warm):
        fn()
    ts = []
    for r in range(reps):
        flush.fill_(r & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def time_hbm_kernels(dsa, q, T, H, D, flush, stream, peaks):
    """The stand-alone HBM-bound kernels, each timed alone (CUDA events,
    median of 5 after 2 warm-ups, L2 flushed before each): the MXFP8 and
    per-vector FP8 quantisers on the workload's FP32 query rows, and KPool
    compression (P = 4) of a 2^20-token FP32 key set.  GB/s from the
    algorithmic bytes (read once, written once)."""
    import torch
    dev = q.device
    out = {}
    x = q.view(T * H, D)
    codes = torch.empty((T * H, D), dtype=torch.uint8, device=dev)
    s_mx = torch.empty((T * H, D // 32), dtype=torch.uint8, device=dev)
    s_row = torch.empty((T * H,), dtype=torch.uint8, device=dev)
    lib = dsa._abi.load()
    st = stream.cuda_stream

    def mx():
        lib.dsa_idx_quantize_mxfp8(x.data_ptr(), 0, T * H, D, 0, codes.data_ptr(), s_mx.data_ptr(), st)

    def f8():
        lib.dsa_idx_quantize_fp8_rows(x.data_ptr(), 0, T * H, D, 0, codes.data_ptr(), s_row.data_ptr(), st)

    n = T * H * D
    for name, fn, nbytes in (("quantize_mxfp8", mx, n * 4 + n + n // 32), ("quantize_fp8_rows", f8, n * 4 + n + T * H)):
        ms = _median_ms(fn, flush, stream)
        out[name] = {"rows": T * H, "ms": ms, "bytes": nbytes, "GB/s": nbytes / ms / 1e6,
                     "frac_of_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"]}
    del codes, s_mx, s_row
    Tk, P = 1 << 20, 4
    kk = torch.randn((Tk, D), device=dev)
    gate = torch.randn(Tk, device=dev).to(torch.bfloat16).view(torch.int16)
    bias = torch.randn(P, device=dev)
    cuk = torch.tensor([0, Tk], dtype=torch.int32, device=dev)
    nbytes = Tk * D * 4 + Tk * 2 + P * 4 + (Tk // P) * D * 2 + 8
    ms = _median_ms(lambda: dsa.kpool_compress(kk, gate, bias, cuk, P), flush, stream)
    out["kpool_compress"] = {"tokens": Tk, "pool": P, "ms": ms, "bytes": nbytes, "GB/s": nbytes / ms / 1e6,
                             "frac_of_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"]}
    return out


def run_hbm_only(args, wl):
    """The HBM-bound kernels alone on the workload's inputs (preprocess in
    the workload's precision, the stand-alone quantisers, KPool compression):
    one JSON line of GB/s figures.  Used for their ncu captures."""
    import torch
    import sparse_attention_indexer_dsa_gb300 as dsa

    torch.cuda.set_device(0)
    devn = torch.device("cuda", 0)
    peaks, _ = load_peaks()
    x = W.make_inputs(wl)
    T, H, D = wl.total_tokens, wl.n_heads, wl.head_dim
    q = torch.from_numpy(x["q"]).to(devn)
    k = torch.from_numpy(x["k"]).to(devn)
    cu = torch.from_numpy(wl.cu_seqlens).to(devn)
    g = torch.from_numpy(x["ln_gamma"]).to(devn) if wl.layernorm else None
    b = torch.from_numpy(x["ln_beta"]).to(devn) if wl.layernorm else None
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=devn)
    stream = torch.cuda.current_stream()
    prec = "mxfp8" if wl.prec == "bf16" else wl.prec
    outs = dsa.preprocess(q, k, cu, wl.max_seqlen, g, b, 1e-6, wl.rope_dim, wl.rope_base, False, True, prec)
    ms = _median_ms(lambda: dsa.preprocess(q, k, cu, wl.max_seqlen, g, b, 1e-6, wl.rope_dim, wl.rope_base, False,
                                           True, prec, out=outs), flush, stream)
    nb = T * H * D * 4 + T * D * 4 + T * H * D + T * H * D // 32 + T * D + T * D // 32
    line = {"mode": "hbm-kernels", "workload": describe(wl, prec),
            "preprocess": {"ms": ms, "bytes": nb, "GB/s": nb / ms / 1e6, "frac_of_hbm": nb / ms / 1e6 / peaks["hbm_gbs"]}}
    line.update(time_hbm_kernels(dsa, q, T, H, D, flush, stream, peaks))
    print(json.dumps(line), flush=True)


def run_reference(args, wl):
    world, rank, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    x = W.make_inputs(wl)
    n_rows = max(8, args.ref_rows // max(1, args.steps))   # the whole run stays within about a minute
    for _ in range(args.warmup):
        oracle_sample_rate(wl, x, max(1, n_rows // 4), seed=99)
    times, done = [], 0
    for s in range(args.steps):
        _, dt, rows = oracle_sample_rate(wl, x, n_rows, seed=s)
        times.append(dt)
        done += rows
    n_rows = done // args.steps
    value = done / sum(times)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded PCG64)",
        "config": {"workload": describe(wl), "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_rows} query rows per step at seeded uniform positions, plus the "
                                   "key-side LayerNorm/RoPE/quantisation those rows need"},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_native(args, wl):
    import torch
    import sparse_attention_indexer_dsa_gb300 as dsa

    world, rank, local = dist_setup(args.gpus)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    devn = torch.device("cuda", torch.cuda.current_device())
    peaks, peak_kind = load_peaks()
    x = W.make_inputs(wl, seed=wl.seed + rank)
    T, H, D, K = wl.total_tokens, wl.n_heads, wl.head_dim, wl.index_topk
    cu_np = wl.cu_seqlens
    # resident inputs
    q = torch.from_numpy(x["q"]).to(devn)
    k = torch.from_numpy(x["k"]).to(devn)
    w = torch.from_numpy(x["w"]).to(devn)
    g = torch.from_numpy(x["ln_gamma"]).to(devn) if wl.layernorm else None
    b = torch.from_numpy(x["ln_beta"]).to(devn) if wl.layernorm else None
    cu = torch.from_numpy(cu_np).to(devn)
    prec = wl.prec
    ws = dsa.workspace(T, len(wl.doc_lens), wl.max_seqlen, H, D, K, 1, prec, devn)
    q_op = torch.empty((T * H, D), dtype=torch.uint8, device=devn)
    k_op = torch.empty((T, D), dtype=torch.uint8, device=devn)
    q_sc = torch.empty((T * H, D // 32), dtype=torch.uint8, device=devn)
    k_sc = torch.empty((T, D // 32), dtype=torch.uint8, device=devn)
    idx = torch.empty((T, K), dtype=torch.int32, device=devn)
    sco = torch.empty((T, K), dtype=torch.float32, device=devn)
    lens = torch.empty((T,), dtype=torch.int32, device=devn)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=devn)
    stream = torch.cuda.current_stream()

    nvtx = torch.cuda.nvtx   # named ranges for nsys/ncu timelines (no effect without a profiler)

    def pre():
        with nvtx.range("dsa_idx_preprocess"):
            dsa.preprocess(q, k, cu, wl.max_seqlen, g, b, 1e-6, wl.rope_dim, wl.rope_base, False, True,
                           prec, out=(q_op, q_sc, k_op, k_sc))

    def score():
        with nvtx.range("dsa_idx_score_topk"):
            dsa.score_topk(q_op, q_sc, k_op, k_sc, w, cu, wl.max_seqlen, H, K, prec, ws=ws,
                           out=(idx, sco, lens))

    for _ in range(args.warmup):
        pre()
        score()
    torch.cuda.synchronize()
    st = dsa.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(devn.index)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.5)    # nvidia-smi's start-up holds the NVIDIA kernel driver for a moment: keep it out of the timed loop
    t_wall0 = time.perf_counter()
    for s in range(args.steps):
        flush.fill_(s & 0xFF)                      # L2 flush, outside the events
        with nvtx.range(f"step {s}"):
            ev[s][0].record(stream)
            pre()
            ev[s][1].record(stream)
            score()
            ev[s][2].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    pre_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    sc_ms = [ev[s][1].elapsed_time(ev[s][2]) for s in range(args.steps)]
    step_ms = [a + c for a, c in zip(pre_ms, sc_ms)]
    total_ms = sum(step_ms)
    total_ms = reduce_max_over_ranks(total_ms, devn)
    st = dsa.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed steps")

    # end to end through the public API with host buffers (pinned), every step:
    # the host -> device copy of the step's inputs and the device -> host copy
    # of its top-k indices run on two copy streams, overlapping the compute of
    # the neighbouring steps (two device buffer sets, ordered by events)
    hq = torch.from_numpy(x["q"]).pin_memory()
    hk = torch.from_numpy(x["k"]).pin_memory()
    hw = torch.from_numpy(x["w"]).pin_memory()
    hidx = [torch.empty((T, K), dtype=torch.int32).pin_memory() for _ in range(2)]
    hlen = [torch.empty((T,), dtype=torch.int32).pin_memory() for _ in range(2)]
    h2d = hq.numel() * 4 + hk.numel() * 4 + hw.numel() * 4
    d2h = hidx[0].numel() * 4 + hlen[0].numel() * 4
    q2 = [q, torch.empty_like(q)]
    k2 = [k, torch.empty_like(k)]
    w2 = [w, torch.empty_like(w)]
    idx2 = [idx, torch.empty_like(idx)]
    lens2 = [lens, torch.empty_like(lens)]
    s_in, s_out = torch.cuda.Stream(device=devn), torch.cuda.Stream(device=devn)
    in_done = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n, e_start=None):
        if e_start is not None:
            s_in.wait_event(e_start)
            s_out.wait_event(e_start)
        for s in range(n):
            bi = s & 1
            if s >= 2:
                s_in.wait_event(used[bi])        # step s-2 is done with this buffer set
            with torch.cuda.stream(s_in):
                q2[bi].copy_(hq, non_blocking=True)
                k2[bi].copy_(hk, non_blocking=True)
                w2[bi].copy_(hw, non_blocking=True)
                in_done[bi].record(s_in)
            stream.wait_event(in_done[bi])
            if s >= 2:
                stream.wait_event(out_done[bi])  # step s-2's indices are on the host
            dsa.preprocess(q2[bi], k2[bi], cu, wl.max_seqlen, g, b, 1e-6, wl.rope_dim, wl.rope_base, False,
                           True, prec, out=(q_op, q_sc, k_op, k_sc))
            dsa.score_topk(q_op, q_sc, k_op, k_sc, w2[bi], cu, wl.max_seqlen, H, K, prec, ws=ws,
                           out=(idx2[bi], sco, lens2[bi]))
            used[bi].record(stream)
            s_out.wait_event(used[bi])
            with torch.cuda.stream(s_out):
                hidx[bi].copy_(idx2[bi], non_blocking=True)
                hlen[bi].copy_(lens2[bi], non_blocking=True)
                out_done[bi].record(s_out)
        stream.wait_event(out_done[(n - 1) & 1])

    e2e_run(2)                                   # untimed: first use of the copy streams
    torch.cuda.synchronize()
    # as many steps as the device-timed loop: the first step's input copy (the
    # pipeline fill) and the last step's output copy (the drain) cannot overlap
    # any compute and are part of the measurement
    e2e_steps = max(4, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max_over_ranks(e0.elapsed_time(e1) / e2e_steps, devn)
    st = dsa.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the end-to-end steps")

    # optional BF16 scoring of the same workload (score kernel only)
    bf16 = None
    if not args.no_bf16:
        qb = torch.empty((T * H, D), dtype=torch.bfloat16, device=devn)
        kb = torch.empty((T, D), dtype=torch.bfloat16, device=devn)
        dsa.preprocess(q, k, cu, wl.max_seqlen, g, b, 1e-6, wl.rope_dim, wl.rope_base, False, True, "bf16",
                       out=(qb, None, kb, None))
        for _ in range(2):
            dsa.score_topk(qb, None, kb, None, w, cu, wl.max_seqlen, H, K, "bf16", ws=ws, out=(idx, sco, lens))
        bt = []
        for s in range(3):
            flush.fill_(s)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            dsa.score_topk(qb, None, kb, None, w, cu, wl.max_seqlen, H, K, "bf16", ws=ws, out=(idx, sco, lens))
            a1.record(stream)
            torch.cuda.synchronize()
            bt.append(a0.elapsed_time(a1))
        bms = statistics.median(bt)
        bf16 = {"score_ms": bms, "tflops": wl.flops() / bms / 1e9,
                "frac_of_bf16_peak": wl.flops() / bms / 1e9 / peaks["bf16_tflops"],
                "peak_tflops": peaks["bf16_tflops"], "peak_kind": peak_kind}

    hbm_kernels = None if args.no_hbm else time_hbm_kernels(dsa, q, T, H, D, flush, stream, peaks)

    # the ranking-order pass (DSA_FLAG_SORT_BY_SCORE): the same call in score
    # order against index order on the same operands, medians of 5 (L2 flushed)
    ranking = None
    if not args.no_rank:
        def call(order):
            return lambda: dsa.score_topk(q_op, q_sc, k_op, k_sc, w, cu, wl.max_seqlen, H, K, prec, ws=ws,
                                          out=(idx, sco, lens), order=order)
        ms_idx = _median_ms(call("index"), flush, stream)
        ms_score = _median_ms(call("score"), flush, stream)
        rows_bytes = 2 * T * K * 8                      # each row read and written once (index + score)
        extra = ms_score - ms_idx
        ranking = {"index_order_ms": ms_idx, "score_order_ms": ms_score, "ranking_pass_ms": extra,
                   "rows": T, "width": K, "bytes": rows_bytes,
                   "GB/s": rows_bytes / extra / 1e6 if extra > 0 else None}
        st = dsa.read_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {st} after the ranking-order calls")

    if rank != 0:
        return
    flops = wl.flops()
    sc_avg = statistics.mean(sc_ms)
    achieved = flops / sc_avg / 1e9                      # TFLOP/s
    fp8_peak, fp8_src = measure_fp8_peak(devn)
    pre_bytes = T * H * D * 4 + T * D * 4 + T * H * D + T * H * D // 32 + T * D + T * D // 32
    tr = traffic_record()
    value = job_rate(world, T, args.steps, total_ms)
    cpu_rate, cpu_dt, _ = (None, None, None)
    if not args.no_cpu and world == 1:   # the oracle baseline: rank 0 at N = 1 only
        cpu_rate, cpu_dt, _ = oracle_sample_rate(wl, x, args.ref_rows)
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (MXFP8) operands, fp32 accumulate",
        "data": "synthetic (seeded PCG64), resident in HBM",
        "config": {"workload": describe(wl),
                   "global_batch": world * T, "seq_len": T, "l2": "flushed (256 MB write) before every step",
                   "parallelism": f"replicas x{world}"},
        "tflops": achieved, "frac_of_fp8_peak": achieved / fp8_peak,
        "score_topk_ms": sc_avg, "preprocess_ms": statistics.mean(pre_ms),
        "preprocess": {"bytes": pre_bytes, "GB/s": pre_bytes / statistics.mean(pre_ms) / 1e6,
                       "frac_of_hbm": pre_bytes / statistics.mean(pre_ms) / 1e6 / peaks["hbm_gbs"]},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp8_peak,
                     "peak_source": fp8_src,
                     "kernel": "score_topk call (work list + key-scale layout + fused kernel; the fused "
                               "kernel is 99.7 % of it), events on the launch stream",
                     "traffic": tr["bytes_per_launch"] if tr else None,
                     "traffic_source": tr["scaled_to"] if tr else None},
        "bf16_scoring": bf16,
        "hbm_kernels": hbm_kernels,
        "ranking_order": ranking,
        "e2e": {"value": job_rate(world, T, 1, e2e_ms), "unit": "queries/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "path": "pinned host q,k,w -> dsa_idx_preprocess -> dsa_idx_score_topk -> host top-k indices; "
                        "copies on two copy streams overlap the neighbouring steps' compute (two buffer sets); "
                        "the first step's input copy and the last step's output copy are not overlapped"},
        # per step: dsa_idx_preprocess (1 kernel); dsa_idx_score_topk (work list,
        # MXFP8 key-scale layout, fused kernel)
        "gpu_launches": (4 if prec == "mxfp8" else 3) * args.steps,
        "clocks": clk,
        # host clock around the timed loop: the K steps plus the L2 flush before
        # each one (a 256 MB write) and the launch overhead
        "timed_loop_wall_s": t_wall,
        "cpu_baseline": None if cpu_rate is None else {
            "value": cpu_rate, "unit": "queries/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{args.ref_rows} query rows of the target at seeded uniform positions "
                      f"({cpu_dt:.1f} s), plus the key-side preprocessing they need"},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="target")
    ap.add_argument("--ref-rows", type=int, default=3072)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-hbm", action="store_true", help="skip timing the stand-alone HBM-bound kernels")
    ap.add_argument("--no-rank", action="store_true", help="skip timing the ranking-order pass")
    ap.add_argument("--hbm-only", action="store_true",
                    help="time only the HBM-bound kernels on the workload and print their GB/s")
    ap.add_argument("--table", action="store_true",
                    help="time every configuration and print a markdown table instead of the JSON line")
    args = ap.parse_args()
    wl = W.config(args.workload)
    if args.table:
        run_table(args)
    elif args.hbm_only:
        run_hbm_only(args, wl)
    elif args.impl == "reference":
        run_reference(args, wl)
    else:
        run_native(args, wl)


if __name__ == "__main__":
    main()
