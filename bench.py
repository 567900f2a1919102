"""Benchmark: DSA prefill query-tokens/s on one GB300 (or N, as weak-scaling
replicas), with the dominant kernel's roofline fraction and the fp64 oracle
timed on the host cores beside it.

A step is one pass of the whole path over one batch: local metadata for
every CP view, split of q / q_idx / w, then per view the indexer + top-k and
the sparse attention, then the rerange of the outputs.  Inputs are resident
in HBM before the timed region (``value``); ``e2e`` repeats the step through
pinned host buffers with the copies inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--mode in-seq|round-robin|head-tail]
Under torchrun each rank runs its own batch (weak scaling); rank 0 prints
one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "DSA prefill query-tokens/s (indexer+top-k+sparse attn), % of roofline"
UNIT = "query-tokens/s"
DEFAULT_WORKLOAD = W.MIXED_16.name
AUX_WORKLOAD = W.LONG_8K.name
L2_BYTES = 126 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.ALL))
    ap.add_argument("--mode", choices=["in-seq", "round-robin", "head-tail"], default=None)
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--core-only", action="store_true",
                    help="skip the e2e and aux legs (workload sweeps; the default run keeps them)")
    ap.add_argument("--aux-workload", default=AUX_WORKLOAD, choices=sorted(W.ALL),
                    help="workload of the aux legs (byte kernels, NEXT-row variants)")
    ap.add_argument("--unfused", action="store_true",
                    help="split q and rerange the outputs as separate passes instead of in the attention")
    ap.add_argument("--view-streams", type=int, default=2,
                    help="streams the CP views are spread over (their kernels' tails overlap)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------------ work model

def positions(wl):
    """in-request position of every flat token"""
    return np.concatenate([np.arange(n) for n in wl.lengths])


def algorithmic(wl, compress_ratio: int = 1):
    """FLOPs (indexer, attention) and bytes per batch of the a3-a5 core, as
    counted for the roofline: indexer sum over causal pairs of HI*DI*2,
    attention sum over tokens of min(p+1, topk)*H*(D+Dv)*2 (with compressed KV
    at ratio c the keys of position p are its floor((p+1)/c) entries); bytes =
    q, q_idx, w, kv, k_idx read once, output written once, top-k indices
    written and read."""
    n = np.floor((positions(wl).astype(np.float64) + 1) / compress_ratio)
    f_idx = float(np.sum(n) * wl.HI * wl.DI * 2)
    f_att = float(np.sum(np.minimum(n, wl.topk)) * wl.H * (wl.D + wl.Dv) * 2)
    T = wl.num_tokens
    per_tok = (wl.H * wl.D * 2 + wl.HI * wl.DI * 2 + wl.HI * 4 + (wl.D * 2 + wl.DI * 2) / compress_ratio
               + wl.H * wl.Dv * 2 + 2 * wl.topk * 4)
    return f_idx, f_att, float(T * per_tok)


def view_attention_flops(wl, cp, mode):
    """attention FLOPs of each CP view (one kernel launch per view)"""
    p = positions(wl)
    _, tpr = (-(-wl.num_tokens // cp) * cp, -(-wl.num_tokens // cp))
    out = []
    for r in range(cp):
        if mode == W.IN_SEQ_SPLIT:
            g = np.arange(r * tpr, min((r + 1) * tpr, wl.num_tokens))
        elif mode == W.HEAD_TAIL:  # a head chunk of ceil(tpr/2) rows, a tail chunk of floor(tpr/2)
            h, t = (tpr + 1) // 2, tpr // 2
            g = np.concatenate([np.arange(r * h, (r + 1) * h), np.arange(cp * h + (cp - 1 - r) * t, cp * h + (cp - r) * t)])
            g = g[g < wl.num_tokens]
        else:
            g = np.arange(r, wl.num_tokens, cp)
        out.append(float(np.sum(np.minimum(p[g] + 1, wl.topk)) * wl.H * (wl.D + wl.Dv) * 2))
    return out


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ oracle (CPU) arm

def oracle_rows(wl, mode, n_seconds, seed=123, max_rows=None):
    """Time the fp64 oracle on a seeded sample of query rows drawn uniformly
    from all CP views of the workload; returns (rows, seconds, description)."""
    from oracle import dsa_oracle as O
    T = wl.num_tokens
    rng = np.random.default_rng(seed)
    # inputs: the oracle needs every key row but only the sampled query rows
    gen = torch.Generator().manual_seed(wl.seed + 1000)
    kv = torch.randn((T, wl.D), generator=gen).to(torch.bfloat16).to(torch.float64).numpy()
    k_idx = torch.randn((T, wl.DI), generator=gen).to(torch.bfloat16).to(torch.float64).numpy()
    sink = torch.randn(wl.H, generator=gen).numpy().astype(np.float64) if wl.sink else None
    qsl = wl.query_start_loc()
    cp = wl.cp_size
    mds = [O.build_local_metadata(qsl, wl.seq_lens(), cp, r, mode) for r in range(cp)]
    rows, t_total = 0, 0.0
    order = rng.permutation(T)
    for g in order:
        g = int(g)
        q = torch.randn((wl.H, wl.D), generator=gen).to(torch.bfloat16).to(torch.float64).numpy()
        qi = torch.randn((wl.HI, wl.DI), generator=gen).to(torch.bfloat16).to(torch.float64).numpy()
        w = (torch.randn(wl.HI, generator=gen) * wl.w_std).numpy().astype(np.float64)
        r = next(rr for rr in range(cp) if g in mds[rr]["local_token_pos"])
        i = mds[r]["local_token_pos"].index(g)
        t0 = time.perf_counter()
        md = mds[r]
        q_loc = {i: q}
        qi_loc = {i: qi}
        w_loc = {i: w}
        O.view_row(md, i, q_loc, qi_loc, w_loc, kv, k_idx, wl.topk, wl.scale, wl.Dv, sink)
        t_total += time.perf_counter() - t0
        rows += 1
        if t_total >= n_seconds or (max_rows and rows >= max_rows):
            break
    desc = (f"{rows} query rows drawn uniformly from all {cp} views of {wl.name}; per row: indexer over its "
            f"causal keys, top-{wl.topk}, attention of {wl.H} heads, fp64 numpy")
    return rows, t_total, desc


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, wl, mode, rank):
    if rank != 0:
        return
    per_step = []
    rows_total = 0
    for s in range(args.warmup + args.steps):
        rows, secs, desc = oracle_rows(wl, mode, n_seconds=max(2.0, args.cpu_seconds / max(1, args.steps)),
                                       seed=1000 + s)
        if s >= args.warmup:
            per_step.append(secs)
            rows_total += rows
    value = rows_total / sum(per_step)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(per_step),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, mode),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl, mode):
    return {"workload": wl.name, "lengths": list(wl.lengths) if len(wl.lengths) <= 16 else len(wl.lengths),
            "num_tokens": wl.num_tokens, "cp_size": wl.cp_size, "mode": W.MODE_NAMES[mode], "heads": wl.H,
            "latent_dim": wl.D, "value_dim": wl.Dv, "indexer_heads": wl.HI, "indexer_dim": wl.DI, "topk": wl.topk,
            "sink": wl.sink, "l2": "flushed between steps (256 MiB write) and per-step inputs > L2"}


# ------------------------------------------------------------------ GPU arm

def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def default_mode(wl):
    """The split mode a workload is benched in: round-robin where the workload
    lists it (the pages' load-balanced split), else its first mode."""
    return W.ROUND_ROBIN if W.ROUND_ROBIN in wl.modes else wl.modes[0]


def e2e_leg(args, wl, mode, dev, x, pk):
    """End to end from page-locked host buffers through the public calls
    (HostStreamedPrefill: per view, the copy engines take its rows of q and
    q_idx up while earlier views compute and bring finished views' outputs
    back into token order), every batch's copies inside the timed region; and
    the same copies on their own, timed the same way (what bounds it)."""
    import sparse_attention_prefill_cp_gb300 as dsa
    from sparse_attention_prefill_cp_gb300.pipeline import HostStreamedPrefill

    host = {}
    for k, v in x.items():
        if v is None:
            host[k] = None
            continue
        h = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
        h.copy_(v)
        host[k] = h
    out_host = torch.empty((wl.num_tokens, wl.H, wl.Dv), dtype=torch.bfloat16, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = out_host.numel() * out_host.element_size()
    streamed = HostStreamedPrefill(wl.lengths, wl.cp_size, mode, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale,
                                   dev, depth=3)
    for _ in range(2):  # warm-up
        streamed.submit(host, out_host)
    torch.cuda.synchronize()
    n = max(2, args.e2e_steps)
    e0 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(streamed.h2d)
    for _ in range(n):
        last = streamed.submit(host, out_host)
    e1 = streamed.done_event(last)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n
    dsa.dsa_poll_device_error()

    # the same bytes through the copy engines alone, on the same two copy
    # streams: full-token inputs, then per chunk its q, q_idx and w rows up
    # and its output rows down (a chunk's read-back after its upload)
    full = {k: torch.empty_like(x[k]) for k in ("kv", "k_idx")}
    qc, qic, wc, oc = streamed.q_c[0], streamed.qi_c[0], streamed.w_c[0], streamed.out_c[0]
    up, down = streamed.h2d, streamed.d2h

    def copies():
        with torch.cuda.stream(up):
            for k, t in full.items():
                t.copy_(host[k], non_blocking=True)
        for (t0, t1) in streamed.chunks:
            n = t1 - t0
            with torch.cuda.stream(up):
                qc[:n].copy_(host["q"][t0:t1], non_blocking=True)
                qic[:n].copy_(host["q_idx"][t0:t1], non_blocking=True)
                wc[:n].copy_(host["w"][t0:t1], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(up)
            down.wait_event(ev)
            with torch.cuda.stream(down):
                out_host[t0:t1].copy_(oc[:n], non_blocking=True)

    copies()
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(up)
    for _ in range(n):
        copies()
    down.wait_stream(up)
    c1.record(down)
    torch.cuda.synchronize()
    copy_ms = c0.elapsed_time(c1) / n
    chunk_tokens, n_chunks = streamed.chunk_tokens, len(streamed.chunks)
    del streamed, full, host, out_host
    torch.cuda.empty_cache()
    return {
        "value": wl.num_tokens / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
        "ms_per_step": e2e_ms, "batches": n,
        "how": "page-locked host inputs -> device -> output back to page-locked host, every batch: full-token inputs "
               "(kv, k_idx, sink) up first, then the token stream in chunks of contiguous rows: a chunk's q, q_idx "
               "and w go up while earlier chunks compute (every view's slots in the chunk: dsa_indexer_topk_rows, "
               "dsa_sparse_attn_prefill_rows) and its output rows come back; HostStreamedPrefill, 3 chunk buffer "
               "sets, views over 2 compute streams",
        "chunk_tokens": chunk_tokens, "chunks_per_batch": n_chunks,
        "copies_only_ms_per_step": copy_ms,
        "copies_gbs": (h2d + d2h) / (copy_ms / 1e3) / 1e9,
    }


def aux_legs(args, wl, mode, dev, pk):
    """Byte-moving steps and the NEXT-row variants, each timed on its own
    (cold L2, outside the timed step) on ``wl``."""
    import sparse_attention_prefill_cp_gb300 as dsa
    from sparse_attention_prefill_cp_gb300.pipeline import DSAPrefill

    x = W.draw_inputs(wl, device=dev)
    pipe = DSAPrefill(wl.lengths, wl.cp_size, mode, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale, dev,
                      view_streams=args.view_streams, fused=True)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def timed(fn, reps=5):
        fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def step():
        return pipe.run(x["q"], x["kv"], x["q_idx"], x["k_idx"], x["w"], x["sink"])

    def fused_core():
        hs = pipe._head_sharded_buffer()
        for r in range(wl.cp_size):
            dsa.dsa_indexer_topk(pipe.md[r], pipe.qi_split[r], x["k_idx"], pipe.w_split[r], pipe.topk,
                                 pipe.max_kv_len, pipe.topk_idx[r], pipe.workspace)
            dsa.dsa_sparse_attn_prefill_headsharded(pipe.md[r], pipe.q_split[r], x["kv"], pipe.topk_idx[r],
                                                    pipe.scale, pipe.Dv, wl.cp_size, hs, x["sink"])

    step()
    T, pad = wl.num_tokens, pipe.pad
    split_bytes = (T + pad) * (wl.H * wl.D * 2 + wl.HI * wl.DI * 2 + wl.HI * 4)
    out_bytes = 2 * T * wl.H * wl.Dv * 2
    aux = {"workload": wl.name, "mode": W.MODE_NAMES[mode]}

    def split_all():  # a2 as its own pass, q included
        for t, dst in ((x["q"], pipe.q_split), (x["q_idx"], pipe.qi_split), (x["w"], pipe.w_split)):
            dsa.dsa_cp_split(t, wl.cp_size, mode, -1, dst)

    for name, fn, nbytes in (("a2_split", split_all, split_bytes),
                             ("a6_rerange", lambda: dsa.dsa_cp_rerange(pipe.out_split, wl.num_tokens, wl.cp_size, mode,
                                                                       pipe.out), out_bytes),
                             ("a2a_heads", pipe.all_to_all_heads, out_bytes)):
        ms = timed(fn)
        aux[name] = {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms / 1e3) / 1e9,
                     "frac_hbm": nbytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"]}
    aux["a3_a5_headsharded_ms"] = timed(fused_core, reps=3)
    aux["a1_metadata_ms"] = timed(pipe.metadata)  # every view's build_cp_local_metadata

    # compressed KV: the same queries over floor(T / c) compressed entries
    # (the first rows of kv and k_idx stand for them), the a3-a5 core timed
    # with its metadata, against the roofline of its own work
    for c in (4, 128):
        rows = wl.num_tokens // c
        pc = DSAPrefill(wl.lengths, wl.cp_size, mode, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale, dev,
                        view_streams=args.view_streams, fused=True, compress_ratio=c)
        pc.run(x["q"], x["kv"][:rows], x["q_idx"], x["k_idx"][:rows], x["w"], x["sink"])

        def core_c(pc=pc, rows=rows):
            pc.metadata()
            pc._q = x["q"]
            pc.views(x["kv"][:rows], x["k_idx"][:rows], x["sink"], torch.cuda.current_stream())

        ms = timed(core_c, reps=3)
        fi, fa, by = algorithmic(wl, c)
        roof_c = max((fi + fa) / (pk["bf16_tflops"] * 1e12), by / (pk["hbm_gbs"] * 1e9))
        aux[f"a3_a5_compressed_c{c}"] = {"ms": ms, "flops": fi + fa, "roofline_frac": roof_c / (ms / 1e3)}
        del pc
    # FP8 latent-KV cache: quantise / dequantise as HBM passes (bytes read +
    # written), and the a3-a5 core over the cache (dequantisation + views)
    cache = dsa.dsa_kv_fp8_quantize(x["kv"], wl.Dv)
    kv_rows = torch.empty_like(x["kv"])
    fp8_bytes = x["kv"].shape[0] * (wl.D * 2 + cache.shape[1])
    for name, fn in (("kv_fp8_quantize", lambda: dsa.dsa_kv_fp8_quantize(x["kv"], wl.Dv, cache)),
                     ("kv_fp8_dequantize", lambda: dsa.dsa_kv_fp8_dequantize(cache, wl.D, wl.Dv, kv_rows))):
        ms = timed(fn)
        aux[name] = {"ms": ms, "bytes": fp8_bytes, "gbs": fp8_bytes / (ms / 1e3) / 1e9,
                     "frac_hbm": fp8_bytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"]}

    # the same two passes over 2^20 rows (1.2 GB of bf16 rows): long enough to
    # run at HBM rate (the workload's own KV is too small for that)
    big_kv = torch.randn((1 << 20, wl.D), device=dev).to(torch.bfloat16)
    big_cache = dsa.dsa_kv_fp8_quantize(big_kv, wl.Dv)
    big_rows = torch.empty_like(big_kv)
    big_bytes = big_kv.shape[0] * (wl.D * 2 + big_cache.shape[1])
    for name, fn in (("kv_fp8_quantize_1M_rows", lambda: dsa.dsa_kv_fp8_quantize(big_kv, wl.Dv, big_cache)),
                     ("kv_fp8_dequantize_1M_rows", lambda: dsa.dsa_kv_fp8_dequantize(big_cache, wl.D, wl.Dv, big_rows))):
        ms = timed(fn)
        aux[name] = {"ms": ms, "bytes": big_bytes, "gbs": big_bytes / (ms / 1e3) / 1e9,
                     "frac_hbm": big_bytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"]}
    del big_kv, big_cache, big_rows

    def fp8_core():
        rows = dsa.dsa_kv_fp8_dequantize(cache, wl.D, wl.Dv, kv_rows)
        pipe.views(rows, x["k_idx"], x["sink"], torch.cuda.current_stream())

    pipe._q = x["q"]
    aux["a3_a5_fp8kv_ms"] = timed(fp8_core, reps=3)
    # the same core with the attention reading the cache itself (its gather
    # dequantises the selected rows; no bf16 copy of the rows)
    pd = DSAPrefill(wl.lengths, wl.cp_size, mode, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale, dev,
                    view_streams=args.view_streams, fused=True, kv_fp8=True, kv_fp8_direct=True)
    pd.run(x["q"], cache, x["q_idx"], x["k_idx"], x["w"], x["sink"])

    def fp8_direct_core():
        pd._q = x["q"]
        pd.views(cache, x["k_idx"], x["sink"], torch.cuda.current_stream())

    aux["a3_a5_fp8kv_direct_ms"] = timed(fp8_direct_core, reps=3)
    del pd
    # FP8 index rows: q_I and k_I quantised (HBM passes, bytes read + written),
    # and the a3-a5 core with the indexer over them beside the same core over
    # bf16 index rows, timed the same way
    q8, k8 = dsa.dsa_indexer_fp8_rows(x["q_idx"]), dsa.dsa_indexer_fp8_rows(x["k_idx"])
    idx8_bytes = x["q_idx"].numel() * 2 + q8.numel() + x["k_idx"].numel() * 2 + k8.numel()
    ms = timed(lambda: (dsa.dsa_indexer_fp8_rows(x["q_idx"], q8), dsa.dsa_indexer_fp8_rows(x["k_idx"], k8)))
    aux["index_fp8_quantize"] = {"ms": ms, "bytes": idx8_bytes, "gbs": idx8_bytes / (ms / 1e3) / 1e9,
                                 "frac_hbm": idx8_bytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"]}
    p8 = DSAPrefill(wl.lengths, wl.cp_size, mode, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale, dev,
                    view_streams=args.view_streams, fused=True, index_fp8=True)
    p8.run(x["q"], x["kv"], q8, k8, x["w"], x["sink"])
    aux["a3_a5_fp8index_ms"] = timed(lambda: p8.views(x["kv"], k8, x["sink"], torch.cuda.current_stream()), reps=3)
    pipe._q = x["q"]
    aux["a3_a5_bf16index_ms"] = timed(lambda: pipe.views(x["kv"], x["k_idx"], x["sink"],
                                                         torch.cuda.current_stream()), reps=3)
    del p8

    # sliding window (W = 128 original rows under the same softmax): the a3-a5
    # core with dsa_swa_index and the attention over the extended rows (view
    # layout), against the roofline of its own work
    window = 128
    pw = DSAPrefill(wl.lengths, wl.cp_size, mode, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale, dev,
                    view_streams=args.view_streams, window=window)
    pw.run(x["q"], x["kv"], x["q_idx"], x["k_idx"], x["w"], x["sink"])
    dsa.dsa_cp_split(x["q"], wl.cp_size, mode, -1, pw.q_split)
    ms = timed(lambda: pw.views(x["kv"], x["k_idx"], x["sink"], torch.cuda.current_stream()), reps=3)
    cnt = pw.ext_counts.float().sum().item()  # rows the attention of every view covers
    fi, _, by = algorithmic(wl)
    fa_w = cnt * wl.H * (wl.D + wl.Dv) * 2
    roof_w = max((fi + fa_w) / (pk["bf16_tflops"] * 1e12), by / (pk["hbm_gbs"] * 1e9))
    aux[f"a3_a5_swa_w{window}"] = {"ms": ms, "flops": fi + fa_w, "roofline_frac": roof_w / (ms / 1e3)}
    del pw

    def unfused_step():  # the whole step with the split of q and the rerange as passes of their own
        pipe.fused = False
        try:
            step()
        finally:
            pipe.fused = True

    aux["step_unfused_ms"] = timed(unfused_step, reps=3)
    aux["note"] = ("a2a_heads: all views' [tpr][H][Dv] outputs -> [cp][T][H/cp][Dv] head-sharded; "
                   "a3_a5_headsharded_ms: the core with that permutation fused into the attention stores; "
                   "kv_fp8_*: the FP8 latent-KV cache (E4M3, per-128-column scales, bf16 rope); "
                   "a3_a5_fp8kv_ms: the core over that cache (one dequantisation, then the views); "
                   "a3_a5_fp8kv_direct_ms: the core with the attention reading the cache; "
                   "step_unfused_ms: a whole step with a2 (q) and a6 as passes of their own; "
                   "a1_metadata_ms: every view's metadata (one launch per view); "
                   "a3_a5_compressed_c*: metadata + core over compressed KV at ratio c (T / c entries); "
                   "index_fp8_quantize: q_I and k_I to FP8 index rows; a3_a5_fp8index_ms / a3_a5_bf16index_ms: "
                   "the core with the indexer over FP8 / bf16 index rows; a3_a5_swa_w128: the core with a "
                   "128-row sliding window over the original KV (extended rows, view layout)")
    dsa.dsa_poll_device_error()
    del pipe, x
    torch.cuda.empty_cache()
    return aux


def run_ours(args, wl, mode, rank, world):
    import sparse_attention_prefill_cp_gb300 as dsa
    from sparse_attention_prefill_cp_gb300.pipeline import DSAPrefill

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dsa.load()
    x = W.draw_inputs(wl, device=dev, seed_offset=rank)
    fused = not args.unfused
    pipe = DSAPrefill(wl.lengths, wl.cp_size, mode, wl.H, wl.D, wl.Dv, wl.HI, wl.DI, wl.topk, wl.scale, dev,
                      view_streams=args.view_streams, fused=fused)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    # attention launches timed live with events on the launching stream
    attn_events = []

    def step(events=None):
        return pipe.run(x["q"], x["kv"], x["q_idx"], x["k_idx"], x["w"], x["sink"], events=events)

    for _ in range(args.warmup):
        step()
    dsa.dsa_poll_device_error()

    def timed_steps(n, record_attention):
        pipe.attention_events = attn_events if record_attention else None
        evs = []
        for _ in range(n):
            flush.zero_()  # evict L2 between steps (outside the timed events)
            ev = {k: torch.cuda.Event(enable_timing=True) for k in ("start", "core_start", "core_end", "end")}
            step(ev)
            evs.append(ev)
        torch.cuda.synchronize()
        pipe.attention_events = None
        return ([ev["start"].elapsed_time(ev["end"]) for ev in evs],
                [ev["core_start"].elapsed_time(ev["core_end"]) for ev in evs])

    sampler = ClockSampler(dev.index) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # the timed steps (the bench value), views spread over --view-streams streams
    step_ms, core_ms = timed_steps(args.steps, record_attention=pipe.view_streams == 1)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    dsa.dsa_poll_device_error()
    t_rank = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    # With several view streams the attention launches share SMs with the next
    # view's indexer, so their event times do not describe the kernel: its
    # launches are then timed in a second pass of the same steps on one stream.
    core_ms_one_stream = None
    if pipe.view_streams > 1:
        n_streams = pipe.view_streams
        pipe.view_streams = 1
        _, core_ms_one_stream = timed_steps(args.steps, record_attention=True)
        pipe.view_streams = n_streams
        dsa.dsa_poll_device_error()

    # dominant kernel: the attention launches
    per_view_flops = view_attention_flops(wl, wl.cp_size, mode)
    attn_ms = [e0.elapsed_time(e1) for (_, e0, e1) in attn_events]
    per_view = [statistics.mean([e0.elapsed_time(e1) for (rr, e0, e1) in attn_events if rr == r])
                for r in range(wl.cp_size)]
    attn_flops = [per_view_flops[r] for (r, _, _) in attn_events]
    pk = peaks()
    achieved = (sum(attn_flops) / (sum(attn_ms) / 1e3)) / 1e12
    launches = pipe.launches_per_step() * args.steps
    core_region_s = sum(core_ms_one_stream or core_ms) / 1e3

    e2e = aux = None
    if not args.core_only:
        del pipe, flush
        torch.cuda.empty_cache()
        e2e = e2e_leg(args, wl, mode, dev, x, pk)
        del x
        torch.cuda.empty_cache()
        wl_aux = W.ALL[args.aux_workload]
        aux = aux_legs(args, wl_aux, default_mode(wl_aux), dev, pk)

    if rank != 0:
        return
    f_idx, f_att, bytes_core = algorithmic(wl)
    total_tokens = world * args.steps * wl.num_tokens
    value = total_tokens / t_rank
    burst, sustained = pk["bf16_tflops"], pk["bf16_tflops_sustained"]
    roof_s = max((f_idx + f_att) / (burst * 1e12), bytes_core / (pk["hbm_gbs"] * 1e9))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_rank / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 inputs, shapes of the workload)",
        "config": dict(config_of(wl, mode), view_streams=args.view_streams, fused_split_rerange=fused),
        "roofline": {"bound": "tensor", "kernel": "sparse_attn_kernel", "achieved": achieved,
                     "peak": burst, "unit": "TFLOP/s", "frac": achieved / burst,
                     "peak_source": f"{pk['source']} bf16 burst (cuBLAS, MEASURED_PEAKS.json bf16_tflops)",
                     "frac_of_sustained_peak": achieved / sustained,
                     "traffic": None,
                     "traffic_note": "DRAM bytes per launch are taken by ncu on a smaller capture (profiles/)",
                     "launch_ms": statistics.mean(attn_ms), "flops_per_launch": statistics.mean(attn_flops),
                     "launches": len(attn_ms), "timed_region_s": core_region_s,
                     "launches_timed": ("in the timed steps" if core_ms_one_stream is None else
                                        "in a second pass of the same steps with the views on one stream")},
        "core": {"what": "a3-a5 (indexer + top-k + sparse attention, all views)",
                 "ms_per_step": statistics.mean(core_ms), "value": wl.num_tokens / (statistics.mean(core_ms) / 1e3),
                 "roofline_frac": roof_s / (statistics.mean(core_ms) / 1e3),
                 "roofline_ms": roof_s * 1e3, "flops": f_idx + f_att, "flops_indexer": f_idx, "flops_attention": f_att,
                 "peak": "bf16 burst",
                 "view_streams": args.view_streams,
                 "ms_per_step_one_stream": (statistics.mean(core_ms_one_stream) if core_ms_one_stream else None)},
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": launches,
        "aux": aux,
        "views": {"attn_ms": per_view, "max_over_mean": max(per_view) / statistics.mean(per_view),
                  "note": "attention time of each CP view; on one GPU per rank the slowest sets the pace"},
    }
    if not args.no_cpu_baseline:
        rows, secs, desc = oracle_rows(wl, mode, n_seconds=args.cpu_seconds)
        line["cpu_baseline"] = {"value": rows / secs, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    wl = W.ALL[args.workload]
    mode = default_mode(wl) if args.mode is None else {"in-seq": W.IN_SEQ_SPLIT, "round-robin": W.ROUND_ROBIN,
                                                        "head-tail": W.HEAD_TAIL}[args.mode]
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, wl, mode, rank)
        else:
            run_ours(args, wl, mode, rank, world)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
