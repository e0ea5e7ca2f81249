"""Benchmark: segmented paged prefill at 128K over 64 layers, and ragged decode.

One step = one pass of the hot path over a 131072-token sequence through 64
layers (64 query / 8 KV heads, D=128, pages of 128): per layer, append K/V
into the segments (local heads keep only their window), prefill attention for
all 131072 positions, then trim the local heads to what decoding needs.
value = useful (kept-key) FLOPs per step / step time. The ragged-decode
workload (32 requests, 2K-32K log-uniform contexts, one token appended per
request per step) is measured alongside and reported as GB/s of algorithmic
K/V bytes.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SegPaged prefill ms & useful TFLOP/s at 128K (1 GB300); decode GB/s vs HBM peak"
UNIT = "TFLOP/s"
N_INPUT_SETS = 4
# DRAM read+write bytes per prefill launch of the 64-layer step, weighted by
# layer kind, from one one-pass ncu capture of the current prefill kernel on
# full-size layers (--case prefill-128k-layers); None once the kernel changes.
PREFILL_TRAFFIC_PER_LAUNCH = 5.05e9


def useful_flops_layer(w, layer, n):
    """4*D * sum over query heads and positions of |visible keys|."""
    W = w.window[layer]
    G = w.group
    tot = 0
    for h in range(w.hkv):
        if w.head_class[layer][h] == 0:
            keys = n * (n + 1) // 2
        else:
            m = min(n, W)
            keys = m * (m + 1) // 2 + (n - m) * W
        tot += G * keys
    return 4 * w.head_dim * tot


def decode_bytes(w, lens):
    """Kept K/V bytes the decode step must read, plus q and o."""
    W = w.window[0]
    b = 0
    for n in lens:
        for h in range(w.hkv):
            keys = n if w.head_class[0][h] == 0 else min(n, W)
            b += keys * w.head_dim * 2 * 2
    b += 2 * len(lens) * w.hq * w.head_dim * 2
    return b


class Clocks:
    """nvidia-smi sampling during a timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7:
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
                except ValueError:
                    pass
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i] == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(value, world, device=None):
    """The largest of every rank's value (one all-reduce; the value itself on
    one rank). The step time of N replicas is the slowest rank's."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replicas_value(units_per_rank, world, ms_per_step):
    """Whole-job throughput of N independent replicas: all ranks' units over
    the slowest rank's time, in units per microsecond (TFLOP/s for FLOPs)."""
    return world * units_per_rank / (ms_per_step * 1e-3) / 1e12


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), \
            d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world):
    import numpy as np
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    w = I.long_128k_64layer(seed=0)
    n = w.seq_lens[0]
    L, hq, hkv, D, P = w.num_layers, w.hq, w.hkv, w.head_dim, w.page_size

    # seeded inputs, generated on the device; layer l uses set l % N_INPUT_SETS
    sets = []
    for s in range(N_INPUT_SETS):
        q = I.normal_bf16(w.seed, I.tensor_stream(I._Q, s), (n, hq, D), device=dev)
        k = I.normal_bf16(w.seed, I.tensor_stream(I._K, s), (n, hkv, D), device=dev)
        v = I.normal_bf16(w.seed, I.tensor_stream(I._V, s), (n, hkv, D), device=dev)
        sets.append((q, k, v))
    cu = np.array([0, n], np.int32)
    q_pos = np.arange(n, dtype=np.int32)
    o = torch.empty((n, hq, D), dtype=torch.bfloat16, device=dev)

    # pool: every global head of every layer keeps 1024 pages; local heads keep
    # the whole layer until its trim, then about W/P + 1 pages
    pages_per_head = n // P
    n_glob = sum(sum(1 for c in w.head_class[l] if c == 0) for l in range(L))
    num_pages = n_glob * pages_per_head + (L * hkv) * (4096 // P + 2) + hkv * pages_per_head + 64
    kp = torch.empty((num_pages, P, D), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    h = S.SegKV(L, hq, hkv, D, w.head_class, w.window, P, 1, n, kp, vp)
    flops = [useful_flops_layer(w, l, n) for l in range(L)]
    step_flops = sum(flops)

    ev_pf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(L)]
    ev_ap = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(L)]

    def step(timed):
        h.free_seq(0)
        for l in range(L):
            q, k, v = sets[l % N_INPUT_SETS]
            if timed:
                ev_ap[l][0].record(stream)
            h.append(l, k, v, cu, [0], stream)
            if timed:
                ev_ap[l][1].record(stream)
                ev_pf[l][0].record(stream)
            h.prefill_attn(l, q, cu, q_pos, [0], o, None, stream)
            if timed:
                ev_pf[l][1].record(stream)
            h.trim(l, [0])

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    if h.status() != 0:
        raise RuntimeError("device status after warm-up: " + S.segkv_last_error(h.handle))

    clk = Clocks(dev.index)
    clk.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    pf_ms, ap_ms = [], []
    t0.record(stream)
    for _ in range(args.steps):
        step(True)
        torch.cuda.synchronize()
        pf_ms.append(sum(a.elapsed_time(b) for a, b in ev_pf))
        ap_ms.append(sum(a.elapsed_time(b) for a, b in ev_ap))
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    if h.status() != 0:
        raise RuntimeError("device status after timed steps: " + S.segkv_last_error(h.handle))
    ms_step = total_ms / args.steps
    prefill_ms = statistics.median(pf_ms)
    append_ms = statistics.median(ap_ms)
    value = replicas_value(step_flops, world, ms_step)

    hbm, bf16_burst, bf16_sus, peak_src = measured_peaks()
    achieved = step_flops / (prefill_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": bf16_sus,
                "unit": "TFLOP/s", "frac": round(achieved / bf16_sus, 4),
                "peak_kind": f"bf16 sustained ({peak_src}); kernel runs inside a ~{ms_step:.0f} ms step",
                "frac_of_burst": round(achieved / bf16_burst, 4),
                "kernel": "prefill_kernel<128>", "per_launch_flops_mean": step_flops / L,
                "traffic": PREFILL_TRAFFIC_PER_LAUNCH,
                "traffic_note": "DRAM read+write bytes per launch (ncu, full-size layers weighted by "
                                "kind); algorithmic bytes per launch are 4.83e9"}

    out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic: seeded splitmix64 + Box-Muller N(0,1), rounded to bf16",
           "config": {"workload": "128k-64layer prefill", "layers": L, "hq": hq, "hkv": hkv,
                      "head_dim": D, "page_size": P, "context": n,
                      "global_kv_heads_total": n_glob, "input_sets": N_INPUT_SETS,
                      "l2": "inputs larger than L2 (Q is 2 GiB per layer); no flush",
                      "parallelism": "replicas" if world > 1 else "single GPU"},
           "prefill_ms": round(prefill_ms, 3), "append_ms": round(append_ms, 3),
           "useful_tflop_per_step": round(step_flops / 1e12, 3),
           "prefill_useful_tflops": round(achieved, 2),
           "roofline": roofline, "clocks": clocks,
           # per layer: append and prefill, each after a plan-copy kernel (both plans
           # travel through the upload ring at this size)
           "gpu_launches": 4 * L * args.steps}

    del h
    torch.cuda.synchronize()
    cpu = rank == 0 and not args.no_cpu
    if not args.no_e2e:
        out["e2e"] = run_e2e(args, dev, stream, w, sets, cu, q_pos, step_flops, num_pages)
    if cpu:
        out["cpu_baseline"] = cpu_baseline(sets, w, budget_s=args.cpu_seconds)
    if not args.no_decode:
        out["rope_shift"] = run_rope(dev, stream, hbm)
        out["pd_transfer"] = run_transfer(dev, stream, hbm)
        out["sparse_ffn_routing"] = run_routing(dev, stream, bf16_burst, peak_src)
        out["prefill_configs"] = run_prefill_configs(dev, stream, bf16_burst, peak_src, cpu=cpu)
    if not args.no_dense:
        out["dense"] = run_dense(args, dev, stream, sets, cu, q_pos, o, prefill_ms)
        out["context_sweep"] = run_context_sweep(dev, stream, sets)
    if not args.no_decode:
        out["decode"] = run_decode(args, dev, stream, hbm, peak_src, cpu=cpu)
    out["summary"] = summary(out, bf16_burst, bf16_sus, hbm)
    return out


def summary(out, bf16_burst, bf16_sus, hbm):
    """The headline figures of every workload in one short object, printed
    last in the JSON line."""
    r = out["roofline"]
    sm = {"128k_64layer": {"prefill_s": round(out["prefill_ms"] / 1e3, 4),
                           "tflops": r["achieved"], "frac_sustained": r["frac"],
                           "frac_burst": r["frac_of_burst"]}}
    if "cpu_baseline" in out:
        sm["128k_64layer"]["cpu_oracle_tflops"] = round(out["cpu_baseline"]["value"], 4)
        sm["cpu_cores"] = out["cpu_baseline"]["cores"]
    for name, d in out.get("prefill_configs", {}).items():
        if not isinstance(d, dict):
            continue
        e = {"ms": d["prefill_ms"], "tflops": d["useful_tflops"], "frac_burst": d["frac_of_burst"]}
        if "cpu_oracle" in d:
            e["cpu_oracle_ms"] = d["cpu_oracle"]["ms_full_layer"]
            e["cpu_oracle_tflops"] = d["cpu_oracle"]["tflops"]
        sm[name] = e
    if "decode" in out:
        d = out["decode"]
        sm["ragged_decode"] = {"us": d["decode_us_median"], "gbs": d["gbs_median"],
                               "frac_hbm": d["frac"], "back_to_back_gbs": d["back_to_back_gbs"],
                               "back_to_back_frac": d["back_to_back_frac"],
                               "step_us_with_append": d["step_us_median"],
                               "tokens_per_s": d["tokens_per_s"],
                               "multi_query_t4_frac": d["multi_query_t4"]["frac"]}
        if "cpu_oracle" in d:
            sm["ragged_decode"]["cpu_oracle_gbs"] = d["cpu_oracle"]["gbs"]
    if "dense" in out:
        sm["dense_speedup_128k_64layer"] = out["dense"]["speedup_segpaged_vs_dense"]
    if "context_sweep" in out:
        c = out["context_sweep"]
        sm["speedup_vs_context"] = {"n": c["n"], "shallow": c["shallow"]["speedup_vs_dense"],
                                    "deep_g1": c["deep_g1"]["speedup_vs_dense"],
                                    "monotone": c["shallow"]["monotone"] and c["deep_g1"]["monotone"]}
    if "e2e" in out:
        sm["e2e_tflops"] = out["e2e"]["value"]
    if "rope_shift" in out:
        sm["rope_frac_hbm"] = out["rope_shift"]["frac_hbm"]
        sm["transfer_gbs"] = {"export": out["pd_transfer"]["export_gbs"],
                              "import": out["pd_transfer"]["import_gbs"]}
        sm["sparse_ffn_frac_burst"] = out["sparse_ffn_routing"]["roofline_ffn"]["frac"]
    return sm


def run_dense(args, dev, stream, sets, cu, q_pos, o, sparse_prefill_ms):
    """The same library with every head global (full causal), on 4 layers;
    layers are identical, so the 64-layer time is 16x theirs."""
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    w = I.long_128k_64layer(seed=0, all_global=True)
    n, P, D = w.seq_lens[0], w.page_size, w.head_dim
    Ld = 4
    kp = torch.empty((w.hkv * (n // P) + 8, P, D), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    h = S.SegKV(Ld, w.hq, w.hkv, D, w.head_class[:Ld], w.window[:Ld], P, 1, n, kp, vp)
    flops = useful_flops_layer(w, 0, n)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Ld)]
    # warm-up one layer
    q, k, v = sets[0]
    h.append(0, k, v, cu, [0], stream)
    h.prefill_attn(0, q, cu, q_pos, [0], o, None, stream)
    h.free_seq(0)
    torch.cuda.synchronize()
    for l in range(Ld):
        q, k, v = sets[l % len(sets)]
        h.append(l, k, v, cu, [0], stream)
        evs[l][0].record(stream)
        h.prefill_attn(l, q, cu, q_pos, [0], o, None, stream)
        evs[l][1].record(stream)
        h.free_seq(0)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    per_layer = statistics.median(ms)
    return {"layers_timed": Ld, "prefill_ms_per_layer": round(per_layer, 3),
            "prefill_ms_64_layers_extrapolated": round(per_layer * 64, 1),
            "useful_tflops": round(flops / (per_layer * 1e-3) / 1e12, 2),
            "speedup_segpaged_vs_dense": round(per_layer * 64 / sparse_prefill_ms, 2),
            "note": "all heads global, full causal; 4 identical layers timed, x16"}


def oracle_decode_timing(w, k, v, cu, step0):
    """Time the fp64 oracle on one whole decode step of the ragged-decode
    workload (every request and query head: step 0's token attending to its
    context plus itself) and report it in the GPU path's unit, GB/s of
    algorithmic K/V bytes."""
    import numpy as np
    import torch

    import oracle

    qq, kk, vv = (t.cpu() for t in step0)
    B = len(w.seq_lens)
    cu = np.asarray(cu, np.int64)
    ks, vs = [], []
    for b in range(B):
        ks += [k[cu[b]:cu[b + 1]].cpu(), kk[b:b + 1]]
        vs += [v[cu[b]:cu[b + 1]].cpu(), vv[b:b + 1]]
    lens = np.array(w.seq_lens, np.int64) + 1
    offs = np.concatenate([[0], np.cumsum(lens)[:-1]])
    W = w.window[0]
    start = np.array([[0 if w.head_class[0][hh] == 0 else max(0, int(n) - W) for hh in range(w.hkv)]
                      for n in lens], np.int32)
    kc, vc = torch.cat(ks), torch.cat(vs)
    t0 = time.perf_counter()
    rc, _, _ = oracle.attention(qq, kc, vc, np.arange(B, dtype=np.int32),
                                (lens - 1).astype(np.int32), offs, lens, w.head_class[0], W, start)
    secs = time.perf_counter() - t0
    assert rc == 0
    nbytes = decode_bytes(w, lens.tolist())
    return {"gbs": round(nbytes / secs / 1e9, 4), "us_per_step": round(1e6 * secs, 1),
            "sample": "one whole decode step (32 requests x 32 query heads)", "cores": host_cores()}


def run_context_sweep(dev, stream, sets, contexts=(8192, 16384, 32768, 65536, 131072)):
    """Speed-up of segmented over dense prefill against context length, on
    the 128K workload's layer shape (64/8 heads, D=128, pages of 128): a
    shallow layer (all 8 KV heads local, window 4096), a deep layer (KV head
    0 global, 7 local with window 1024) and the dense layer of the same
    library (all 8 heads global, full causal), each timed alone on the first
    n tokens of the same inputs."""
    import numpy as np
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    q, k, v = sets[0]
    hq, hkv, D, P = q.shape[1], k.shape[1], q.shape[2], 128
    kinds = {"shallow": ([1] * hkv, 4096), "deep_g1": ([0] + [1] * (hkv - 1), 1024),
             "dense": ([0] * hkv, 1 << 30)}
    out = {"n": list(contexts)}
    res = {kk: [] for kk in kinds}
    for n in contexts:
        cu = np.array([0, n], np.int32)
        qp = np.arange(n, dtype=np.int32)
        o = torch.empty((n, hq, D), dtype=torch.bfloat16, device=dev)
        for kind, (hc, W) in kinds.items():
            kp = torch.empty((hkv * (n // P) + 8, P, D), dtype=torch.bfloat16, device=dev)
            h = S.SegKV(1, hq, hkv, D, [hc], [min(W, n)], P, 1, n, kp, torch.empty_like(kp))
            h.append(0, k[:n], v[:n], cu, [0], stream)
            reps = 3 if n >= 65536 else 10
            h.prefill_attn(0, q[:n], cu, qp, [0], o, None, stream)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                h.prefill_attn(0, q[:n], cu, qp, [0], o, None, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            if h.status() != 0:
                raise RuntimeError("device status in the context sweep: " +
                                   S.segkv_last_error(h.handle))
            ms = e0.elapsed_time(e1) / reps
            wl = I.Workload(kind, 1, hq, hkv, D, P, [hc], [min(W, n)], [n])
            res[kind].append((ms, useful_flops_layer(wl, 0, n)))
            h.close()
            del kp
        del o
    torch.cuda.empty_cache()
    dense = [ms for ms, _ in res["dense"]]
    for kind in ("shallow", "deep_g1"):
        sp = [d / ms for (ms, _), d in zip(res[kind], dense)]
        out[kind] = {"seg_ms": [round(ms, 3) for ms, _ in res[kind]],
                     "useful_tflops": [round(f / (ms * 1e-3) / 1e12, 1) for ms, f in res[kind]],
                     "speedup_vs_dense": [round(x, 2) for x in sp],
                     "monotone": all(b > a for a, b in zip(sp, sp[1:]))}
    out["dense"] = {"ms": [round(x, 3) for x in dense],
                    "useful_tflops": [round(f / (ms * 1e-3) / 1e12, 1) for ms, f in res["dense"]]}
    return out


def run_decode(args, dev, stream, hbm, peak_src, cpu=False):
    import numpy as np
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    w = I.ragged_decode(seed=0, steps=128)
    B, P, D = len(w.seq_lens), w.page_size, w.head_dim
    steps = w.decode_steps
    max_len = max(w.seq_lens) + steps + 8  # + the multi-query tokens
    num_pages = sum((n + steps + 8) // P + 2 for n in w.seq_lens) * w.hkv + 64
    kp = torch.empty((num_pages, P, D), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    h = S.SegKV(1, w.hq, w.hkv, D, w.head_class, w.window, P, B, max_len, kp, vp)
    q, k, v, cu, qp = I.prefill_tensors(w, 0, device=dev)
    ids = list(range(B))
    h.append(0, k, v, cu, ids, stream)
    h.trim(0, ids)
    del q
    qd = [I.decode_step_tensors(w, s, device=dev) for s in range(steps)]
    cpu_oracle = oracle_decode_timing(w, k, v, cu, qd[0]) if cpu else None
    del k, v
    ws = torch.empty(h.workspace_size(S.SEGKV_WS_DECODE, B, B) // 4 + 64, dtype=torch.float32,
                     device=dev)
    o = torch.empty((B, w.hq, D), dtype=torch.bfloat16, device=dev)
    lens = list(w.seq_lens)
    one = np.arange(B + 1, dtype=np.int32)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    lens_at = [[x + s + 1 for x in lens] for s in range(steps)]  # lengths after step s
    bytes_step = [decode_bytes(w, ls) for ls in lens_at]
    torch.cuda.synchronize()
    t_host = time.perf_counter()
    for s in range(steps):
        qq, kk, vv = qd[s]
        ev[s][0].record(stream)
        h.append(0, kk, vv, one, ids, stream)
        ev[s][1].record(stream)
        h.decode_attn(0, qq, lens_at[s], ids, o, ws, stream)
        ev[s][2].record(stream)
    t_host = time.perf_counter() - t_host  # host time to issue all steps
    torch.cuda.synchronize()
    if h.status() != 0:
        raise RuntimeError("device status after decode: " + S.segkv_last_error(h.handle))
    lens = lens_at[-1]
    # back to back: decode is read-only for the segment state, so the last
    # step's call is repeated to time the GPU without host-issue gaps
    reps = 30
    qq = qd[-1][0]
    for _ in range(3):
        h.decode_attn(0, qq, lens, ids, o, ws, stream)
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(reps):
        h.decode_attn(0, qq, lens, ids, o, ws, stream)
    b1.record(stream)
    torch.cuda.synchronize()
    b2b_us = 1e3 * b0.elapsed_time(b1) / reps
    b2b_gbs = decode_bytes(w, lens) / (b2b_us * 1e-6) / 1e9
    # four query tokens per request (speculative decoding): append four
    # tokens each, then time the multi-query call back to back
    T = 4
    kt = I.normal_bf16(w.seed, I.tensor_stream(I._KD, 1, 9999), (B * T, w.hkv, D), device=dev)
    qt = I.normal_bf16(w.seed, I.tensor_stream(I._QD, 1, 9999), (B * T, w.hq, D), device=dev)
    h.append(0, kt, kt, np.arange(0, B * T + 1, T, dtype=np.int32), ids, stream)
    lens_t = [x + T for x in lens]
    ot = torch.empty((B * T, w.hq, D), dtype=torch.bfloat16, device=dev)
    wst_bytes = h.workspace_size(S.SEGKV_WS_DECODE, B * T, B)
    wst = torch.empty(wst_bytes // 4 + 64, dtype=torch.float32, device=dev) if wst_bytes else None
    for _ in range(3):
        h.decode_attn_multi(0, qt, T, lens_t, ids, ot, None, wst, stream)
    b0.record(stream)
    for _ in range(reps):
        h.decode_attn_multi(0, qt, T, lens_t, ids, ot, None, wst, stream)
    b1.record(stream)
    torch.cuda.synchronize()
    multi_us = 1e3 * b0.elapsed_time(b1) / reps
    rows_t = T * w.hq // w.hkv
    multi_kernel = ("prefill_kernel<128>" if not wst_bytes else
                    "decode_mma_kernel + decode_combine_kernel (%d query rows per KV head)" % rows_t
                    if rows_t in (8, 16) else
                    "decode_split_kernel<128,%d> (T*G query rows per KV head)" % rows_t)
    multi_bytes = decode_bytes(w, lens_t) + sum(
        (T - 1) * w.head_dim * 4 for n in lens_t for hh in range(w.hkv) if w.head_class[0][hh])
    warm = 8
    dec_ms = [ev[s][1].elapsed_time(ev[s][2]) for s in range(warm, steps)]
    app_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(warm, steps)]
    step_ms = [ev[s][0].elapsed_time(ev[s][2]) for s in range(warm, steps)]
    gbs = [bytes_step[s] / (dec_ms[s - warm] * 1e-3) / 1e9 for s in range(warm, steps)]
    med = statistics.median(gbs)
    return {"workload": "ragged decode, 32 requests, 2K-32K log-uniform, 128 steps",
            "gbs_median": round(med, 1), "hbm_peak_gbs": hbm, "frac": round(med / hbm, 4),
            "back_to_back_gbs": round(b2b_gbs, 1), "back_to_back_frac": round(b2b_gbs / hbm, 4),
            "back_to_back_us": round(b2b_us, 2),
            "multi_query_t4": {"us": round(multi_us, 2),
                               "gbs": round(multi_bytes / (multi_us * 1e-6) / 1e9, 1),
                               "frac": round(multi_bytes / (multi_us * 1e-6) / 1e9 / hbm, 4),
                               "kernel": multi_kernel},
            "peak_kind": peak_src,
            "decode_us_median": round(1e3 * statistics.median(dec_ms), 2),
            "append_us_median": round(1e3 * statistics.median(app_ms), 2),
            "step_us_median": round(1e3 * statistics.median(step_ms), 2),
            "tokens_per_s": round(B / (statistics.median(step_ms) * 1e-3), 1),
            "bytes_per_step_mean": int(statistics.mean(bytes_step)),
            "host_issue_us_per_step": round(1e6 * t_host / steps, 2),
            "steps_timed": steps - warm,
            "kernels": ["decode_split_kernel<128,4> (split-KV with the merge fused in)"],
            **({"cpu_oracle": cpu_oracle} if cpu_oracle else {})}


def run_rope(dev, stream, hbm):
    """Rotary re-alignment of one 32768-token sequence's cached keys (8 KV
    heads, D=128, pages of 64), every head global so every key is rotated:
    HBM bytes = keys read + keys written."""
    import numpy as np
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    n, hkv, D, P = 32768, 8, 128, 64
    kp = torch.empty((hkv * n // P + 8, P, D), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    h = S.SegKV(1, 32, hkv, D, [[0] * hkv], [n], P, 1, n, kp, vp)
    k = I.normal_bf16(0, I.tensor_stream(I._K, 9), (n, hkv, D), device=dev)
    h.append(0, k, k, np.array([0, n], np.int32), [0], stream)
    for _ in range(3):
        h.rope_shift(0, 0, 1000, 10000.0, D, S.SEGKV_ROPE_HALF, stream=stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record(stream)
    for _ in range(reps):
        h.rope_shift(0, 0, 1000, 10000.0, D, S.SEGKV_ROPE_HALF, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    assert h.status() == 0
    us = 1e3 * e0.elapsed_time(e1) / reps
    nbytes = 2 * n * hkv * D * 2
    return {"workload": "rope re-alignment of one 32768-token sequence, 8 KV heads, D=128",
            "us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "frac_hbm": round(nbytes / (us * 1e-6) / 1e9 / hbm, 4), "bytes": nbytes,
            "kernel": "rope_kernel"}


def run_prefill_configs(dev, stream, bf16_burst, peak_src, cpu=False):
    """Single-layer prefill of the Mistral-shaped 8K sequence and of the
    Llama-70B-shaped varlen batch (4 sequences of 16K-32K, window 2048, key
    sinks): prefill kernel time, tokens/s and useful TFLOP/s; with cpu=True
    also the fp64 oracle on the host cores (the 8K layer in full, the varlen
    batch on sampled query tokens)."""
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    out = {}
    # The leg before this one runs FFN GEMMs at the power limit; measured right
    # after it, the 8K layer took 0.204 ms against 0.182 ms alone. A short
    # pause lets the clocks recover, so that one layer is timed as if alone.
    time.sleep(2.0)
    for w in (I.mistral_8k(), I.llama70b_varlen()):
        q, k, v, cu, qp = I.prefill_tensors(w, 0, device=dev)
        cu, qp = cu.numpy(), qp.numpy()
        P, D = w.page_size, w.head_dim
        pages = sum(n // P + 2 for n in w.seq_lens) * w.hkv + 8
        kp = torch.empty((pages, P, D), dtype=torch.bfloat16, device=dev)
        h = S.SegKV(1, w.hq, w.hkv, D, w.head_class, w.window, P, len(w.seq_lens),
                    max(w.seq_lens), kp, torch.empty_like(kp))
        ids = list(range(len(w.seq_lens)))
        h.append(0, k, v, cu, ids, stream)
        o = torch.empty((int(cu[-1]), w.hq, D), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            h.prefill_attn(0, q, cu, qp, ids, o, None, stream)
        reps = 10
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            h.prefill_attn(0, q, cu, qp, ids, o, None, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if h.status() != 0:
            raise RuntimeError("device status after prefill: " + S.segkv_last_error(h.handle))
        ms = e0.elapsed_time(e1) / reps
        fl = sum(useful_flops_layer(w, 0, n) for n in w.seq_lens)
        tf = fl / (ms * 1e-3) / 1e12
        out[w.name] = {"seq_lens": list(w.seq_lens), "prefill_ms": round(ms, 3),
                       "tokens_per_s": round(int(cu[-1]) / (ms * 1e-3)),
                       "useful_tflop": round(fl / 1e12, 3), "useful_tflops": round(tf, 1),
                       "frac_of_burst": round(tf / bf16_burst, 4)}
        if cpu:
            out[w.name]["cpu_oracle"] = oracle_prefill_timing(
                w, q.cpu(), k.cpu(), v.cpu(), cu, qp,
                sample_rows=None if w.name == "mistral-8k" else 384)
        h.close()
        del q, k, v, o, kp
        torch.cuda.empty_cache()
    out["peak_kind"] = f"bf16 burst ({peak_src}); one layer timed alone, inputs larger than L2"
    return out


def run_routing(dev, stream, bf16_burst, peak_src):
    """Sparse FFN routing on the Mistral-shaped 8K layer: prefill attention
    (with LSE), attention mass per token, top-k choice of a quarter of the
    tokens, and the SwiGLU FFN (hidden 4096, width 14336) on the chosen rows,
    against the dense FFN on every row."""
    import numpy as np
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    w = I.mistral_8k()
    fw = I.mistral_ffn()
    n, P, D = w.seq_lens[0], w.page_size, w.head_dim
    q, k, v, cu, qp = I.prefill_tensors(w, 0, device=dev)
    cu, qp = cu.numpy(), qp.numpy()
    kp = torch.empty(((n // P + 2) * w.hkv, P, D), dtype=torch.bfloat16, device=dev)
    h = S.SegKV(1, w.hq, w.hkv, D, w.head_class, w.window, P, 1, n, kp, torch.empty_like(kp))
    h.append(0, k, v, cu, [0], stream)
    x, r, wg, wu, wd = I.ffn_tensors(fw, device=dev)
    o = torch.empty((n, w.hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.hq, n), device=dev)
    mass = torch.empty((w.hkv, n), device=dev)
    score = torch.empty((n,), device=dev)
    idx = torch.empty((fw.m,), dtype=torch.int32, device=dev)
    res = r.clone()
    rc, wsb = S.segkv_ffn_workspace_size(n, fw.d_model, fw.d_ff)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stages = {
        "prefill": lambda: h.prefill_attn(0, q, cu, qp, [0], o, lse, stream),
        "mass": lambda: h.attn_mass(0, q, cu, qp, [0], lse, mass, stream),
        "topk": lambda: h.topk_tokens(mass, cu, [fw.m], score, idx, stream),
        "sparse_ffn": lambda: h.sparse_ffn(x, res, idx, wg, wu, wd, ws, stream),
        "dense_ffn": lambda: h.sparse_ffn(x, res, None, wg, wu, wd, ws, stream),
    }
    us = {}
    for name, fn in stages.items():
        for _ in range(3):
            fn()
        reps = 10
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        us[name] = 1e3 * e0.elapsed_time(e1) / reps
    if h.status() != 0:
        raise RuntimeError("device status after routing: " + S.segkv_last_error(h.handle))
    att_flops = useful_flops_layer(w, 0, n)
    ffn_flops = 6.0 * fw.m * fw.d_model * fw.d_ff
    dense_flops = 6.0 * n * fw.d_model * fw.d_ff
    sparse_layer = us["prefill"] + us["mass"] + us["topk"] + us["sparse_ffn"]
    dense_layer = us["prefill"] + us["dense_ffn"]
    ffn_tf = ffn_flops / (us["sparse_ffn"] * 1e-6) / 1e12
    return {"workload": "Mistral-shaped 8K layer: prefill, mass, top-k of 2048 tokens, SwiGLU FFN "
                        "4096x14336 on them; dense FFN on all 8192 for comparison",
            "us": {kk: round(vv, 2) for kk, vv in us.items()},
            "prefill_useful_tflops": round(att_flops / (us["prefill"] * 1e-6) / 1e12, 1),
            "mass_tflops": round(att_flops / 2 / (us["mass"] * 1e-6) / 1e12, 1),
            "sparse_ffn_tflops": round(ffn_tf, 1),
            "dense_ffn_tflops": round(dense_flops / (us["dense_ffn"] * 1e-6) / 1e12, 1),
            "roofline_ffn": {"bound": "tensor", "achieved": round(ffn_tf, 1), "peak": bf16_burst,
                             "unit": "TFLOP/s", "frac": round(ffn_tf / bf16_burst, 4),
                             "peak_kind": f"bf16 burst ({peak_src}); GEMMs timed alone"},
            "ffn_share_of_dense_layer": round(us["dense_ffn"] / dense_layer, 3),
            "layer_us_sparse": round(sparse_layer, 1), "layer_us_dense": round(dense_layer, 1),
            "layer_speedup": round(dense_layer / sparse_layer, 3),
            "kernels": ["prefill_kernel<128>", "mass_kernel<128>", "score_sum_kernel",
                        "topk_kernel", "gather_rows_kernel", "ffn_gemm_kernel<0>",
                        "ffn_gemm_kernel<1>"]}


def run_transfer(dev, stream, hbm):
    """Prefill-to-decode transfer of one 32768-token session (1 global + 7
    local heads, window 1024, D=128, pages of 64) after its post-prefill trim:
    bytes moved by segkv_export versus a dense [n, Hkv, D] K/V export, the
    export and import rates, and how many such sessions fit per GB of KV."""
    import numpy as np
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    n, hkv, D, P, W = 32768, 8, 128, 64, 1024
    hc = [[0] + [1] * 7]
    kp = torch.empty((hkv * n // P + 64, P, D), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    src = S.SegKV(1, 32, hkv, D, hc, [W], P, 1, n + 8, kp, vp)
    k = I.normal_bf16(0, I.tensor_stream(I._K, 11), (n, hkv, D), device=dev)
    src.append(0, k, k, np.array([0, n], np.int32), [0], stream)
    src.trim(0, [0])
    buf, hdr = src.export_segment(0, 0, stream)
    kp2 = torch.empty_like(kp)
    vp2 = torch.empty_like(kp)
    dst = S.SegKV(1, 32, hkv, D, hc, [W], P, 1, n + 8, kp2, vp2)

    host_us = {}

    def timed(name, fn, reps=20):
        for _ in range(3):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        host_us[name] = round(1e6 * (time.perf_counter() - t0) / reps, 2)  # issue cost per call
        torch.cuda.synchronize()
        return 1e3 * e0.elapsed_time(e1) / reps

    hnd = src.handle
    header = np.zeros(1 + hkv, np.int32)
    exp_us = timed("export", lambda: S.segkv_export(hnd, 0, 0, buf, header, stream))

    def imp():
        dst.free_seq(0)
        dst.import_segment(0, 0, buf, hdr, stream)
    imp_us = timed("import", imp)
    assert src.status() == 0 and dst.status() == 0
    seg_bytes = buf.numel() * 2
    dense_bytes = n * hkv * D * 2 * 2
    return {"workload": "one 32768-token session, 1 global + 7 local heads (W=1024), D=128, "
                        "after the post-prefill trim",
            "export_bytes": seg_bytes, "dense_bytes": dense_bytes,
            "bytes_ratio_dense_over_segmented": round(dense_bytes / seg_bytes, 3),
            "export_us": round(exp_us, 2),
            "export_gbs": round(2 * seg_bytes / (exp_us * 1e-6) / 1e9, 1),
            "import_us": round(imp_us, 2),
            "import_gbs": round(2 * seg_bytes / (imp_us * 1e-6) / 1e9, 1),
            "kv_sessions_per_gb": {"segmented": round(1e9 / seg_bytes, 2),
                                   "dense": round(1e9 / dense_bytes, 2)},
            "host_issue_us_per_call": host_us,
            "kernels": ["transfer_kernel"]}


def run_e2e(args, dev, stream, w, sets, cu, q_pos, step_flops, num_pages):
    """The same step through the public API from pinned host buffers: every
    layer's Q, K, V copied host->device inside the timed region (a side stream
    copies ahead into three rotating device buffers while the kernels run),
    and the last layer's output copied back."""
    import torch

    import head_segmented_paged_gb300 as S

    n, L, hq, hkv, D, P = w.seq_lens[0], w.num_layers, w.hq, w.hkv, w.head_dim, w.page_size
    host = [tuple(t.to("cpu").pin_memory() for t in s) for s in sets]
    NB = 3  # copies run up to two layers ahead of the kernels
    dbuf = [tuple(torch.empty_like(t) for t in sets[0]) for _ in range(NB)]
    o = torch.empty((n, hq, D), dtype=torch.bfloat16, device=dev)
    o_host = torch.empty((n, hq, D), dtype=torch.bfloat16).pin_memory()
    kp = torch.empty((num_pages, P, D), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    h = S.SegKV(L, hq, hkv, D, w.head_class, w.window, P, 1, n, kp, vp)
    copy_stream = torch.cuda.Stream(device=dev)
    done = [torch.cuda.Event() for _ in range(NB)]
    free = [torch.cuda.Event() for _ in range(NB)]
    h2d = 0
    # per layer: its copies' start and end on the copy stream, and the start
    # and end of its kernels on the compute stream (after the wait on its copy)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    cp_ev = [(ev(), ev()) for _ in range(L)]
    k_ev = [(ev(), ev()) for _ in range(L)]

    def step():
        nonlocal h2d
        h.free_seq(0)
        h2d = 0
        for l in range(L + 1):
            if l < L:  # issue the copy for layer l
                b = l % NB
                copy_stream.wait_event(free[b])
                with torch.cuda.stream(copy_stream):
                    cp_ev[l][0].record(copy_stream)
                    for dst, src in zip(dbuf[b], host[l % N_INPUT_SETS]):
                        dst.copy_(src, non_blocking=True)
                        h2d += src.numel() * src.element_size()
                    cp_ev[l][1].record(copy_stream)
                done[b].record(copy_stream)
            if l >= 1:  # compute layer l-1
                lb = (l - 1) % NB
                stream.wait_event(done[lb])
                k_ev[l - 1][0].record(stream)
                qd, kd, vd = dbuf[lb]
                h.append(l - 1, kd, vd, cu, [0], stream)
                h.prefill_attn(l - 1, qd, cu, q_pos, [0], o, None, stream)
                h.trim(l - 1, [0])
                k_ev[l - 1][1].record(stream)
                free[lb].record(stream)
        o_host.copy_(o, non_blocking=True)

    for b in range(NB):
        free[b].record(stream)
    step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # the host->device rate alone on this machine (one layer's Q, K, V, twice),
    # to tell a copy-bound step from a compute-bound one
    with torch.cuda.stream(copy_stream):
        t0.record(copy_stream)
        for _ in range(2):
            for dst, src in zip(dbuf[0], host[0]):
                dst.copy_(src, non_blocking=True)
        t1.record(copy_stream)
    torch.cuda.synchronize()
    layer_bytes = sum(t.numel() * t.element_size() for t in host[0])
    h2d_gbs = 2 * layer_bytes / (t0.elapsed_time(t1) * 1e-3) / 1e9
    ks = 5
    rates, waits = [], []
    t0.record(stream)
    for _ in range(ks):
        step()
        torch.cuda.synchronize()
        # each layer's copy rate, and how long the kernels waited for copies
        rates += [layer_bytes / (a.elapsed_time(b) * 1e-3) / 1e9 for a, b in cp_ev]
        waits.append(sum(max(0.0, k_ev[l][1].elapsed_time(k_ev[l + 1][0]))
                         for l in range(L - 1)))
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / ks
    rates.sort()
    return {"value": round(step_flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 2), "steps_timed": ks, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": o.numel() * o.element_size(),
            "h2d_gbs_copy_alone": round(h2d_gbs, 1),
            "h2d_gbs_per_layer_in_step": {"median": round(statistics.median(rates), 1),
                                          "p10": round(rates[len(rates) // 10], 1),
                                          "min": round(rates[0], 1)},
            "kernels_waiting_for_copies_ms_per_step": round(statistics.median(waits), 1),
            "note": "pinned host Q/K/V per layer copied inside the timed region on a side stream "
                    "into three rotating device buffers; the last layer's O copied back"}


# ------------------------------------------------------------------ oracle timings per config
def visible_keys(head_class, window, p):
    """Keys a query at position p sees in a head: p+1 (global) or min(p+1, W)."""
    return p + 1 if head_class == 0 else min(p + 1, window)


def rows_flops(w, layer, pos):
    """Useful FLOPs of the query tokens at positions pos (all query heads)."""
    pos = [int(x) for x in pos]
    return sum(4 * w.head_dim * w.group * visible_keys(w.head_class[layer][hh], w.window[layer], p)
               for p in pos for hh in range(w.hkv))


def oracle_prefill_timing(w, q, k, v, cu, qp, sample_rows=None, seed=0):
    """Time the fp64 oracle on a prefill layer (CPU tensors): every query
    token, or sample_rows random tokens spread over the sequences, and
    extrapolate by useful FLOPs to the whole layer."""
    import numpy as np

    import oracle

    cu = np.asarray(cu, np.int64)
    qp = np.asarray(qp, np.int32)
    nseq = len(w.seq_lens)
    row_seq = np.repeat(np.arange(nseq), np.diff(cu)).astype(np.int32)
    tot = int(cu[-1])
    rows = None
    if sample_rows is not None and sample_rows < tot:
        rows = np.sort(np.random.default_rng(seed).choice(tot, sample_rows, replace=False))
    t0 = time.perf_counter()
    rc, _, _ = oracle.attention(q, k, v, row_seq, qp, cu[:-1], np.diff(cu), w.head_class[0],
                                w.window[0], np.zeros((nseq, w.hkv), np.int32), rows=rows)
    secs = time.perf_counter() - t0
    assert rc == 0
    full = sum(useful_flops_layer(w, 0, n) for n in w.seq_lens)
    done = full if rows is None else rows_flops(w, 0, qp[rows])
    rate = done / secs
    return {"tflops": round(rate / 1e12, 5), "seconds": round(secs, 2),
            "ms_full_layer": round(1e3 * full / rate, 1),
            "sample": ("every query token" if rows is None else
                       f"{len(rows)} random query tokens of {tot}, extrapolated by useful FLOPs"),
            "cores": host_cores()}


# ------------------------------------------------------------------ oracle (CPU) arm
def oracle_rate(q_rows, k, v, w, budget_s):
    """Time the oracle on sampled query rows of three layer kinds of the
    128K workload (shallow all-local, deep with no global head, deep with
    one); return useful FLOPs/s over the sample. q_rows(rows) gives those
    rows of Q (bf16, CPU); k, v are the layer's full K and V on the CPU."""
    import numpy as np

    import oracle

    n = w.seq_lens[0]
    kinds = {}
    for l in range(w.num_layers):
        g = sum(1 for c in w.head_class[l] if c == 0)
        kind = "shallow" if l < 8 else ("deep_g1" if g else "deep_g0")
        kinds.setdefault(kind, l)
    rng = np.random.default_rng(0)
    total_flops, total_s = 0, 0.0
    per = {}
    for kind, l in kinds.items():
        t_kind, f_kind, nrows = 0.0, 0, 2
        while t_kind < budget_s / len(kinds):
            pos = np.sort(rng.integers(0, n, nrows)).astype(np.int32)
            qs = q_rows(pos)
            t0 = time.perf_counter()
            rc, _, _ = oracle.attention(qs, k, v, np.zeros(len(pos), np.int32), pos, [0], [n],
                                        w.head_class[l], w.window[l],
                                        np.zeros((1, w.hkv), np.int32))
            dt = time.perf_counter() - t0
            assert rc == 0
            f = 0
            for p in pos:
                for hh in range(w.hkv):
                    vis = p + 1 if w.head_class[l][hh] == 0 else min(p + 1, w.window[l])
                    f += 4 * w.head_dim * w.group * int(vis)
            t_kind += dt
            f_kind += f
            if dt < 1.0:
                nrows *= 2
        per[kind] = {"layer": l, "seconds": round(t_kind, 2), "useful_flops": f_kind}
        total_flops += f_kind
        total_s += t_kind
    return total_flops / total_s, per, total_s


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(sets, w, budget_s=20.0):
    import oracle
    oracle.build()
    q, k, v = sets[0]
    kc, vc = k.to("cpu"), v.to("cpu")

    def q_rows(pos):
        import torch
        return q[torch.as_tensor(pos, dtype=torch.long, device=q.device)].to("cpu")

    rate, per, secs = oracle_rate(q_rows, kc, vc, w, budget_s)
    return {"value": rate / 1e12, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "sample": ("fp64 C++ oracle (OpenMP) on random query rows (all 64 query heads) of one "
                       "shallow, one deep g=0 and one deep g=1 layer of the 128K workload, "
                       f"{secs:.1f} s total; useful FLOPs / CPU time"),
            "per_kind": per}


def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores, on bounded samples of the
    same 128K workload; each step is one sample."""
    import importlib.util

    import oracle

    # the seeded generators only, loaded by path: importing the package would
    # map the CUDA library into a process that runs none of it
    spec = importlib.util.spec_from_file_location(
        "segkv_inputs", os.path.join(ROOT, "head_segmented_paged_gb300", "inputs.py"))
    I = importlib.util.module_from_spec(spec)
    sys.modules["segkv_inputs"] = I  # dataclasses resolve annotations through it
    spec.loader.exec_module(I)
    oracle.build()
    w = I.long_128k_64layer(seed=0)
    n = w.seq_lens[0]
    shape_q = (n, w.hq, w.head_dim)
    k = I.normal_bf16(w.seed, I.tensor_stream(I._K, 0), (n, w.hkv, w.head_dim))
    v = I.normal_bf16(w.seed, I.tensor_stream(I._V, 0), (n, w.hkv, w.head_dim))

    def q_rows(pos):
        return I.normal_bf16_rows(w.seed, I.tensor_stream(I._Q, 0), shape_q, pos)

    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rate(q_rows, k, v, w, per_step / 3)
    rates, secs = [], 0.0
    for _ in range(args.steps):
        r, _, s = oracle_rate(q_rows, k, v, w, per_step)
        rates.append(r)
        secs += s
    value = statistics.median(rates) / 1e12
    cores = host_cores()
    ms_step = 1e3 * secs / max(1, args.steps)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded splitmix64 + Box-Muller N(0,1), rounded to bf16",
            "config": {"workload": "128k-64layer prefill", "layers": w.num_layers, "hq": w.hq,
                       "hkv": w.hkv, "head_dim": w.head_dim, "page_size": w.page_size,
                       "context": n},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: random query rows of one shallow, one deep "
                                       "g=0 and one deep g=1 layer, about "
                                       f"{per_step:.0f} s of CPU work"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_case_128k_layers(args, dev, stream):
    """One layer of each kind of the 128K workload (shallow all-local, deep
    without and with a global head), one prefill launch each; for capturing
    per-launch counters at full size."""
    import numpy as np
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    w = I.long_128k_64layer(seed=0)
    n, P, D = w.seq_lens[0], w.page_size, w.head_dim
    kinds = {}
    for l in range(w.num_layers):
        g = sum(1 for c in w.head_class[l] if c == 0)
        kinds.setdefault("shallow" if l < 8 else ("deep_g1" if g else "deep_g0"), l)
    q = I.normal_bf16(0, I.tensor_stream(I._Q, 0), (n, w.hq, D), device=dev)
    k = I.normal_bf16(0, I.tensor_stream(I._K, 0), (n, w.hkv, D), device=dev)
    v = I.normal_bf16(0, I.tensor_stream(I._V, 0), (n, w.hkv, D), device=dev)
    o = torch.empty_like(q)
    cu = np.array([0, n], np.int32)
    q_pos = np.arange(n, dtype=np.int32)
    out = {"case": args.case}
    for kind, l in sorted(kinds.items(), key=lambda x: x[1]):
        kp = torch.empty((w.hkv * n // P + 8, P, D), dtype=torch.bfloat16, device=dev)
        vp = torch.empty_like(kp)
        h = S.SegKV(1, w.hq, w.hkv, D, [w.head_class[l]], [w.window[l]], P, 1, n, kp, vp)
        h.append(0, k, v, cu, [0], stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h.prefill_attn(0, q, cu, q_pos, [0], o, None, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        assert h.status() == 0
        ms = e0.elapsed_time(e1)
        f = useful_flops_layer(w, l, n)
        out[kind] = {"layer": l, "ms": round(ms, 3), "useful_tflops": round(f / (ms * 1e-3) / 1e12, 1)}
        h.close()
        del kp, vp
    print(json.dumps(out), flush=True)


def run_case(args):
    """Single-kernel cases for profiling: one layer of prefill at 32K tokens
    (64/8 heads, D=128, pages of 128; KV head 0 global, the rest local with
    window 1024, or all global with --case dense-32k), or the ragged decode
    workload. Prints one JSON line with per-launch times."""
    import numpy as np
    import torch

    import head_segmented_paged_gb300 as S
    from head_segmented_paged_gb300 import inputs as I

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    if args.case == "decode":
        out = run_decode(args, dev, stream, *measured_peaks()[::3])
        print(json.dumps({"case": args.case, **out}), flush=True)
        return
    if args.case == "transfer":
        print(json.dumps({"case": args.case, **run_transfer(dev, stream, measured_peaks()[0])}),
              flush=True)
        return
    if args.case == "configs":
        hbm, burst, _, src = measured_peaks()
        print(json.dumps({"case": args.case, **run_prefill_configs(dev, stream, burst, src)}),
              flush=True)
        return
    if args.case == "routing":
        hbm, burst, _, src = measured_peaks()
        print(json.dumps({"case": args.case, **run_routing(dev, stream, burst, src)}), flush=True)
        return
    if args.case == "rope":
        print(json.dumps({"case": args.case, **run_rope(dev, stream, measured_peaks()[0])}),
              flush=True)
        return
    if args.case == "prefill-128k-layers":
        run_case_128k_layers(args, dev, stream)
        return
    n, hq, hkv, D, P = 32768, 64, 8, 128, 128
    glob = args.case == "dense-32k"
    hc = [[0] * 8] if glob else [[0] + [1] * 7]
    w = I.Workload(args.case, 1, hq, hkv, D, P, hc, [n if glob else 1024], [n])
    q = I.normal_bf16(0, I.tensor_stream(I._Q, 0), (n, hq, D), device=dev)
    k = I.normal_bf16(0, I.tensor_stream(I._K, 0), (n, hkv, D), device=dev)
    v = I.normal_bf16(0, I.tensor_stream(I._V, 0), (n, hkv, D), device=dev)
    kp = torch.empty((hkv * n // P + 8, P, D), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    h = S.SegKV(1, hq, hkv, D, hc, w.window, P, 1, n, kp, vp)
    cu = np.array([0, n], np.int32)
    q_pos = np.arange(n, dtype=np.int32)
    o = torch.empty((n, hq, D), dtype=torch.bfloat16, device=dev)
    h.append(0, k, v, cu, [0], stream)
    flops = useful_flops_layer(w, 0, n)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.warmup + args.steps)]
    for i in range(args.warmup + args.steps):
        ev[i][0].record(stream)
        h.prefill_attn(0, q, cu, q_pos, [0], o, None, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert h.status() == 0
    ms = [a.elapsed_time(b) for a, b in ev[args.warmup:]]
    med = statistics.median(ms)
    print(json.dumps({"case": args.case, "prefill_ms": ms, "useful_tflops":
                      round(flops / (med * 1e-3) / 1e12, 1), "useful_flops": flops}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--case", default=None,
                    choices=["prefill-32k", "dense-32k", "decode", "prefill-128k-layers", "rope",
                             "transfer", "routing", "configs"],
                    help="run one kernel's profiling case instead of the benchmark")
    args = ap.parse_args()
    if args.case:
        import __graft_entry__
        __graft_entry__.build()
        run_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    out = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
