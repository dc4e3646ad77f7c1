#!/usr/bin/env python
"""Benchmark: decode attention over a paged KV cache on GB300.

One step = one pass of the whole decode path over one batch (Llama-3-8B GQA
shape by default: B=16 sequences, 32 q / 8 kv heads, d=128, 32K context,
16-token pages, 128 pages kept per q-head):
    kv_meta_build   page min/max metadata        (reads K, writes meta)
    decode_attn_full   exact attention            (reads q, K, V)
    decode_attn_select bound scores, top-K, sparse attention over the pages
The metric is queries/s (a query = one sequence's one-token decode over all
heads of one layer) and the effective GB/s of algorithmic bytes.  Inputs are
seeded synthetic tensors already resident in HBM; K+V (2 GiB) exceed L2, and
the step orders the calls so the exact path's 2 GiB stream sits between the
metadata build and the sparse read of that metadata.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dkv|reference]

Prints one JSON line (rank 0).  Under torchrun each rank decodes its own batch
(weak scaling, no collective on the data path); the time is the max over ranks.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import WORKLOADS, Workload, bits, by_name  # noqa: E402

METRIC = "decode-attn queries/s and effective KV GB/s (% of GB300 8 TB/s HBM roofline)"
DEFAULT_WORKLOAD = "llama3-8b-gqa-b16-n32k"
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["dkv", "reference"], default="dkv")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (small cases for ncu captures)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the e2e, CPU-baseline, 1M-token head-wise and other-workload legs")
    ap.add_argument("--legs", default="all",
                    help="comma list of extra legs to run (e2e, group, paged, pagesize, ratios, "
                         "reuse, tokens, meta8, cpu, headwise, others) or 'all'; for small "
                         "profiling runs")
    args = ap.parse_args()
    legs = {"e2e", "group", "paged", "pagesize", "ratios", "reuse", "tokens", "meta8", "cpu",
            "headwise", "others"}
    args.legs = set() if args.no_extra else (legs if args.legs == "all" else set(args.legs.split(",")))
    unknown = args.legs - legs
    if unknown:
        ap.error(f"unknown legs: {sorted(unknown)}")
    return args


# ------------------------------------------------------------------ helpers
def rank_seed(widx: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling: no rank repeats another's work)."""
    return 42 + widx + 1000 * rank


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: the job is done when every rank is."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_queries_per_s(world: int, batch: int, ms_step: float) -> float:
    """Queries of all ranks (each its own batch) per second of the slowest rank."""
    return world * batch / (ms_step * 1e-3)


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_sha(files=None) -> str:
    """Hash of the kernel sources (all of csrc/, or the listed files in it)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_paged_kv_gb300", "csrc")
    names = files if files else [f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h"))]
    for f in sorted(names):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t["kernels"][kernel_key]
        if e.get("source_sha") != source_sha(e.get("sources")):
            return None
        return e["dram_bytes_per_launch_full_size"]
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        busy = [s for s in sm if smax and s > 0.3 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def step_launches(w: Workload) -> int:
    """The library's kernel launches in one step (meta build, exact, select) on
    workload w, by the library's dispatch rules for these shapes: one metadata
    kernel; the exact call's attention and merge; the select call's per-unit
    selection kernel (selection pages of 16 tokens or more, 256 to 2048 of
    them) or its score, top-K and union kernels (no union kernel with one
    query head per kv head at 16-token pages: the top-K writes the unions),
    then its attention and merge (no merge on a 4-bit cache whose unions fit
    one work item)."""
    P, P16, G = w.P, -(-w.N // 16), w.Hq // w.Hkv
    kk = min(w.top_k, P)
    select = 1 if (w.S >= 16 and 256 <= P <= 2048) else (2 + (0 if G == 1 and w.S == 16 else 1))
    union_sel = min(G * kk, P)
    union_max = min(union_sel * (w.S // 16) if w.S > 16 else union_sel, P16)
    ppc = max(32 if w.d == 128 else 64, -(-union_max // 256))
    merge = 0 if (w.q4 and -(-union_max // ppc) == 1) else 1
    return 1 + 2 + select + 1 + merge


def union_tokens(sel: torch.Tensor, w: Workload, S: int = 0) -> int:
    """Valid tokens of the unique pages (of S tokens, default the workload's)
    gathered per (batch, kv head)."""
    S = S or w.S
    P = (w.N + S - 1) // S
    B, Hq, kk = sel.shape
    mask = torch.zeros(B, w.Hkv, P, dtype=torch.bool, device=sel.device)
    grp = sel.view(B, w.Hkv, w.G * kk).long()
    mask.scatter_(2, grp, True)
    toks = torch.full((P,), S, dtype=torch.int64, device=sel.device)
    toks[-1] = w.N - (P - 1) * S
    return int((mask.long() * toks).sum().item())


def cache_tokens(sel: torch.Tensor, w: Workload, S: int) -> int:
    """Valid tokens of the unique 16-token cache pages that hold the selected
    pages of S < 16 tokens, per (batch, kv head)."""
    P16 = (w.N + 15) // 16
    B, Hq, kk = sel.shape
    mask = torch.zeros(B, w.Hkv, P16, dtype=torch.bool, device=sel.device)
    grp = (sel.view(B, w.Hkv, w.G * kk).long() * S) // 16
    mask.scatter_(2, grp, True)
    toks = torch.full((P16,), 16, dtype=torch.int64, device=sel.device)
    toks[-1] = w.N - (P16 - 1) * 16
    return int((mask.long() * toks).sum().item())


# ------------------------------------------------------------------ GPU arm
def run_dkv(args, rank, world, local):
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc
    from workloads import make_inputs

    dkv.lib()  # fails loudly if the CUDA library is missing
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = by_name(args.workload)
    widx = [x.name for x in WORKLOADS].index(w.name)
    if args.batch:
        w = w.replace(B=args.batch)
    q, K, V = make_inputs(w, seed=rank_seed(widx, rank), device=dev)
    stream = torch.cuda.current_stream(dev)
    if w.q4:
        # (a 4-bit workload: small profiling runs of the step on the 4-bit
        # cache; the headline workload is dense)
        K, V = dkv.kv_quant4(K), dkv.kv_quant4(V)

    ws_full = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, 0), dtype=torch.uint8,
                          device=dev)
    ws_sel = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k),
                         dtype=torch.uint8, device=dev)
    kk = min(w.top_k, w.P)
    out_full = torch.empty(w.B, w.Hq, w.d, dtype=torch.float32, device=dev)
    out_sel = torch.empty_like(out_full)
    sel = torch.empty(w.B, w.Hq, kk, dtype=torch.int32, device=dev)
    calls = ["kv_meta_build", "decode_attn_full", "decode_attn_select"]
    ev = {c: [] for c in calls}

    def step(record=False):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if record else None
        if record:
            e[0].record(stream)
        meta = dkv.kv_meta_build(K)
        if record:
            e[1].record(stream)
        dkv.decode_attn_full(q, K, V, out=out_full, workspace=ws_full)
        if record:
            e[2].record(stream)
        dkv.decode_attn_select(q, K, V, meta, w.top_k, out=out_sel, selected=sel,
                               workspace=ws_sel)
        if record:
            e[3].record(stream)
            for i, c in enumerate(calls):
                ev[c].append((e[i], e[i + 1]))

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    gathered = union_tokens(sel, w)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t0.record(stream)
        for _ in range(args.steps):
            step(record=True)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_step = ms_total / args.steps
    per_call = {c: statistics.mean(a.elapsed_time(b) for a, b in ev[c]) for c in calls}

    status = max(dkv.read_device_status(ws_full), dkv.read_device_status(ws_sel))
    if status != 0:
        raise SystemExit(f"device status {status} during the timed region")

    # The same three calls again, each after an L2 flush (outside its event
    # pair): the select call then reads the metadata the build just wrote from
    # HBM, not from L2.
    flush = L2Flush(dev)
    cold = {c: [] for c in calls}
    for _ in range(max(10, args.steps)):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        flush()
        e[0].record(stream)
        meta = dkv.kv_meta_build(K)
        e[1].record(stream)
        flush()
        e[2].record(stream)
        dkv.decode_attn_full(q, K, V, out=out_full, workspace=ws_full)
        e[3].record(stream)
        flush()
        e[4].record(stream)
        dkv.decode_attn_select(q, K, V, meta, w.top_k, out=out_sel, selected=sel,
                               workspace=ws_sel)
        e[5].record(stream)
        for i, c in enumerate(calls):
            cold[c].append((e[2 * i], e[2 * i + 1]))
    torch.cuda.synchronize()
    per_call_cold = {c: statistics.median(a.elapsed_time(b) for a, b in cold[c]) for c in calls}
    if max(dkv.read_device_status(ws_full), dkv.read_device_status(ws_sel)) != 0:
        raise SystemExit("device status error in the cold-L2 pass")

    bytes_call = {
        "kv_meta_build": acc.meta_bytes(w.B, w.Hkv, w.d, w.N, w.S, q4=w.q4),
        "decode_attn_full": acc.full_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, q4=w.q4),
        "decode_attn_select": acc.select_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, gathered, w.S,
                                               q4=w.q4),
    }
    step_bytes = sum(bytes_call.values())
    peak, peak_kind = peaks()
    kernels = {}
    for c in calls:
        gbs = bytes_call[c] / (per_call[c] * 1e-3) / 1e9
        kernels[c] = {"ms": round(per_call[c], 5), "alg_bytes": bytes_call[c],
                      "GB/s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4),
                      "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}
    kernels_cold = {c: call_stats(per_call_cold[c], bytes_call[c], peak) for c in calls}
    kernels["decode_attn_select"]["gathered_pages"] = gathered // w.S
    kernels["decode_attn_full"]["queries_per_s"] = round(w.B / (per_call["decode_attn_full"] * 1e-3), 1)
    kernels["decode_attn_select"]["queries_per_s"] = round(
        w.B / (per_call["decode_attn_select"] * 1e-3), 1)
    dom = max(calls, key=lambda c: per_call[c])
    dom_gbs = bytes_call[dom] / (per_call[dom] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(dom_gbs, 1),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(dom_gbs / peak, 4),
                "frac_of_8tbs": round(dom_gbs / NOMINAL_HBM_GBS, 4),
                "traffic": ncu_traffic(dom),
                # every call of the step, in the timed region (warm) and each
                # after an L2 flush (cold): ms and fraction of 8 TB/s
                "calls": {c: {"ms": kernels[c]["ms"], "frac_of_8tbs": kernels[c]["frac_of_8tbs"],
                              "ms_cold": kernels_cold[c]["ms"],
                              "frac_of_8tbs_cold": kernels_cold[c]["frac_of_8tbs"]}
                          for c in calls}}
    value = job_queries_per_s(world, w.B, ms_step)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "q4g64/fp16" if w.q4 else w.dtype,
        "data": "synthetic (seeded torch Philox on device; K pages 2% hot, aligned to the group query)",
        "config": {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv,
                   "head_dim": w.d, "context": w.N, "page_size": w.S, "top_k_pages": w.top_k,
                   "step": "kv_meta_build + decode_attn_full + decode_attn_select",
                   "l2": "inputs larger than L2 (2 GiB K+V streamed every step); per-call "
                         "figures also taken each after a write of twice the L2 (kernels_cold)",
                   "parallelism": f"replicas x{world} (each rank its own batch)"},
        "effective_GB_per_s": round(step_bytes / (ms_step * 1e-3) / 1e9, 1),
        "kernels": kernels, "kernels_cold": kernels_cold,
        "kernels_timing": {"kernels": "inside the timed region (back-to-back steps)",
                           "kernels_cold": COLD},
        "roofline": roofline,
        "gpu_launches": args.steps * step_launches(w),
        "clocks": clk.summary(),
    }
    return res, (q, K, V, w, widx, dev, stream, flush)


def group_select_leg(q, K, V, w, dev, stream, flush, reps=10):
    """decode_attn_select with one selection per kv head group (summed bound
    scores) on the bench workload; the same byte count rule (metadata plus the
    unique pages gathered per (batch, kv head))."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc

    meta = dkv.kv_meta_build(K)
    kk = min(w.top_k, w.P)
    ws = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k),
                     dtype=torch.uint8, device=dev)
    out = torch.empty(w.B, w.Hq, w.d, dtype=torch.float32, device=dev)
    sel = torch.empty(w.B, w.Hq, kk, dtype=torch.int32, device=dev)

    def call():
        dkv.decode_attn_select(q, K, V, meta, w.top_k, out=out, selected=sel, workspace=ws,
                               group_select=True)

    ms = time_cold(call, stream, flush, reps)
    gathered = union_tokens(sel, w)
    nbytes = acc.select_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, gathered, w.S)
    peak, _ = peaks()
    res = {"workload": w.name, **call_stats(ms, nbytes, peak), "gathered_pages": gathered // w.S,
           "queries_per_s": round(w.B / (ms * 1e-3), 1), "timing": COLD}
    return res


class L2Flush:
    """Writes a buffer of twice the L2 size: the next call then finds none of
    its inputs (metadata included) in L2."""

    def __init__(self, dev):
        props = torch.cuda.get_device_properties(dev)
        l2 = int(getattr(props, "L2_cache_size", 0) or (129 << 20))
        self.bytes = 2 * l2
        self.buf = torch.empty(self.bytes // 4, dtype=torch.int32, device=dev)
        self.n = 0

    def __call__(self):
        self.n += 1
        self.buf.fill_(self.n)


def time_cold(fn, stream, flush, reps):
    """Median device time of `fn` over `reps` calls, each after an L2 flush
    (outside its event pair), after 3 warm-up calls."""
    for _ in range(3):
        fn()
    pairs = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in pairs)


def call_stats(ms, nbytes, peak):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 5), "alg_bytes": nbytes, "GB/s": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 4),
            "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}


COLD = "cold L2: median of 10 calls, each after a write of twice the L2 size"


def meta8_leg(q, K, V, w, dev, stream, flush, reps=10):
    """8-bit page metadata on the bench workload: its build from the 16-bit
    metadata, and decode_attn_select scoring it (cold L2);
    how many (batch, q-head) rows keep the 16-bit metadata's page set."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc

    meta = dkv.kv_meta_build(K)
    m8 = dkv.kv_meta8_build(meta)
    kk = min(w.top_k, w.P)
    ws = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k),
                     dtype=torch.uint8, device=dev)
    out = torch.empty(w.B, w.Hq, w.d, dtype=torch.float32, device=dev)
    sel = torch.empty(w.B, w.Hq, kk, dtype=torch.int32, device=dev)
    peak, _ = peaks()
    res = {"workload": w.name, "timing": COLD}
    ms = time_cold(lambda: dkv.kv_meta8_build(meta), stream, flush, reps)
    nbytes = acc.meta8_bytes(w.B, w.Hkv, w.d, w.N, w.S)
    gbs = nbytes / (ms * 1e-3) / 1e9
    res["kv_meta8_build"] = {"ms": round(ms, 5), "alg_bytes": nbytes, "GB/s": round(gbs, 1),
                             "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                             "frac_of_measured_hbm": round(gbs / peak, 4)}
    ms = time_cold(lambda: dkv.decode_attn_select(q, K, V, m8, w.top_k, out=out, selected=sel,
                                                  workspace=ws), stream, flush, reps)
    gathered = union_tokens(sel, w)
    nbytes = acc.select8_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, gathered, w.S)
    gbs = nbytes / (ms * 1e-3) / 1e9
    res["decode_attn_select"] = {"ms": round(ms, 5), "alg_bytes": nbytes, "GB/s": round(gbs, 1),
                                 "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                                 "frac_of_measured_hbm": round(gbs / peak, 4),
                                 "gathered_pages": gathered // w.S,
                                 "queries_per_s": round(w.B / (ms * 1e-3), 1)}
    sel16 = dkv.decode_attn_select(q, K, V, meta, w.top_k, return_selected=True)[1]
    same = (torch.sort(sel16, -1)[0] == torch.sort(sel, -1)[0]).all(-1)
    res["rows_with_16bit_page_set"] = round(float(same.float().mean().item()), 4)
    a, b = sel16.view(-1, kk).long(), sel.view(-1, kk).long()
    hit = torch.zeros(w.B * w.Hq, w.P, dtype=torch.bool, device=dev)
    hit.scatter_(1, a, True)
    overlap = hit.gather(1, b).float().mean()
    res["page_overlap_with_16bit"] = round(float(overlap.item()), 4)
    del m8, meta, ws
    return res


def paged_leg(q, K, V, w, dev, stream, flush, reps=10):
    """The bench workload held as a pool of 16-token blocks in shuffled order
    with a block table: exact and sparse attention timed like the contiguous
    cache (cold L2), outputs compared bit for bit."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc

    nb = w.B * w.P
    g = torch.Generator(device=dev).manual_seed(11)
    order = torch.randperm(nb, generator=g, device=dev)
    bt = order.view(w.B, w.P).to(torch.int32).contiguous()

    def pool_of(X):
        pool = torch.empty(nb, w.Hkv, w.S, w.d, dtype=X.dtype, device=dev)
        pool[order] = X.view(w.B, w.Hkv, w.P, w.S, w.d).permute(0, 2, 1, 3, 4).reshape(
            nb, w.Hkv, w.S, w.d)
        return pool

    PK, PV = dkv.PagedCache(pool_of(K), bt, w.N), dkv.PagedCache(pool_of(V), bt, w.N)
    meta = dkv.kv_meta_build(K)
    ws = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k),
                     dtype=torch.uint8, device=dev)
    kk = min(w.top_k, w.P)
    outs = {k: torch.empty(w.B, w.Hq, w.d, dtype=torch.float32, device=dev)
            for k in ("full", "full_paged", "select", "select_paged")}
    sel = torch.empty(w.B, w.Hq, kk, dtype=torch.int32, device=dev)
    calls = {
        "full": lambda: dkv.decode_attn_full(q, K, V, out=outs["full"], workspace=ws),
        "full_paged": lambda: dkv.decode_attn_full(q, PK, PV, out=outs["full_paged"], workspace=ws),
        "select": lambda: dkv.decode_attn_select(q, K, V, meta, w.top_k, out=outs["select"],
                                                 selected=sel, workspace=ws),
        "select_paged": lambda: dkv.decode_attn_select(q, PK, PV, meta, w.top_k,
                                                       out=outs["select_paged"], selected=sel,
                                                       workspace=ws),
    }
    peak, _ = peaks()
    res = {"workload": w.name, "pool_blocks": nb, "timing": COLD}
    for name, fn in calls.items():
        ms = time_cold(fn, stream, flush, reps)
        if name.startswith("full"):
            nbytes = acc.full_bytes(w.B, w.Hq, w.Hkv, w.d, w.N)
        else:
            nbytes = acc.select_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, union_tokens(sel, w), w.S)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 5), "GB/s": round(gbs, 1),
                     "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                     "frac_of_measured_hbm": round(gbs / peak, 4)}
    res["bitwise_equal_to_contiguous"] = bool(
        torch.equal(outs["full"], outs["full_paged"]) and
        torch.equal(outs["select"], outs["select_paged"]))
    del PK, PV
    return res


def page_size_leg(q, K, V, w, dev, stream, flush, reps=10):
    """Selection page sizes S = 4, 8, 16, 32, 64 ("TinyServe" page-size
    variants) on the bench workload at the same token budget (K = budget / S
    pages): metadata build and select, cold L2.  Pages of 4
    or 8 tokens are read as the 16-token cache pages holding them
    (cache_tokens_read); the roofline counts the selected pages' tokens."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc

    budget = w.top_k * w.S
    peak, _ = peaks()
    res = {"workload": w.name, "token_budget": budget, "timing": COLD}
    for S in (4, 8, 16, 32, 64):
        kk = budget // S
        P = (w.N + S - 1) // S
        ws = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, kk, page_size=S),
                         dtype=torch.uint8, device=dev)
        out = torch.empty(w.B, w.Hq, w.d, dtype=torch.float32, device=dev)
        sel = torch.empty(w.B, w.Hq, min(kk, P), dtype=torch.int32, device=dev)
        meta = dkv.kv_meta_build(K, page_size=S)
        calls = {"kv_meta_build": lambda: dkv.kv_meta_build(K, page_size=S),
                 "decode_attn_select": lambda: dkv.decode_attn_select(
                     q, K, V, meta, kk, out=out, selected=sel, workspace=ws, page_size=S)}
        r = {"top_k_pages": kk}
        for name, fn in calls.items():
            ms = time_cold(fn, stream, flush, reps)
            if name == "kv_meta_build":
                nbytes = acc.meta_bytes(w.B, w.Hkv, w.d, w.N, S)
            else:
                nbytes = acc.select_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, union_tokens(sel, w, S), S)
            gbs = nbytes / (ms * 1e-3) / 1e9
            r[name] = {"ms": round(ms, 5), "alg_bytes": nbytes, "GB/s": round(gbs, 1),
                       "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                       "frac_of_measured_hbm": round(gbs / peak, 4)}
        r["gathered_tokens"] = union_tokens(sel, w, S)
        if S < 16:
            r["cache_tokens_read"] = cache_tokens(sel, w, S)
        res[f"S{S}"] = r
        del meta, ws
    return res


def ratio_leg(name, q, K, V, dev, stream, flush, reps=10):
    """Selection ratio K / P in {0.1, 0.2, 0.3, 0.5} at S = 16 ("TinyServe"
    hyper-parameter search: page sizes and selection ratios): select per call
    (cold L2), its algorithmic bytes against the exact call's, and the model
    fraction 1/S + K S / L of the pages' normalised comparison."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc
    from workloads import make_inputs

    w = by_name(name)
    if q is None:
        widx = [x.name for x in WORKLOADS].index(w.name)
        q, K, V = make_inputs(w, seed=42 + widx, device=dev)
    meta = dkv.kv_meta_build(K)
    full_b = acc.full_bytes(w.B, w.Hq, w.Hkv, w.d, w.N)
    peak, _ = peaks()
    res = {"workload": w.name, "page_size": w.S, "pages": w.P, "timing": COLD}
    for ratio in (0.1, 0.2, 0.3, 0.5):
        kk = max(1, round(ratio * w.P))
        ws = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, kk), dtype=torch.uint8,
                         device=dev)
        out = torch.empty(w.B, w.Hq, w.d, dtype=torch.float32, device=dev)
        sel = torch.empty(w.B, w.Hq, kk, dtype=torch.int32, device=dev)
        ms = time_cold(lambda: dkv.decode_attn_select(q, K, V, meta, kk, out=out, selected=sel,
                                                      workspace=ws), stream, flush, reps)
        if dkv.read_device_status(ws) != 0:
            raise SystemExit(f"device status error in the ratio leg ({name}, {ratio})")
        gathered = union_tokens(sel, w)
        nbytes = acc.select_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, gathered, w.S)
        r = {"top_k_pages": kk, **call_stats(ms, nbytes, peak),
             "union_pages_per_unit": round(gathered / w.S / (w.B * w.Hkv), 1),
             "bytes_vs_exact": round(nbytes / full_b, 4),
             "model_1_over_S_plus_KS_over_L": round(1 / w.S + kk * w.S / w.N, 4),
             "queries_per_s": round(w.B / (ms * 1e-3), 1)}
        res[f"r{ratio}"] = r
        del ws
    return res


def reuse_leg(q, K, V, w, dev, stream, steps=16, sigma=0.15):
    """Cross-step page reuse ("TinyServe" 内存效率量化模型构建: a step moves the
    metadata plus rho K new pages; 系统实现意义: hot pages stay resident): a
    decode loop of `steps` steps on the bench workload, each appending one
    token (metadata of its page rebuilt) and selecting with a query that
    drifts by sigma N(0, 1) per step.  Run twice, through the hot-page call
    (pages gathered at the previous step kept in L2) and through the plain
    select; per step time, rho and bytes."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc

    g = torch.Generator(device=dev).manual_seed(77)
    qs, cur = [], q.float()
    for _ in range(steps):
        qs.append(cur.to(q.dtype))
        cur = cur + sigma * torch.randn(cur.shape, generator=g, device=dev)
    N0 = w.N - steps
    kk = min(w.top_k, w.P)
    ws = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k), dtype=torch.uint8,
                     device=dev)
    out = torch.empty(w.B, w.Hq, w.d, dtype=torch.float32, device=dev)
    sels = [torch.empty(w.B, w.Hq, kk, dtype=torch.int32, device=dev) for _ in range(steps)]
    lens = [torch.full((w.B,), N0 + t + 1, dtype=torch.int32, device=dev) for t in range(steps)]
    peak, _ = peaks()
    res = {"workload": w.name, "steps": steps, "query_drift_sigma": sigma,
           "timing": "each loop after an L2 flush; per step = loop time / steps"}
    flush = L2Flush(dev)
    for mode in ("hot", "plain"):
        meta = dkv.kv_meta_build(K, seq_lens=lens[0])
        hot = dkv.hot_state(w.B, w.Hkv, w.N, dev) if mode == "hot" else None

        def loop():
            for t in range(steps):
                if t > 0:
                    dkv.kv_meta_append(K, meta, seq_lens=lens[t])
                dkv.decode_attn_select(qs[t], K, V, meta, w.top_k, out=out, selected=sels[t],
                                       workspace=ws, seq_lens=lens[t], hot=hot, step=t + 1)

        loop()  # warm-up (and the selections the counters are checked against)
        if hot is not None:
            hot.zero_()
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        loop()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        if dkv.read_device_status(ws) != 0:
            raise SystemExit("device status error in the reuse leg")
        r = {"ms_per_step": round(ms, 5), "queries_per_s": round(w.B / (ms * 1e-3), 1)}
        if hot is not None:
            loads, hits = dkv.hot_stats(hot)
            first = union_tokens(sels[0], w) // w.S
            r["pages_gathered"] = loads
            r["pages_held_from_previous_step"] = hits
            # rho over steps 2.. (step 1 has no previous step)
            r["rho"] = round(1.0 - hits / max(1, loads - first), 4)
        res[mode] = r
        del meta, hot
    # bytes per step (steps 2..): metadata + the pages gathered (algorithmic),
    # and the pages new to the step (the rho K S term of the pages' model)
    loads, hits = res["hot"]["pages_gathered"], res["hot"]["pages_held_from_previous_step"]
    first = union_tokens(sels[0], w) // w.S
    per_step_pages = (loads - first) / (steps - 1)
    page_bytes = 2 * 16 * w.d * 2
    meta_b = acc.meta_bytes(w.B, w.Hkv, w.d, w.N, w.S) - w.B * w.Hkv * w.N * w.d * 2
    res["bytes_per_step"] = {
        "metadata": int(meta_b), "gathered_pages": int(per_step_pages * page_bytes),
        "new_pages_rho_K_S": int((per_step_pages - hits / (steps - 1)) * page_bytes)}
    gbs = (meta_b + per_step_pages * page_bytes) / (res["plain"]["ms_per_step"] * 1e-3) / 1e9
    res["plain"]["GB/s_algorithmic"] = round(gbs, 1)
    res["plain"]["frac_of_8tbs"] = round(gbs / NOMINAL_HBM_GBS, 4)
    res["hot_vs_plain_time"] = round(res["hot"]["ms_per_step"] / res["plain"]["ms_per_step"], 4)
    return res


def token_leg(q, K, V, w, dev, stream, flush, reps=10):
    """Token-level sparse attention on the bench workload, keeping the top 10%
    of the tokens per q-head (cold L2)."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc

    ktok = w.N // 10
    ws = torch.zeros(dkv.workspace_bytes_tokens(w.B, w.Hq, w.Hkv, w.d, w.N, ktok),
                     dtype=torch.uint8, device=dev)
    out = torch.empty(w.B, w.Hq, w.d, dtype=torch.float32, device=dev)

    def call():
        dkv.decode_attn_topk_tokens(q, K, V, ktok, out=out, workspace=ws)

    ms = time_cold(call, stream, flush, reps)
    nbytes = acc.token_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, ktok)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, _ = peaks()
    return {"workload": w.name, "top_k_tokens": ktok, "ms": round(ms, 5), "alg_bytes": nbytes,
            "GB/s": round(gbs, 1), "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
            "frac_of_measured_hbm": round(gbs / peak, 4),
            "queries_per_s": round(w.B / (ms * 1e-3), 1), "timing": COLD}


def headwise_leg(dev, stream):
    """1M-token context, 8 kv heads: exact attention all heads at once and one
    kv head at a time (HeadInfer), bitwise-equal outputs.  The 4 GiB working
    set is over 4x the L2, so calls are timed back to back."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc
    from workloads import make_inputs

    w = WORKLOADS[3]
    q, K, V = make_inputs(w, seed=45, device=dev)
    ws = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, 0), dtype=torch.uint8,
                     device=dev)
    ws1 = torch.zeros(dkv.workspace_bytes(w.B, w.G, 1, w.d, w.N, 0), dtype=torch.uint8,
                      device=dev)
    out = torch.empty(w.B, w.Hq, w.d, device=dev)
    out_hw = torch.empty_like(out)

    def all_heads():
        dkv.decode_attn_full(q, K, V, out=out, workspace=ws)

    def head_wise():
        for h in range(w.Hkv):
            dkv.decode_attn_full(q[:, h * w.G:(h + 1) * w.G], K[:, h:h + 1], V[:, h:h + 1],
                                 out=out_hw[:, h * w.G:(h + 1) * w.G], workspace=ws1)

    res = {}
    nbytes = acc.full_bytes(w.B, w.Hq, w.Hkv, w.d, w.N)
    peak, _ = peaks()
    for name, fn in [("all_heads", all_heads), ("head_wise_8_calls", head_wise)]:
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                     "frac_of_measured_hbm": round(gbs / peak, 4),
                     "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}
    res["bitwise_equal"] = bool(torch.equal(out, out_hw))
    res["workload"] = w.name
    del q, K, V
    torch.cuda.empty_cache()
    return res


def workload_leg(name, dev, stream, flush, reps=10):
    """Per-call device times and GB/s on another workload: the 1.3B-MHA shape
    (dense bf16) or the OPT-30B shape in the 4-bit format (quantise K and V,
    then metadata, exact and page-sparse attention over the 4-bit cache)."""
    import decode_attention_paged_kv_gb300 as dkv
    from decode_attention_paged_kv_gb300 import accounting as acc
    from workloads import make_inputs

    w = by_name(name)
    widx = [x.name for x in WORKLOADS].index(w.name)
    q, K, V = make_inputs(w, seed=42 + widx, device=dev)
    kk = min(w.top_k, w.P)
    ws_full = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, 0), dtype=torch.uint8,
                          device=dev)
    ws_sel = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k),
                         dtype=torch.uint8, device=dev)
    out_full = torch.empty(w.B, w.Hq, w.d, device=dev)
    out_sel = torch.empty_like(out_full)
    sel = torch.empty(w.B, w.Hq, kk, dtype=torch.int32, device=dev)
    state = {}
    calls = []
    if w.q4:
        def quant():
            state["K"], state["V"] = dkv.kv_quant4(K), dkv.kv_quant4(V)
        calls.append(("kv_quant4 (K and V)", quant,
                      2 * acc.quant4_bytes(w.B * w.Hkv * w.N, w.d)))
    else:
        state["K"], state["V"] = K, V

    def meta():
        state["meta"] = dkv.kv_meta_build(state["K"])

    def full():
        dkv.decode_attn_full(q, state["K"], state["V"], out=out_full, workspace=ws_full)

    def select():
        dkv.decode_attn_select(q, state["K"], state["V"], state["meta"], w.top_k, out=out_sel,
                               selected=sel, workspace=ws_sel)

    # the same selection over 8-bit metadata (built from the 16-bit one)
    out_sel8, sel8 = torch.empty_like(out_sel), torch.empty_like(sel)

    def meta8():
        state["meta8"] = dkv.kv_meta8_build(state["meta"])

    def select8():
        dkv.decode_attn_select(q, state["K"], state["V"], state["meta8"], w.top_k,
                               out=out_sel8, selected=sel8, workspace=ws_sel)

    calls += [("kv_meta_build", meta, acc.meta_bytes(w.B, w.Hkv, w.d, w.N, w.S, q4=w.q4)),
              ("decode_attn_full", full, acc.full_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, q4=w.q4)),
              ("decode_attn_select", select, None),
              ("kv_meta8_build", meta8, acc.meta8_bytes(w.B, w.Hkv, w.d, w.N, w.S)),
              ("decode_attn_select (8-bit metadata)", select8, "select8")]
    if not w.q4:
        # token-level sparse attention keeping the top 10% of the tokens per head
        ktok = max(1, w.N // 10)
        ws_tok = torch.zeros(dkv.workspace_bytes_tokens(w.B, w.Hq, w.Hkv, w.d, w.N, ktok),
                             dtype=torch.uint8, device=dev)
        out_tok = torch.empty_like(out_full)

        def tokens():
            dkv.decode_attn_topk_tokens(q, K, V, ktok, out=out_tok, workspace=ws_tok)

        calls.append(("decode_attn_topk_tokens (10%)", tokens,
                      acc.token_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, ktok)))
    for _ in range(3):
        for _, fn, _ in calls:
            fn()
    torch.cuda.synchronize()
    gathered = union_tokens(sel, w)
    # Each call on a cold L2 (its inputs, metadata included, come from HBM).
    times = {c: time_cold(fn, stream, flush, reps) for c, fn, _ in calls}
    if max(dkv.read_device_status(ws_full), dkv.read_device_status(ws_sel)) != 0:
        raise SystemExit(f"device status error on {w.name}")
    peak, _ = peaks()
    res = {"workload": w.name, "dtype": w.dtype, "kv_format": "q4g64" if w.q4 else "dense",
           "top_k_pages": w.top_k, "gathered_pages": gathered // w.S, "timing": COLD}
    for c, _, nbytes in calls:
        if nbytes is None:
            nbytes = acc.select_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, gathered, w.S, q4=w.q4)
        elif nbytes == "select8":
            nbytes = acc.select8_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, union_tokens(sel8, w), w.S,
                                       q4=w.q4)
        gbs = nbytes / (times[c] * 1e-3) / 1e9
        res[c] = {"ms": round(times[c], 5), "alg_bytes": nbytes, "GB/s": round(gbs, 1),
                  "frac_of_measured_hbm": round(gbs / peak, 4),
                  "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}
    res["decode_attn_full"]["queries_per_s"] = round(w.B / (times["decode_attn_full"] * 1e-3), 1)
    del q, K, V, state
    torch.cuda.empty_cache()
    return res


def e2e_leg(q, K, V, w, dev, stream, steps, chunks=8):
    """The same step through the public API with host inputs: every step copies
    q, K, V from pinned host memory and reads the outputs back.  The batch goes
    in `chunks` parts: a copy stream brings part c + 1 over while the compute
    stream runs part c (meta + exact + sparse on its sequences) and copies its
    outputs back, so only the last part's compute is not hidden by the copy."""
    import decode_attention_paged_kv_gb300 as dkv

    hq = q.cpu().pin_memory()
    hK = K.cpu().pin_memory()
    hV = V.cpu().pin_memory()
    kk = min(w.top_k, w.P)
    ho = torch.empty(w.B, w.Hq, w.d, dtype=torch.float32).pin_memory()
    hs = torch.empty_like(ho).pin_memory()
    hsel = torch.empty(w.B, w.Hq, kk, dtype=torch.int32).pin_memory()
    dq, dK, dV = torch.empty_like(q), torch.empty_like(K), torch.empty_like(V)
    ws_full = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, 0), dtype=torch.uint8,
                          device=dev)
    ws_sel = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k),
                         dtype=torch.uint8, device=dev)
    of, osl = torch.empty(w.B, w.Hq, w.d, device=dev), torch.empty(w.B, w.Hq, w.d, device=dev)
    sel = torch.empty(w.B, w.Hq, kk, dtype=torch.int32, device=dev)
    copy_stream = torch.cuda.Stream(device=dev)
    bounds = [(w.B * c) // chunks for c in range(chunks + 1)]
    parts = [(b0, b1) for b0, b1 in zip(bounds[:-1], bounds[1:]) if b1 > b0]

    def step():
        copy_stream.wait_stream(stream)  # the previous step is done with the buffers
        ready = []
        with torch.cuda.stream(copy_stream):
            for b0, b1 in parts:
                dq[b0:b1].copy_(hq[b0:b1], non_blocking=True)
                dK[b0:b1].copy_(hK[b0:b1], non_blocking=True)
                dV[b0:b1].copy_(hV[b0:b1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                ready.append(ev)
        for (b0, b1), ev in zip(parts, ready):
            stream.wait_event(ev)
            qc, Kc, Vc = dq[b0:b1], dK[b0:b1], dV[b0:b1]
            meta = dkv.kv_meta_build(Kc)
            dkv.decode_attn_full(qc, Kc, Vc, out=of[b0:b1], workspace=ws_full)
            dkv.decode_attn_select(qc, Kc, Vc, meta, w.top_k, out=osl[b0:b1], selected=sel[b0:b1],
                                   workspace=ws_sel)
            ho[b0:b1].copy_(of[b0:b1], non_blocking=True)
            hs[b0:b1].copy_(osl[b0:b1], non_blocking=True)
            hsel[b0:b1].copy_(sel[b0:b1], non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    n = max(3, min(steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    h2d = (hq.numel() * 2 + hK.numel() * 2 + hV.numel() * 2)
    d2h = ho.numel() * 4 + hs.numel() * 4 + hsel.numel() * 4
    return {"value": round(w.B / (ms * 1e-3), 1), "unit": "queries/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipeline": f"{len(parts)} batch parts, copy of part c + 1 under compute of part c"}


# ------------------------------------------------------------------ CPU oracle
def oracle_step(qs, Ks, Vs, w):
    """The oracle's pass over the given sequences: page metadata, exact
    attention, bound scores, top-K and attention over the selected pages."""
    import oracle

    is16 = int(w.dtype == "fp16")
    scale = 1.0 / math.sqrt(w.d)
    mn, mx = oracle.meta(Ks, w.S, is16)
    oracle.attention(qs, Ks, Vs, w.S, scale, is16)
    r = oracle.scores(qs, mn, mx, is16)
    sel = oracle.topk(r, w.top_k)
    oracle.attention(qs, Ks, Vs, w.S, scale, is16, sel=sel)


def cpu_baseline_leg(q, K, V, w, min_seconds=10.0, max_reps=40):
    """The oracle timed on the host cores over the whole batch, repeated until
    at least `min_seconds` of CPU work."""
    import oracle
    oracle.build()
    qs, Ks, Vs = bits(q.cpu()), bits(K.cpu()), bits(V.cpu())
    reps, t0 = 0, time.perf_counter()
    while reps < max_reps and (reps == 0 or time.perf_counter() - t0 < min_seconds):
        oracle_step(qs, Ks, Vs, w)
        reps += 1
    secs = time.perf_counter() - t0
    return {"value": round(reps * w.B / secs, 3), "unit": "queries/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"the whole batch ({w.B} sequences, all heads; meta + exact + sparse) "
                      f"x {reps} = {secs:.1f} s"}


def run_reference(args, rank, world, local):
    """The oracle as the reference arm, on the same workload and metric: each
    step decodes one sequence of the workload (all heads) on the host cores."""
    import oracle
    from workloads import make_inputs

    oracle.build()
    w = by_name(args.workload)
    widx = [x.name for x in WORKLOADS].index(w.name)
    one = w.replace(B=1)  # one sequence, drawn on the CPU (the oracle's own inputs)
    q, K, V = make_inputs(one, seed=42 + widx)
    qs, Ks, Vs = bits(q), bits(K), bits(V)
    for _ in range(max(1, args.warmup)):
        oracle_step(qs, Ks, Vs, one)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(qs, Ks, Vs, one)
    tot = time.perf_counter() - t0
    value = args.steps / tot
    sample = f"per step: sequence 0 of the workload (all heads): meta + exact + sparse"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "queries/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name},
            "cpu_baseline": {"value": round(value, 4), "unit": "queries/s",
                             "cores": oracle.threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "queries/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    rank, world, local = dist_info()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world, local)), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    if by_name(args.workload).q4 and args.legs:
        raise SystemExit("a 4-bit workload runs the step alone: add --no-extra")
    res, (q, K, V, w, widx, dev, stream, flush) = run_dkv(args, rank, world, local)
    if args.legs and rank == 0:
        L = args.legs
        if "e2e" in L:
            res["e2e"] = e2e_leg(q, K, V, w, dev, stream, args.steps)
        if "group" in L:
            res["group_select"] = group_select_leg(q, K, V, w, dev, stream, flush)
        if "paged" in L:
            res["paged"] = paged_leg(q, K, V, w, dev, stream, flush)
        if "pagesize" in L:
            res["page_sizes"] = page_size_leg(q, K, V, w, dev, stream, flush)
        if "ratios" in L:
            res["select_ratios"] = [ratio_leg(w.name, q, K, V, dev, stream, flush),
                                    ratio_leg(WORKLOADS[1].name, None, None, None, dev, stream,
                                              flush)]
        if "reuse" in L:
            res["reuse"] = reuse_leg(q, K, V, w, dev, stream)
        if "tokens" in L:
            res["topk_tokens"] = token_leg(q, K, V, w, dev, stream, flush)
        if "meta8" in L:
            res["meta8"] = meta8_leg(q, K, V, w, dev, stream, flush)
        if "cpu" in L:
            res["cpu_baseline"] = cpu_baseline_leg(q, K, V, w)
        del q, K, V
        torch.cuda.empty_cache()
        if "headwise" in L:
            res["headwise_1m"] = headwise_leg(dev, stream)
        if "others" in L:
            res["other_workloads"] = [workload_leg(n, dev, stream, flush)
                                      for n in (WORKLOADS[1].name, WORKLOADS[4].name)]
    if rank == 0:
        # the per-call summary last, where a tail of the line shows it
        res["per_call"] = res["roofline"]["calls"]
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
