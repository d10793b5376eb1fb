#!/usr/bin/env python
"""Benchmark of the DFlash2 draft tail on GB300: draft blocks/s and µs per call.

One step = one dflash2_draft_tail call (5 conv layers -> LM-head contraction with fused
top-16 + log-sum-exp -> merge -> transitions + Viterbi) over one batch of the page-shape
workload (block 8, hidden 5120, vocab 248,320, K=16, rank 256), inputs resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Device timing: the call is captured in a CUDA graph; before every step a 256 MiB buffer is
written to flush L2 (129 MB), then the step is bracketed by CUDA events on its stream.
The dominant kernel (the LM-head contraction) is timed the same way on its own for the
roofline. `e2e` times the public call with pinned host buffers: the step's inputs
(hidden, anchor) copied in and its results (path ids, path indices, scores) copied out
inside the timed region, each direction as one copy of a contiguous buffer. Under torchrun every rank runs its own replica (replicas only).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "draft blocks/s (B=1, block 8, hidden 5120, vocab 248320, K=16, rank 256, 5 conv layers)"


def metric_name(sh) -> str:
    """The metric of a workload's line (METRIC for the page shape at B=1)."""
    return (f"draft blocks/s (B={sh.batch}, block {sh.block}, hidden {sh.hidden}, vocab {sh.vocab}, "
            f"K={sh.top_k}, rank {sh.rank}, {sh.layers} conv layers)")

UNIT = "blocks/s"
FLUSH_BYTES = 256 << 20


def make_flush(torch, dev):
    """L2 flush between steps: write a 256 MiB buffer (twice L2), then read another one, so the
    step starts with a cold L2 that holds no dirty lines left by the flush itself."""
    wbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    rbuf = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        wbuf.fill_(1)
        rbuf.sum()
    return flush


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, help="workload (2: B=1 page shape)")
    ap.add_argument("--no-extra", action="store_true", help="skip the B=8/B=32 lines and the CPU baseline")
    ap.add_argument("--kernel", choices=["lmhead", "conv"], default=None,
                    help="time one kernel alone (profiling case) instead of the whole tail")
    ap.add_argument("--rows", type=int, default=8, help="--kernel: rows of the contraction")
    ap.add_argument("--vocab", type=int, default=62080, help="--kernel: vocabulary size")
    ap.add_argument("--oracle-child", type=int, default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.path = tempfile.mktemp(prefix="dflash2_clocks_", suffix=".csv")
        self.proc = None
        self.marks = []

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append(dict(ts=ts, index=int(parts[1]), sm=float(parts[2]), smax=float(parts[3]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], swp=parts[9]))
            except Exception:
                continue
        os.unlink(self.path)
        mine = [r for r in rows if r["index"] == self.index] or rows
        if len(self.marks) >= 2:
            t0, t1 = self.marks[0] - 0.05, self.marks[-1] + 0.05
            inside = [r for r in mine if t0 <= r["ts"] <= t1]
            mine = inside or mine
        if not mine:
            return None
        reasons = set()
        for r in mine:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                            ("swp", "sw_power_cap")):
                if r[k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in mine), "sm_max_mhz": max(r["smax"] for r in mine),
                "reasons": sorted(reasons), "samples": len(mine)}


# ---------------------------------------------------------------------------------- workload

def make_workload(config: int):
    import synth
    rc = synth.recipe(config)
    inp = synth.make_inputs(rc)
    return rc, inp


def synth_uniforms(B: int, T: int):
    """Seeded uniform draws [B, T] in [0, 1) for the sampling walk."""
    import synth
    return synth.uniform(7, 40, B * T).reshape(B, T)


def lmhead_alg_bytes(sh, M):
    """Algorithmic bytes of one LM-head contraction launch: the weight stream, the rows,
    and the partials written (per-partition top-16 + (max, sum) per row)."""
    return sh.vocab * sh.hidden * 2 + M * sh.hidden * 2


def tail_roofline_us(sh, M, bw_gbs, tflops):
    flop = 2.0 * M * sh.hidden * sh.vocab
    return max(flop / (tflops * 1e12), sh.vocab * sh.hidden * 2 / (bw_gbs * 1e9)) * 1e6


def traffic_record(M: int):
    """DRAM bytes per launch of the LM-head kernel from the committed ncu summary, if it was
    taken on the current kernel source (hash match) and for this row count; otherwise None."""
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", "lmhead_topk_b1_page.md")).read()
        src = os.path.join(ROOT, "block_drafter_dflash2_gb300", "csrc")
        h = hashlib.sha256()
        for name in ("tc_gemm.cuh", "ptx.cuh", "lmhead_tc.cu"):
            h.update(open(os.path.join(src, name), "rb").read())
        m_hash = re.search(r"^source_sha256: (\w+)", text, re.M)
        m_traffic = re.search(rf"^traffic_bytes_full_launch_M{M}: (\d+)", text, re.M)
        if not m_hash or m_hash.group(1) != h.hexdigest() or not m_traffic:
            return None
        return int(m_traffic.group(1))
    except Exception:
        return None


# ---------------------------------------------------------------------------------- ranks

def max_over_ranks(x: float, device) -> float:
    """Largest value of x over all ranks (the slowest rank's time); x itself with one rank."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, world: int, slowest_ms: float) -> float:
    """Whole-job units per second when every rank processes units_per_rank in its own time
    and the job ends with the slowest rank (replicas, no data exchange)."""
    return world * units_per_rank / (slowest_ms * 1e-3)


# ---------------------------------------------------------------------------------- ours

def run_ours(args, rank, world, local_rank):
    import torch
    import block_drafter_dflash2_gb300 as df2

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    df2.load()
    bw, tf, tf_sus, peak_kind = peaks()
    rc, inp = make_workload(args.config)
    sh = rc.shape
    B, T, H, K = sh.batch, sh.block, sh.hidden, sh.top_k
    M = B * T

    def up(a):
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    d = {k: up(inp[k]) for k in ("hidden", "lm_head", "U", "V", "conv_w", "anchor")}
    shape = df2.Shape.make(B, T, H, sh.vocab, K, sh.rank, sh.layers)
    ws = torch.zeros(df2.workspace_size(shape), dtype=torch.uint8, device=dev)
    flush = make_flush(torch, dev)
    out = dict(pid=torch.empty((B, T), dtype=torch.int32, device=dev),
               pix=torch.empty((B, T), dtype=torch.int32, device=dev),
               score=torch.empty((B,), dtype=torch.float32, device=dev))
    stream = torch.cuda.Stream(device=dev)

    def call(hidden, anchor, shp=shape, o=out, s=stream):
        df2.draft_tail(shp, hidden, d["lm_head"], d["U"], d["V"], d["conv_w"], anchor, o["pid"], o["pix"],
                       o["score"], ws, stream=s)

    def timed(fn, steps, warm):
        """Per-step device time (ms) of fn on `stream`, L2 flushed before every step."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for _ in range(warm):
                flush()
                fn()
            torch.cuda.synchronize(dev)
            for e0, e1 in evs:
                flush()
                e0.record(stream)
                fn()
                e1.record(stream)
            torch.cuda.synchronize(dev)
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    # correctness of the captured call before timing it
    with torch.cuda.stream(stream):
        call(d["hidden"], d["anchor"])
    torch.cuda.synchronize(dev)
    assert df2.read_device_error(ws, stream) == 0, "device error word set"
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call(d["hidden"], d["anchor"])

    clocks = ClockSampler(local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush()
            graph.replay()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark()
    step_ms = timed(graph.replay, args.steps, 0)
    clocks.mark()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    total_ms = sum(step_ms)
    t_max = max_over_ranks(total_ms, dev)
    clk = clocks.stop()

    def graphed(fn):
        """fn captured in its own CUDA graph: times the kernels, not the host call."""
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g.replay

    # each stage on its own; the dominant kernel (the LM-head contraction with its fused
    # epilogue) gives the roofline figure
    z = torch.empty_like(d["hidden"])
    ids = torch.empty((M, K), dtype=torch.int32, device=dev)
    lp = torch.empty((M, K), dtype=torch.float32, device=dev)
    conv_ms = timed(graphed(lambda: df2.conv(shape, d["hidden"], d["conv_w"], z, ws, stream=stream)),
                    min(args.steps, 50), 3)
    lm_ms = timed(graphed(lambda: df2.lmhead_partials(shape, z, d["lm_head"], ws, stream=stream)), args.steps, 3)
    merge_ms = timed(graphed(lambda: df2.merge_partials(shape, ids, lp, None, ws, stream=stream)),
                     min(args.steps, 50), 3)
    walk_ms = timed(graphed(lambda: df2.viterbi(shape, d["anchor"], ids, lp, d["U"], d["V"], out["pid"], out["pix"],
                                                out["score"], ws, stream=stream)), min(args.steps, 50), 3)

    # end to end through the public call, host buffers in and out: the step's inputs (hidden
    # rows, then the anchor ids) sit in one pinned buffer and its results (path ids, path
    # indices, scores) in one device buffer, as a caller would lay them out, so each
    # direction is one copy of the same bytes
    hid_bytes = inp["hidden"].nbytes
    in_bytes = hid_bytes + inp["anchor"].nbytes
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    h_in[:hid_bytes].copy_(torch.from_numpy(inp["hidden"].view(np.uint8).reshape(-1)))
    h_in[hid_bytes:].copy_(torch.from_numpy(np.ascontiguousarray(inp["anchor"]).view(np.uint8).reshape(-1)))
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    d_hidden = d_in[:hid_bytes].view(torch.int16).view(B, T, H)
    d_anchor = d_in[hid_bytes:].view(torch.int32)
    n_out = 2 * B * T + B
    d_out = torch.empty(n_out, dtype=torch.int32, device=dev)
    h_out = torch.empty(n_out, dtype=torch.int32).pin_memory()
    e2e_o = dict(pid=d_out[:B * T].view(B, T), pix=d_out[B * T:2 * B * T].view(B, T),
                 score=d_out[2 * B * T:].view(torch.float32))

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        call(d_hidden, d_anchor, o=e2e_o)
        h_out.copy_(d_out, non_blocking=True)

    e2e_ms = timed(e2e_step, args.steps, 3)
    assert np.array_equal(h_out[:B * T].numpy().reshape(B, T), out["pid"].cpu().numpy())
    e2e_total = max_over_ranks(sum(e2e_ms), dev)

    extra = {}
    if not args.no_extra and world == 1:
        # the same workload with the context gate H(h_t): gate rows contracted in the LM-head
        # pass (R extra columns), applied to the transitions in the walk
        gw = up(inp["gate_w"])
        gate_o = torch.empty((B, T, sh.rank), dtype=torch.float32, device=dev)

        def call_g():
            df2.draft_tail_gated(shape, d["hidden"], d["lm_head"], d["U"], d["V"], d["conv_w"], gw, d["anchor"],
                                 out["pid"], out["pix"], out["score"], ws, gate=gate_o, stream=stream)
        with torch.cuda.stream(stream):
            call_g()
        torch.cuda.synchronize(dev)
        assert df2.read_device_error(ws, stream) == 0
        gg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gg, stream=stream):
            call_g()
        ms_adj = timed(graph.replay, args.steps, 3)  # the ungated tail again, right before
        us_adj = statistics.mean(ms_adj) * 1e3
        msg = timed(gg.replay, args.steps, 3)
        usg = statistics.mean(msg) * 1e3
        extra["B=1 gated"] = {"us_per_call": round(usg, 2), "blocks_per_s": round(B / (usg * 1e-6), 1),
                              "tail_roofline_frac": round(tail_roofline_us(sh, M, bw, tf) / usg, 4),
                              "over_ungated_us": round(usg - us_adj, 2), "ungated_adjacent_us": round(us_adj, 2)}

        # and with the walk sampling a path at temperature 1 (fixed seeded uniforms)
        u_d = up(np.asarray(synth_uniforms(B, T), dtype=np.float32))

        def call_s():
            df2.draft_tail_sampled(shape, d["hidden"], d["lm_head"], d["U"], d["V"], d["conv_w"], d["anchor"], 1.0,
                                   u_d, out["pid"], out["pix"], out["score"], ws, stream=stream)
        with torch.cuda.stream(stream):
            call_s()
        torch.cuda.synchronize(dev)
        assert df2.read_device_error(ws, stream) == 0
        gs = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gs, stream=stream):
            call_s()
        ms_adj = timed(graph.replay, args.steps, 3)
        us_adj = statistics.mean(ms_adj) * 1e3
        mss = timed(gs.replay, args.steps, 3)
        uss = statistics.mean(mss) * 1e3
        extra["B=1 sampled T=1"] = {"us_per_call": round(uss, 2), "blocks_per_s": round(B / (uss * 1e-6), 1),
                                    "over_viterbi_us": round(uss - us_adj, 2), "viterbi_adjacent_us": round(us_adj, 2)}

    # the other workloads of the metric, each on its own seeded inputs (weights included):
    # B=8 with planted peaks, B=32 with duplicated anchors, and the B=64 block-16 stress case
    # (1024 rows into the LM head: past the ridge, tensor-bound)
    if not args.no_extra and world == 1:
        for cfg in (3, 4, 5):
            rc_c, inp_c = make_workload(cfg)
            sh_c = rc_c.shape
            Bc, Tc = sh_c.batch, sh_c.block
            Mc = Bc * Tc
            dc = {k: up(inp_c[k]) for k in ("hidden", "lm_head", "U", "V", "conv_w", "anchor")}
            del inp_c
            shp2 = df2.Shape.make(Bc, Tc, H, sh_c.vocab, K, sh_c.rank, sh_c.layers)
            ws2 = torch.zeros(df2.workspace_size(shp2), dtype=torch.uint8, device=dev)
            o2 = dict(pid=torch.empty((Bc, Tc), dtype=torch.int32, device=dev),
                      pix=torch.empty((Bc, Tc), dtype=torch.int32, device=dev),
                      score=torch.empty((Bc,), dtype=torch.float32, device=dev))

            def call2(shp2=shp2, o2=o2, ws2=ws2, dc=dc):
                df2.draft_tail(shp2, dc["hidden"], dc["lm_head"], dc["U"], dc["V"], dc["conv_w"], dc["anchor"],
                               o2["pid"], o2["pix"], o2["score"], ws2, stream=stream)
            with torch.cuda.stream(stream):
                call2()
            torch.cuda.synchronize(dev)
            assert df2.read_device_error(ws2, stream) == 0
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2, stream=stream):
                call2()
            ms2 = timed(g2.replay, args.steps, 3)
            z2 = torch.empty_like(dc["hidden"])
            cv2 = timed(graphed(lambda: df2.conv(shp2, dc["hidden"], dc["conv_w"], z2, ws2, stream=stream)), 20, 3)
            lm2 = timed(graphed(lambda: df2.lmhead_partials(shp2, z2, dc["lm_head"], ws2, stream=stream)),
                        args.steps, 3)
            us = statistics.mean(ms2) * 1e3
            lmu = statistics.mean(lm2) * 1e3
            roof = tail_roofline_us(sh_c, Mc, bw, tf)
            roof_sus = tail_roofline_us(sh_c, Mc, bw, tf_sus)
            lm_tflops = 2.0 * Mc * H * sh_c.vocab / (lmu * 1e-6) / 1e12
            extra[f"B={Bc}"] = {
                "workload": rc_c.name, "block": Tc, "rows": Mc,
                "us_per_call": round(us, 2), "blocks_per_s": round(Bc / (us * 1e-6), 1),
                "tail_roofline_us": round(roof, 1), "tail_roofline_frac": round(roof / us, 4),
                "tail_roofline_frac_sustained_bf16": round(roof_sus / us, 4),
                "bound": "tensor" if 2.0 * Mc * H * sh_c.vocab / (tf * 1e12) > sh_c.vocab * H * 2 / (bw * 1e9)
                else "hbm",
                "lmhead_us": round(lmu, 2), "conv_us": round(statistics.mean(cv2) * 1e3, 2),
                "lmhead_hbm_gbs": round(lmhead_alg_bytes(sh_c, Mc) / (lmu * 1e-6) / 1e9, 1),
                "lmhead_tflops": round(lm_tflops, 1),
                "lmhead_tensor_frac_burst": round(lm_tflops / tf, 4),
                "lmhead_tensor_frac_sustained": round(lm_tflops / tf_sus, 4)}
            del dc, ws2, g2, z2
            torch.cuda.empty_cache()

    us = total_ms / args.steps * 1e3
    lm_us = statistics.mean(lm_ms) * 1e3
    achieved = lmhead_alg_bytes(sh, M) / (lm_us * 1e-6) / 1e9
    value = replica_throughput(B * args.steps, world, t_max)
    e2e_val = replica_throughput(B * args.steps, world, e2e_total)
    # one tail call: the conv chain (all layers, one cooperative launch), the LM-head
    # contraction, and the merge fused with the transitions and the walk
    launches_per_step = (1 if sh.layers > 0 else 0) + 2
    # the LM head's roofline: its weight stream against the copy bandwidth, or past the ridge its
    # contraction against the bf16 tensor peak; above one row chunk the CTA-pair kernel runs
    flop = 2.0 * M * sh.hidden * sh.vocab
    tensor_bound = flop / (tf * 1e12) > lmhead_alg_bytes(sh, M) / (bw * 1e9)
    lm_kernel = ("tc_gemm_pair_kernel<EpiTopK> (CTA-pair LM-head contraction + fused top-16/lse)" if M > 128
                 else "tc_gemm_kernel<EpiTopK> (LM-head contraction + fused top-16/lse)")
    if tensor_bound:
        lm_tf = flop / (lm_us * 1e-6) / 1e12
        roofline = {"bound": "tensor", "achieved": round(lm_tf, 1), "peak": tf, "unit": "TFLOP/s",
                    "frac": round(lm_tf / tf, 4), "traffic": traffic_record(M), "kernel": lm_kernel,
                    "peak_source": f"{peak_kind} bf16_tflops"}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": bw, "unit": "GB/s",
                    "frac": round(achieved / bw, 4), "traffic": traffic_record(M), "kernel": lm_kernel,
                    "peak_source": f"{peak_kind} hbm_gbs"}
    line = {
        "metric": metric_name(sh), "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded Philox inputs, random weights)",
        "config": {"workload": rc.name, "batch": B, "block": T, "hidden": H, "vocab": sh.vocab, "top_k": K,
                   "rank": sh.rank, "conv_layers": sh.layers, "parallelism": "replicas" if world > 1 else "single",
                   "timing": "CUDA graph replay, CUDA events per step",
                   "l2": "flushed before every step (256 MiB write, then a 256 MiB read)"},
        "us_per_call": round(us, 2),
        "us_per_call_p10_p90": [round(float(np.percentile(step_ms, 10)) * 1e3, 2),
                                round(float(np.percentile(step_ms, 90)) * 1e3, 2)],
        "tail_roofline_frac": round(tail_roofline_us(sh, M, bw, tf) / us, 4),
        "stages_us": {"conv_5_layers": round(statistics.mean(conv_ms) * 1e3, 2), "lmhead": round(lm_us, 2),
                      "merge": round(statistics.mean(merge_ms) * 1e3, 2),
                      "transition_walk": round(statistics.mean(walk_ms) * 1e3, 2)},
        "roofline": roofline,
        "e2e": {"value": round(e2e_val, 2), "unit": UNIT,
                "h2d_bytes_per_step": int(in_bytes), "d2h_bytes_per_step": int(n_out * 4),
                "us_per_call": round(e2e_total / args.steps * 1e3, 2)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "also": extra,
    }
    return line, rc, inp


def run_kernel_case(args):
    """Profiling case: the LM-head contraction with its fused epilogue alone, on `rows` page-shape
    rows and a `vocab`-row head (default 62,080 rows = 636 MB, larger than L2)."""
    import torch
    import synth
    import block_drafter_dflash2_gb300 as df2
    df2.load()
    dev = torch.device("cuda", 0)
    conv = args.kernel == "conv"
    rows, block = (args.rows // 8, 8) if conv else (args.rows, 1)
    rc = synth.scaled_recipe(synth.recipe(2), batch=rows, block=block, vocab=args.vocab if not conv else 64,
                             layers=5 if conv else 0)
    sh = rc.shape
    inp = synth.make_inputs(rc)
    z = torch.from_numpy(inp["hidden"].view(np.int16)).to(dev)
    w = torch.from_numpy(inp["lm_head"].view(np.int16)).to(dev)
    cw = torch.from_numpy(inp["conv_w"].view(np.int16)).to(dev)
    y = torch.empty_like(z)
    shape = df2.Shape.make(rows, block, sh.hidden, sh.vocab, sh.top_k, sh.rank, sh.layers)
    ws = torch.zeros(df2.workspace_size(shape), dtype=torch.uint8, device=dev)
    flush = make_flush(torch, dev)
    ms = []
    for i in range(args.warmup + args.steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if conv:
            df2.conv(shape, z, cw, y, ws)
        else:
            df2.lmhead_partials(shape, z, w, ws)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            ms.append(e0.elapsed_time(e1))
    assert df2.read_device_error(ws) == 0
    us = statistics.mean(ms) * 1e3
    if conv:
        print(json.dumps({"kernel": "conv (5 layers)", "rows": rows * block, "hidden": sh.hidden, "us": round(us, 2)}),
              flush=True)
        return
    print(json.dumps({"kernel": "lmhead_partials", "rows": args.rows, "vocab": sh.vocab, "hidden": sh.hidden,
                      "us": round(us, 2), "alg_gbs": round(lmhead_alg_bytes(sh, args.rows) / (us * 1e-6) / 1e9, 1),
                      "tflops": round(2.0 * args.rows * sh.hidden * sh.vocab / (us * 1e-6) / 1e12, 1)}), flush=True)


# ---------------------------------------------------------------------------------- oracle

def oracle_shard_step(rc, inp, shard: int, n_shards: int):
    """One bounded sample of the workload for the CPU oracle: the whole tail (conv, logits,
    lse, full-sort top-K, transitions, Viterbi) on vocabulary shard `shard` of `n_shards`."""
    from oracle import core as O
    import synth
    sh = rc.shape
    Vs = sh.vocab // n_shards
    v0 = shard * Vs
    sub = dict(inp)
    sub["lm_head"] = inp["lm_head"][v0:v0 + Vs]
    sub["U"] = inp["U"][v0:v0 + Vs]
    sub["V"] = inp["V"][v0:v0 + Vs]
    sub["anchor"] = (np.asarray(inp["anchor"]) % Vs).astype(np.int32)
    sh2 = synth.Shape(**{**sh.__dict__, "vocab": Vs})
    return O.draft_tail(sub, sh2)


def oracle_child(config: int) -> None:
    """Child process of the CPU baseline: one full block of the workload through the oracle, timed
    after the inputs are generated; prints the seconds. BLAS threads are fixed by the parent's
    environment before numpy loads."""
    from oracle import core as O
    rc, inp = make_workload(config)
    t0 = time.perf_counter()
    O.draft_tail(inp, rc.shape)
    print(json.dumps({"seconds": time.perf_counter() - t0}), flush=True)


def oracle_block_seconds(config: int, threads: int) -> float:
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", str(config)], env=env,
                         capture_output=True, text=True, check=True)
    return float(json.loads(out.stdout.strip().splitlines()[-1])["seconds"])


def cpu_machine() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline(rc, config: int):
    """The oracle on the host: one full block single-threaded (the plain, slow CPU implementation,
    one BLAS thread) and with BLAS on every host core."""
    cores = os.cpu_count() or 1
    t1 = oracle_block_seconds(config, 1)
    tn = oracle_block_seconds(config, cores)
    return {"value": round(1.0 / t1, 5), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"one full block of {rc.name} (all {rc.shape.block} slots, whole vocabulary) through the "
                      f"numpy float64 oracle, one thread: {t1:.1f} s; CPU: {cpu_machine()}",
            "all_cores": {"value": round(1.0 / tn, 5), "cores": cores, "seconds": round(tn, 2)}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    rc, inp = make_workload(args.config)
    # calibrate the per-step sample: a vocabulary shard sized so warm-up + timed steps stay
    # within a few minutes
    n_shards = 64
    t0 = time.perf_counter()
    oracle_shard_step(rc, inp, 0, n_shards)
    t_one = time.perf_counter() - t0
    budget = 150.0
    while n_shards > 1 and t_one * 2 * (args.steps + args.warmup) < budget:
        n_shards //= 2
        t_one *= 2
    for i in range(args.warmup):
        oracle_shard_step(rc, inp, i % n_shards, n_shards)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_shard_step(rc, inp, i % n_shards, n_shards)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps / n_shards / total
    sample = (f"each step: the oracle's whole tail on 1/{n_shards} of the vocabulary "
              f"({rc.shape.vocab // n_shards} tokens) for all {rc.shape.block} slots of {rc.name}; "
              f"blocks counted as steps/{n_shards}")
    return {"impl": "reference", "metric": metric_name(rc.shape), "value": round(value, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Philox inputs, random weights)",
            "config": {"workload": rc.name, "batch": rc.shape.batch, "block": rc.shape.block},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.oracle_child is not None:
        oracle_child(args.oracle_child)
        return
    if args.kernel:
        run_kernel_case(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line, rc, inp = run_ours(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_extra:
        del inp
        line["cpu_baseline"] = cpu_baseline(rc, args.config)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
