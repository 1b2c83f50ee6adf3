#!/usr/bin/env python
"""KDA fwd+bwd throughput on GB300: one JSON line on rank 0.

A step is one pass of the whole hot path over one batch: kda_fwd (writing the saved set) followed
by kda_bwd (saved mode) on the 4doc workload (16384 tokens in documents of 8192/4096/3072/1024,
64 heads, d = 128, raw gate, no fused L2 norm), inputs already resident in HBM.  Timing: W warm-up
steps, then K steps bracketed by a barrier and torch.cuda.synchronize(), CUDA events on the
launching stream, max over ranks.  The inputs are larger than L2 (q, k, v, a, dO ~2.1 GB), so no
flush is needed between steps.

Also reported: per-kernel device time (CUDA events around each launch, a second pass of K
steps), the dominant kernel's roofline position, an end-to-end number through the public API
with host buffers (pinned H2D of every input and D2H of the parameter gradients inside every
step), SM clocks sampled during the timed region, and the FP64 oracle timed on the host cores on
a bounded sample of the same workload.

--impl reference times the oracle (the reference arm for this build) on the same workload,
metric and unit, each step a bounded sample (a subset of heads), scaled to the full workload.
Multi-GPU (torchrun, one process per GPU): every rank runs its own copy of the workload (the
path shards by heads / documents with no exchange), so scaling is weak.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "4doc"
PAGES_MS = 4.2789  # 4doc:raw:off:saved fwd+bwd on GB300 (sm_103a), the chunked KDA package page


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-profile", action="store_true", help="skip the per-kernel event pass")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-configuration rows")
    ap.add_argument("--no-protocol", action="store_true",
                    help="skip the pages' protocol pass (15 samples of 20 steps)")
    ap.add_argument("--only", choices=["conv", "walk"], default=None,
                    help="run only the conv (16384 x 8192, fwd + bwd) or the transfer-walk "
                         "formats (4 documents x 8 fragments x 16 heads) a few times and print "
                         "their times (profiling targets)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max_ms(ms, world, device):
    """Max over ranks of a per-rank time (the slowest rank sets the step time)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, max_ms):
    """Whole-job tokens/s: every rank processes its own batch (weak scaling)."""
    return world * tokens_per_rank / (max_ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------------------------
# clocks sampled during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------------
# algorithmic bytes per kernel launch (method inputs and outputs a kernel must touch; workspace
# intermediates excluded), per token-head, in the bench's I/O formats: q, k, v, beta, dO bf16;
# gate fp32; outputs o, dq, dk, dv, dbeta, dg fp32 (parity-grade outputs)


def alg_bytes_per_token_head(kernel, out_bytes=4):
    """Method inputs and outputs the kernel must touch, per token-head; out_bytes = bytes of one
    o / dq / dk / dv / dbeta element (4: fp32 outputs, 2: bf16 outputs, the inputs' format)."""
    qkv, beta, gate, dO = 3 * 256, 2, 512, 256
    o, dqkv, dbeta, dg = 128 * out_bytes, 3 * 128 * out_bytes, out_bytes, 512
    table = {
        "k_intra_fwd": qkv + beta + gate,                    # reads the chunk inputs
        "k_chain_fwd": o,                                    # writes o
        "k_chain_bwd": dO,                                   # reads dO
        "k_bwd_gemms_tc": dO,                                # reads dO
        "k_bwd_intra": qkv + beta + gate + dqkv + dbeta + dg,  # reads inputs, writes grads
    }
    return table.get(kernel)


def step_bytes_per_token_head(out_bytes):
    """Algorithmic bytes of a whole fwd (and fwd+bwd) per token-head: q, k, v, beta, gate in,
    o out; the backward reads them and dO again and writes dq, dk, dv, dbeta, dg.  out_bytes = 2
    (outputs in the inputs' bf16 format) gives 1,538 / 4,358 B; 4 (the library's fp32 outputs)
    1,794 / 5,384 B."""
    inputs = 3 * 256 + 2 + 512
    fwd = inputs + 128 * out_bytes
    bwd = inputs + 256 + 3 * 128 * out_bytes + out_bytes + 512
    return fwd, fwd + bwd


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it is for the kernel's current code."""
    path = os.path.join(ROOT, "profiles", "traffic_4doc.txt")
    if not os.path.exists(path):
        return None
    from linear_attention_chunked_gb300 import build as b
    sha = b.source_digest(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#"):
            k, w, s, byts = parts[:4]
            if k == kernel and w == workload and s == sha:
                return float(byts)
    return None


# ---------------------------------------------------------------------------------------------
# per-configuration rows: fwd and fwd+bwd ms with the pages' protocol (median of 15 samples, each
# 20 back-to-back calls / 20)

# (workload, backward mode, chunk groups per document: 0 = one serial chain per document)
ROWS = [("m2", "saved", 0), ("R2", "saved", 0), ("R2", "saved", 48), ("R2fast", "saved", 0),
        ("1doc", "saved", 0), ("1doc", "saved", 64), ("4doc", "saved", 0), ("4doc", "replay", 0),
        ("longpack", "saved", 0)]


def _time_calls(fn, samples=15, calls=20):
    import torch
    fn()
    torch.cuda.synchronize()
    out = []
    for _ in range(samples):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(calls):
            fn()
        b.record()
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b) / calls)
    return statistics.median(out)


# per token-head: method inputs and outputs (q, k, v, beta, gate, o; + dO, dq, dk, dv, dbeta, dg)
# with bf16 outputs (the inputs' format) and with the fp32 outputs every bench run writes, and FLOPs of
# the chunked method with 64-token chunks, head dim 128
BYTES_FWD, BYTES_FWD_BWD = step_bytes_per_token_head(2)        # 1,538 / 4,358
BYTES_FWD_F32, BYTES_FWD_BWD_F32 = step_bytes_per_token_head(4)  # 1,794 / 5,384
FLOP_FWD, FLOP_FWD_BWD = 180224, 540672


def run_rows(dev, hbm_gbs, bf16_tflops):
    import torch
    from linear_attention_chunked_gb300 import inputs, kda
    rows = {}
    for name, mode, G in ROWS:
        w = inputs.WORKLOADS[name]
        x = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inputs.workload_inputs(name).items()}
        kw = dict(gate=w.gate, A_log=x["A_log"], dt_bias=x["dt_bias"], l2norm=w.l2norm)
        if w.fragments:
            frag, doc_frag = [], [0]
            for L in w.lens:
                pieces = inputs.fragment_lens(L, w.fragments)
                frag += pieces
                doc_frag.append(doc_frag[-1] + len(pieces))
            fcu = inputs.cu_from_lens(frag).to(dev)
            dfr = torch.tensor(doc_frag, dtype=torch.int32, device=dev)
            a = (x["q"], x["k"], x["v"], x["beta"], x["g"], fcu)
            T, F, H = w.T, len(frag), w.H
            wsf, svb = kda.kda_workspace_size(T, F, H, kda.KDA_OP_FWD)
            wsb, _ = kda.kda_workspace_size(T, F, H, kda.KDA_OP_BWD_SAVED)
            ws = torch.empty(max(wsf, wsb), dtype=torch.uint8, device=dev)
            saved = torch.empty(svb, dtype=torch.uint8, device=dev)
            st = {}

            def fwd():
                M, B = kda.kda_fragment_summary(*a, mode=kda.KDA_FRAG_FWD, ws=ws, **kw)
                S_in, S_fin = kda.kda_transfer_walk(dfr, M, B)
                o, _, _ = kda.kda_fwd(*a, h0=S_in, saved=saved, ws=ws, **kw)
                st.update(M=M, B=B, S_in=S_in)

            def fwd_bwd():
                fwd()
                C = kda.kda_fragment_summary(*a, mode=kda.KDA_FRAG_BWD, dO=x["dO"], ws=ws, **kw)
                dS_end, dh0 = kda.kda_transfer_walk(dfr, st["M"], C, reverse=True)
                kda.kda_bwd(*a, x["dO"], saved=saved, h0=st["S_in"], dht=dS_end, want_dh0=False,
                            ws=ws, **kw)
        else:
            a = (x["q"], x["k"], x["v"], x["beta"], x["g"], x["cu_seqlens"])
            T, N, H = w.T, w.N, w.H
            replay = mode == "replay"
            kw["group_chunks"] = G
            wsf, svb = kda.kda_workspace_size(T, N, H, kda.KDA_OP_FWD, group_chunks=G)
            wsb, _ = kda.kda_workspace_size(T, N, H, kda.KDA_OP_BWD_REPLAY if replay else
                                            kda.KDA_OP_BWD_SAVED, group_chunks=G)
            ws = torch.empty(max(wsf, wsb), dtype=torch.uint8, device=dev)
            saved = None if replay else torch.empty(svb, dtype=torch.uint8, device=dev)

            def fwd():
                kda.kda_fwd(*a, saved=saved, save=not replay, ws=ws, **kw)

            def fwd_bwd():
                fwd()
                kda.kda_bwd(*a, x["dO"], saved=saved, want_dh0=False, ws=ws, **kw)
        f_ms = _time_calls(fwd)
        fb_ms = _time_calls(fwd_bwd)
        # roofline position of the row: algorithmic bytes and FLOPs per token-head (method I/O and
        # chunked-method FLOPs; replay adds one forward's FLOPs) against the measured peaks
        th = w.T * w.H
        fb_flop = FLOP_FWD_BWD + (FLOP_FWD if mode == "replay" else 0)
        rows[f"{w.row}:{mode}" + (f":groups{G}" if G else "")] = {
            "T": w.T, "H": w.H, "fwd_ms": round(f_ms, 4), "fwd_bwd_ms": round(fb_ms, 4),
            "fwd_bwd_tokens_per_s": round(w.T / (fb_ms / 1e3)),
            "fwd_byte_frac": round(th * BYTES_FWD / (f_ms * 1e6) / hbm_gbs, 4),
            "fwd_bwd_byte_frac": round(th * BYTES_FWD_BWD / (fb_ms * 1e6) / hbm_gbs, 4),
            "fwd_byte_frac_fp32_out": round(th * BYTES_FWD_F32 / (f_ms * 1e6) / hbm_gbs, 4),
            "fwd_bwd_byte_frac_fp32_out": round(th * BYTES_FWD_BWD_F32 / (fb_ms * 1e6) / hbm_gbs, 4),
            "fwd_bwd_flop_frac": round(th * fb_flop / (fb_ms * 1e9) / bf16_tflops, 4)}
        if w.fragments:
            rows[f"{w.row}:walk"] = walk_formats(st["M"], st["B"], dfr)
        del x, ws, saved
        torch.cuda.empty_cache()
    rows["conv:qkv"] = conv_row(dev, hbm_gbs)
    return rows


def walk_formats(M, B, dfr):
    """Each transfer-walk product format: forward-walk ms on the long-pack summaries (pages'
    protocol), and max|S_in - S_in(FP32 FMA walk)| / rms on the same shapes with a contractive
    random M (the long-pack M has decayed to ~0 over 15,000 tokens, which would make every
    format agree)."""
    import torch
    from linear_attention_chunked_gb300 import kda
    gen = torch.Generator("cpu").manual_seed(0)
    Mr = (torch.randn(M.shape, generator=gen) * 0.05).to(M.device)
    ref, _ = kda.kda_transfer_walk(dfr, Mr, B, precision=kda.KDA_WALK_FP32)
    out = {}
    for name, prec in kda.WALK_PRECISIONS.items():
        S_in, _ = kda.kda_transfer_walk(dfr, Mr, B, precision=prec)
        torch.cuda.synchronize()
        diff = float((S_in - ref).abs().max() / ref.pow(2).mean().sqrt().clamp_min(1e-30))
        ms = _time_calls(lambda: kda.kda_transfer_walk(dfr, M, B, precision=prec))
        out[name] = {"ms": round(ms, 4), "vs_fp32_walk": diff}
    return out


def conv_row(dev, hbm_gbs):
    """The width-4 causal conv1d + SiLU over q, k and v together (C = 3 x 64 heads x 128) of the
    4doc pack, bf16 in and out: fwd and fwd+bwd ms and the HBM fraction of their algorithmic bytes
    (fwd: x in, y out; bwd: x and dy in, dx out; 2 bytes each per channel-token)."""
    import torch
    from linear_attention_chunked_gb300 import inputs, kda
    w_ = inputs.WORKLOADS["4doc"]
    T, C = w_.T, 3 * w_.H * 128
    c = inputs.conv_inputs(w_.lens, C, seed=0)
    x, wt, b, cu = (c[k].to(dev) for k in ("x", "w", "bias", "cu_seqlens"))
    dy = c["dy"].bfloat16().to(dev)
    ws = torch.empty(max(kda.kda_conv_workspace_size(T, len(w_.lens), C), 256), dtype=torch.uint8,
                     device=dev)
    y = torch.empty_like(x)

    def fwd():
        kda.kda_conv_fwd(x, wt, cu, bias=b, y=y)

    def fwd_bwd():
        fwd()
        kda.kda_conv_bwd(x, wt, cu, dy, bias=b, ws=ws)
    f_ms, fb_ms = _time_calls(fwd), _time_calls(fwd_bwd)
    fb, bb = T * C * 4, T * C * 6
    return {"T": T, "C": C, "fwd_ms": round(f_ms, 4), "fwd_bwd_ms": round(fb_ms, 4),
            "fwd_byte_frac": round(fb / (f_ms * 1e6) / hbm_gbs, 4),
            "fwd_bwd_byte_frac": round((fb + bb) / (fb_ms * 1e6) / hbm_gbs, 4)}


# ---------------------------------------------------------------------------------------------


def bench_config(w, world):
    """The `config` object of both arms' JSON lines (same keys, same values)."""
    return {"workload": f"{w.row}:saved", "T": w.T, "H": w.H, "docs": list(w.lens), "d": 128,
            "chunk": 64, "gate": w.gate, "l2norm": bool(w.l2norm),
            "outputs": "fp32 (o, dq, dk, dv, dbeta, dg / da, dA_log, dt_bias, states)",
            "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}


def oracle_sample(w):
    """Heads of the workload the FP64 oracle runs per sample: one head per host core, so the
    N x heads (document, head) chains keep every core busy (the oracle schedules chains over
    os.cpu_count() threads, longest documents first)."""
    cores = os.cpu_count() or 1
    heads = list(range(max(1, min(w.H, cores))))
    return heads, cores


def run_reference(args, rank, world):
    """The reference arm: the FP64 oracle on all host cores, a bounded sample per step."""
    if rank != 0:
        return
    import numpy as np  # noqa: F401
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from harness import oracle_fwd_bwd
    from linear_attention_chunked_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    inp = inputs.workload_inputs(args.workload)
    oracle.build()
    heads, cores = oracle_sample(w)
    for _ in range(args.warmup):
        oracle_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, heads=heads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, heads=heads)
    dt = (time.perf_counter() - t0) / args.steps
    full_s = dt * w.H / len(heads)  # seconds per full-workload step
    value = w.T / full_s
    line = {
        "impl": "reference", "metric": f"KDA fwd+bwd tokens/s (H={w.H},d=128)",
        "value": value, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": full_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"heads 0..{len(heads) - 1} of {w.H} per step "
                                   f"({w.N * len(heads)} (document, head) chains on {cores} "
                                   f"threads), fwd+bwd token by token, {dt:.2f} s per sample, "
                                   f"scaled by {w.H}/{len(heads)}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, inp):
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from harness import oracle_fwd_bwd
    oracle.build()
    heads, cores = oracle_sample(w)
    t0 = time.perf_counter()
    oracle_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, heads=heads)
    dt = time.perf_counter() - t0
    value = w.T * len(heads) / w.H / dt
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"heads 0..{len(heads) - 1} of {w.H} ({w.N * len(heads)} (document, head) "
                      f"chains on {cores} threads; fwd+bwd, FP64 token by token), {dt:.1f} s, "
                      f"scaled to {w.H} heads"}


def run_only(what):
    """Small fixed workloads of the conv or the walk formats (targets for ncu captures)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from linear_attention_chunked_gb300 import inputs, kda
    dev = torch.device("cuda", 0)
    out = {"only": what}
    if what == "conv":
        lens, C = [8192, 4096, 3072, 1024], 8192
        c = inputs.conv_inputs(lens, C, seed=0)
        x, w, b, cu = (c[k].to(dev) for k in ("x", "w", "bias", "cu_seqlens"))
        dy = c["dy"].bfloat16().to(dev)
        ws = torch.empty(kda.kda_conv_workspace_size(sum(lens), len(lens), C), dtype=torch.uint8,
                         device=dev)
        y = torch.empty_like(x)
        f = lambda: kda.kda_conv_fwd(x, w, cu, bias=b, y=y)  # noqa: E731
        g = lambda: kda.kda_conv_bwd(x, w, cu, dy, bias=b, ws=ws)  # noqa: E731
        for _ in range(3):  # launch order fwd, bwd (+ reduce) x 3, then the timing loops
            f()
            g()
        n = sum(lens) * C
        f_ms, g_ms = _time_calls(f, 5, 20), _time_calls(g, 5, 20)
        out.update(fwd_ms=f_ms, bwd_ms=g_ms, fwd_gbs=n * 4 / f_ms / 1e6, bwd_gbs=n * 6 / g_ms / 1e6)
    else:
        gen = torch.Generator("cpu").manual_seed(0)
        M = (torch.randn((32, 16, 128, 128), generator=gen) * 0.05).to(dev)
        B = torch.randn((32, 16, 128, 128), generator=gen).to(dev)
        dfr = torch.tensor([0, 8, 16, 24, 32], dtype=torch.int32, device=dev)
        for _ in range(2):  # launch order: every format forward then reverse, twice; then timing
            for name, prec in kda.WALK_PRECISIONS.items():
                for rev in (False, True):
                    kda.kda_transfer_walk(dfr, M, B, precision=prec, reverse=rev)
        for name, prec in kda.WALK_PRECISIONS.items():
            out[name] = _time_calls(lambda: kda.kda_transfer_walk(dfr, M, B, precision=prec), 5, 20)
    torch.cuda.synchronize()
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.only:
        run_only(args.only)
        return
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    from linear_attention_chunked_gb300 import inputs, kda

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    w = inputs.WORKLOADS[args.workload]
    cpu_inp = inputs.workload_inputs(args.workload)
    inp = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in cpu_inp.items()}
    T, N, H = w.T, w.N, w.H
    wsf, svb = kda.kda_workspace_size(T, N, H, kda.KDA_OP_FWD)
    wsb, _ = kda.kda_workspace_size(T, N, H, kda.KDA_OP_BWD_SAVED)
    ws = torch.empty(max(wsf, wsb), dtype=torch.uint8, device=dev)
    saved = torch.empty(svb, dtype=torch.uint8, device=dev)
    # fp32 outputs (the library's parity-grade default: rounding o / dq to bf16 alone exceeds the
    # error bounds on the heavy-tailed raw-gate workloads)
    f32 = torch.float32

    def make_outputs():
        out = dict(o=torch.empty((T, H, 128), dtype=f32, device=dev),
                   ht=torch.empty((N, H, 128, 128), dtype=f32, device=dev),
                   dq=torch.empty((T, H, 128), dtype=f32, device=dev),
                   dk=torch.empty((T, H, 128), dtype=f32, device=dev),
                   dv=torch.empty((T, H, 128), dtype=f32, device=dev),
                   dbeta=torch.empty((T, H), dtype=f32, device=dev),
                   dg=torch.empty((T, H, 128), dtype=f32, device=dev))
        if w.gate == "raw":
            out["dA_log"] = torch.empty((H,), dtype=f32, device=dev)
            out["ddt_bias"] = torch.empty((H, 128), dtype=f32, device=dev)
        return out

    outs = make_outputs()
    grad_keys = [k for k in outs if k not in ("o", "ht")]
    kw = dict(gate=w.gate, l2norm=w.l2norm)

    def step(x, out):
        a = (x["q"], x["k"], x["v"], x["beta"], x["g"], x["cu_seqlens"])
        kda.kda_fwd(*a, A_log=x["A_log"], dt_bias=x["dt_bias"], o=out["o"], ht=out["ht"],
                    saved=saved, ws=ws, **kw)
        kda.kda_bwd(*a, x["dO"], saved=saved, A_log=x["A_log"], dt_bias=x["dt_bias"],
                    want_dh0=False, out={k: out[k] for k in grad_keys}, ws=ws, **kw)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step(inp, outs)
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps; an event every 20 steps gives the pages' samples ----
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = kda.kda_launch_counter()
    barrier()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True)]
    evs[0].record(stream)
    for i in range(args.steps):
        step(inp, outs)
        if (i + 1) % 20 == 0 or i + 1 == args.steps:
            evs.append(torch.cuda.Event(enable_timing=True))
            evs[-1].record(stream)
    torch.cuda.synchronize()
    barrier()
    ck = clocks.stop()
    launches = kda.kda_launch_counter() - launches0
    ms = reduce_max_ms(evs[0].elapsed_time(evs[-1]) / args.steps, world, dev)
    value = job_throughput(T, world, ms)

    # ---- the pages' protocol: median of 15 samples, each 20 back-to-back steps / 20 ----
    protocol = None
    if not args.no_protocol:
        proto_ms = _time_calls(lambda: step(inp, outs), samples=15, calls=20)
        proto_ms = reduce_max_ms(proto_ms, world, dev)
        protocol = {"samples": 15, "calls_per_sample": 20, "median_ms_per_step": proto_ms,
                    "value": job_throughput(T, world, proto_ms), "unit": "tokens/s"}

    hbm, bf16, src = load_peaks()
    step_roof = {
        "bound": "hbm", "peak": hbm, "unit": "GB/s", "peak_source": src,
        "bf16_out_bytes_per_token_head": BYTES_FWD_BWD,
        "frac": T * H * BYTES_FWD_BWD / (ms * 1e6) / hbm,
        "fp32_out_bytes_per_token_head": BYTES_FWD_BWD_F32,
        "frac_fp32_out": T * H * BYTES_FWD_BWD_F32 / (ms * 1e6) / hbm,
        "flop_per_token_head": FLOP_FWD_BWD,
        "flop_frac": T * H * FLOP_FWD_BWD / (ms * 1e9) / bf16,
    }

    # ---- per-kernel device time (second pass, CUDA events around every launch) ----
    kernels, roof = {}, None
    if not args.no_profile:
        kda.kda_profile_enable(True)
        for _ in range(args.steps):
            step(inp, outs)
        torch.cuda.synchronize()
        kda.kda_profile_enable(False)
        prof = kda.kda_profile_collect()
        kernels = {k: {"ms_per_step": v[0] / args.steps, "launches_per_step": v[1] / args.steps}
                   for k, v in prof.items() if v[1]}
        dom = max(kernels, key=lambda k: kernels[k]["ms_per_step"])
        per_th = alg_bytes_per_token_head(dom, out_bytes=4)
        if per_th is not None:
            launch_ms = kernels[dom]["ms_per_step"] / kernels[dom]["launches_per_step"]
            byts = per_th * T * H
            achieved = byts / (launch_ms / 1e3) / 1e9
            byts2 = alg_bytes_per_token_head(dom, out_bytes=2) * T * H
            roof = {"kernel": dom, "scope": "dominant kernel alone (the step's fraction is "
                                             "step_roofline)",
                    "bound": "hbm", "achieved": achieved, "peak": hbm,
                    "unit": "GB/s", "frac": achieved / hbm, "peak_source": src,
                    "alg_bytes_per_launch": byts, "alg_bytes_model": "fp32 outputs (as written)",
                    "achieved_bf16_out_model": byts2 / (launch_ms / 1e3) / 1e9,
                    "frac_bf16_out_model": byts2 / (launch_ms / 1e3) / 1e9 / hbm,
                    "launch_ms": launch_ms,
                    "traffic": traffic_for(dom, args.workload)}

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in cpu_inp.items()}
        res_host = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values() if torch.is_tensor(v))
        d2h = sum(v.numel() * v.element_size() for v in res_host.values())

        # an input / output pipeline: inputs and outputs double-buffered on the device; step i+1's
        # host-to-device copies and step i-1's device-to-host copies of every result (o, ht, dq,
        # dk, dv, dbeta, dg and the parameter gradients) run while step i computes, each
        # direction spread over NCOPY streams (every tensor cut into NCOPY contiguous pieces) so
        # that several copy engines share it.  Every step's copies lie inside the timed region.
        NCOPY = 4
        ibufs = [inp, {k_: (v_.clone() if torch.is_tensor(v_) else v_) for k_, v_ in inp.items()}]
        obufs = [outs, make_outputs()]
        h2d_streams = [torch.cuda.Stream(dev) for _ in range(NCOPY)]
        d2h_streams = [torch.cuda.Stream(dev) for _ in range(NCOPY)]
        ev = lambda: [[torch.cuda.Event() for _ in range(NCOPY)] for _ in range(2)]  # noqa: E731
        copied, out_free = ev(), ev()  # per buffer and copy stream
        in_free = [torch.cuda.Event(), torch.cuda.Event()]   # the step reading buffer b is done
        computed = [torch.cuda.Event(), torch.cuda.Event()]  # outputs of buffer b written

        def pieces(t):
            flat = t.view(-1)
            n = flat.numel()
            return [flat[i * n // NCOPY:(i + 1) * n // NCOPY] for i in range(NCOPY)]

        pin_in = {k_: pieces(v_) for k_, v_ in host.items() if torch.is_tensor(v_)}
        pin_out = {k_: pieces(v_) for k_, v_ in res_host.items()}
        dev_in = [{k_: pieces(bf[k_]) for k_ in pin_in} for bf in ibufs]
        dev_out = [{k_: pieces(bf[k_]) for k_ in pin_out} for bf in obufs]

        def copy_in(b):
            for i, cs in enumerate(h2d_streams):
                cs.wait_event(in_free[b])
                with torch.cuda.stream(cs):
                    for k_ in pin_in:
                        dev_in[b][k_][i].copy_(pin_in[k_][i], non_blocking=True)
                    copied[b][i].record(cs)

        def copy_out(b):
            for i, cs in enumerate(d2h_streams):
                cs.wait_event(computed[b])
                with torch.cuda.stream(cs):
                    for k_ in pin_out:
                        pin_out[k_][i].copy_(dev_out[b][k_][i], non_blocking=True)
                    out_free[b][i].record(cs)

        def run(i):
            b = i % 2
            for j in range(NCOPY):
                stream.wait_event(copied[b][j])
                stream.wait_event(out_free[b][j])  # step i-2's results have left this buffer
            step(ibufs[b], obufs[b])
            in_free[b].record(stream)
            computed[b].record(stream)
            copy_out(b)

        def e2e_steps(n, start):
            for cs in h2d_streams + d2h_streams:
                cs.wait_event(start)
            for b in (0, 1):  # nothing pending on the buffers at the start
                in_free[b].record(stream)
                for j in range(NCOPY):
                    out_free[b][j].record(stream)
            copy_in(0)
            for i in range(n):
                if i + 1 < n:
                    copy_in((i + 1) % 2)
                run(i)
            for cs in d2h_streams:  # the last results are on the host before the end
                stream.wait_stream(cs)

        s0 = torch.cuda.Event()
        s0.record(stream)
        e2e_steps(2, s0)  # warm-up
        torch.cuda.synchronize()
        barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        e2e_steps(args.steps, a0)
        a1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = reduce_max_ms(a0.elapsed_time(a1) / args.steps, world, dev)
        e2e = {"value": job_throughput(T, world, ems), "unit": "tokens/s", "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "returned": sorted(res_host), "copy_streams_per_direction": NCOPY}
        del ibufs, obufs, host, res_host

    rows = None
    if rank == 0 and not args.no_rows:
        rows = run_rows(dev, hbm, bf16)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, cpu_inp)

    if rank == 0:
        line = {
            "metric": f"KDA fwd+bwd tokens/s (H={H},d=128)", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": ((value / world) / (T / (PAGES_MS / 1e3))
                            if args.workload == "4doc" else None),
            "dtype": "f32", "data": "synthetic",
            "config": bench_config(w, world),
            "pages_protocol": protocol,
            "step_roofline": step_roof,
            "clocks": ck,
            "gpu_launches": launches,
            "kernels": kernels,
            "roofline": roof,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "rows": rows,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
