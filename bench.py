"""Benchmark of the block-drafter hot path: draft tokens/s of (draft block + constrained argmax + verify).

Default workload: text speculative mode at the 4B-target drafter shape, batch 1, context 2048, block 16
(1 anchor + 15 proposals), vocabulary 151936, unconstrained, greedy verification against a synthetic target
row whose agreement prefix is Geometric(0.25).  The context K/V is prepared once before timing (its time is
reported separately).  All inputs are seeded synthetic data; the drafter weights (1.83 GB streamed per
block) are far larger than the 129 MB L2, so every step reads them from HBM.

The line's `roofline` is the whole step's: algorithmic bytes (HBM-bound workloads) or flops (tensor-bound ones)
per step over the measured step time.  The default run also times the batched fixed-width workload (32 requests,
L = 381) and reports its tensor-core fraction under `batched`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
  python bench.py --sweep          # the 32-point throughput sweep, one JSON line per point

N > 1 runs N independent replicas (one per rank, launched by torchrun): the path has no exchange step.
Prints ONE JSON line (rank 0), or one per point with --sweep.
"""
from __future__ import annotations

import argparse
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

METRIC = "draft tokens/s per GB300 (fwd+constrain+verify)"


def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, kind)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        burst = float(p["bf16_tflops"])
        return float(p["hbm_gbs"]), burst, float(p.get("bf16_tflops_sustained", burst)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def legal_counts(wl):
    """Legal ids of each drafted position 1..L-1 and the set of LM-head rows any position needs."""
    s, L = wl.shape, wl.block_len
    if wl.layout is None:
        return np.full(L - 1, s.vocab, dtype=np.int64), s.vocab
    lay = wl.layout
    off, rng = lay["class_off"], lay["class_ranges"]
    per_class, rows = [], set()
    full = False
    for c in range(len(off) - 1):
        n = 0
        for k in range(off[c], off[c + 1]):
            lo, hi = int(rng[2 * k]), int(rng[2 * k + 1])
            n += hi - lo
        per_class.append(n)
    used = set(int(c) for c in lay["pos_class"][1:L])
    for c in used:
        if per_class[c] >= s.vocab:
            full = True
        for k in range(off[c], off[c + 1]):
            rows.update(range(int(rng[2 * k]), int(rng[2 * k + 1])))
    counts = np.array([per_class[int(c)] for c in lay["pos_class"][1:L]], dtype=np.int64)
    return counts, (s.vocab if full else len(rows))


def algorithmic_work(wl, fp8=False):
    """Minimum bytes and flops of one step (every request's block): drafter layer weights, the LM-head rows some
    position can select, the context K/V reads; 2 flops per multiply-add of the projections, the LM-head columns
    of the legal ids and the attention (4 (T_b + L) L h per q head and layer).  fp8: one byte per weight plus one
    exponent byte per 128 weights for the streamed matrices (the unconstrained LM head included)."""
    s, B, L = wl.shape, wl.batch, wl.block_len
    layer_params = (s.qkv_rows * s.d_model + s.d_model * s.n_q_heads * s.head_dim + 2 * s.d_ff * s.d_model
                    + s.d_model * s.d_ff)
    counts, lm_rows = legal_counts(wl)
    ctx = wl.ctx_len.astype(np.int64)
    wb = 1 + 1 / 128 if fp8 else 2
    lmb = wb if (fp8 and wl.layout is None) else 2
    bytes_ = {"layers": int(s.n_layers * layer_params * wb), "lm_head": int(lm_rows * s.d_model * lmb),
              "kv": int(ctx.sum()) * s.n_layers * 2 * s.n_kv_heads * s.head_dim * 2}
    flops = {"layers": 2 * B * L * layer_params * s.n_layers, "lm_head": 2 * B * int(counts.sum()) * s.d_model,
             "attention": 4 * int((ctx + L).sum()) * L * s.head_dim * s.n_q_heads * s.n_layers}
    return bytes_, flops


def profiled_traffic(workload):
    """DRAM bytes per step (dram__bytes_read.sum + dram__bytes_write.sum over every kernel of one step) from the
    committed ncu summary, or None when no summary covers this workload or a kernel of the step has changed since
    its counters were taken (the row's `current` cell is not `yes`)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_per_step.md")
    try:
        for ln in open(path):
            cells = [c.strip() for c in ln.strip().strip("|").split("|")]
            if len(cells) >= 5 and cells[0] == workload:
                return int(float(cells[2])) if cells[4] == "yes" else None
    except (OSError, ValueError):
        pass
    return None


class ClockSampler:
    def __init__(self, out_path):
        self.out_path = out_path
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.out_path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self, gpu_index=0):
        try:
            rows = [ln.split(",") for ln in open(self.out_path) if ln.strip()]
        except Exception:
            rows = []
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9 and r[0].strip() == str(gpu_index)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(elapsed_ms, world, device):
    """The timed region's length as the slowest rank saw it (all ranks get the same number)."""
    if world == 1:
        return float(elapsed_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_step, steps, elapsed_ms):
    """Whole-job draft tokens/s: every replica drafts `tokens_per_step` per step; time = slowest rank."""
    return world * tokens_per_step * steps / (elapsed_ms / 1e3)


def run_oracle_block(om, wl, kv, target, layout):
    import oracle
    t0 = time.perf_counter()
    hid = oracle.draft_block(om, kv, wl.t_cap, wl.ctx_len, wl.anchor, wl.mask_id, wl.block_len)
    toks, _, _ = oracle.constrain_argmax(om, hid, wl.batch, wl.block_len, layout=layout)
    if layout is None:
        oracle.verify(0, toks, target)
    else:
        oracle.verify(1, toks, layout=layout, rule=layout["rule"], pad_id=layout["pad_id"])
    return time.perf_counter() - t0


def oracle_sample(wl, w, kv_np, target):
    """The oracle as it stands on one block of request 0 (a bounded sample of the workload)."""
    import dataclasses
    import oracle
    om = oracle.Model(wl.shape, w)
    one = dataclasses.replace(wl, batch=1, ctx_len=wl.ctx_len[:1], anchor=wl.anchor[:1], t_cap=int(wl.ctx_len[0]))
    kv1 = np.ascontiguousarray(kv_np[:, :1, :, :, :one.t_cap])
    lay = wl.layout
    return om, one, kv1, (target[:1] if target is not None else None), lay


class StepRunner:
    """One workload on one drafter: device inputs, the step as one CUDA graph (draft, LM head + argmax, verify:
    the calls' kernels keep their programmatic-dependent-launch overlap across call boundaries) for the timed
    steps, and the same step as three graphs with CUDA events between them for the per-call breakdown."""

    def __init__(self, pkg, dr, wl, dev, prepare=True, kv_seed=None):
        import torch
        import synth
        self.pkg, self.dr, self.wl, self.dev = pkg, dr, wl, dev
        s, B, L = wl.shape, wl.batch, wl.block_len
        self.stream = torch.cuda.current_stream(dev)
        self.prepare_ms = None
        if prepare:
            feats = synth.make_features(s, int(wl.row_off[-1]), wl.seed + 1)
            fd, row_off_d, _ = dr.prepare_context(B, wl.row_off, feats)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            pkg.fpd_prepare_context(dr.handle, B, int(wl.row_off[-1]), row_off_d, None, fd, dr.kv_store, dr.t_cap,
                                    dr.workspace, dr.ws_bytes, self.stream)
            e1.record(self.stream)
            torch.cuda.synchronize()
            self.prepare_ms = e0.elapsed_time(e1)
            del fd, feats
        else:
            # a prepared context stands in as seeded N(0, 1) bf16 K/V drawn on the device
            g = torch.Generator(device=dev).manual_seed(int(kv_seed if kv_seed is not None else wl.seed + 5))
            kv = dr.kv_view(B)
            for l in range(s.n_layers):
                kv[l].normal_(generator=g)
        self.ctx_len = torch.from_numpy(wl.ctx_len).to(dev)
        self.anchor = torch.from_numpy(wl.anchor).to(dev)
        self.hidden = torch.empty(B * L, s.d_model, dtype=torch.bfloat16, device=dev)
        self.tokens = torch.empty(B, L - 1, dtype=torch.int32, device=dev)
        self.accept = torch.empty(B, dtype=torch.int32, device=dev)
        self.committed = torch.empty(B, L, dtype=torch.int32, device=dev)
        self.valid = torch.empty(B, dtype=torch.int32, device=dev)
        self.lay_d = self.rule_d = None
        if wl.layout is not None:
            self.lay_d, self.rule_d = pkg.Drafter.layout(wl.layout, B, L, dev)
        # target rows: Geometric(p) agreement with the drafter's own ids (text mode)
        self.do_draft(self.stream)
        self.do_argmax(self.stream)
        torch.cuda.synchronize()
        self.target_np = self.target = None
        if wl.layout is None:
            self.target_np, _ = synth.make_target_rows(self.tokens.cpu().numpy(), s.vocab, wl.geo_p or 0.25,
                                                       wl.seed + 2)
            self.target = torch.from_numpy(self.target_np).to(dev)

    def do_draft(self, st):
        wl, dr = self.wl, self.dr
        self.pkg.fpd_draft_block(dr.handle, wl.batch, wl.block_len, dr.kv_store, dr.t_cap, self.ctx_len, self.anchor,
                                 wl.mask_id, self.hidden, None, dr.workspace, dr.ws_bytes, st)

    def do_argmax(self, st):
        wl, dr = self.wl, self.dr
        self.pkg.fpd_constrain_argmax(dr.handle, wl.batch, wl.block_len, self.hidden, self.lay_d, self.tokens, None,
                                      dr.workspace, dr.ws_bytes, st)

    def do_verify(self, st):
        wl = self.wl
        if wl.layout is None:
            self.pkg.fpd_verify(0, wl.batch, wl.block_len, self.tokens, self.target, None, None, -1, self.accept,
                                self.committed, self.valid, st)
        else:
            self.pkg.fpd_verify(1, wl.batch, wl.block_len, self.tokens, None, self.lay_d, self.rule_d,
                                wl.layout["pad_id"], self.accept, self.committed, self.valid, st)

    def capture(self, warmup):
        import torch
        for _ in range(max(3, warmup)):   # eager warm-up (also counts the kernels one step launches)
            n0 = self.pkg.fpd_kernel_launches()
            self.do_draft(self.stream)
            self.do_argmax(self.stream)
            self.do_verify(self.stream)
            self.launches_per_step = self.pkg.fpd_kernel_launches() - n0
        torch.cuda.synchronize()
        cap = torch.cuda.Stream(self.dev)
        self.graphs = []
        for fn in (self.do_draft, self.do_argmax, self.do_verify):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                fn(torch.cuda.current_stream(self.dev))
            self.graphs.append(g)
        self.g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_step, stream=cap):
            st = torch.cuda.current_stream(self.dev)
            self.do_draft(st)
            self.do_argmax(st)
            self.do_verify(st)
        for _ in range(max(3, warmup)):
            self.step()
            self.step_parts()
        torch.cuda.synchronize()

    def step(self):
        self.g_step.replay()

    def step_parts(self, ev=None):
        g_draft, g_argmax, g_verify = self.graphs
        if ev is not None:
            ev[0].record(self.stream)
        g_draft.replay()
        if ev is not None:
            ev[1].record(self.stream)
        g_argmax.replay()
        if ev is not None:
            ev[2].record(self.stream)
        g_verify.replay()

    def time_steps(self, steps, barrier=lambda: None):
        """Device time of `steps` back-to-back steps (the one-graph step), then, after that timed region, the mean
        draft and LM-head call times from as many three-graph steps with events between the calls."""
        import torch
        t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        t0e.record(self.stream)
        for _ in range(steps):
            self.step()
        t1e.record(self.stream)
        torch.cuda.synchronize()
        barrier()
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
        for i in range(steps):
            self.step_parts(ev[i])
        torch.cuda.synchronize()
        draft_ms = float(np.mean([a.elapsed_time(b) for a, b, _ in ev]))
        lm_ms = float(np.mean([b.elapsed_time(c) for _, b, c in ev]))
        return t0e.elapsed_time(t1e), draft_ms, lm_ms


def roofline_of(wl, ms_per_step, draft_ms, lm_ms, traffic=None, fp8=False):
    """The step's roofline: HBM-bound when the bytes take longer than the flops at the measured peaks."""
    hbm, tc_burst, tc_sus, kind = peaks()
    by, fl = algorithmic_work(wl, fp8)
    B_tot, F_tot = sum(by.values()), sum(fl.values())
    sec = ms_per_step * 1e-3
    lm_bytes = by["lm_head"] + wl.batch * (wl.block_len - 1) * wl.shape.d_model * 2
    calls = {
        "fpd_draft_block": {"ms": draft_ms, "achieved_gbs": (by["layers"] + by["kv"]) / (draft_ms * 1e-3) / 1e9,
                            "achieved_tflops": (fl["layers"] + fl["attention"]) / (draft_ms * 1e-3) / 1e12},
        "fpd_constrain_argmax": {"ms": lm_ms, "achieved_gbs": lm_bytes / (lm_ms * 1e-3) / 1e9,
                                 "achieved_tflops": fl["lm_head"] / (lm_ms * 1e-3) / 1e12},
    }
    if B_tot / (hbm * 1e9) >= F_tot / (tc_burst * 1e12):
        for c in calls.values():
            c["frac"] = c["achieved_gbs"] / hbm
        ach = B_tot / sec / 1e9
        return {"bound": "hbm", "kernel": "whole step (draft block + constrained argmax + verify)",
                "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_kind": f"{kind} copy bandwidth", "traffic": traffic, "algorithmic_bytes": B_tot,
                "bytes_parts": by, "calls": calls}
    for c in calls.values():
        c["frac"] = c["achieved_tflops"] / tc_sus
    ach = F_tot / sec / 1e12
    return {"bound": "tensor", "kernel": "whole step (draft block + constrained argmax + verify)",
            "achieved": ach, "peak": tc_sus, "unit": "TFLOP/s", "frac": ach / tc_sus,
            "frac_of_burst": ach / tc_burst, "peak_kind": f"{kind} bf16 cuBLAS, sustained (steps run back to back)",
            "traffic": traffic, "algorithmic_flops": F_tot, "flops_parts": fl, "calls": calls}


def workload_config(name, wl):
    import synth
    s = wl.shape
    return {"workload": name, "batch": wl.batch, "block_len": wl.block_len,
            "context": wl.ctx_len.tolist() if wl.batch <= 4 else [int(wl.ctx_len.min()), int(wl.ctx_len.max())],
            "d_model": s.d_model, "layers": s.n_layers, "vocab": s.vocab,
            "layout": "unconstrained" if wl.layout is None else synth.CONFIGS[wl.name]["layout"],
            "l2": "inputs larger than L2 (1.83 GB weights streamed per step)"}


def run_batched_extra(pkg, w, dev, steps=10, warmup=3):
    """The batched fixed-width workload (32 requests, L = 381) timed after the main line: its tensor fraction."""
    import synth
    wl = synth.make_workload("primitive_fixedwidth_b32")
    dr = pkg.Drafter(wl.shape, w, wl.batch, wl.block_len, wl.t_cap, device=dev)
    r = StepRunner(pkg, dr, wl, dev)
    r.capture(warmup)
    ms, dms, lms = r.time_steps(steps)
    rf = roofline_of(wl, ms / steps, dms, lms)
    out = {"workload": "primitive_fixedwidth_b32", "ms_per_step": ms / steps,
           "value": wl.batch * (wl.block_len - 1) * steps / (ms * 1e-3), "unit": "draft tokens/s",
           "prepare_ms": r.prepare_ms, "bound": rf["bound"], "achieved": rf["achieved"], "unit_roofline": rf["unit"],
           "frac": rf["frac"], "frac_of_burst": rf.get("frac_of_burst"), "peak": rf["peak"],
           "weights": "the main workload's synthetic draw (values do not change the work)"}
    del r
    dr.close()
    return out


def run_fp8_extra(pkg, w, wl, dev, steps=20, warmup=3):
    """The same workload on the model's 8-bit weight copies (fpd_model_enable_fp8): the streamed GEMMs read E4M3
    weights and quantise their inputs per 128 elements; the HBM roofline counts the 8-bit bytes."""
    dr = pkg.Drafter(wl.shape, w, wl.batch, wl.block_len, wl.t_cap, device=dev, fp8=True)
    r = StepRunner(pkg, dr, wl, dev)
    r.capture(warmup)
    ms, dms, lms = r.time_steps(steps)
    assert pkg.fpd_device_status(r.stream) == 0, "device-side check failed (8-bit run)"
    rf = roofline_of(wl, ms / steps, dms, lms, fp8=True)
    out = {"ms_per_step": ms / steps, "value": wl.batch * (wl.block_len - 1) * steps / (ms * 1e-3),
           "unit": "draft tokens/s", "draft_ms": dms, "lm_head_ms": lms, "bound": rf["bound"],
           "achieved": rf["achieved"], "unit_roofline": rf["unit"], "frac": rf["frac"], "peak": rf["peak"],
           "algorithmic_bytes": rf.get("algorithmic_bytes"),
           "weights": "E4M3 codes + one power-of-two exponent per 128 elements (a different model from the bf16 "
                      "line: its activations are quantised too)"}
    del r
    dr.close()
    return out


def run_sweep(pkg, steps, warmup):
    """The 32-point sweep: batch {1,4,16,64} x context {512,2048,8192,16384} x block {16 text, 385 special}.
    Each point's context K/V is drawn on the device (seed 5000 + point index); the LM head, attention and
    verification run exactly as in the named workloads."""
    import torch
    import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = synth.CONFIGS["text_4b_b1"]["shape"]
    w = synth.make_weights(s, 5000)
    points = [(B, T, L) for L in (16, 385) for B in (1, 4, 16, 64) for T in (512, 2048, 8192, 16384)]
    dr = pkg.Drafter(s, w, 64, 385, 16384, device=dev)
    for idx, (B, T, L) in enumerate(points):
        base = "text_4b_b1" if L == 16 else "primitive_special_b1"
        wl = synth.make_workload(base, batch=B, t_ctx=T, seed=5000 + idx)
        r = StepRunner(pkg, dr, wl, dev, prepare=False, kv_seed=5000 + idx)
        r.capture(warmup)
        ms, dms, lms = r.time_steps(steps)
        rf = roofline_of(wl, ms / steps, dms, lms)
        assert pkg.fpd_device_status(r.stream) == 0, "device-side check failed"
        line = {"metric": METRIC, "value": B * (L - 1) * steps / (ms * 1e-3), "unit": "draft tokens/s",
                "n_gpus": 1, "steps": steps, "warmup": warmup, "ms_per_step": ms / steps, "higher_is_better": True,
                "dtype": "bf16", "data": "synthetic", "sweep_point": idx,
                "config": workload_config(f"sweep_B{B}_T{T}_L{L}", wl),
                "blocks_per_s": B * steps / (ms * 1e-3), "roofline": rf, "gpu_launches": r.launches_per_step * steps}
        print(json.dumps(line), flush=True)
        del r
        torch.cuda.synchronize()
    dr.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="text_4b_b1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-batched", action="store_true", help="skip the batched workload's extra measurement")
    ap.add_argument("--sweep", action="store_true", help="time the 32-point sweep, one line per point")
    ap.add_argument("--no-fp8", action="store_true", help="skip the 8-bit-weight measurement of the workload")
    ap.add_argument("--fp8", action="store_true", help="time the workload on the 8-bit weight copies (main line)")
    args = ap.parse_args()

    import torch
    import synth

    if args.sweep:
        import block_diffusion_speculative_non_gb300 as pkg
        run_sweep(pkg, min(args.steps, 10), args.warmup)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)

    wl = synth.make_workload(args.workload)
    s = wl.shape
    L, B = wl.block_len, wl.batch
    draft_tokens_per_step = B * (L - 1)
    config = workload_config(args.workload, wl)
    if args.fp8:
        config["weights"] = "8-bit E4M3 copies of the streamed matrices (fpd_model_enable_fp8)"

    if args.impl == "reference":
        # the CPU oracle, as it stands, on the host cores: rank 0 only
        if rank != 0:
            return
        import oracle
        oracle.build()
        w = synth.make_weights(s, wl.seed)
        kv = synth.make_kv_store(s, B, wl.t_cap, wl.seed + 5)
        om, one, kv1, _, lay = oracle_sample(wl, w, kv, None)
        target = None
        if lay is None:
            rng = np.random.default_rng(wl.seed + 9)
            target = rng.integers(0, s.vocab, (1, L)).astype(np.int32)
        for _ in range(max(0, min(args.warmup, 1))):
            run_oracle_block(om, one, kv1, target, lay)
        times = [run_oracle_block(om, one, kv1, target, lay) for _ in range(args.steps)]
        t = float(np.sum(times))
        v = args.steps * (L - 1) / t
        cores = oracle.num_threads()
        line = {"metric": METRIC, "value": v, "unit": "draft tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "impl": "reference",
                "cpu_baseline": {"value": v, "unit": "draft tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": "one block of request 0 per step (draft + constrained argmax + verify)"},
                "e2e": {"value": v, "unit": "draft tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import block_diffusion_speculative_non_gb300 as pkg
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    w = synth.make_weights(s, wl.seed)
    dr = pkg.Drafter(s, w, B, L, wl.t_cap, device=dev, fp8=args.fp8)
    r = StepRunner(pkg, dr, wl, dev)
    r.capture(args.warmup)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    clock_fd, clock_path = tempfile.mkstemp(prefix=f"fpd_bench_clocks_r{rank}_", suffix=".csv")
    os.close(clock_fd)
    with ClockSampler(clock_path) as cs:
        elapsed_ms, draft_ms, lm_ms = r.time_steps(args.steps, barrier)
    launches = r.launches_per_step * args.steps      # graph replays: the kernels of one step, K times
    assert pkg.fpd_device_status(r.stream) == 0, "device-side check failed"
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    ms_per_step = elapsed_ms / args.steps
    value = replica_throughput(world, draft_tokens_per_step, args.steps, elapsed_ms)

    # ---- end to end through the C ABI with host buffers: H2D of the step's inputs, D2H of its results --------
    a_h = torch.from_numpy(wl.anchor.copy()).pin_memory()
    t_h = torch.from_numpy(r.target_np.copy()).pin_memory() if r.target_np is not None else None
    acc_h = torch.empty(B, dtype=torch.int32).pin_memory()
    com_h = torch.empty(B, L, dtype=torch.int32).pin_memory()
    h2d = a_h.numel() * 4 + (t_h.numel() * 4 if t_h is not None else 0)
    d2h = acc_h.numel() * 4 + com_h.numel() * 4
    e2e_steps = max(10, args.steps // 2)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        r.anchor.copy_(a_h, non_blocking=True)
        if t_h is not None:
            r.target.copy_(t_h, non_blocking=True)
        r.step()
        acc_h.copy_(r.accept, non_blocking=True)
        com_h.copy_(r.committed, non_blocking=True)
        r.stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_value = world * draft_tokens_per_step * e2e_steps / e2e_s

    roofline = roofline_of(wl, ms_per_step, draft_ms, lm_ms, None if args.fp8 else profiled_traffic(args.workload),
                           fp8=args.fp8 and B * L <= 16)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            import oracle
            oracle.build()
            # the oracle's inputs come from the seeded generators only (timing sample, values irrelevant)
            kv_np = synth.make_kv_store(s, 1, int(wl.ctx_len[0]), wl.seed + 5)
            tgt_np = np.random.default_rng(wl.seed + 9).integers(0, s.vocab, (1, L)).astype(np.int32)
            om, one, kv1, tgt1, lay = oracle_sample(wl, w, kv_np, tgt_np)
            dt = run_oracle_block(om, one, kv1, tgt1, lay)
            cpu = {"value": (L - 1) / dt, "unit": "draft tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                   "sample": "one block of request 0 (draft + constrained argmax + verify), fp64 oracle"}
        except Exception as e:  # the baseline is reported, never required
            cpu = {"value": None, "unit": "draft tokens/s", "cores": None, "kind": "oracle", "sample": f"failed: {e}"}

    prepare_ms = r.prepare_ms
    del r
    dr.close()
    fp8 = None
    if rank == 0 and world == 1 and B * L <= 16 and not args.no_fp8 and not args.fp8:
        fp8 = run_fp8_extra(pkg, w, wl, dev)
    batched = None
    if rank == 0 and world == 1 and B * L < 300 and not args.no_batched:
        batched = run_batched_extra(pkg, w, dev)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "draft tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f8e4m3 x f8e4m3 -> f32" if args.fp8 and B * L <= 16 else "bf16",
                "data": "synthetic", "config": config,
                "blocks_per_s": world * B * args.steps / (elapsed_ms / 1e3), "prepare_ms": prepare_ms,
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "draft tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": int(launches), "clocks": cs.summary(local_rank)}
        if fp8 is not None:
            line["fp8"] = fp8
        if batched is not None:
            line["batched"] = batched
        print(json.dumps(line), flush=True)
    try:
        os.remove(clock_path)
    except OSError:
        pass
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
