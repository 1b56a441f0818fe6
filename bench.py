"""Benchmark of the gated delta-rule state update on GB300.

Headline workload (one "step"): the batched decode step, 64 sequences x 48
value heads (16 key heads), kd = vd = 128, fp32 state -- one launch of the
token-serial kernel over 3072 heads, 406.9 MB of algorithmic HBM traffic.
Three state sets (3 x 201 MB, larger than the 129 MB L2) rotate between
steps, so every step reads its state from HBM.

Also timed (the "parts" object): the M-token verify launch (32 x 48 heads,
M = 2, 4, 8, with and without per-token checkpoints) and the prefill of
8 x 4096 tokens x 48 heads.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]
Multi-GPU: launched by torchrun, one rank per GPU; each rank decodes its own
64-sequence batch (rank_workload: weak scaling, no collective on the data
path; only the timing is reduced over ranks).
"""

from __future__ import annotations

import argparse
import ctypes
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdn_inputs  # noqa: E402

METRIC = "GDN head-steps/sec and achieved HBM GB/s (% of 8 TB/s) at 1 GB300"
UNIT = "head-steps/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
NSETS = 3
E2E_SETS = 8    # pinned input buffers the end-to-end leg reads in turn
D = 128


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- bytes

def decode_bytes(B, kh, vh, M=1, ckpt=False):
    """Algorithmic HBM bytes of one launch over M tokens: the state read
    once and written once (plus M checkpoints), the token inputs read and o
    written once."""
    state = B * vh * D * D * 4
    qk = 2 * B * M * kh * D * 4
    vo = 2 * B * M * vh * D * 4
    gb = 2 * B * M * vh * 4
    return 2 * state + (M * state if ckpt else 0) + qk + vo + gb


# FP32 issue floor of the token-serial update: per head-token and state
# element, two fused multiply-adds (S^T k and S^T q), one multiply (the
# decay) and one fused multiply-add (the rank-1 update) -- 4 FP32 lane
# operations for the 7 flops per element of the definition (decay 1, S^T k
# 2, rank-1 update 2, S^T q 2).  The GB300 has
# 152 SMs x 128 FP32 lanes; at the measured maximum SM clock that is
# 152 * 128 * clock lane operations per second.
FP32_LANE_OPS_PER_ELEM = 4
SMS = 152
FP32_LANES_PER_SM = 128


def fp32_floor_s(head_tokens, sm_mhz):
    lane_ops = head_tokens * FP32_LANE_OPS_PER_ELEM * D * D
    return lane_ops / (SMS * FP32_LANES_PER_SM * sm_mhz * 1e6)


# ------------------------------------------------------------- clocks

CLOCK_FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,"
                "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background."""

    def __init__(self):
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + CLOCK_FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(
                    parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            self.rows.append((ts, parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1, uuid=None):
        rows = [p for ts, p in self.rows]
        if uuid:
            mine = [p for p in rows if uuid.lower() in p[1].lower()]
            rows = mine or rows
        inwin = [p for (ts, p) in self.rows if t0 <= ts <= t1 and p in rows]
        use = inwin or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "note": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[2]) for p in use if num(p[2]) is not None]
        mx = [num(p[3]) for p in use if num(p[3]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap")
        reasons = sorted({n for p in use for n, v in zip(names, p[6:10])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_in_timed_window": len(inwin),
                "window": "timed" if inwin else "whole run (timed region "
                          "shorter than the sampling period)"}


# ------------------------------------------------------------ multi-rank

def rank_workload(rank, **overrides):
    """The headline batch that `rank` decodes: 64 sequences x 48 heads of
    its own (the workload's seed plus 1000 x rank), so ranks share no data
    and the data path needs no collective; rank 0's batch is the
    single-GPU workload.  `overrides` change the sizes (tests)."""
    kw = dict(gdn_inputs.WORKLOADS["decode_b64"])
    kw.update(overrides)
    return gdn_inputs.make_inputs(
        gdn_inputs.WORKLOAD_SEED["decode_b64"] + 1000 * rank, **kw)


def aggregate(ms_local, units_local, dist=None, device=None):
    """Whole-job rate: the slowest rank's time and the units all ranks
    processed.  Returns (ms_max, total_units, units_per_second)."""
    import torch
    if dist is None or not dist.is_initialized():
        return ms_local, units_local, units_local / (ms_local * 1e-3)
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    u = torch.tensor([units_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    ms, units = float(t.item()), float(u.item())
    return ms, units, units / (ms * 1e-3)


# --------------------------------------------------------------- timing

def time_launches(torch, fn, n, stream):
    """Average device time of fn() over n launches, CUDA events on stream."""
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(n):
        fn(i)
    ev1.record(stream)
    ev1.synchronize()
    return ev0.elapsed_time(ev1) / n


def kernel_traffic(kernel_src_files, name):
    """Per-launch DRAM bytes from the committed ncu summary, or None when the
    kernel source changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        fields = dict(tok.split("=", 1) for tok in open(path).read().split()
                      if "=" in tok)
    except OSError:
        return None
    h = hashlib.sha256()
    for f in kernel_src_files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if fields.get("source_sha256", "")[:16] != h.hexdigest()[:16]:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------- CPU baseline

def cpu_baseline(inp, seconds=10.0):
    """The oracle, as it is, on the host cores: sequences of the headline
    workload, one token each, repeated for about `seconds`."""
    import oracle
    oracle.build()
    nseq = min(8, inp.B)
    sub = inp.heads(range(nseq), range(inp.vh))
    heads = sub.B * sub.vh
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.run_inputs(sub)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": heads * calls / el, "unit": UNIT,
            "cores": oracle.threads(), "kind": "oracle",
            "sample": f"decode_b64 sequences 0-{nseq - 1} x {sub.vh} heads "
                      f"({heads} head-steps per call), {calls} calls in "
                      f"{el:.1f} s",
            "gbs": decode_bytes(sub.B, sub.kh, sub.vh) * calls / el / 1e9}


def cpu_configs(seconds=2.0):
    """The oracle on the other workloads (one sequence, one token; one
    sequence, 64 chained tokens; 32 sequences x M tokens, each repeated for
    about `seconds`; the 8 x 4096-token prefill once): head-steps/s per
    workload."""
    import oracle
    oracle.build()

    def rate(run, head_steps):
        calls, t0 = 0, time.perf_counter()
        while True:
            run()
            calls += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return head_steps * calls / el, calls, el

    out = {"cores": oracle.threads(), "kind": "oracle", "unit": UNIT}
    for name in ("decode_b1", "decode_b1_t64"):
        w = gdn_inputs.make_workload(name)
        r, c, el = rate(lambda w=w: oracle.run_inputs(w), w.B * w.vh * w.T)
        out[name] = {"value": r, "sample": f"{c} calls in {el:.1f} s"}
    vin = gdn_inputs.make_workload("verify_b32")
    for M in (2, 4, 8):
        sub = vin.tokens(0, M)
        r, c, el = rate(lambda sub=sub: oracle.run_inputs(sub, ckpt=True),
                        sub.B * sub.vh * M)
        out[f"verify_b32_m{M}_ckpt"] = {"value": r,
                                        "sample": f"{c} calls in {el:.1f} s"}
    # the long-sequence prefill in full (8 x 4096 tokens x 48 heads, one
    # call: the token-serial definition, which the chunked form regroups)
    pre = gdn_inputs.make_workload("prefill_b8_t4096")
    t0 = time.perf_counter()
    oracle.run_inputs(pre)
    el = time.perf_counter() - t0
    out["prefill_b8_t4096"] = {"value": pre.B * pre.T * pre.vh / el,
                               "sample": f"1 call in {el:.1f} s"}
    return out


# ------------------------------------------------------------ reference

def run_reference(args, rank, world):
    """--impl reference: the CPU oracle timed as the reference arm."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    inp = gdn_inputs.make_workload("decode_b64")
    one = inp.heads([0], range(inp.vh))
    t0 = time.perf_counter()
    oracle.run_inputs(one)
    t1 = time.perf_counter() - t0
    budget = 90.0 / max(1, args.steps + args.warmup)
    nseq = int(max(1, min(inp.B, budget // max(t1, 1e-6))))
    sub = inp.heads(range(nseq), range(inp.vh))
    for _ in range(args.warmup):
        oracle.run_inputs(sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run_inputs(sub)
    el = time.perf_counter() - t0
    heads = sub.B * sub.vh
    value = heads * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "decode_b64 (sampled: %d of 64 sequences x 48 "
                   "heads per step)" % nseq, "B": 64, "kh": 16, "vh": 48,
                   "kd": 128, "vd": 128, "seed": inp.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                         "cores": oracle.threads(),
                         "sample": f"{nseq} sequences x 48 heads per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def tens_fn(torch, dev):
    return lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def verify_parts(torch, gdn, tens, stream, hbm_peak, parts, steps,
                 warmup=5, sm_mhz=2070.0, case=None):
    """The M-token verify launches, M = 2, 4, 8, without and with per-token
    checkpoints, on 32 sequences x 48 heads (the verify workload) and on
    64 sequences x 48 heads (the batched decode size); each timed over
    max(20, min(200, steps)) launches after `warmup` untimed ones, with
    three state sets in turn (each larger than L2 at B = 64, 100 MB at
    B = 32).  Besides the HBM fraction each entry gives the FP32 issue floor
    and the fraction of max(HBM floor, FP32 floor).  `case` (a part name
    such as "verify_b64_m8") runs that one configuration only (profiling)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    for wname in ("verify_b32", "verify_b64"):
        if case is not None and not case.startswith(wname + "_"):
            continue
        if wname == "verify_b32":
            vin = gdn_inputs.make_workload("verify_b32")
        else:
            vin = gdn_inputs.make_inputs(gdn_inputs.SEED_BASE + 5, B=64, T=8,
                                         kh=16, vh=48)
        Sv = [tens(vin.S) for _ in range(NSETS)]
        ck = torch.empty((8,) + tuple(vin.S.shape), device=dev)
        for M in (2, 4, 8):
            sub = vin.tokens(0, M)
            toks = [tuple(tens(x) for x in (sub.q, sub.k, sub.v, sub.g,
                                            sub.beta)) for _ in range(NSETS)]
            vo = torch.empty(sub.B, M, sub.vh, D, device=dev)
            for use_ck in (False, True):
                pname = f"{wname}_m{M}{'_ckpt' if use_ck else ''}"
                if case is not None and case != pname:
                    continue

                def vstep(i, M=M, use_ck=use_ck):
                    s = Sv[i % NSETS]
                    gdn.gdn_step_m(s, s, ck[:M] if use_ck else None,
                                   *toks[i % NSETS], vo, M=M, stream=stream)
                n = max(20, min(200, steps))
                for i in range(warmup):
                    vstep(i)
                vms = time_launches(torch, vstep, n, stream)
                nb = decode_bytes(sub.B, sub.kh, sub.vh, M, use_ck)
                ht = sub.B * sub.vh * M
                hbm_floor = nb / (hbm_peak * 1e9)
                fp_floor = fp32_floor_s(ht, sm_mhz)
                parts[pname] = {
                    "ms": vms, "head_steps_per_s": ht / (vms * 1e-3),
                    "gbs": nb / (vms * 1e-3) / 1e9,
                    "frac_of_measured_hbm": nb / (vms * 1e-3) / 1e9 / hbm_peak,
                    "bytes_per_launch": nb,
                    "flops_per_launch": ht * 7 * D * D,
                    "fp32_lane_ops_per_launch": ht * FP32_LANE_OPS_PER_ELEM * D * D,
                    "fp32_floor_us": fp_floor * 1e6,
                    "hbm_floor_us": hbm_floor * 1e6,
                    "frac_of_max_floor": max(hbm_floor, fp_floor) / (vms * 1e-3)}
        rname = f"{wname}_rollback_m8"
        if case is None or case == rname:
            # per-sequence rollback after an 8-token verify: sequence b keeps
            # m[b] of the 8 tokens (seeded, 0..8), i.e. S[b] = snap[b] or
            # ckpt[m[b] - 1][b]; one state read and one written per launch
            snap = tens(vin.S)
            rng = np.random.default_rng(gdn_inputs.SEED_BASE + 6)
            m_dev = torch.from_numpy(
                rng.integers(0, 9, size=vin.B).astype(np.int32)).to(dev)

            def rstep(i):
                gdn.gdn_rollback_seq(Sv[i % NSETS], 8, m_dev, snap, ck, vin.kh,
                                     stream=stream)
            for i in range(warmup):
                rstep(i)
            rms = time_launches(torch, rstep, max(20, min(200, steps)), stream)
            rbytes = 2 * Sv[0].numel() * 4
            parts[rname] = {
                "ms": rms, "gbs": rbytes / (rms * 1e-3) / 1e9,
                "frac_of_measured_hbm": rbytes / (rms * 1e-3) / 1e9 / hbm_peak,
                "bytes_per_launch": rbytes,
                "note": "gdn_rollback_seq after an 8-token verify: each "
                        "sequence's state restored from the snapshot or one "
                        "of its 8 checkpoints (accepted counts 0..8, seeded)"}
            del snap
        del Sv, ck
        torch.cuda.empty_cache()


def small_decode_parts(torch, gdn, tens, stream, parts, steps):
    """Latency of the small decode cases (one sequence x 48 heads, state
    6.3 MB, L2-resident): one gdn_step per call; 64 chained gdn_step calls
    with fresh inputs each token; the same 64 tokens as one gdn_step_m
    launch.  Times are CUDA-event averages over back-to-back launches on one
    stream (launch gaps included)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    one = gdn_inputs.make_workload("decode_b1")
    S1 = tens(one.S)
    ins = tuple(tens(x) for x in (one.q, one.k, one.v, one.g, one.beta))
    o1 = torch.empty(1, 1, one.vh, D, device=dev)
    f = lambda i: gdn.gdn_step(S1, *ins, o1, stream=stream)
    for i in range(20):
        f(i)
    n = max(200, min(2000, steps))
    ms = time_launches(torch, f, n, stream)
    # the same call through the C ABI with its arguments prepared once: what
    # a C or C++ caller pays per call (the library's argument checks and the
    # launch), without the Python binding's tensor checks
    lib = gdn.load()
    sh = gdn.Shape(1, one.kh, one.vh, D, D)
    ptrs = [t.data_ptr() for t in (S1,) + ins + (o1,)]
    raw_stream = stream.cuda_stream
    byref_sh = ctypes.byref(sh)

    def raw(i):
        if lib.gdn_step(byref_sh, *ptrs, raw_stream) != gdn.GDN_OK:
            raise RuntimeError("gdn_step refused the decode_b1 call")
    for i in range(20):
        raw(i)
    ms_raw = time_launches(torch, raw, n, stream)
    parts["decode_b1"] = {
        "us_per_call": ms * 1e3, "head_steps_per_s": one.vh / (ms * 1e-3),
        "us_per_call_c_abi": ms_raw * 1e3,
        "head_steps_per_s_c_abi": one.vh / (ms_raw * 1e-3),
        "note": "gdn_step, B=1 x 48 heads, back-to-back launches: through "
                "the Python binding, and through the C ABI with arguments "
                "prepared once (argument checks and launch every call)"}

    ch = gdn_inputs.make_workload("decode_b1_t64")
    T = ch.T
    q, k, v, g, beta = (tens(x) for x in (ch.q, ch.k, ch.v, ch.g, ch.beta))
    per_tok = [tuple(x[:, t:t + 1].contiguous() for x in (q, k, v, g, beta))
               for t in range(T)]
    Sc = tens(ch.S)
    oc = torch.empty(1, 1, ch.vh, D, device=dev)
    chain = lambda i: gdn.gdn_step(Sc, *per_tok[i % T], oc, stream=stream)
    for i in range(T):
        chain(i)
    ms = time_launches(torch, chain, 10 * T, stream)
    # the same 64 chained steps captured once in a CUDA graph and replayed
    # (the per-call host work of the binding and the library is then gone)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for t in range(T):
            gdn.gdn_step(Sc, *per_tok[t], oc)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in range(T):
            gdn.gdn_step(Sc, *per_tok[t], oc)
    cur = torch.cuda.current_stream()
    for _ in range(3):
        graph.replay()
    msg = time_launches(torch, lambda i: graph.replay(), 20, cur) / T
    om = torch.empty(1, T, ch.vh, D, device=dev)
    Sm = tens(ch.S)
    multi = lambda i: gdn.gdn_step_m(Sm, Sm, None, q, k, v, g, beta, om,
                                     M=T, stream=stream)
    for i in range(5):
        multi(i)
    msm = time_launches(torch, multi, 50, stream)
    parts["decode_b1_t64"] = {
        "us_per_step_chained": ms * 1e3,
        "head_steps_per_s_chained": ch.vh / (ms * 1e-3),
        "us_per_step_chained_graph": msg * 1e3,
        "us_per_launch_m64": msm * 1e3,
        "us_per_token_m64": msm * 1e3 / T,
        "head_steps_per_s_m64": ch.vh * T / (msm * 1e-3),
        "note": "64 tokens, B=1 x 48 heads: 64 chained gdn_step calls "
                "(launched one by one, and replayed from a CUDA graph), and "
                "one gdn_step_m launch over the same 64 tokens"}
    del S1, Sc, Sm, graph


def layer_parts(torch, gdn, tens, stream, hbm_peak, parts, steps,
                warmup=5):
    """The layer core on 64 sequences x 48 heads, one token: prologue +
    update (gdn_layer_step_m), then the same followed by the gated RMSNorm."""
    dev = torch.device("cuda", torch.cuda.current_device())
    L = gdn_inputs.make_layer_inputs(gdn_inputs.SEED_BASE + 100, B=64, T=1)
    SL = [tens(L.S) for _ in range(NSETS)]
    hL = [tens(L.hist), tens(L.hist)]
    lx, lw, la, lb = (tens(t) for t in (L.x, L.conv_w, L.a, L.b))
    lA, ldt = tens(L.A_log), tens(L.dt_bias)
    lo = torch.empty(64, 1, 48, D, device=dev)

    lws = torch.empty(gdn.gdn_layer_workspace(64, 16, 48, 1),
                      dtype=torch.uint8, device=dev)

    def lstep(i):
        s_ = SL[i % NSETS]
        gdn.gdn_layer_step_m(s_, s_, None, hL[i % 2], hL[(i + 1) % 2], lx,
                             lw, la, lb, lA, ldt, lo, L.kh, lws,
                             stream=stream)
    for i in range(warmup):
        lstep(i)
    n = max(20, min(200, steps))
    lms = time_launches(torch, lstep, n, stream)
    conv_dim = 2 * 16 * D + 48 * D
    lbytes = decode_bytes(64, 16, 48) + 64 * 4 * (conv_dim + 6 * conv_dim)
    parts["layer_decode_b64"] = {
        "ms": lms, "head_steps_per_s": 64 * 48 / (lms * 1e-3),
        "gbs": lbytes / (lms * 1e-3) / 1e9,
        "frac_of_measured_hbm": lbytes / (lms * 1e-3) / 1e9 / hbm_peak,
        "bytes_per_launch": lbytes,
        "note": "raw projections in: layer prologue (conv1d+SiLU with "
                "history, q/k norm, gates) then the update, two launches"}
    # the same, followed by the gated RMSNorm in place on o
    _, zn, wn = gdn_inputs.make_gate_norm_inputs(
        gdn_inputs.SEED_BASE + 101, 64, 1, 48)
    lz, lwn = tens(zn), tens(wn)

    def lnstep(i):
        lstep(i)
        gdn.gdn_gated_rmsnorm_m(lo, lz, lwn, lo, stream=stream)
    for i in range(warmup):
        lnstep(i)
    lnms = time_launches(torch, lnstep, n, stream)
    lnbytes = lbytes + 3 * 64 * 48 * D * 4
    parts["layer_norm_decode_b64"] = {
        "ms": lnms, "head_steps_per_s": 64 * 48 / (lnms * 1e-3),
        "gbs": lnbytes / (lnms * 1e-3) / 1e9,
        "frac_of_measured_hbm": lnbytes / (lnms * 1e-3) / 1e9 / hbm_peak,
        "bytes_per_launch": lnbytes,
        "note": "raw projections in, normalised output out: layer "
                "prologue, update, gated RMSNorm in place; three launches"}
    del SL, hL
    torch.cuda.empty_cache()


def prefill_parts(torch, gdn, tens, stream, peaks, parts):
    """Time the 8 x 4096-token prefill in its three precisions."""
    pin_ = gdn_inputs.make_workload("prefill_b8_t4096")
    pq, pk, pv, pg, pb = (tens(x) for x in
                          (pin_.q, pin_.k, pin_.v, pin_.g, pin_.beta))
    Sp = tens(pin_.S)
    po = torch.empty(pin_.B, pin_.T, pin_.vh, D, device=pq.device)

    toks = pin_.B * pin_.T
    flops = 7 * D * D * toks * pin_.vh
    # executed tensor-core flops of the chunked form per 64-token chunk
    # and head: [K;Q]K^T 2*128*64*128; S^T [K;Q]^T 2*128*128*128;
    # (V^T - Y diag(gamma)) (T diag(beta))^T 2*128*64*64; Delta^T P^T
    # 2*128*64*64; Delta^T K~ 2*128*128*64
    tc_flops = (2 * 128 * 64 * 128 + 2 * 128 * 128 * 128 +
                2 * 128 * 64 * 64 + 2 * 128 * 64 * 64 +
                2 * 128 * 128 * 64) * (pin_.T // 64) * pin_.B * pin_.vh
    # algorithmic HBM bytes: q, k, v, g, beta read and o written once, the
    # state read and written once
    hbm_bytes = (4 * pin_.B * pin_.T * (2 * pin_.kh * D + 2 * pin_.vh * D +
                                        2 * pin_.vh) +
                 2 * 4 * pin_.B * pin_.vh * D * D)
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    for prec, name, reps in ((gdn.GDN_PREC_FP32, "fp32", 3),
                             (gdn.GDN_PREC_BF16X3, "bf16x3", 10),
                             (gdn.GDN_PREC_BF16, "bf16", 10)):
        def pstep(i, prec=prec):
            gdn.gdn_prefill(Sp, pq, pk, pv, pg, pb, po, precision=prec,
                            stream=stream)
        for i in range(3):
            pstep(i)
        pms = time_launches(torch, pstep, reps, stream)
        entry = {
            "ms": pms, "tokens_per_s": toks / (pms * 1e-3),
            "head_steps_per_s": toks * pin_.vh / (pms * 1e-3),
            "tflops_fp32_equiv": flops / (pms * 1e-3) / 1e12}
        hbm_floor = hbm_bytes / (hbm_peak * 1e9)
        entry.update({"bytes_per_launch": hbm_bytes,
                      "hbm_floor_us": hbm_floor * 1e6})
        if prec == gdn.GDN_PREC_FP32:
            fp_floor = fp32_floor_s(toks * pin_.vh, 2070.0)
            entry.update({"fp32_floor_us": fp_floor * 1e6,
                          "frac_of_max_floor": max(hbm_floor, fp_floor) / (pms * 1e-3),
                          "note": "token-serial fp32 path"})
        else:
            mult = 3 if prec == gdn.GDN_PREC_BF16X3 else 1
            ach = tc_flops * mult / (pms * 1e-3) / 1e12
            peak = float(peaks.get("bf16_tflops_sustained",
                                   peaks.get("bf16_tflops", 1900.0)))
            tensor_floor = tc_flops * mult / (peak * 1e12)
            entry.update({"tensor_tflops": ach, "tensor_peak_tflops": peak,
                          "tensor_frac": ach / peak,
                          "tensor_floor_us": tensor_floor * 1e6,
                          "frac_of_max_floor":
                              max(hbm_floor, tensor_floor) / (pms * 1e-3),
                          "note": "chunk-parallel form on tcgen05; "
                                  "executed MMA flops (x3 for split-bf16); "
                                  "frac_of_max_floor against the larger of "
                                  "the HBM and tensor floors"})
        parts[f"prefill_b8_t4096_{name}"] = entry
    del pq, pk, pv, pg, pb, Sp, po


# ------------------------------------------------------------- main arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-parts", action="store_true",
                    help="skip the verify / prefill sub-measurements")
    ap.add_argument("--no-cpu", action="store_true",
                    help="skip the CPU-baseline leg")
    ap.add_argument("--case", default=None,
                    help="with --only verify: one configuration, e.g. "
                         "verify_b64_m8 or verify_b64_m2_ckpt (profiling)")
    ap.add_argument("--only", choices=["prefill", "layer", "verify", "small"],
                    default=None,
                    help="time only the prefill, layer or verify parts (used "
                         "for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import gated_deltanet_linear_gb300 as gdn
    from gated_deltanet_linear_gb300 import _build
    _build.build()
    gdn.load()

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()


    if args.only is not None:
        parts = {}
        sampler = ClockSampler()
        sampler.start()
        time.sleep(0.3)
        t0 = time.time()
        if args.only == "prefill":
            prefill_parts(torch, gdn, tens_fn(torch, dev), stream, peaks, parts)
        elif args.only == "verify":
            verify_parts(torch, gdn, tens_fn(torch, dev), stream, hbm_peak,
                         parts, args.steps, max(5, args.warmup), sm_max,
                         args.case)
        elif args.only == "small":
            small_decode_parts(torch, gdn, tens_fn(torch, dev), stream, parts,
                               args.steps)
        else:
            layer_parts(torch, gdn, tens_fn(torch, dev), stream, hbm_peak,
                        parts, args.steps, max(5, args.warmup))
        t1 = time.time()
        sampler.stop()
        print(json.dumps({"only": args.only, "parts": parts,
                          "clocks": sampler.summary(t0, t1, None)}), flush=True)
        return 0

    # ---- headline workload: batched decode step
    inp = rank_workload(rank)
    B, kh, vh = inp.B, inp.kh, inp.vh
    tens = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    S0 = tens(inp.S)
    states = [S0.clone() for _ in range(NSETS)]
    del S0
    # token inputs and outputs rotate with the state sets (their own
    # buffers per set), so no step finds them in L2 from the step before
    tok_sets = [tuple(tens(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
                for _ in range(NSETS)]
    o_sets = [torch.empty(B, 1, vh, D, device=dev) for _ in range(NSETS)]
    o = o_sets[0]

    def step(i):
        gdn.gdn_step(states[i % NSETS], *tok_sets[i % NSETS], o_sets[i % NSETS],
                     stream=stream)

    sampler = ClockSampler()
    sampler.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        step(i)
    barrier()
    t_wall0 = time.time()
    ms_local = time_launches(torch, step, args.steps, stream)
    t_wall1 = time.time()
    barrier()
    bytes_step = decode_bytes(B, kh, vh)
    heads_per_step = B * vh
    ms, _, value = aggregate(ms_local, heads_per_step, dist, dev)
    achieved_gbs = bytes_step / (ms_local * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers: the step's
    # inputs q | k | v | g | beta sit back to back in one pinned host buffer
    # and o goes to another; the kernel reads the inputs and writes o over
    # the host link itself (gdn_step takes page-locked host token buffers),
    # so the transfers overlap the state streaming and no copy is issued.
    # (One copy engine transfer in, then the kernel, measured 91.5 us
    # against 70.2 us this way.)
    parts_in = (inp.q, inp.k, inp.v, inp.g, inp.beta)
    sizes = [x.size for x in parts_in]           # each a multiple of 4 floats
    # E2E_SETS packed input buffers in turn, so that no step finds its
    # inputs still in L2 from an earlier step
    h_sets = []
    for _ in range(E2E_SETS):
        h_pack = torch.empty(sum(sizes), dtype=torch.float32).pin_memory()
        h_in, off = [], 0
        for x, n_ in zip(parts_in, sizes):
            h_pack[off:off + n_] = torch.from_numpy(np.ascontiguousarray(x).ravel())
            h_in.append(h_pack[off:off + n_].view(x.shape))
            off += n_
        h_sets.append(h_in)
    h_o = torch.empty(tuple(o.shape), dtype=torch.float32).pin_memory()
    h2d = h_pack.numel() * 4
    d2h = h_o.numel() * 4

    def e2e_step(i):
        gdn.gdn_step(states[i % NSETS], *h_sets[i % E2E_SETS], h_o,
                     stream=stream)

    for i in range(args.warmup):
        e2e_step(i)
    barrier()
    ms_e2e, _, e2e_value = aggregate(
        time_launches(torch, e2e_step, args.steps, stream), heads_per_step,
        dist, dev)
    e2e = {"value": e2e_value, "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": ms_e2e,
           "note": "the kernel reads q, k, v, g, beta from a pinned host "
                   "buffer (8 in turn) and writes o into another over the "
                   "host link, every step; the recurrent state stays "
                   "resident on the device"}

    # ---- parts: verify launches and prefill (rank 0 only, N = 1 shapes)
    parts = {}
    launches = args.steps  # headline timed region: one kernel per step
    if not args.no_parts and rank == 0:
        # reference point: a plain copy of the same 201 MB state (gdn_mark),
        # same rotation of state sets, i.e. the same bytes as the headline
        # step without its arithmetic and token inputs
        snaps = [torch.empty_like(states[0]) for _ in range(NSETS)]

        def cstep(i):
            gdn.gdn_mark(states[i % NSETS], snaps[(i + 1) % NSETS], kh,
                         stream=stream)
        for i in range(5):
            cstep(i)
        cms = time_launches(torch, cstep, max(20, min(200, args.steps)), stream)
        cbytes = 2 * states[0].numel() * 4
        parts["state_copy_b64"] = {
            "ms": cms, "gbs": cbytes / (cms * 1e-3) / 1e9,
            "frac_of_measured_hbm": cbytes / (cms * 1e-3) / 1e9 / hbm_peak,
            "bytes_per_launch": cbytes,
            "note": "gdn_mark copy of the headline state (201.3 MB read + "
                    "201.3 MB written): the practical ceiling for this size"}
        del snaps
        torch.cuda.empty_cache()
        del states
        torch.cuda.empty_cache()
        verify_parts(torch, gdn, tens, stream, hbm_peak, parts, args.steps,
                     sm_mhz=sm_max)
        small_decode_parts(torch, gdn, tens, stream, parts, args.steps)
        layer_parts(torch, gdn, tens, stream, hbm_peak, parts, args.steps)
        prefill_parts(torch, gdn, tens, stream, peaks, parts)

    sampler.stop()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = sampler.summary(t_wall0, t_wall1, uuid)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    cpu = None
    if world == 1 and not args.no_cpu:
        cpu = cpu_baseline(inp)
        cpu["other_workloads"] = cpu_configs()

    traffic = kernel_traffic(["gated_deltanet_linear_gb300/csrc/gdn_decode.cu"],
                             "gdn_steps_decode_b64.traffic.txt")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": "decode_b64: batched decode step, B=64 "
                   "sequences x vh=48 value heads (kh=16), kd=vd=128, fp32 "
                   "state", "B": B, "kh": kh, "vh": vh, "kd": D, "vd": D,
                   "seed": inp.seed,
                   "l2": f"{NSETS} rotating state sets of "
                         f"{B * vh * D * D * 4 / 1e6:.0f} MB (> 129 MB L2)",
                   "bytes_per_step": bytes_step},
        "hbm_gbs": achieved_gbs,
        "hbm_frac_of_8tbs": achieved_gbs / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs,
                     "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved_gbs / hbm_peak,
                     "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "gdn_step_c32_kernel"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "parts": parts,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
