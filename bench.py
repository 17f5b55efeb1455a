#!/usr/bin/env python3
"""Throughput of the fused causal MHA path on GB300, one JSON line on stdout.

A step is one pass of the hot path over one batch of synthetic input, every
configuration of the workload table once, inputs resident in HBM:
  * bf16 causal prefill on the large-logit workload B=4, H=32, S=4096, D=128
    (Q, K ~ N(0, 3^2), V ~ N(0, 1)) -- the headline: `value` and `roofline`;
  * the same inputs with causal=0 (`prefill_noncausal`);
  * bf16 causal prefill B=1, H=32, S=2048, D=128 (`prefill_s2048`);
  * bf16 causal prefill B=2, H=16, S=16384, D=64 (`prefill_d64`);
  * f16 causal prefill on the large-logit shape (`prefill_f16`) and bf16
    causal prefill with key padding, lengths U{1024..4096} (`prefill_varlen`);
  * bf16 single-query decode on B=16, H=32, D=128 with cached lengths drawn
    uniformly from [512, 8192] -- one mha_decode call (split + merge), in
    the `decode` object.
Prefill throughput counts 2*B*H*S^2*D flops per causal call (4*B*H*S^2*D
without the mask; key padding counts each row's valid keys) over the device
time of that configuration's launches, measured with CUDA events on the
launching stream; decode counts algorithmic bytes (K and V read once, q read
and O written).  Every configuration's inputs are larger than the 129 MB L2
except the S=2048 one (50 MB of Q, K, V), which follows a launch of another
configuration that streams more than L2 through it, so no flush is needed.

--impl reference times the fp64 CPU oracle (the reference arm of this build)
on bounded samples of the headline prefill workload, on the host cores.
--gpus N (N > 1) without a launcher starts N ranks itself (torch.distributed.run).
"""
from __future__ import annotations

import argparse
import datetime
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

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

METRIC = "causal MHA prefill TFLOPS (% BF16 peak); decode mmha HBM GB/s (% peak)"
PREFILL_WORKLOAD = "prefill_bf16_b4h32s4096d128_qk3"
DECODE_WORKLOAD = "decode_bf16_b16h32d128_len512_8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch measured with ncu (dram__bytes_read.sum + dram__bytes_write.sum) on the
# named workload, valid only while the kernel source hashes to the recorded value.  Each record
# comes from a one-pass capture (those metrics only) of the `--only prefill | decode |
# projections ... --steps 1 --warmup 1 --profile` bench command for that workload.
PREFILL_SRC = ['causal_head_attention_mha_gb300/csrc/prefill_bf16.cu',
               'causal_head_attention_mha_gb300/csrc/ptx.cuh']
DECODE_SRC = ['causal_head_attention_mha_gb300/csrc/decode.cu']
GEMM_SRC = ['causal_head_attention_mha_gb300/csrc/gemm_bf16.cu',
            'causal_head_attention_mha_gb300/csrc/ptx.cuh']
TRAFFIC = [
    # kernel, workload, causal, sources, sha256 of the sources, bytes per launch
    ("prefill_bf16", PREFILL_WORKLOAD, True, PREFILL_SRC,
     "4b16b779af583ecbe033acd248a3aa91760027bc0fe100fa345cb03f55d3d09e", 521016832),
    ("prefill_bf16", PREFILL_WORKLOAD, False, PREFILL_SRC,
     "4b16b779af583ecbe033acd248a3aa91760027bc0fe100fa345cb03f55d3d09e", 528776192),
    ("prefill_bf16", "prefill_bf16_b1h32s2048d128", True, PREFILL_SRC,
     "4b16b779af583ecbe033acd248a3aa91760027bc0fe100fa345cb03f55d3d09e", 50631424),
    ("prefill_bf16", "prefill_bf16_b2h16s16384d64", True, PREFILL_SRC,
     "4b16b779af583ecbe033acd248a3aa91760027bc0fe100fa345cb03f55d3d09e", 351610368),
    ("prefill_f16", "prefill_f16_b4h32s4096d128_qk3", True, PREFILL_SRC,
     "4b16b779af583ecbe033acd248a3aa91760027bc0fe100fa345cb03f55d3d09e", 521415424),
    ("prefill_bf16", "prefill_varlen_bf16_b4h32s4096d128", True, PREFILL_SRC,
     "4b16b779af583ecbe033acd248a3aa91760027bc0fe100fa345cb03f55d3d09e", 843763712),
    # the split kernel's bytes plus the merge kernel's
    ("decode", DECODE_WORKLOAD, True, DECODE_SRC,
     "51a3bd6f99e0087d667f1f6f42c299a03ac35889771e1e3c211f81a163af275f", 1202752000),
    ("decode", "decode_f16_b16h32d128_len512_8192", True, DECODE_SRC,
     "51a3bd6f99e0087d667f1f6f42c299a03ac35889771e1e3c211f81a163af275f", 1293512192),
    ("qkv_proj", "qkv_bf16_b4s4096hid4096_h32d128", True, GEMM_SRC,
     "121503fab5ccd8ded0b5056bad7dfec04dadac8327c2730c7dea06a290ca1de1", 1045314048),
    ("out_proj_rows", "outproj_bf16_b4h32s4096d128_n4096", True, GEMM_SRC,
     "121503fab5ccd8ded0b5056bad7dfec04dadac8327c2730c7dea06a290ca1de1", 389191424),
    ("out_proj", "outproj_bf16_b4h32s4096d128_n4096", True, GEMM_SRC,
     "121503fab5ccd8ded0b5056bad7dfec04dadac8327c2730c7dea06a290ca1de1", 393275392),
]


def source_sha(rels):
    h = hashlib.sha256()
    for rel in rels:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_for(kernel, workload, causal=True):
    """Recorded DRAM bytes per launch of `kernel` on `workload`, or None when no
    capture of this workload exists or the source changed since it was taken."""
    for k, w, c, files, sha, nbytes in TRAFFIC:
        if k != kernel or w != workload or c != causal:
            continue
        if sha is None or nbytes is None:
            return None
        return nbytes if source_sha(files) == sha else None
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ ranks (weak scaling)
RANK_SEED_STRIDE = 1000


def rank_seed(base_seed, rank):
    """Seed of a rank's own batch: every rank runs the same shape on different data."""
    return base_seed + RANK_SEED_STRIDE * rank


def max_over_ranks(values, dist, device):
    """Element-wise maximum over ranks of per-rank timings; every rank gets the result."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(world, units_per_rank, seconds):
    """Units processed by all ranks over the slowest rank's time."""
    return world * units_per_rank / seconds


def launch_percentiles(ms_list):
    """p50 / p95 of per-launch device times given in ms, returned in us."""
    v = sorted(ms_list)
    def q(f):
        return 1e3 * v[min(len(v) - 1, int(round(f * (len(v) - 1))))]
    return {"us_p50": q(0.5), "us_p95": q(0.95)}


def prefill_flops(B, H, S, D, causal=True):
    return (2.0 if causal else 4.0) * B * H * S * S * D


def valid_keys(x, rows, causal=True):
    """Keys each flat row (b*H + h)*S + i attends to: min(i + 1, L_b) causal,
    L_b otherwise (L_b = S without key padding)."""
    rows = np.asarray(rows)
    i = rows % x.S
    L = x.key_lens[rows // (x.H * x.S)] if x.key_lens is not None else x.S
    return np.minimum(i + 1, L) if causal else np.broadcast_to(L, rows.shape)


def prefill_flops_varlen(H, S, D, key_lens, causal=True):
    """Useful flops (two products, 2 flops per multiply-add) with key padding."""
    L = np.asarray(key_lens, np.float64)
    per_seq = L * (L + 1) / 2 + (S - L) * L if causal else S * L
    return 4.0 * H * D * float(np.sum(per_seq))


def decode_bytes(B, H, D, seqlens):
    return 2.0 * float(np.sum(seqlens)) * H * D * 2 + 2.0 * B * H * D * 2


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of the SM clock, power and throttle reasons while the
    GPU works; `mark` notes host times so the samples of the timed region can
    be told from those of the soak before it."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index, interval_ms=50):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.marks = {}

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def mark(self, name):
        self.marks[name] = datetime.datetime.now()

    @staticmethod
    def parse(text):
        """(timestamp, sm MHz, max sm MHz, power W, active reasons) per CSV row."""
        out = []
        for r in text.strip().splitlines():
            f = [x.strip() for x in r.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                sm, smax = float(f[2]), float(f[3])
            except ValueError:
                continue
            try:
                pw = float(f[4])
            except ValueError:
                pw = None
            reasons = {n for n, v in zip(ClockSampler.REASONS, f[6:10]) if v.lower() == "active"}
            out.append((ts, sm, smax, pw, reasons))
        return out

    @staticmethod
    def summarise(rows, t0=None, t1=None):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [r[1] for r in rows]
        load = [r for r in rows if r[1] > 0.5 * max(sm)] or rows
        reasons = sorted(set().union(*(r[4] for r in load)))
        pw = [r[3] for r in load if r[3] is not None]
        d = {"sm_mhz": statistics.median(r[1] for r in load), "sm_max_mhz": max(r[2] for r in rows),
             "reasons": reasons, "samples": len(rows), "samples_under_load": len(load),
             "power_w_max": max(pw) if pw else None}
        if t0 is not None and t1 is not None:
            timed = [r for r in rows if t0 <= r[0] <= t1]
            d["samples_timed"] = len(timed)
            d["sm_mhz_timed"] = statistics.median(r[1] for r in timed) if timed else None
            d["reasons_timed"] = sorted(set().union(*(r[4] for r in timed))) if timed else []
        return d

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            text, _ = self.proc.communicate()
        return self.summarise(self.parse(text), self.marks.get("timed_start"),
                              self.marks.get("timed_end"))


# ------------------------------------------------------------------ CPU oracle timing
def oracle_sample_tflops(x, target_s, causal=True, seed=0, max_rows=None, workload=PREFILL_WORKLOAD):
    """Time the fp64 oracle on random rows of the prefill workload for about target_s."""
    import oracle
    rng = np.random.default_rng(seed)
    total_rows = x.B * x.H * x.S
    max_rows = total_rows if max_rows is None else max_rows

    def run(n):
        rows = np.sort(rng.choice(total_rows, size=n, replace=False))
        flops = float(np.sum(4.0 * valid_keys(x, rows, causal) * x.D))
        t0 = time.perf_counter()
        res = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal, rows=rows,
                               key_lens=x.key_lens)
        return time.perf_counter() - t0, flops, res.threads

    dt, _, _ = run(2048)
    per_row = max(dt / 2048, 1e-7)
    n = int(min(max_rows, max(64, target_s / per_row)))
    dt, flops, threads = run(n)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} random query rows of {workload} ({'causal' if causal else 'not causal'}), "
                      f"fp64 C oracle, {dt:.1f} s"}


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    w = si.WORKLOADS[args.prefill_workload]
    x = si.workload_inputs(args.prefill_workload)
    rng = np.random.default_rng(123)
    total_rows = x.B * x.H * x.S
    budget_per_step = min(1.0, 150.0 / max(1, args.steps + args.warmup))

    def step(n):
        rows = np.sort(rng.choice(total_rows, size=n, replace=False))
        t0 = time.perf_counter()
        res = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, True, rows=rows,
                               key_lens=x.key_lens)
        return time.perf_counter() - t0, float(np.sum(4.0 * valid_keys(x, rows) * x.D)), res.threads

    dt, _, _ = step(32)
    n = int(max(16, min(100000, budget_per_step / max(dt / 32, 1e-6))))
    for _ in range(args.warmup):
        step(n)
    tot_t = tot_f = 0.0
    threads = 0
    for _ in range(args.steps):
        dt, fl, threads = step(n)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.prefill_workload, "B": w["B"], "H": w["H"], "S": w["S"],
                   "D": w["D"], "causal": True, "sample_rows_per_step": n},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n} random query rows per step of {args.prefill_workload}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
# The prefill configurations of one step, in launch order: (key in the JSON line,
# workload, causal).  The first is the headline (`value`).  The S = 2048 inputs
# fit in L2; the launch before them streams more than L2 through it.
PREFILL_CASES = [
    ("prefill", PREFILL_WORKLOAD, True),
    ("prefill_noncausal", PREFILL_WORKLOAD, False),
    ("prefill_s2048", "prefill_bf16_b1h32s2048d128", True),
    ("prefill_d64", "prefill_bf16_b2h16s16384d64", True),
    ("prefill_f16", "prefill_f16_b4h32s4096d128_qk3", True),
    ("prefill_varlen", "prefill_varlen_bf16_b4h32s4096d128", True),
]


class PrefillCase:
    """Device-resident inputs and outputs of one prefill configuration of the step."""

    def __init__(self, mha, key, workload, causal, rank, dev, shared=None):
        import torch
        self.key, self.workload, self.causal = key, workload, causal
        w = si.WORKLOADS[workload]
        self.dtype = w["dtype"]
        tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[self.dtype]
        self.varlen = "key_len_lo" in w
        if shared is not None:  # the same inputs as another case (causal=0 on the headline data)
            self.x, self.Q, self.K, self.V = shared.x, shared.Q, shared.K, shared.V
        else:
            self.x = si.prefill_inputs(w["B"], w["H"], w["S"], w["D"], rank_seed(w["seed"], rank),
                                       qk_std=w["qk_std"], dtype=self.dtype)
            self.Q, self.K, self.V = (torch.from_numpy(t.bits.view(np.int16)).view(tdt).to(dev)
                                      for t in (self.x.Q, self.x.K, self.x.V))
        x = self.x
        self.O = torch.empty_like(self.Q)
        self.LSE = torch.empty((x.B, x.H, x.S), dtype=torch.float32, device=dev)
        self.KL = None
        if self.varlen:
            x.key_lens = si.prefill_key_lens(x.B, rank_seed(w["seed"], rank), w["key_len_lo"],
                                             w["key_len_hi"])
            self.KL = torch.from_numpy(x.key_lens).to(dev)
            self.flops = prefill_flops_varlen(x.H, x.S, x.D, x.key_lens, causal)
            self.fn = mha.mha_fwd_varlen_f16 if self.dtype == "f16" else mha.mha_fwd_varlen
        else:
            self.flops = prefill_flops(x.B, x.H, x.S, x.D, causal)
            self.fn = mha.mha_fwd_f16 if self.dtype == "f16" else mha.mha_fwd
        self.kernel_family = "prefill_" + self.dtype
        self.kernel = (f"prefill_{self.dtype}{'_varlen' if self.varlen else ''}_kernel"
                       f"<{x.D}, {'causal' if causal else 'not causal'}>")

    def __call__(self, stream, O=None, LSE=None, Q=None, K=None, V=None):
        args = (self.Q if Q is None else Q, self.K if K is None else K, self.V if V is None else V)
        kw = dict(O=self.O if O is None else O, LSE=self.LSE if LSE is None else LSE,
                  scale=self.x.scale, causal=self.causal, stream=stream)
        if self.varlen:
            self.fn(*args, self.KL, **kw)
        else:
            self.fn(*args, **kw)

    def config(self):
        x, w = self.x, si.WORKLOADS[self.workload]
        c = {"workload": self.workload, "B": x.B, "H": x.H, "S": x.S, "D": x.D,
             "causal": self.causal, "dtype": self.dtype, "qk_std": w["qk_std"],
             "flops_per_step": self.flops}
        if self.varlen:
            c["key_lens"] = [int(v) for v in x.key_lens]
            c["flops_count"] = "each row's valid keys, min(i + 1, L_b)"
        return c


def run_ours(args, rank, world, dist):
    import torch
    import causal_head_attention_mha_gb300 as mha

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mha.load_library()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)

    do_prefill = args.only in ("both", "prefill")
    do_decode = args.only in ("both", "decode")
    # the prefill configurations of the step: every one by default, or the one named
    if args.only == "both" and args.prefill_workload == PREFILL_WORKLOAD:
        plan = PREFILL_CASES
    else:
        plan = [("prefill", args.prefill_workload, not args.noncausal)]
    cases = []
    if do_prefill:
        for key, wl, causal in plan:
            shared = next((c for c in cases if c.workload == wl), None)
            cases.append(PrefillCase(mha, key, wl, causal, rank, dev, shared))
    wd = si.WORKLOADS[args.decode_workload]
    ddt = wd.get("dtype", "bf16")
    dec = mha.mha_decode_f16 if ddt == "f16" else mha.mha_decode
    if do_decode:
        xd = si.decode_inputs(wd["B"], wd["H"], wd["D"], rank_seed(wd["seed"], rank), wd["len_lo"],
                              wd["len_hi"], dtype=ddt)
        tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[ddt]
        q, Kc, Vc = (torch.from_numpy(t.bits.view(np.int16)).view(tdt).to(dev)
                     for t in (xd.q, xd.Kc, xd.Vc))
        sl = torch.from_numpy(xd.seqlens).to(dev)
        Od = torch.empty_like(q)
        dbytes = decode_bytes(xd.B, xd.H, xd.D, xd.seqlens)
        nsplit = mha.mha_decode_num_splits(xd.B, xd.H)

    def decode():
        dec(q, Kc, Vc, sl, O=Od, scale=xd.scale, stream=stream)

    def step(evs=None):
        for i, c in enumerate(cases):
            if evs is not None:
                evs[i].record(stream)
            c(stream)
        if evs is not None:
            evs[len(cases)].record(stream)
        if do_decode:
            decode()
        if evs is not None:
            evs[len(cases) + 1].record(stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---------------- warm-up
    for _ in range(args.warmup):
        step()
    barrier()
    st = mha.mha_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {mha.mha_status_string(st)}")

    # ---------------- clock soak: back-to-back steps for about args.soak seconds, sampled
    # together with the timed region, so the clock record has samples under load
    clock = ClockSampler(local)
    soak_steps = 0
    if not args.profile:
        clock.start()
        time.sleep(0.2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        barrier()
        one = max(e0.elapsed_time(e1) / 1e3, 1e-5)
        soak_steps = int(math.ceil(args.soak / one))
        for _ in range(soak_steps):
            step()
        barrier()

    # ---------------- timed region (device-resident inputs)
    K_ = args.steps
    nev = len(cases) + 2
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(K_)]
    barrier()
    clock.mark("timed_start")
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(K_):
        step(evs[k])
    t_end.record(stream)
    barrier()
    clock.mark("timed_end")
    clocks = clock.stop() if not args.profile else None
    st = mha.mha_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {mha.mha_status_string(st)}")
    per_case = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / 1e3 for i in range(len(cases))]
    td = sum(e[len(cases)].elapsed_time(e[len(cases) + 1]) for e in evs) / 1e3
    total = t_start.elapsed_time(t_end) / 1e3
    reduced = max_over_ranks(per_case + [td, total], dist, dev)
    per_case, td, total = reduced[:len(cases)], reduced[-2], reduced[-1]
    launches = K_ * (len(cases) + (((1 + (nsplit > 1)) if do_decode else 0)))

    # ---------------- end to end: pinned host buffers, copies inside the timed region
    # Every step copies its inputs from pinned host memory and reads its result
    # back.  Two device buffer sets and three streams let step k+1's inputs go
    # up and step k-1's result come back while step k computes (the link moves
    # ~210 GB/s each way, so the copies, not the kernels, set this rate).
    def pipelined(E, copy_in, compute, copy_out):
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_done = [torch.cuda.Event() for _ in range(E)]
        cmp_done = [torch.cuda.Event() for _ in range(E)]
        out_done = [torch.cuda.Event() for _ in range(E)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier()
        t0.record(s_in)
        for k in range(E):
            b = k & 1
            if k >= 2:
                s_in.wait_event(cmp_done[k - 2])  # buffer set b no longer read
            with torch.cuda.stream(s_in):
                copy_in(b)
            in_done[k].record(s_in)
            stream.wait_event(in_done[k])
            if k >= 2:
                stream.wait_event(out_done[k - 2])  # buffer set b's result read back
            compute(b)
            cmp_done[k].record(stream)
            s_out.wait_event(cmp_done[k])
            with torch.cuda.stream(s_out):
                copy_out(b)
            out_done[k].record(s_out)
        t1.record(s_out)
        barrier()
        return t0.elapsed_time(t1) / 1e3

    e2e = None
    head = cases[0] if cases else None
    if not args.no_e2e:
        E = min(K_, args.e2e_steps)
        h2d = d2h = 0
        ep = ed = 0.0
        if head is not None:
            hQ, hK, hV = (torch.from_numpy(t.bits.view(np.int16)).pin_memory()
                          for t in (head.x.Q, head.x.K, head.x.V))
            hO = torch.empty(head.Q.shape, dtype=torch.int16).pin_memory()
            hL = torch.empty(head.LSE.shape, dtype=torch.float32).pin_memory()
            h2d += 3 * hQ.numel() * 2
            d2h += hO.numel() * 2 + hL.numel() * 4
            pb = [(head.Q, head.K, head.V, head.O, head.LSE),
                  tuple(torch.empty_like(t) for t in (head.Q, head.K, head.V, head.O, head.LSE))]

            def p_in(b):
                for dst, src in zip(pb[b][:3], (hQ, hK, hV)):
                    dst.view(torch.int16).copy_(src, non_blocking=True)

            def p_cmp(b):
                q_, k_, v_, o_, l_ = pb[b]
                head(stream, O=o_, LSE=l_, Q=q_, K=k_, V=v_)

            def p_out(b):
                hO.copy_(pb[b][3].view(torch.int16), non_blocking=True)
                hL.copy_(pb[b][4], non_blocking=True)

            ep = pipelined(E, p_in, p_cmp, p_out)
            del pb
        if do_decode:
            hq = torch.from_numpy(xd.q.bits.view(np.int16)).pin_memory()
            hKc = torch.from_numpy(xd.Kc.bits.view(np.int16)).pin_memory()
            hVc = torch.from_numpy(xd.Vc.bits.view(np.int16)).pin_memory()
            hsl = torch.from_numpy(xd.seqlens).pin_memory()
            hOd = torch.empty(q.shape, dtype=torch.int16).pin_memory()
            h2d += (hq.numel() + hKc.numel() + hVc.numel()) * 2 + hsl.numel() * 4
            d2h += hOd.numel() * 2
            db = [(q, Kc, Vc, sl, Od),
                  tuple(torch.empty_like(t) for t in (q, Kc, Vc, sl, Od))]

            def d_in(b):
                for dst, src in zip(db[b][:3], (hq, hKc, hVc)):
                    dst.view(torch.int16).copy_(src, non_blocking=True)
                db[b][3].copy_(hsl, non_blocking=True)

            def d_cmp(b):
                q_, kc_, vc_, sl_, od_ = db[b]
                dec(q_, kc_, vc_, sl_, O=od_, scale=xd.scale, stream=stream)

            def d_out(b):
                hOd.copy_(db[b][4].view(torch.int16), non_blocking=True)

            ed = pipelined(E, d_in, d_cmp, d_out)
            del db
        ep, ed = max_over_ranks([ep, ed], dist, dev)
        e2e = {"value": (whole_job_rate(world, E * head.flops, ep) / 1e12) if head else None,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": E,
               "workload": head.workload if head else None,
               "decode_gbs": (whole_job_rate(world, E * dbytes, ed) / 1e9) if do_decode else None,
               "path": "pinned host -> cudaMemcpyAsync (copy-in stream) -> C-ABI call (compute "
                       "stream) -> cudaMemcpyAsync (read-back stream) -> pinned host; two "
                       "device buffer sets, so step k+1's inputs go up and step k-1's result "
                       "comes back while step k computes"}

    if rank != 0:
        return 0

    def prefill_roofline(c, t):
        per_launch_s = t / K_
        achieved = c.flops / per_launch_s / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": traffic_for(c.kernel_family, c.workload, c.causal),
                "peak_source": f"bf16_tflops (burst), of {peak_src}",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "kernel": c.kernel, "us_per_launch": 1e6 * per_launch_s,
                **launch_percentiles([e[cases.index(c)].elapsed_time(e[cases.index(c) + 1])
                                      for e in evs])}

    line = {"impl": "ours", "metric": METRIC}
    cfg = {"workload": head.workload if head else args.decode_workload,
           "l2": "inputs larger than L2 (no flush); the S=2048 inputs (50 MB) follow a launch "
                 "that streams more than L2",
           "parallelism": f"replicas x{world}"}
    if head is not None:
        line.update({"value": whole_job_rate(world, K_ * head.flops, per_case[0]) / 1e12,
                     "unit": "TFLOP/s"})
        cfg["prefill"] = head.config()
        line["roofline"] = prefill_roofline(head, per_case[0])
        for c, t in zip(cases[1:], per_case[1:]):
            line[c.key] = {"value": whole_job_rate(world, K_ * c.flops, t) / 1e12,
                           "unit": "TFLOP/s", "config": c.config(),
                           "roofline": prefill_roofline(c, t)}
    if do_decode:
        gbs = whole_job_rate(world, K_ * dbytes, td) / 1e9
        cfg["decode"] = {"workload": args.decode_workload, "B": xd.B, "H": xd.H, "D": xd.D,
                         "len_range": [wd["len_lo"], wd["len_hi"]],
                         "total_tokens": int(xd.seqlens.sum()), "splits": nsplit,
                         "bytes_per_step": dbytes}
        line["decode"] = {"value": gbs, "unit": "GB/s", "bound": "hbm",
                          "achieved": dbytes / (td / K_) / 1e9, "peak": peaks["hbm_gbs"],
                          "frac": dbytes / (td / K_) / 1e9 / peaks["hbm_gbs"],
                          "traffic": traffic_for("decode", args.decode_workload),
                          "peak_source": f"hbm_gbs, of {peak_src}",
                          "us_per_call": 1e6 * td / K_,
                          **launch_percentiles([e[len(cases)].elapsed_time(e[len(cases) + 1])
                                                for e in evs])}
        if head is None:
            line.update({"value": gbs, "unit": "GB/s"})
    if clocks is not None and clocks.get("sm_mhz"):
        clocks["soak_steps"] = soak_steps
        clocks["ms_per_step_x_sm_mhz"] = 1e3 * total / K_ * clocks["sm_mhz"]
    line.update({
        "n_gpus": world, "steps": K_, "warmup": args.warmup, "ms_per_step": 1e3 * total / K_,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": head.dtype if head else ddt,
        "data": "synthetic", "config": cfg, "clocks": clocks, "e2e": e2e,
        "gpu_launches": launches,
    })
    if not args.no_cpu_baseline and world == 1 and head is not None:
        line["cpu_baseline"] = oracle_sample_tflops(head.x, args.cpu_seconds, causal=head.causal,
                                                    workload=head.workload)
    print(json.dumps(line), flush=True)
    return 0


QKV_WORKLOAD = "qkv_bf16_b4s4096hid4096_h32d128"
OUTPROJ_WORKLOAD = "outproj_bf16_b4h32s4096d128_n4096"


def run_projections(args, rank, world, dist):
    """--only projections: the two GEMMs around attention (mha_qkv_proj, then
    mha_out_proj) on the bench's layer shape, device-resident inputs, each
    kernel timed with CUDA events on the launching stream; `value` is their
    combined TFLOP/s (2 * M * K * N flops per GEMM).  Not part of the default step."""
    import torch
    import causal_head_attention_mha_gb300 as mha

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mha.load_library()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)

    def dev16(t):
        return torch.from_numpy(t.bits.view(np.int16)).view(torch.bfloat16).to(dev)

    wq, wo = si.WORKLOADS[QKV_WORKLOAD], si.WORKLOADS[OUTPROJ_WORKLOAD]
    xq = si.projection_inputs(wq["B"], wq["S"], wq["hidden"], wq["H"], wq["D"],
                              rank_seed(wq["seed"], rank))
    xo = si.out_projection_inputs(wo["B"], wo["H"], wo["S"], wo["D"], wo["n_out"],
                                  rank_seed(wo["seed"], rank))
    X, Wqkv = dev16(xq.X), dev16(xq.W)
    shp = (xq.B, xq.H, xq.S, xq.D)
    Q, K, V = (torch.empty(shp, dtype=torch.bfloat16, device=dev) for _ in range(3))
    O, Wo = dev16(xo.O), dev16(xo.W)
    O_rows = O.permute(0, 2, 1, 3).contiguous()  # the same O as [B, S, H, D]
    Y = torch.empty((xo.B, xo.S, xo.n_out), dtype=torch.bfloat16, device=dev)
    M = xq.B * xq.S
    f_qkv = 2.0 * M * xq.hidden * 3 * xq.H * xq.D
    f_out = 2.0 * xo.B * xo.S * xo.H * xo.D * xo.n_out

    def step(ev):
        ev[0].record(stream)
        mha.mha_qkv_proj(X, Wqkv, xq.H, xq.D, Q=Q, K=K, V=V, stream=stream)
        ev[1].record(stream)
        mha.mha_out_proj(O, Wo, Y=Y, stream=stream)
        ev[2].record(stream)
        mha.mha_out_proj(O_rows, Wo, Y=Y, stream=stream, o_layout="bshd")
        ev[3].record(stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    barrier()
    if mha.mha_get_device_status(stream) != 0:
        raise RuntimeError("device status after warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clock = ClockSampler(local)
    if not args.profile:
        clock.start()
        time.sleep(0.3)
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for ev in evs:
        step(ev)
    t1.record(stream)
    barrier()
    clocks = clock.stop() if not args.profile else None
    if mha.mha_get_device_status(stream) != 0:
        raise RuntimeError("device status after timed region")
    tq = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    to = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    tr = sum(e[2].elapsed_time(e[3]) for e in evs) / 1e3
    total = t0.elapsed_time(t1) / 1e3
    tq, to, tr, total = max_over_ranks([tq, to, tr, total], dist, dev)
    if rank != 0:
        return 0
    K_ = args.steps
    peak = peaks["bf16_tflops"]

    def roof(name, flops, t, j, traffic):
        a = flops / (t / K_) / 1e12
        return {"bound": "tensor", "achieved": a, "peak": peak, "unit": "TFLOP/s",
                "frac": a / peak, "frac_of_sustained": a / peaks["bf16_tflops_sustained"],
                "traffic": traffic, "peak_source": f"bf16_tflops (burst), of {peak_src}",
                "kernel": name, "us_per_launch": 1e6 * t / K_,
                **launch_percentiles([e[j].elapsed_time(e[j + 1]) for e in evs])}

    line = {"impl": "ours", "metric": "attention projections TFLOP/s (% BF16 peak)",
            "value": whole_job_rate(world, K_ * (f_qkv + f_out), tq + to) / 1e12,
            "unit": "TFLOP/s", "n_gpus": world, "steps": K_, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / K_, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{QKV_WORKLOAD} + {OUTPROJ_WORKLOAD}",
                       "l2": "inputs larger than L2 (no flush)",
                       "parallelism": f"replicas x{world}",
                       "qkv": {"M": M, "K": xq.hidden, "N": 3 * xq.H * xq.D, "flops": f_qkv},
                       "out": {"M": xo.B * xo.S, "K": xo.H * xo.D, "N": xo.n_out,
                               "flops": f_out}},
            "roofline": roof("qkv_proj_kernel", f_qkv, tq, 0, traffic_for("qkv_proj", QKV_WORKLOAD)),
            "out_proj": roof("out_proj_kernel", f_out, to, 1,
                             traffic_for("out_proj", OUTPROJ_WORKLOAD)),
            # the same product with O already in [B, S, H, D] (mha_fwd_ex o_layout 1)
            "out_proj_rows": roof("out_proj_rows_kernel", f_out, tr, 2,
                                  traffic_for("out_proj_rows", OUTPROJ_WORKLOAD)),
            "clocks": clocks, "gpu_launches": 3 * K_}
    print(json.dumps(line), flush=True)
    return 0


def free_port():
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def launch_ranks(n):
    """Run this script as n ranks on this node (one process per GPU), the way
    torch.distributed.run starts them; returns the launcher's exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def run_dry(args, rank, world):
    """--dry-run: the multi-rank host path without any CUDA call.  Every rank
    builds its own seeded batch of the headline prefill recipe (a small slice),
    joins a gloo group, and the timing reduction runs over dummy times; rank 0
    prints each rank's seed and input digest."""
    import torch
    import torch.distributed as tdist
    dist = None
    if world > 1:
        tdist.init_process_group("gloo")
        dist = tdist
    try:
        w = si.WORKLOADS[PREFILL_WORKLOAD]
        seed = rank_seed(w["seed"], rank)
        x = si.prefill_inputs(1, 1, 64, w["D"], seed, qk_std=w["qk_std"])
        digest = hashlib.sha256(x.Q.bits.tobytes()).hexdigest()
        ranks = [None] * world
        if dist is not None:
            dist.all_gather_object(ranks, {"rank": rank, "seed": seed, "q_sha256": digest})
        else:
            ranks = [{"rank": rank, "seed": seed, "q_sha256": digest}]
        t = max_over_ranks([1.0 + rank], dist, torch.device("cpu"))[0]
        if rank == 0:
            print(json.dumps({"dry_run": True, "n_gpus": world, "ranks": ranks,
                              "max_time_over_ranks": t}), flush=True)
        return 0
    finally:
        if dist is not None:
            tdist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1,
                    help="ranks (one GPU each); without a launcher, N > 1 starts them itself")
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--only", choices=("both", "prefill", "decode", "projections"),
                    default="both")
    ap.add_argument("--prefill-workload", default=PREFILL_WORKLOAD,
                    choices=[k for k, w in si.WORKLOADS.items()
                             if w["kind"] == "prefill" and w["dtype"] in ("bf16", "f16")],
                    help="prefill workload (default: every configuration of the step, the "
                         "headline first; a workload named here runs alone)")
    ap.add_argument("--noncausal", action="store_true",
                    help="with --only prefill: the named workload with causal=0")
    ap.add_argument("--decode-workload", default=DECODE_WORKLOAD,
                    choices=[k for k, w in si.WORKLOADS.items() if w["kind"] == "decode"],
                    help="decode workload of the step (bf16 or f16)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of back-to-back steps before the timed region, sampled "
                         "with the clocks")
    ap.add_argument("--profile", action="store_true", help="no clock sampling (for ncu runs)")
    ap.add_argument("--dry-run", action="store_true",
                    help="the multi-rank host path only (seeds, reduction), no CUDA")
    args = ap.parse_args()
    if args.warmup < 3 and not args.profile:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return launch_ranks(args.gpus)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match WORLD_SIZE={world}")
    if args.dry_run:
        return run_dry(args, rank, world)
    dist = None
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        if args.only == "projections":
            return run_projections(args, rank, world, dist)
        return run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
