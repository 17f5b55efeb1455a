#!/usr/bin/env python3
"""Throughput of the fused causal MHA path on GB300, one JSON line on stdout.

A step is one pass of the hot path over one batch of synthetic input:
  * bf16 causal prefill on the large-logit workload B=4, H=32, S=4096, D=128
    (Q, K ~ N(0, 3^2), V ~ N(0, 1)) -- one mha_fwd call, O and LSE written;
  * bf16 single-query decode on B=16, H=32, D=128 with cached lengths drawn
    uniformly from [512, 8192] -- one mha_decode call (split + merge).
`value` is the prefill throughput in TFLOP/s, counting 2*B*H*S^2*D flops per
causal call, over the prefill kernels' device time; the decode throughput
(algorithmic bytes: K and V read once, q read and O written) is reported in
the `decode` object.  Inputs (384 MiB for prefill, ~1.1 GiB of cache for
decode) are larger than the 129 MB L2, so no flush is needed between steps.

--impl reference times the fp64 CPU oracle (the reference arm of this build)
on bounded samples of the same prefill workload, on the host cores.
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
# named workload, valid only while the kernel source hashes to the recorded value.  The prefill
# records come from one-pass captures (those metrics only) of `bench.py --only prefill
# --prefill-workload <workload> --steps 1 --warmup 1 --profile`; the profiles named beside
# them hold the full captures of the same kernels.
TRAFFIC = {
    # profiles/prefill_bf16_d128_causal_b4h32s4096.md
    "prefill": {"kernel": "prefill_bf16", "workload": PREFILL_WORKLOAD,
                "files": ['causal_head_attention_mha_gb300/csrc/prefill_bf16.cu', 'causal_head_attention_mha_gb300/csrc/ptx.cuh'],
                "sha256": "34663ef60bd3ed993f66174c07c2bef1729c78e4dbf944c1358b3a7d8c979462", "bytes_per_launch": 519273728},
    # profiles/prefill_bf16_d64_causal_b2h16s16384.md
    "prefill_d64": {"kernel": "prefill_bf16", "workload": "prefill_bf16_b2h16s16384d64",
                    "files": ['causal_head_attention_mha_gb300/csrc/prefill_bf16.cu', 'causal_head_attention_mha_gb300/csrc/ptx.cuh'],
                    "sha256": "34663ef60bd3ed993f66174c07c2bef1729c78e4dbf944c1358b3a7d8c979462", "bytes_per_launch": 345352960},
    # profiles/prefill_f16_d128_causal_b4h32s4096.md
    "prefill_f16": {"kernel": "prefill_f16", "workload": "prefill_f16_b4h32s4096d128_qk3",
                    "files": ['causal_head_attention_mha_gb300/csrc/prefill_bf16.cu', 'causal_head_attention_mha_gb300/csrc/ptx.cuh'],
                    "sha256": "34663ef60bd3ed993f66174c07c2bef1729c78e4dbf944c1358b3a7d8c979462", "bytes_per_launch": 522228992},
    # key padding, B4 H32 S4096 D128 (one capture of the same bench command, dram metrics only)
    "prefill_varlen": {"kernel": "prefill_bf16", "workload": "prefill_varlen_bf16_b4h32s4096d128",
                       "files": ['causal_head_attention_mha_gb300/csrc/prefill_bf16.cu', 'causal_head_attention_mha_gb300/csrc/ptx.cuh'],
                       "sha256": "34663ef60bd3ed993f66174c07c2bef1729c78e4dbf944c1358b3a7d8c979462", "bytes_per_launch": 453030656},
    # profiles/decode_split_d128_b16h32_len512_8192.md (split kernel; merge adds ~4 MB)
    "decode": {"kernel": "decode", "workload": DECODE_WORKLOAD, "files": ['causal_head_attention_mha_gb300/csrc/decode.cu'],
               "sha256": "4a57a2900bce4d3d7c8d88f0f7cc6c14a2b81669d8e7139e37f15245594dfa2a", "bytes_per_launch": 1201886720},
    # profiles/decode_split_f16_d128_b16h32_len512_8192.md
    "decode_f16": {"kernel": "decode", "workload": "decode_f16_b16h32d128_len512_8192",
                   "files": ['causal_head_attention_mha_gb300/csrc/decode.cu'],
                   "sha256": "4a57a2900bce4d3d7c8d88f0f7cc6c14a2b81669d8e7139e37f15245594dfa2a", "bytes_per_launch": 1292623616},
    # profiles/proj_gemm_bf16_b4s4096_h32d128.md (the projection kernels; these figures from one
    # one-pass DRAM capture of `bench.py --only projections --steps 1 --warmup 1 --profile`)
    "qkv_proj": {"kernel": "qkv_proj", "workload": "qkv_bf16_b4s4096hid4096_h32d128",
                 "files": ['causal_head_attention_mha_gb300/csrc/gemm_bf16.cu', 'causal_head_attention_mha_gb300/csrc/ptx.cuh'],
                 "sha256": "d4365aeeda8876f4d66ac37b9eb57eae1df6b69289171a103464038b9ac0cc00", "bytes_per_launch": 1354212608},
    "out_proj_rows": {"kernel": "out_proj_rows", "workload": "outproj_bf16_b4h32s4096d128_n4096",
                      "files": ['causal_head_attention_mha_gb300/csrc/gemm_bf16.cu', 'causal_head_attention_mha_gb300/csrc/ptx.cuh'],
                      "sha256": "d4365aeeda8876f4d66ac37b9eb57eae1df6b69289171a103464038b9ac0cc00", "bytes_per_launch": 396940544},
    "out_proj": {"kernel": "out_proj", "workload": "outproj_bf16_b4h32s4096d128_n4096",
                 "files": ['causal_head_attention_mha_gb300/csrc/gemm_bf16.cu', 'causal_head_attention_mha_gb300/csrc/ptx.cuh'],
                 "sha256": "d4365aeeda8876f4d66ac37b9eb57eae1df6b69289171a103464038b9ac0cc00", "bytes_per_launch": 404913152},
}


def source_sha(rels):
    h = hashlib.sha256()
    for rel in rels:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_for(kernel, workload):
    """Recorded DRAM bytes per launch of `kernel` on `workload`, or None when no
    capture of this workload exists or the source changed since it was taken."""
    for t in TRAFFIC.values():
        if t["kernel"] != kernel or t["workload"] != workload:
            continue
        if t["sha256"] is None or t["bytes_per_launch"] is None:
            return None
        return t["bytes_per_launch"] if source_sha(t["files"]) == t["sha256"] else None
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
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            text, _ = self.proc.communicate()
        rows = [r.split(",") for r in text.strip().splitlines() if r.count(",") >= 8]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


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
            "sample": f"{n} random query rows of {workload} (causal), "
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
def run_ours(args, rank, world, dist):
    import torch
    import causal_head_attention_mha_gb300 as mha

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mha.load_library()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)

    torch_dtype = {"bf16": torch.bfloat16, "f16": torch.float16}

    def dev16(t, dtype):
        return torch.from_numpy(t.bits.view(np.int16)).view(torch_dtype[dtype]).to(dev)

    do_prefill = args.only in ("both", "prefill")
    do_decode = args.only in ("both", "decode")
    wp = si.WORKLOADS[args.prefill_workload]
    wd = si.WORKLOADS[args.decode_workload]
    pdt, ddt = wp["dtype"], wd.get("dtype", "bf16")
    varlen = "key_len_lo" in wp
    if varlen:
        fwd = mha.mha_fwd_varlen_f16 if pdt == "f16" else mha.mha_fwd_varlen
    else:
        fwd = mha.mha_fwd_f16 if pdt == "f16" else mha.mha_fwd
    dec = mha.mha_decode_f16 if ddt == "f16" else mha.mha_decode
    # each rank works on its own batch (weak scaling, no collective on the data path)
    if do_prefill:
        xp = si.prefill_inputs(wp["B"], wp["H"], wp["S"], wp["D"], rank_seed(wp["seed"], rank),
                               qk_std=wp["qk_std"], dtype=pdt)
        Q, K, V = dev16(xp.Q, pdt), dev16(xp.K, pdt), dev16(xp.V, pdt)
        O = torch.empty_like(Q)
        LSE = torch.empty((xp.B, xp.H, xp.S), dtype=torch.float32, device=dev)
        if varlen:
            xp.key_lens = si.prefill_key_lens(xp.B, rank_seed(wp["seed"], rank), wp["key_len_lo"],
                                              wp["key_len_hi"])
            KL = torch.from_numpy(xp.key_lens).to(dev)
            flops = prefill_flops_varlen(xp.H, xp.S, xp.D, xp.key_lens, True)
        else:
            flops = prefill_flops(xp.B, xp.H, xp.S, xp.D, True)
    if do_decode:
        xd = si.decode_inputs(wd["B"], wd["H"], wd["D"], rank_seed(wd["seed"], rank), wd["len_lo"],
                              wd["len_hi"], dtype=ddt)
        q, Kc, Vc = dev16(xd.q, ddt), dev16(xd.Kc, ddt), dev16(xd.Vc, ddt)
        sl = torch.from_numpy(xd.seqlens).to(dev)
        Od = torch.empty_like(q)
        dbytes = decode_bytes(xd.B, xd.H, xd.D, xd.seqlens)
        nsplit = mha.mha_decode_num_splits(xd.B, xd.H)

    def prefill():
        if varlen:
            fwd(Q, K, V, KL, O=O, LSE=LSE, scale=xp.scale, causal=True, stream=stream)
        else:
            fwd(Q, K, V, O=O, LSE=LSE, scale=xp.scale, causal=True, stream=stream)

    def decode():
        dec(q, Kc, Vc, sl, O=Od, scale=xd.scale, stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---------------- warm-up
    for _ in range(args.warmup):
        if do_prefill:
            prefill()
        if do_decode:
            decode()
    barrier()
    st = mha.mha_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {mha.mha_status_string(st)}")

    # ---------------- timed region (device-resident inputs)
    K_ = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K_)]
    clock = ClockSampler(local)
    if not args.profile:
        clock.start()
        time.sleep(0.3)
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(K_):
        evs[k][0].record(stream)
        if do_prefill:
            prefill()
        evs[k][1].record(stream)
        if do_decode:
            decode()
        evs[k][2].record(stream)
    t_end.record(stream)
    barrier()
    clocks = clock.stop() if not args.profile else None
    st = mha.mha_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {mha.mha_status_string(st)}")
    tp = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3  # s, prefill launches
    td = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3  # s, decode launches
    total = t_start.elapsed_time(t_end) / 1e3
    tp, td, total = max_over_ranks([tp, td, total], dist, dev)
    launches = K_ * ((1 if do_prefill else 0) + ((1 + (nsplit > 1)) if do_decode else 0))

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
    if not args.no_e2e:
        E = min(K_, args.e2e_steps)
        h2d = d2h = 0
        ep = ed = 0.0
        if do_prefill:
            hQ, hK, hV = (torch.from_numpy(t.bits.view(np.int16)).pin_memory()
                          for t in (xp.Q, xp.K, xp.V))
            hO = torch.empty(Q.shape, dtype=torch.int16).pin_memory()
            hL = torch.empty(LSE.shape, dtype=torch.float32).pin_memory()
            h2d += 3 * hQ.numel() * 2
            d2h += hO.numel() * 2 + hL.numel() * 4
            pb = [(Q, K, V, O, LSE),
                  tuple(torch.empty_like(t) for t in (Q, K, V, O, LSE))]

            def p_in(b):
                for dst, src in zip(pb[b][:3], (hQ, hK, hV)):
                    dst.view(torch.int16).copy_(src, non_blocking=True)

            def p_cmp(b):
                q_, k_, v_, o_, l_ = pb[b]
                if varlen:
                    fwd(q_, k_, v_, KL, O=o_, LSE=l_, scale=xp.scale, causal=True, stream=stream)
                else:
                    fwd(q_, k_, v_, O=o_, LSE=l_, scale=xp.scale, causal=True, stream=stream)

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
        e2e = {"value": (whole_job_rate(world, E * flops, ep) / 1e12) if do_prefill else None,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": E,
               "decode_gbs": (whole_job_rate(world, E * dbytes, ed) / 1e9) if do_decode else None,
               "path": "pinned host -> cudaMemcpyAsync (copy-in stream) -> C-ABI call (compute "
                       "stream) -> cudaMemcpyAsync (read-back stream) -> pinned host; two "
                       "device buffer sets, so step k+1's inputs go up and step k-1's result "
                       "comes back while step k computes"}

    if rank != 0:
        return 0

    line = {"impl": "ours", "metric": METRIC}
    cfg = {"workload": args.prefill_workload if do_prefill else args.decode_workload,
           "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}
    if do_prefill:
        value = whole_job_rate(world, K_ * flops, tp) / 1e12
        per_launch_s = tp / K_
        achieved = flops / per_launch_s / 1e12
        line.update({"value": value, "unit": "TFLOP/s"})
        cfg.update({"prefill": {"B": xp.B, "H": xp.H, "S": xp.S, "D": xp.D, "causal": True,
                                "qk_std": wp["qk_std"], "flops_per_step": flops}})
        if varlen:
            # flops count each row's valid keys: min(i + 1, L_b)
            cfg["prefill"]["key_lens"] = [int(v) for v in xp.key_lens]
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                    "traffic": traffic_for("prefill_" + pdt, args.prefill_workload),
                    "peak_source": f"bf16_tflops (burst), of {peak_src}",
                    "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                    "kernel": f"prefill_{pdt}{'_varlen' if varlen else ''}_kernel<{xp.D}, causal>", "us_per_launch": 1e6 * per_launch_s,
                    **launch_percentiles([e[0].elapsed_time(e[1]) for e in evs])}
        line["roofline"] = roofline
    if do_decode:
        gbs = whole_job_rate(world, K_ * dbytes, td) / 1e9
        cfg.update({"decode": {"B": xd.B, "H": xd.H, "D": xd.D, "len_range": [512, 8192],
                               "total_tokens": int(xd.seqlens.sum()), "splits": nsplit,
                               "bytes_per_step": dbytes}})
        line["decode"] = {"value": gbs, "unit": "GB/s", "bound": "hbm",
                          "achieved": dbytes / (td / K_) / 1e9, "peak": peaks["hbm_gbs"],
                          "frac": dbytes / (td / K_) / 1e9 / peaks["hbm_gbs"],
                          "traffic": traffic_for("decode", args.decode_workload), "peak_source": f"hbm_gbs, of {peak_src}",
                          "us_per_call": 1e6 * td / K_,
                          **launch_percentiles([e[1].elapsed_time(e[2]) for e in evs])}
        if not do_prefill:
            line.update({"value": gbs, "unit": "GB/s"})
    line.update({
        "n_gpus": world, "steps": K_, "warmup": args.warmup, "ms_per_step": 1e3 * total / K_,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": pdt if do_prefill else ddt,
        "data": "synthetic", "config": cfg, "clocks": clocks, "e2e": e2e,
        "gpu_launches": launches,
    })
    if not args.no_cpu_baseline and world == 1 and do_prefill:
        line["cpu_baseline"] = oracle_sample_tflops(xp, args.cpu_seconds, workload=args.prefill_workload)
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


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--only", choices=("both", "prefill", "decode", "projections"),
                    default="both")
    ap.add_argument("--prefill-workload", default=PREFILL_WORKLOAD,
                    choices=[k for k, w in si.WORKLOADS.items()
                             if w["kind"] == "prefill" and w["dtype"] in ("bf16", "f16")],
                    help="prefill workload of the step, bf16 or f16 (default: the headline one)")
    ap.add_argument("--decode-workload", default=DECODE_WORKLOAD,
                    choices=[k for k, w in si.WORKLOADS.items() if w["kind"] == "decode"],
                    help="decode workload of the step (bf16 or f16)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--profile", action="store_true", help="no clock sampling (for ncu runs)")
    args = ap.parse_args()
    if args.warmup < 3 and not args.profile:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
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
