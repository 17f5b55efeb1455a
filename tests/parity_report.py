"""Measured errors of the GPU path against the fp64 oracle on the five workloads,
plus the f16 and key-padding prefill workloads of the bench.

Not a test (pytest does not collect it): it prints one markdown row per
workload with the largest absolute error of O, its relative Frobenius error
and the largest LSE error, next to the tolerances the parity tests enforce
(fp32: max-abs <= 1e-4; 16-bit: max-abs <= 2e-2, rel-Frobenius <= 5e-3;
LSE <= 1e-3).  Small workloads are compared in full; the large prefill
workloads on sampled rows (every tile edge plus random rows of random
heads), as the parity tests do.  Run on a GPU machine:

    python tests/parity_report.py
"""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import oracle  # noqa: E402
import seeded_inputs as si  # noqa: E402
from gpu_util import dev_tensor, errors, sample_rows  # noqa: E402


def prefill_row(name, causal, rows_per_bh=None):
    import causal_head_attention_mha_gb300 as mha
    x = si.workload_inputs(name)
    w = si.WORKLOADS[name]
    if w["dtype"] == "f32":
        O, L = mha.mha_fwd_f32(dev_tensor(x.Q, torch.float32), dev_tensor(x.K, torch.float32),
                               dev_tensor(x.V, torch.float32), scale=x.scale, causal=causal)
    elif x.key_lens is not None:
        kl = torch.from_numpy(np.ascontiguousarray(x.key_lens, dtype=np.int32)).cuda()
        O, L = mha.mha_fwd_varlen(dev_tensor(x.Q, torch.bfloat16), dev_tensor(x.K, torch.bfloat16),
                                  dev_tensor(x.V, torch.bfloat16), kl, scale=x.scale, causal=causal)
    else:
        tdt = torch.float16 if w["dtype"] == "f16" else torch.bfloat16
        fn = mha.mha_fwd_f16 if w["dtype"] == "f16" else mha.mha_fwd
        O, L = fn(dev_tensor(x.Q, tdt), dev_tensor(x.K, tdt), dev_tensor(x.V, tdt), scale=x.scale,
                  causal=causal)
    O = O.float().cpu().numpy().reshape(-1, x.D)
    L = L.cpu().numpy().reshape(-1)
    if rows_per_bh is None:
        rows = np.arange(x.B * x.H * x.S)
        Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal,
                                  key_lens=x.key_lens)
        Or, Lr = Or.reshape(-1, x.D), Lr.reshape(-1)
    else:
        rows = sample_rows(x.B, x.H, x.S, 8, rows_per_bh, seed=7)
        Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal, rows=rows,
                                  key_lens=x.key_lens)
    max_abs, frob = errors(O[rows], Or)
    lse = float(np.max(np.abs(L[rows] - Lr)))
    what = "all rows" if rows_per_bh is None else f"{len(rows)} sampled rows"
    return max_abs, frob, lse, what


def decode_row(name):
    import causal_head_attention_mha_gb300 as mha
    z = si.workload_inputs(name)
    O = mha.mha_decode(dev_tensor(z.q, torch.bfloat16), dev_tensor(z.Kc, torch.bfloat16),
                       dev_tensor(z.Vc, torch.bfloat16), torch.from_numpy(z.seqlens).cuda(),
                       scale=z.scale)
    Or, _ = oracle.decode(z.q.values, z.Kc.values, z.Vc.values, z.seqlens, z.scale)
    max_abs, frob = errors(O.float().cpu().numpy(), Or)
    return max_abs, frob, None, "all rows"


def main():
    torch.cuda.set_device(0)
    rows = [
        ("1. fp32 B1 H2 S128 D64, causal", lambda: prefill_row("prefill_f32_b1h2s128d64", True)),
        ("2. bf16 B1 H32 S2048 D128, causal",
         lambda: prefill_row("prefill_bf16_b1h32s2048d128", True, rows_per_bh=256)),
        ("3. bf16 B4 H32 S4096 D128 qk3, causal",
         lambda: prefill_row("prefill_bf16_b4h32s4096d128_qk3", True, rows_per_bh=192)),
        ("3. bf16 B4 H32 S4096 D128 qk3, causal=0",
         lambda: prefill_row("prefill_bf16_b4h32s4096d128_qk3", False, rows_per_bh=192)),
        ("4. decode bf16 B16 H32 D128", lambda: decode_row("decode_bf16_b16h32d128_len512_8192")),
        ("5. bf16 B2 H16 S16384 D64, causal",
         lambda: prefill_row("prefill_bf16_b2h16s16384d64", True, rows_per_bh=256)),
        ("f16 B4 H32 S4096 D128 qk3, causal",
         lambda: prefill_row("prefill_f16_b4h32s4096d128_qk3", True, rows_per_bh=192)),
        ("key padding bf16 B4 H32 S4096 D128, causal",
         lambda: prefill_row("prefill_varlen_bf16_b4h32s4096d128", True, rows_per_bh=192)),
    ]
    print("| Workload | max-abs | rel-Frobenius | LSE max-abs | compared |")
    print("|---|---:|---:|---:|---|")
    for name, fn in rows:
        max_abs, frob, lse, what = fn()
        lse_s = "—" if lse is None else f"{lse:.2e}"
        print(f"| {name} | {max_abs:.2e} | {frob:.2e} | {lse_s} | {what} |", flush=True)


if __name__ == "__main__":
    main()
