"""Helpers shared by the GPU tests: device copies of seeded inputs, error metrics.

Tolerances (fixed for the floating-point paths):
  fp32 path : max |O - O_ref| <= 1e-4
  bf16 path : max |O - O_ref| <= 2e-2 and ||O - O_ref||_F / ||O_ref||_F <= 5e-3
  LSE       : max |LSE - LSE_ref| <= 1e-3 (both paths)
"""
import numpy as np
import torch

TOL_F32_ABS = 1e-4
TOL_BF16_ABS = 2e-2
TOL_BF16_FROB = 5e-3
TOL_LSE = 1e-3


def dev_tensor(t, dtype, device="cuda"):
    """seeded_inputs.Tensor -> torch tensor on the device (bf16 / f16 from its bit patterns)."""
    if dtype in (torch.bfloat16, torch.float16):
        return torch.from_numpy(t.bits.view(np.int16)).view(dtype).to(device)
    return torch.from_numpy(np.ascontiguousarray(t.values)).to(device)


def errors(out, ref):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = out - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    nref = float(np.linalg.norm(ref))
    frob = float(np.linalg.norm(diff)) / nref if nref > 0 else float(np.linalg.norm(diff))
    return max_abs, frob


def assert_bf16_close(O, Oref, L=None, Lref=None, what=""):
    max_abs, frob = errors(O, Oref)
    assert np.all(np.isfinite(O)), f"{what}: non-finite output"
    assert max_abs <= TOL_BF16_ABS, f"{what}: max-abs {max_abs:.3e}"
    assert frob <= TOL_BF16_FROB, f"{what}: rel-Frobenius {frob:.3e}"
    if L is not None:
        lerr = float(np.max(np.abs(np.asarray(L, np.float64) - Lref)))
        assert lerr <= TOL_LSE, f"{what}: LSE {lerr:.3e}"
    return max_abs, frob


def sample_rows(B, H, S, n_bh, rows_per_bh, seed, tile=128):
    """Flat row ids (b*H+h)*S+i: random rows plus every tile edge and the tail."""
    rng = np.random.default_rng(seed)
    bhs = rng.choice(B * H, size=min(n_bh, B * H), replace=False)
    bhs = np.unique(np.concatenate([bhs, [0, B * H - 1]]))
    edges = sorted({0, 1, S - 1, S - 2} | {t for k in range(0, S, tile)
                                             for t in (k, k + tile - 1) if t < S})
    out = []
    for bh in bhs:
        r = rng.choice(S, size=min(rows_per_bh, S), replace=False)
        pick = np.unique(np.concatenate([r, np.array(edges[:: max(1, len(edges) // 64)])]))
        out.append(bh * S + pick)
    return np.concatenate(out).astype(np.int64)
