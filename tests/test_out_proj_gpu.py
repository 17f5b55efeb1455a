"""The output projection (mha_out_proj) against the fp64 oracle (GPU only).

Y = concat_h(O_h) W_O with O in the [B, H, S, D] layout attention writes.
Tolerance (the method fixes none; derived from the arithmetic, as for the
Q/K/V projection): bf16 products accumulated in fp32 and rounded to bf16, so
|Y - ref| <= 2^-8 |ref| + 2^-13 sum_k |a_k w_k|, relative Frobenius <= 5e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import dev_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import causal_head_attention_mha_gb300 as mha
    mha.load_library()
    torch.cuda.set_device(0)
    yield
    assert mha.mha_get_device_status() == 0


def mha():
    import causal_head_attention_mha_gb300 as m
    return m


def _check(Y, O, W, rows=None, what=""):
    """Y: GPU [B, S, N]; O [B, H, S, D], W [H*D, N]: float32 values; rows: (b, s) pairs."""
    if rows is not None:
        O = O[rows[:, 0], :, rows[:, 1], :][:, :, None, :]      # [R, H, 1, D]
    R = oracle.out_projection(O, W)
    B, H, S, D = O.shape
    A = np.abs(O.astype(np.float64)).transpose(0, 2, 1, 3).reshape(B * S, H * D)
    extra = (2.0 ** -13) * (A @ np.abs(W.astype(np.float64))).reshape(R.shape)
    g = Y.float().cpu().numpy()
    if rows is not None:
        g = g[rows[:, 0], rows[:, 1]][:, None, :]
    assert np.all(np.isfinite(g)), what
    err = np.abs(g - R)
    bound = 2.0 ** -8 * np.abs(R) + extra
    assert np.all(err <= bound), f"{what}: worst excess {float(np.max(err - bound)):.3e}"
    frob = float(np.linalg.norm(g - R) / max(np.linalg.norm(R), 1e-30))
    assert frob <= 5e-3, f"{what}: rel-Frobenius {frob:.3e}"


SHAPES = [
    (1, 1, 100, 64, 32),      # one partial row tile, one 32-column chunk
    (2, 3, 130, 128, 288),    # S tail in both sequences, 1.1 column tiles
    (1, 2, 1, 64, 64),        # a single row
    (3, 5, 257, 64, 544),     # tails everywhere, K = 320 (5 steps)
    (2, 8, 1024, 128, 512),   # 32 row tiles x 2 column tiles: several tiles per CTA
]


@pytest.mark.parametrize("B,H,S,D,N", SHAPES)
def test_out_proj_full(B, H, S, D, N):
    x = si.out_projection_inputs(B, H, S, D, N, seed=5000 + S + N)
    Y = mha().mha_out_proj(dev_tensor(x.O, torch.bfloat16), dev_tensor(x.W, torch.bfloat16))
    assert Y.shape == (B, S, N) and Y.dtype == torch.bfloat16
    _check(Y, x.O.values, x.W.values, what=f"B{B} H{H} S{S} D{D} N{N}")


def test_out_proj_workload_sampled():
    """The full-size output projection (B4 H32 S4096 D128 -> 4096) on sampled rows."""
    x = si.workload_inputs("outproj_bf16_b4h32s4096d128_n4096")
    Y = mha().mha_out_proj(dev_tensor(x.O, torch.bfloat16), dev_tensor(x.W, torch.bfloat16))
    rng = np.random.default_rng(6)
    rows = np.stack([rng.integers(0, x.B, 96), rng.integers(0, x.S, 96)], axis=1)
    rows = np.concatenate([rows, [[0, 0], [x.B - 1, x.S - 1], [1, 127], [2, 128]]])
    _check(Y, x.O.values, x.W.values, rows=rows, what="out-projection workload")
    assert torch.isfinite(Y.float()).all()


def test_out_proj_head_order_one_hot():
    """O one-hot at (b, h, s, d): Y is zero except row (b, s), which is row
    h*D + d of W exactly; a head-order or layout slip moves or loses it."""
    B, H, S, D, N = 2, 4, 200, 64, 96
    x = si.out_projection_inputs(B, H, S, D, N, seed=10)
    O = np.zeros((B, H, S, D), np.float32)
    O[1, 2, 150, 17] = 1.0
    Y = mha().mha_out_proj(torch.from_numpy(O).to(torch.bfloat16).cuda(),
                           dev_tensor(x.W, torch.bfloat16))
    g = Y.float().cpu().numpy()
    assert np.array_equal(g[1, 150], x.W.values[2 * D + 17])
    g[1, 150] = 0.0
    assert not np.any(g)


def test_out_proj_after_attention():
    """The attention output feeds the projection directly (same layout)."""
    p = si.prefill_inputs(2, 4, 300, 128, seed=77)
    w = si.out_projection_inputs(2, 4, 300, 128, 256, seed=78)
    t = torch.bfloat16
    O, _ = mha().mha_fwd(dev_tensor(p.Q, t), dev_tensor(p.K, t), dev_tensor(p.V, t),
                         scale=p.scale, causal=True)
    Y = mha().mha_out_proj(O, dev_tensor(w.W, t))
    _check(Y, O.float().cpu().numpy(), w.W.values, what="attention -> projection")


def test_out_proj_deterministic():
    x = si.out_projection_inputs(2, 4, 300, 128, 256, seed=13)
    Od, Wd = dev_tensor(x.O, torch.bfloat16), dev_tensor(x.W, torch.bfloat16)
    a = mha().mha_out_proj(Od, Wd)
    b = mha().mha_out_proj(Od, Wd)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
