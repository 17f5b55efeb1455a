"""The fused Q/K/V projection (mha_qkv_proj) against the fp64 oracle (GPU only).

Tolerance (the method fixes none for this product; derived from the
arithmetic): each output is a dot product of bf16 values accumulated in fp32
and rounded to bf16, so |out - ref| <= 2^-8 |ref| (twice the round-to-nearest
bound of the output) + 2^-13 sum_k |x_k w_k| (fp32 accumulation), and the
relative Frobenius error <= 5e-3 as for attention.
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


def _check(out, X, W, H, D, rows=None, what=""):
    """out: GPU (Q, K, V); X, W: float32 values; rows: optional (b, s) pairs."""
    Xs = X if rows is None else X[rows[:, 0], rows[:, 1]][None]
    Qr, Kr, Vr = oracle.qkv_projection(Xs, W, H, D)
    absprod = np.abs(Xs.astype(np.float64)).reshape(-1, Xs.shape[-1]) @ np.abs(W.astype(np.float64))
    bound_extra = (2.0 ** -13) * absprod.reshape(Xs.shape[0], Xs.shape[1], 3, H, D).transpose(2, 0, 3, 1, 4)
    for c, (G, R) in enumerate(zip(out, (Qr, Kr, Vr))):
        g = G.float().cpu().numpy()
        if rows is not None:
            g = g[rows[:, 0], :, rows[:, 1], :][None].transpose(0, 2, 1, 3)
        err = np.abs(g - R)
        assert np.all(np.isfinite(g)), what
        assert np.all(err <= 2.0 ** -8 * np.abs(R) + bound_extra[c]), \
            f"{what} {'QKV'[c]}: worst excess {float(np.max(err - 2.0 ** -8 * np.abs(R) - bound_extra[c])):.3e}"
        frob = float(np.linalg.norm(g - R) / max(np.linalg.norm(R), 1e-30))
        assert frob <= 5e-3, f"{what} {'QKV'[c]}: rel-Frobenius {frob:.3e}"


SHAPES = [
    (1, 100, 72, 2, 64),     # one partial row tile, ragged K, 1.5 column tiles
    (2, 130, 256, 3, 128),   # row tail, 4.5 column tiles
    (1, 1, 8, 1, 64),        # a single row, K below one step
    (3, 257, 520, 5, 64),    # tails everywhere
    (2, 1024, 512, 8, 128),  # 192 tiles: several tiles per CTA, both accumulator buffers
]


@pytest.mark.parametrize("B,S,hid,H,D", SHAPES)
def test_qkv_proj_full(B, S, hid, H, D):
    x = si.projection_inputs(B, S, hid, H, D, seed=4000 + S + hid)
    out = mha().mha_qkv_proj(dev_tensor(x.X, torch.bfloat16), dev_tensor(x.W, torch.bfloat16), H, D)
    assert all(t.shape == (B, H, S, D) and t.dtype == torch.bfloat16 for t in out)
    _check(out, x.X.values, x.W.values, H, D, what=f"B{B} S{S} hidden{hid} H{H} D{D}")


def test_qkv_proj_workload_sampled():
    """The full-size projection (B4 S4096 hidden 4096, H32 D128) on sampled rows."""
    x = si.workload_inputs("qkv_bf16_b4s4096hid4096_h32d128")
    out = mha().mha_qkv_proj(dev_tensor(x.X, torch.bfloat16), dev_tensor(x.W, torch.bfloat16),
                             x.H, x.D)
    rng = np.random.default_rng(5)
    rows = np.stack([rng.integers(0, x.B, 96), rng.integers(0, x.S, 96)], axis=1)
    rows = np.concatenate([rows, [[0, 0], [x.B - 1, x.S - 1], [1, 127], [2, 128]]])
    _check(out, x.X.values, x.W.values, x.H, x.D, rows=rows, what="projection workload")
    for t in out:
        assert torch.isfinite(t.float()).all()


def test_qkv_proj_layout_one_hot():
    """X one-hot at (b, s, k): every output is zero except row (b, s), which
    holds row k of W split into Q, K, V heads exactly (products by 1, sums of
    zeros)."""
    B, S, hid, H, D = 2, 200, 64, 4, 64
    x = si.projection_inputs(B, S, hid, H, D, seed=9)
    X = np.zeros((B, S, hid), np.float32)
    X[1, 150, 17] = 1.0
    Xt = torch.from_numpy(X).to(torch.bfloat16).cuda()
    out = mha().mha_qkv_proj(Xt, dev_tensor(x.W, torch.bfloat16), H, D)
    row = x.W.values[17].reshape(3, H, D)
    for c, t in enumerate(out):
        g = t.float().cpu().numpy()
        assert np.array_equal(g[1, :, 150, :], row[c])
        g[1, :, 150, :] = 0.0
        assert not np.any(g)


def test_qkv_proj_deterministic():
    x = si.projection_inputs(2, 300, 256, 4, 128, seed=12)
    Xd, Wd = dev_tensor(x.X, torch.bfloat16), dev_tensor(x.W, torch.bfloat16)
    a = mha().mha_qkv_proj(Xd, Wd, 4, 128)
    b = mha().mha_qkv_proj(Xd, Wd, 4, 128)
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))
