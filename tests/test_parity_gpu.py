"""CUDA path against the fp64 oracle on the same seeded inputs (GPU only).

Small shapes are compared element by element on every output; the full-size
workloads are compared on sampled rows (every tile edge plus random rows),
in the launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import (TOL_F32_ABS, TOL_LSE, assert_bf16_close, dev_tensor, errors, sample_rows)

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


# ------------------------------------------------------------------ fp32 path
@pytest.mark.parametrize("B,H,S,D,causal", [
    (1, 2, 128, 64, True),      # the fp32 workload
    (1, 2, 128, 64, False),
    (2, 3, 1, 64, True), (1, 2, 127, 128, True), (1, 1, 129, 64, False),
    (2, 1, 255, 128, True), (1, 2, 300, 64, True),
])
def test_f32_prefill_full(B, H, S, D, causal):
    seed = 1001 if (B, H, S, D) == (1, 2, 128, 64) else 500 + S + D
    x = si.prefill_inputs(B, H, S, D, seed=seed, dtype="f32")
    O, L = mha().mha_fwd_f32(dev_tensor(x.Q, torch.float32), dev_tensor(x.K, torch.float32),
                             dev_tensor(x.V, torch.float32), scale=x.scale, causal=causal)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal)
    err, _ = errors(O.cpu().numpy(), Or)
    lerr, _ = errors(L.cpu().numpy(), Lr)
    assert err <= TOL_F32_ABS, err
    assert lerr <= TOL_LSE, lerr


# ------------------------------------------------------------------ bf16 prefill, small
SMALL = [
    (1, 1, 1, 128), (1, 2, 128, 128), (2, 3, 300, 128), (1, 2, 257, 64), (2, 2, 383, 64),
    (1, 1, 640, 128), (1, 3, 129, 64), (3, 1, 520, 64),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("qk_std", [1.0, 3.0])
@pytest.mark.parametrize("B,H,S,D", SMALL)
def test_bf16_prefill_full(B, H, S, D, causal, qk_std):
    x = si.prefill_inputs(B, H, S, D, seed=900 + S + D + int(qk_std), qk_std=qk_std)
    O, L = mha().mha_fwd(dev_tensor(x.Q, torch.bfloat16), dev_tensor(x.K, torch.bfloat16),
                         dev_tensor(x.V, torch.bfloat16), scale=x.scale, causal=causal)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal)
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr,
                      what=f"B{B} H{H} S{S} D{D} causal={causal} std={qk_std}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_bf16_prefill_many_items_per_cta(causal, D):
    """Every output compared on a workload with several 256-row work items
    per CTA of the persistent grid (B*H*ceil(S/256) = 960 items), so the K/V
    ring and every barrier phase carry over from item to item; S = 600 also
    leaves the last query block of each head without its second tile."""
    x = si.prefill_inputs(8, 40, 600, D, seed=5150 + D)
    O, L = mha().mha_fwd(dev_tensor(x.Q, torch.bfloat16), dev_tensor(x.K, torch.bfloat16),
                         dev_tensor(x.V, torch.bfloat16), scale=x.scale, causal=causal)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal)
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr,
                      what=f"B8 H40 S600 D{D} causal={causal}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("B,H,S,causal", [(4, 40, 512, True), (4, 32, 768, False),
                                           (4, 40, 384, False), (4, 40, 300, False),
                                           (8, 16, 700, True), (4, 40, 1000, True)])
def test_prefill_wide_item_schedule(B, H, S, causal, dtype):
    """Plain D = 128 shapes whose item schedule takes the wide groups (the
    host's load model picks them on this GPU), every output compared.  There
    tile A of each item starts while tile B finishes the item before, also
    after items whose last query block has no tile B (S = 384, 300) and after
    ragged tiles (S = 300, 700, 1000)."""
    if not mha().mha_prefill_wide_schedule(B, H, S, 128, causal=causal):
        pytest.skip("the narrow groups are chosen on this GPU's SM count")
    f16 = dtype == torch.float16
    x = si.prefill_inputs(B, H, S, 128, seed=7300 + S, dtype="f16" if f16 else "bf16")
    fwd = mha().mha_fwd_f16 if f16 else mha().mha_fwd
    O, L = fwd(dev_tensor(x.Q, dtype), dev_tensor(x.K, dtype), dev_tensor(x.V, dtype),
               scale=x.scale, causal=causal)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal)
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr,
                      what=f"wide schedule B{B} H{H} S{S} causal={causal} {dtype}")


def _scale_keys(t, lo, hi, factor):
    """K with keys lo..hi-1 multiplied by a power of two (exact in bf16)."""
    v = t.values.copy()
    v[:, :, lo:hi, :] *= factor
    bits = si.bf16_bits(v)
    return si.Tensor(si.bf16_to_f32(bits), bits)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("which", ["later_keys_dominate", "first_keys_dominate",
                                   "second_half_dominates"])
def test_bf16_prefill_reference_moves(causal, D, which):
    """Scores of some keys far above the others (x64): with later keys larger,
    a row's reference maximum has to move by far more than 64 (log2 units)
    after its first tile, which takes the kernel's re-do path (the tile's
    weights redone with its true maximum, O rescaled); with the first keys
    larger, later tiles underflow against the reference.  With only keys
    192..255 larger (the second half of key tile 1), the first half of that
    tile stays within the bound and is handed to the tensor core before the
    second half is found to pass it: the second half is redone and O, which
    by then includes the first half's product, is rescaled after that
    product completes."""
    S = 300
    x = si.prefill_inputs(1, 2, S, D, seed=777 + D)
    lo, hi = {"later_keys_dominate": (128, S), "first_keys_dominate": (0, 128),
              "second_half_dominates": (192, 256)}[which]
    K = _scale_keys(x.K, lo, hi, 64.0)
    O, L = mha().mha_fwd(dev_tensor(x.Q, torch.bfloat16), dev_tensor(K, torch.bfloat16),
                         dev_tensor(x.V, torch.bfloat16), scale=x.scale, causal=causal)
    Or, Lr = oracle.attention(x.Q.values, K.values, x.V.values, x.scale, causal)
    assert float(np.max(Lr)) > 60.0  # the logits really are large
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr,
                      what=f"{which} D{D} causal={causal}")


def test_bf16_prefill_without_lse_and_canary():
    x = si.prefill_inputs(1, 2, 200, 128, seed=4242)
    Q, K, V = (dev_tensor(t, torch.bfloat16) for t in (x.Q, x.K, x.V))
    n = Q.numel()
    buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    O = buf[:n].view(Q.shape)
    mha().mha_fwd(Q, K, V, O=O, scale=x.scale, causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert torch.all(buf[n:] == 7.0), "write past the end of O"
    Or, _ = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, True)
    assert_bf16_close(O.float().cpu().numpy(), Or)


def test_bf16_prefill_deterministic():
    x = si.prefill_inputs(2, 4, 1000, 128, seed=31337)
    Q, K, V = (dev_tensor(t, torch.bfloat16) for t in (x.Q, x.K, x.V))
    O1, L1 = mha().mha_fwd(Q, K, V, scale=x.scale, causal=True)
    O2, L2 = mha().mha_fwd(Q, K, V, scale=x.scale, causal=True)
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1, L2)


# ------------------------------------------------------------------ bf16 prefill, full size
FULL = [
    ("prefill_bf16_b1h32s2048d128", True),
    ("prefill_bf16_b4h32s4096d128_qk3", True),
    ("prefill_bf16_b4h32s4096d128_qk3", False),
    ("prefill_bf16_b2h16s16384d64", True),
]


@pytest.mark.parametrize("name,causal", FULL)
def test_bf16_prefill_workload_sampled(name, causal):
    x = si.workload_inputs(name)
    Q, K, V = (dev_tensor(t, torch.bfloat16) for t in (x.Q, x.K, x.V))
    O, L = mha().mha_fwd(Q, K, V, scale=x.scale, causal=causal)
    rows = sample_rows(x.B, x.H, x.S, n_bh=12, rows_per_bh=96, seed=7)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal, rows=rows)
    Og = O.view(-1, x.D)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    Lg = L.view(-1)[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_bf16_close(Og, Or, Lg, Lr, what=f"{name} causal={causal}")
    # properties checked on every row, not only the sampled ones
    assert torch.isfinite(O.float()).all()
    assert torch.isfinite(L).all()


# Long D = 128 sequences take the wide item groups, where tile A's first S
# product of an item is issued in the previous item's last step
LONG_WIDE = [
    (2, 16, 16384, True, torch.bfloat16),
    (2, 16, 16384, False, torch.bfloat16),
    (1, 32, 8192, False, torch.bfloat16),
    (2, 16, 16384, True, torch.float16),
]


@pytest.mark.parametrize("B,H,S,causal,dtype", LONG_WIDE)
def test_prefill_long_wide_sampled(B, H, S, causal, dtype):
    """Sampled rows (random rows and tile edges of sampled heads, so the first
    tiles of many items) of long D = 128 prefills against the oracle."""
    if not mha().mha_prefill_wide_schedule(B, H, S, 128, causal=causal):
        pytest.skip("the narrow groups are chosen on this GPU's SM count")
    f16 = dtype == torch.float16
    x = si.prefill_inputs(B, H, S, 128, seed=8100 + S + int(causal), qk_std=3.0 if f16 else 1.0,
                          dtype="f16" if f16 else "bf16")
    Q, K, V = (dev_tensor(t, dtype) for t in (x.Q, x.K, x.V))
    fwd = mha().mha_fwd_f16 if f16 else mha().mha_fwd
    O, L = fwd(Q, K, V, scale=x.scale, causal=causal)
    rows = sample_rows(x.B, x.H, x.S, n_bh=8, rows_per_bh=64, seed=11)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal, rows=rows)
    Og = O.view(-1, x.D)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    Lg = L.view(-1)[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_bf16_close(Og, Or, Lg, Lr, what=f"B{B} H{H} S{S} causal={causal} {dtype}")
    assert torch.isfinite(O.float()).all()
    assert torch.isfinite(L).all()


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("B,H,D,lens", [
    (3, 4, 128, [1, 200, 77]),
    (5, 2, 64, [64, 0, 513, 1, 1000]),
    (1, 8, 128, [4096]),
    (7, 3, 128, [33, 129, 2049, 5, 0, 700, 1]),
])
def test_decode_small(B, H, D, lens):
    z = si.decode_inputs(B, H, D, seed=77 + B + D, seqlens=np.array(lens, np.int32))
    O = mha().mha_decode(dev_tensor(z.q, torch.bfloat16), dev_tensor(z.Kc, torch.bfloat16),
                         dev_tensor(z.Vc, torch.bfloat16),
                         torch.from_numpy(z.seqlens).cuda(), scale=z.scale)
    Or, _ = oracle.decode(z.q.values, z.Kc.values, z.Vc.values, z.seqlens, z.scale)
    Og = O.float().cpu().numpy()
    assert_bf16_close(Og, Or, what=f"decode {lens}")
    for b, Lb in enumerate(lens):
        if Lb == 0:
            assert np.all(Og[b] == 0.0)


def test_decode_workload_full():
    z = si.workload_inputs("decode_bf16_b16h32d128_len512_8192")
    O = mha().mha_decode(dev_tensor(z.q, torch.bfloat16), dev_tensor(z.Kc, torch.bfloat16),
                         dev_tensor(z.Vc, torch.bfloat16),
                         torch.from_numpy(z.seqlens).cuda(), scale=z.scale)
    Or, _ = oracle.decode(z.q.values, z.Kc.values, z.Vc.values, z.seqlens, z.scale)
    assert_bf16_close(O.float().cpu().numpy(), Or, what="decode workload")
    O2 = mha().mha_decode(dev_tensor(z.q, torch.bfloat16), dev_tensor(z.Kc, torch.bfloat16),
                          dev_tensor(z.Vc, torch.bfloat16),
                          torch.from_numpy(z.seqlens).cuda(), scale=z.scale)
    assert torch.equal(O.view(torch.int16), O2.view(torch.int16)), "decode not deterministic"


def test_decode_matches_last_causal_row():
    """Cross-entry consistency: decode over L keys = row L-1 of causal prefill."""
    H, D, L = 4, 128, 300
    x = si.prefill_inputs(1, H, L, D, seed=606)
    O, _ = mha().mha_fwd(dev_tensor(x.Q, torch.bfloat16), dev_tensor(x.K, torch.bfloat16),
                         dev_tensor(x.V, torch.bfloat16), scale=x.scale, causal=True)
    q = dev_tensor(x.Q, torch.bfloat16)[0, :, L - 1, :].contiguous().view(1, H, D)
    Kc = dev_tensor(x.K, torch.bfloat16)[0].transpose(0, 1).contiguous()  # [L, H, D]
    Vc = dev_tensor(x.V, torch.bfloat16)[0].transpose(0, 1).contiguous()
    Od = mha().mha_decode(q, Kc, Vc, torch.tensor([L], dtype=torch.int32, device="cuda"),
                          scale=x.scale)
    diff = (Od[0].float() - O[0, :, L - 1].float()).abs().max().item()
    assert diff <= 2 * 2e-2, diff
