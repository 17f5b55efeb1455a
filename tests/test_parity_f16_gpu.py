"""f16 entry points (mha_fwd_f16, mha_decode_f16) against the fp64 oracle (GPU only).

The same checks as the bf16 path, on f16 inputs: element by element on small
shapes (several tiles, ragged tails, several work items per CTA), on sampled
rows of the full-size f16 bench workload, moves of the reference maximum
(f16 weights are kept <= 2^15: the f16 kernel takes each tile's row maximum and
moves the reference, rescaling O, when the scores jump by more than 15.9 log2
units), and decode.  The tolerances are
the bf16 ones (f16 keeps more mantissa bits, so they are looser for it).
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_bf16_close, dev_tensor, sample_rows

pytestmark = pytest.mark.gpu
F16 = torch.float16


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


def _prefill(x, causal, K=None):
    K = x.K if K is None else K
    return mha().mha_fwd_f16(dev_tensor(x.Q, F16), dev_tensor(K, F16), dev_tensor(x.V, F16),
                             scale=x.scale, causal=causal)


SMALL = [(1, 2, 128, 128), (2, 3, 300, 128), (1, 2, 257, 64), (2, 2, 383, 64), (3, 1, 520, 64),
         (1, 1, 640, 128), (1, 1, 1, 64)]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("qk_std", [1.0, 3.0])
@pytest.mark.parametrize("B,H,S,D", SMALL)
def test_f16_prefill_full(B, H, S, D, causal, qk_std):
    x = si.prefill_inputs(B, H, S, D, seed=1900 + S + D + int(qk_std), qk_std=qk_std, dtype="f16")
    O, L = _prefill(x, causal)
    assert O.dtype == F16
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal)
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr,
                      what=f"f16 B{B} H{H} S{S} D{D} causal={causal} std={qk_std}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_f16_prefill_many_items_per_cta(causal, D):
    x = si.prefill_inputs(8, 40, 600, D, seed=6150 + D, dtype="f16")
    O, L = _prefill(x, causal)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal)
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr,
                      what=f"f16 B8 H40 S600 D{D} causal={causal}")


def _scale_keys_f16(t, lo, hi, factor):
    """K with keys lo..hi-1 multiplied by a power of two (exact in f16 here)."""
    v = t.values.copy()
    v[:, :, lo:hi, :] *= factor
    bits = si.f16_bits(v)
    out = si.Tensor(si.f16_to_f32(bits), bits)
    assert np.array_equal(out.values, v)
    return out


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("factor", [8.0, 64.0])
@pytest.mark.parametrize("which", ["later_keys_dominate", "first_keys_dominate"])
def test_f16_prefill_reference_moves(causal, D, factor, which):
    """Keys scaled by 8 push later scores ~20-30 (log2 units) above an item's
    first-tile reference, past the f16 headroom of 15.9: the reference moves and
    O is rescaled; by 64 the jump is larger still, and with the first keys
    scaled the later tiles underflow against the reference."""
    S = 300
    x = si.prefill_inputs(1, 2, S, D, seed=1777 + D, dtype="f16")
    lo, hi = (128, S) if which == "later_keys_dominate" else (0, 128)
    K = _scale_keys_f16(x.K, lo, hi, factor)
    O, L = _prefill(x, causal, K)
    Or, Lr = oracle.attention(x.Q.values, K.values, x.V.values, x.scale, causal)
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr,
                      what=f"f16 {which} x{factor} D{D} causal={causal}")


def _f16_tensor(v):
    bits = si.f16_bits(v)
    out = si.Tensor(si.f16_to_f32(bits), bits)
    assert np.array_equal(out.values, v)
    return out


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_f16_prefill_some_rows_of_a_warp_move(causal, D):
    """Only a few rows of each 32-row warp see their scores jump past the f16
    headroom in later key tiles: query feature 0 is 200 on rows 3, 40, 77,
    131, 170 and 250, and key feature 0 is 0 on keys 0..127 and 1 after, so
    those rows' scores rise by 200 * scale * log2(e) (25 to 36, log2 units)
    while every other row's change is below 1.  The rows that must move take
    their warp along (each row to its own tile maximum + 8): the moving rows
    and the rows moved with them must both match the oracle."""
    S = 300
    x = si.prefill_inputs(1, 2, S, D, seed=2711 + D, dtype="f16")
    q = x.Q.values.copy()
    k = x.K.values.copy()
    rows = [3, 40, 77, 131, 170, 250]
    q[:, :, rows, 0] = 200.0
    k[:, :, :128, 0] = 0.0
    k[:, :, 128:, 0] = 1.0
    Q, K = _f16_tensor(q), _f16_tensor(k)
    O, L = mha().mha_fwd_f16(dev_tensor(Q, F16), dev_tensor(K, F16), dev_tensor(x.V, F16),
                             scale=x.scale, causal=causal)
    Or, Lr = oracle.attention(Q.values, K.values, x.V.values, x.scale, causal)
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr,
                      what=f"f16 some rows move D{D} causal={causal}")


def test_f16_prefill_deterministic():
    x = si.prefill_inputs(2, 4, 1000, 128, seed=41337, dtype="f16")
    Q, K, V = (dev_tensor(t, F16) for t in (x.Q, x.K, x.V))
    O1, L1 = mha().mha_fwd_f16(Q, K, V, scale=x.scale, causal=True)
    O2, L2 = mha().mha_fwd_f16(Q, K, V, scale=x.scale, causal=True)
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1, L2)


@pytest.mark.parametrize("causal", [True, False])
def test_f16_prefill_workload_sampled(causal):
    name = "prefill_f16_b4h32s4096d128_qk3"
    x = si.workload_inputs(name)
    O, L = _prefill(x, causal)
    rows = sample_rows(x.B, x.H, x.S, n_bh=12, rows_per_bh=96, seed=8)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal, rows=rows)
    Og = O.view(-1, x.D)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    Lg = L.view(-1)[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_bf16_close(Og, Or, Lg, Lr, what=f"{name} causal={causal}")
    assert torch.isfinite(O.float()).all()
    assert torch.isfinite(L).all()


def test_f16_and_bf16_entry_points_reject_each_others_tensors():
    x = si.prefill_inputs(1, 1, 64, 64, seed=3, dtype="f16")
    Q = dev_tensor(x.Q, F16)
    with pytest.raises(ValueError):
        mha().mha_fwd(Q, Q, Q)
    with pytest.raises(ValueError):
        mha().mha_fwd_f16(Q.to(torch.bfloat16), Q.to(torch.bfloat16), Q.to(torch.bfloat16))


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("B,H,D,lens", [
    (3, 4, 128, [1, 200, 77]),
    (5, 2, 64, [64, 0, 513, 1, 1000]),
    (7, 3, 128, [33, 129, 2049, 5, 0, 700, 1]),
])
def test_f16_decode_small(B, H, D, lens):
    z = si.decode_inputs(B, H, D, seed=177 + B + D, seqlens=np.array(lens, np.int32), dtype="f16")
    O = mha().mha_decode_f16(dev_tensor(z.q, F16), dev_tensor(z.Kc, F16), dev_tensor(z.Vc, F16),
                             torch.from_numpy(z.seqlens).cuda(), scale=z.scale)
    assert O.dtype == F16
    Or, _ = oracle.decode(z.q.values, z.Kc.values, z.Vc.values, z.seqlens, z.scale)
    Og = O.float().cpu().numpy()
    assert_bf16_close(Og, Or, what=f"f16 decode {lens}")
    for b, Lb in enumerate(lens):
        if Lb == 0:
            assert np.all(Og[b] == 0.0)


def test_f16_decode_workload_full():
    z = si.workload_inputs("decode_f16_b16h32d128_len512_8192")
    O = mha().mha_decode_f16(dev_tensor(z.q, F16), dev_tensor(z.Kc, F16), dev_tensor(z.Vc, F16),
                             torch.from_numpy(z.seqlens).cuda(), scale=z.scale)
    Or, _ = oracle.decode(z.q.values, z.Kc.values, z.Vc.values, z.seqlens, z.scale)
    assert_bf16_close(O.float().cpu().numpy(), Or, what="f16 decode workload")


def test_f16_decode_matches_last_causal_row():
    """Cross-entry consistency on f16: decode over L keys = row L-1 of causal prefill."""
    H, D, L = 4, 128, 300
    x = si.prefill_inputs(1, H, L, D, seed=1606, dtype="f16")
    O, _ = _prefill(x, True)
    q = dev_tensor(x.Q, F16)[0, :, L - 1, :].unsqueeze(0).contiguous()
    Kc = dev_tensor(x.K, F16)[0].permute(1, 0, 2).contiguous()
    Vc = dev_tensor(x.V, F16)[0].permute(1, 0, 2).contiguous()
    Od = mha().mha_decode_f16(q, Kc, Vc, torch.tensor([L], dtype=torch.int32, device="cuda"),
                              scale=x.scale)
    diff = (Od[0].float() - O[0, :, L - 1, :].float()).abs().max().item()
    assert diff <= 2e-2, diff
