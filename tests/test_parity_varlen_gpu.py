"""Key padding (mha_fwd_varlen, mha_fwd_varlen_f16) against the fp64 oracle (GPU only).

Sequence b has key_lens[b] valid keys; the oracle excludes keys j >= L_b the
same way (pinned in tests/oracle_pins.py).  Compared element by element on
shapes with several tiles and ragged tails, key lengths of 0, 1, shorter than
the causal diagonal, not a multiple of the 128-key tile, and the full S; plus
properties that need no oracle: with every L_b = S the result is mha_fwd's,
bit for bit, and the padding keys' K and V rows do not matter, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_bf16_close, dev_tensor

pytestmark = pytest.mark.gpu
TYPES = {"bf16": torch.bfloat16, "f16": torch.float16}


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


def _run(x, kl, causal, dtype, K=None, V=None):
    t = TYPES[dtype]
    fn = mha().mha_fwd_varlen_f16 if dtype == "f16" else mha().mha_fwd_varlen
    K = x.K if K is None else K
    V = x.V if V is None else V
    return fn(dev_tensor(x.Q, t), dev_tensor(K, t), dev_tensor(V, t),
              torch.as_tensor(np.asarray(kl, np.int32)).cuda(), scale=x.scale, causal=causal)


def _compare(x, kl, causal, O, L, what):
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal,
                              key_lens=np.clip(np.asarray(kl), 0, x.S))
    Og, Lg = O.float().cpu().numpy(), L.cpu().numpy()
    empty = ~np.isfinite(Lr)
    assert np.all(Lg[empty] == -np.inf), f"{what}: empty rows must have LSE = -inf"
    assert np.all(Og[empty] == 0.0), f"{what}: empty rows must have O = 0"
    assert_bf16_close(Og[~empty], Or[~empty], Lg[~empty], Lr[~empty], what=what)


CASES = [
    (4, 2, 300, 128, [300, 1, 129, 0]),
    (3, 2, 383, 64, [200, 383, 64]),
    (2, 3, 640, 128, [513, 128]),
    (5, 1, 257, 64, [1, 2, 255, 256, 257]),
    (1, 2, 1, 128, [1]),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,S,D,kl", CASES)
def test_varlen_prefill_full(B, H, S, D, kl, causal, dtype):
    x = si.prefill_inputs(B, H, S, D, seed=2900 + S + D + B, qk_std=2.0, dtype=dtype)
    O, L = _run(x, kl, causal, dtype)
    _compare(x, kl, causal, O, L, f"{dtype} B{B} H{H} S{S} D{D} lens={kl} causal={causal}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_varlen_many_items_per_cta(causal, D):
    """B*H*ceil(S/256) = 960 items with random key lengths (some 0): item
    shapes vary from item to item across the persistent grid."""
    B, H, S = 8, 40, 600
    x = si.prefill_inputs(B, H, S, D, seed=7150 + D)
    kl = np.random.default_rng(D).integers(0, S + 1, size=B)
    kl[0], kl[1] = 0, S
    O, L = _run(x, kl, causal, "bf16")
    _compare(x, kl, causal, O, L, f"varlen B{B} H{H} S{S} D{D} causal={causal}")


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_full_length_equals_plain(causal):
    x = si.prefill_inputs(2, 4, 700, 128, seed=515)
    O1, L1 = _run(x, [700, 700], causal, "bf16")
    t = torch.bfloat16
    O2, L2 = mha().mha_fwd(dev_tensor(x.Q, t), dev_tensor(x.K, t), dev_tensor(x.V, t),
                           scale=x.scale, causal=causal)
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1, L2)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [True, False])
def test_varlen_padding_keys_do_not_matter(causal, dtype):
    B, H, S, D = 2, 2, 520, 64
    kl = [131, 390]
    x = si.prefill_inputs(B, H, S, D, seed=616, dtype=dtype)
    O1, L1 = _run(x, kl, causal, dtype)
    rng = np.random.default_rng(3)
    K2 = x.K.values.copy()
    V2 = x.V.values.copy()
    for b, Lb in enumerate(kl):
        K2[b, :, Lb:] = 40.0 * rng.standard_normal(K2[b, :, Lb:].shape)
        V2[b, :, Lb:] = 1000.0
    to16 = si.f16_bits if dtype == "f16" else si.bf16_bits
    back = si.f16_to_f32 if dtype == "f16" else si.bf16_to_f32
    Kt = si.Tensor(back(to16(K2)), to16(K2))
    Vt = si.Tensor(back(to16(V2)), to16(V2))
    O2, L2 = _run(x, kl, causal, dtype, K=Kt, V=Vt)
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1, L2)


def test_varlen_lengths_outside_the_range_are_clamped():
    x = si.prefill_inputs(3, 1, 200, 64, seed=88)
    O1, L1 = _run(x, [250, -7, 99], True, "bf16")
    O2, L2 = _run(x, [200, 0, 99], True, "bf16")
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1, L2)


def test_varlen_rejects_missing_lengths():
    x = si.prefill_inputs(1, 1, 64, 64, seed=4)
    t = torch.bfloat16
    with pytest.raises(ValueError):
        mha().mha_fwd_varlen(dev_tensor(x.Q, t), dev_tensor(x.K, t), dev_tensor(x.V, t),
                             torch.zeros(2, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_workload_sampled(causal):
    """The full-size key-padding workload the benchmark can time, on sampled rows."""
    from gpu_util import sample_rows
    x = si.workload_inputs("prefill_varlen_bf16_b4h32s4096d128")
    O, L = _run(x, x.key_lens, causal, "bf16")
    rows = sample_rows(x.B, x.H, x.S, n_bh=12, rows_per_bh=96, seed=9)
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, causal, rows=rows,
                              key_lens=x.key_lens)
    Og = O.view(-1, x.D)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    Lg = L.view(-1)[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_bf16_close(Og, Or, Lg, Lr, what=f"varlen workload causal={causal}")
    assert torch.isfinite(O.float()).all()
