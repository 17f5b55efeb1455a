"""The shared input generator: determinism and bf16 / f16 rounding."""
import numpy as np
import torch

import seeded_inputs as si


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 37,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, -1e-40], np.float32)])
    ours = si.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = si.bf16_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_f16_rounding_pins():
    # hand-checked IEEE half patterns: exact values, ties to even, largest
    # finite, smallest subnormal, and overflow to infinity
    x = np.array([1.0, -2.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 65504.0, 2.0 ** -24,
                  2.0 ** -25, 65520.0], np.float32)
    want = np.array([0x3C00, 0xC000, 0x3C00, 0x3C02, 0x7BFF, 0x0001, 0x0000, 0x7C00], np.uint16)
    assert np.array_equal(si.f16_bits(x), want)
    back = np.array([1.0, -2.0, 1.0, 1.0 + 2.0 ** -9, 65504.0, 2.0 ** -24, 0.0, np.inf], np.float32)
    assert np.array_equal(si.f16_to_f32(want), back)


def test_f16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(100000).astype(np.float32) * 37
    ours = si.f16_bits(x)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    t = si.make_tensor(7, si.STREAM_V, (3, 5), 2.0, "f16")
    assert t.bits.dtype == np.uint16 and np.array_equal(t.values, si.f16_to_f32(t.bits))


def test_streams_are_deterministic_and_distinct():
    a = si.prefill_inputs(1, 2, 8, 4, seed=5)
    b = si.prefill_inputs(1, 2, 8, 4, seed=5)
    assert np.array_equal(a.Q.bits, b.Q.bits) and np.array_equal(a.V.values, b.V.values)
    assert not np.array_equal(a.Q.values, a.K.values)
    d = si.decode_inputs(4, 2, 8, seed=3, len_lo=5, len_hi=9)
    assert d.seqlens.dtype == np.int32 and d.seqlens.min() >= 5 and d.seqlens.max() <= 9
    assert d.Kc.shape == (int(d.seqlens.sum()), 2, 8)


def test_large_logit_workload_std():
    w = si.WORKLOADS["prefill_bf16_b4h32s4096d128_qk3"]
    x = si.make_tensor(w["seed"], si.STREAM_Q, (1 << 16,), w["qk_std"], "bf16").values
    assert abs(float(x.std()) - 3.0) < 0.05
