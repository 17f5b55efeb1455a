"""Decode does not depend on how a row's keys are split across thread blocks.

Page 1 ("Week 4 CUDA notes", section 2.2) warns that a row split over
blocks must have its normalisation reconciled across them; the decode
kernel merges the splits' (m, l, o) by log-sum-exp.  Here the same rows are
evaluated with 1, 2, 7 and 64 splits through mha_decode_ex: each result
must match the fp64 oracle within the bf16 tolerances, and the results must
agree with each other.  Split counts above a sequence's length leave most
splits empty (their maximum is -inf), which the merge must ignore.

A second check covers batches larger than the decode kernel's on-device
length sort (more than 1024 sequences), where blocks take sequences in
index order and sum the offsets straight from seqlens.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import TOL_BF16_ABS, assert_bf16_close, dev_tensor, errors

pytestmark = pytest.mark.gpu


def _dev(z, dtype):
    return (dev_tensor(z.q, dtype), dev_tensor(z.Kc, dtype), dev_tensor(z.Vc, dtype),
            torch.from_numpy(z.seqlens).cuda())


@pytest.mark.parametrize("D,dtype", [(128, torch.bfloat16), (64, torch.bfloat16),
                                     (128, torch.float16)])
def test_decode_same_rows_at_several_split_counts(D, dtype):
    import causal_head_attention_mha_gb300 as mha
    lens = [0, 1, 2, 63, 127, 1000, 4999, 8192]
    z = si.decode_inputs(len(lens), 4, D, seed=4242 + D, seqlens=np.array(lens, np.int32),
                         dtype="f16" if dtype == torch.float16 else "bf16")
    q, Kc, Vc, sl = _dev(z, dtype)
    Oo, _ = oracle.decode(z.q.values, z.Kc.values, z.Vc.values, z.seqlens, z.scale)
    outs = {}
    for n in (1, 2, 7, 64):
        O = mha.mha_decode_ex(q, Kc, Vc, sl, scale=z.scale, nsplit=n)
        assert mha.mha_get_device_status() == 0
        outs[n] = O.float().cpu().numpy()
        assert_bf16_close(outs[n], Oo, what=f"decode nsplit={n} D={D}")
        assert np.all(outs[n][0] == 0), "an empty sequence gives O = 0"
    # the automatic choice is one of these paths too
    auto = mha.mha_decode_ex(q, Kc, Vc, sl, scale=z.scale, nsplit=0).float().cpu().numpy()
    ref_auto = (mha.mha_decode_f16 if dtype == torch.float16 else mha.mha_decode)(
        q, Kc, Vc, sl, scale=z.scale).float().cpu().numpy()
    assert np.array_equal(auto, ref_auto), "nsplit=0 is mha_decode's own choice"
    for a in outs:
        for b in outs:
            if a < b:
                max_abs, _ = errors(outs[a], outs[b])
                assert max_abs <= TOL_BF16_ABS, (a, b, max_abs)


def test_decode_rejects_bad_split_counts():
    import causal_head_attention_mha_gb300 as mha
    z = si.decode_inputs(2, 2, 64, seed=5, seqlens=np.array([3, 4], np.int32))
    q, Kc, Vc, sl = _dev(z, torch.bfloat16)
    for n in (-1, 65):
        with pytest.raises(mha.MHAError):
            mha.mha_decode_ex(q, Kc, Vc, sl, scale=z.scale, nsplit=n)


def test_decode_more_sequences_than_the_length_sort():
    import causal_head_attention_mha_gb300 as mha
    B, H, D = 1100, 2, 64
    rng = np.random.default_rng(77)
    lens = rng.integers(0, 41, size=B).astype(np.int32)
    z = si.decode_inputs(B, H, D, seed=78, seqlens=lens)
    q, Kc, Vc, sl = _dev(z, torch.bfloat16)
    Oo, _ = oracle.decode(z.q.values, z.Kc.values, z.Vc.values, z.seqlens, z.scale)
    for n in (0, 3):
        O = mha.mha_decode_ex(q, Kc, Vc, sl, scale=z.scale, nsplit=n)
        assert mha.mha_get_device_status() == 0
        On = O.float().cpu().numpy()
        assert_bf16_close(On, Oo, what=f"B={B} nsplit={n}")
        assert np.all(On[lens == 0] == 0)
