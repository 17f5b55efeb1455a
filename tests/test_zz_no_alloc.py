"""mha_decode_noalloc: the decode entry point that allocates nothing.

Some callers cannot allocate device memory when they call: a serving loop
that plans all of its device memory up front and treats a later allocation
as a failure, a device or driver mode without memory-pool support (where
mha_decode's cudaMallocAsync fails), or code that runs while its process's
allocator is busy.  For them the library keeps the split partials in a fixed
device array.  This file is collected last on purpose, so a run that stops at
its first failure has already run every other test.

Every check calls the entry point through the C ABI (ctypes on libmha.so).
mha_decode runs the same kernels with the same split count, so the two must
agree bit for bit; both are also compared with the fp64 oracle.  The array
keeps whatever the previous call left in it, so the same shape is called
twice in a row on new inputs, after a larger call has filled more of it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_bf16_close, dev_tensor

pytestmark = pytest.mark.gpu
MHA_OK = 0
SCRATCH_BYTES = 2 * 1024 * 1024  # MHA_DECODE_NOALLOC_SCRATCH_BYTES


def _inputs(B, H, D, lens, seed):
    z = si.decode_inputs(B, H, D, seed=seed, seqlens=np.array(lens, np.int32))
    dev = (dev_tensor(z.q, torch.bfloat16), dev_tensor(z.Kc, torch.bfloat16),
           dev_tensor(z.Vc, torch.bfloat16), torch.from_numpy(z.seqlens).cuda())
    return z, dev


def _call_noalloc(lib, q, Kc, Vc, sl, O, scale):
    B, H, D = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mha_decode_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(Kc.data_ptr()),
                                  ctypes.c_void_p(Vc.data_ptr()), ctypes.c_void_p(sl.data_ptr()),
                                  ctypes.c_void_p(O.data_ptr()), B, H, D, ctypes.c_float(scale),
                                  ctypes.c_void_p(stream))


def _check_call(mha, lib, B, H, D, lens, seed, ref_nsplit=0):
    """One mha_decode_noalloc call against mha_decode_ex (split count ref_nsplit, 0 =
    automatic, i.e. mha_decode) bit for bit, and against the oracle."""
    z, (q, Kc, Vc, sl) = _inputs(B, H, D, lens, seed)
    O_ref = mha.mha_decode_ex(q, Kc, Vc, sl, scale=z.scale, nsplit=ref_nsplit)
    O = torch.full_like(q, float("nan"))
    assert _call_noalloc(lib, q, Kc, Vc, sl, O, z.scale) == MHA_OK
    assert mha.mha_get_device_status() == MHA_OK
    same = torch.equal(O.view(torch.int16), O_ref.view(torch.int16))
    assert same, f"noalloc differs from mha_decode, B{B} H{H} D{D} seed {seed}"
    Oo, _ = oracle.decode(z.q.values, z.Kc.values, z.Vc.values, z.seqlens, z.scale)
    assert_bf16_close(O.float().cpu().numpy(), Oo, what=f"noalloc vs oracle B{B} H{H} D{D}")


def test_noalloc_decode_bitwise_equal_to_mha_decode_on_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import causal_head_attention_mha_gb300 as mha
    lib = mha.load_library()
    torch.cuda.set_device(0)
    rng = np.random.default_rng(5)
    big = (16, 32, 128, rng.integers(512, 8193, size=16).tolist())  # the decode workload's shape
    small = (5, 8, 64, [70, 0, 1300, 1, 257])                       # ragged, an empty sequence
    for B, H, D, _ in (big, small):
        assert mha.mha_decode_num_splits(B, H) > 1  # the scratch array is really used
    # the larger call first (it fills more of the array), then the small shape
    # twice in a row on new inputs, then the large shape again
    _check_call(mha, lib, *big, seed=1004)
    _check_call(mha, lib, *small, seed=99)
    _check_call(mha, lib, *small, seed=100)
    _check_call(mha, lib, *big, seed=1005)


def test_noalloc_decode_lowers_splits_to_fit_the_array():
    """A shape whose automatic split count needs more than the array: the call uses
    the largest split count that fits instead of failing."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import causal_head_attention_mha_gb300 as mha
    lib = mha.load_library()
    B, D = 1, 128
    H = next(h for h in range(64, 65535, 64)
             if mha.mha_decode_num_splits(B, h) > 1
             and B * h * mha.mha_decode_num_splits(B, h) * (D + 2) * 4 > SCRATCH_BYTES)
    fit = max(1, SCRATCH_BYTES // (4 * B * H * (D + 2)))
    assert fit < mha.mha_decode_num_splits(B, H)
    _check_call(mha, lib, B, H, D, [37], seed=7, ref_nsplit=fit)
