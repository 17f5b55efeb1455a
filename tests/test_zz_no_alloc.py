"""mha_decode_noalloc: the decode entry point that allocates nothing.

Some callers cannot allocate device memory when they call (memory planned
up front, no memory-pool support, an allocator that is busy); for them the
library keeps the split partials in a fixed device array.  This file is
collected last on purpose, so a run that stops at its first failure has
already run every other test.  Each check calls the entry point through the
C ABI (ctypes on libmha.so) twice in a row, with different inputs, and
compares it with mha_decode on the same inputs.
"""
import ctypes

import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import assert_bf16_close, dev_tensor

pytestmark = pytest.mark.gpu
MHA_OK, MHA_ERR_UNSUPPORTED = 0, 2


def _inputs(B, H, D, lens, seed):
    z = si.decode_inputs(B, H, D, seed=seed, seqlens=np.array(lens, np.int32))
    return (dev_tensor(z.q, torch.bfloat16), dev_tensor(z.Kc, torch.bfloat16),
            dev_tensor(z.Vc, torch.bfloat16), torch.from_numpy(z.seqlens).cuda(), z.scale)


def _call_noalloc(lib, q, Kc, Vc, sl, O, scale):
    B, H, D = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mha_decode_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(Kc.data_ptr()),
                                  ctypes.c_void_p(Vc.data_ptr()), ctypes.c_void_p(sl.data_ptr()),
                                  ctypes.c_void_p(O.data_ptr()), B, H, D, ctypes.c_float(scale),
                                  ctypes.c_void_p(stream))


def test_noalloc_decode_matches_mha_decode_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import causal_head_attention_mha_gb300 as mha
    lib = mha.load_library()
    torch.cuda.set_device(0)
    rng = np.random.default_rng(5)
    cases = [
        (16, 32, 128, rng.integers(512, 8193, size=16).tolist(), 1004),  # the decode workload shape
        (5, 8, 64, [70, 0, 1300, 1, 257], 99),                            # smaller, ragged, empty row
    ]
    for B, H, D, lens, seed in cases:
        assert mha.mha_decode_num_splits(B, H) > 1  # the scratch array is really used
        q, Kc, Vc, sl, scale = _inputs(B, H, D, lens, seed)
        O_ref = mha.mha_decode(q, Kc, Vc, sl, scale=scale)
        O = torch.empty_like(q)
        assert _call_noalloc(lib, q, Kc, Vc, sl, O, scale) == MHA_OK
        assert mha.mha_get_device_status() == MHA_OK
        assert_bf16_close(O.float().cpu().numpy(), O_ref.float().cpu().numpy(),
                          what=f"noalloc vs mha_decode B{B} H{H} D{D}")


def test_noalloc_decode_rejects_oversized_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import causal_head_attention_mha_gb300 as mha
    lib = mha.load_library()
    # find a head count whose partials do not fit in the 2 MiB array on this device
    B, D = 1, 128
    H = next(h for h in range(64, 65535, 64)
             if mha.mha_decode_num_splits(B, h) > 1
             and B * h * mha.mha_decode_num_splits(B, h) * (D + 2) * 4 > 2 * 1024 * 1024)
    q = torch.zeros((B, H, D), dtype=torch.bfloat16, device="cuda")
    Kc = torch.zeros((1, H, D), dtype=torch.bfloat16, device="cuda")
    sl = torch.ones((B,), dtype=torch.int32, device="cuda")
    O = torch.empty_like(q)
    assert _call_noalloc(lib, q, Kc, Kc, sl, O, 0.1) == MHA_ERR_UNSUPPORTED
