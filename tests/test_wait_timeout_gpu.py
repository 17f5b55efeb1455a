"""Failure detection on the GPU without a fault: a bounded wait runs out.

The library's fault-injection hook makes every CTA of the next prefill
launch withhold one internal signal; the tensor-core issuer's wait for it
runs out after a short limit, the kernel records MHA_ERR_TIMEOUT, drains its
in-flight copies and MMAs, frees tensor memory and returns.  The host reads
the status, and the same context then computes a correct result.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_bf16_close, dev_tensor

pytestmark = pytest.mark.gpu
MHA_ERR_TIMEOUT = 5


def test_withheld_signal_times_out_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import causal_head_attention_mha_gb300 as mha
    torch.cuda.set_device(0)
    x = si.prefill_inputs(1, 2, 512, 128, seed=2024)
    Q, K, V = (dev_tensor(t, torch.bfloat16) for t in (x.Q, x.K, x.V))
    assert mha.mha_get_device_status() == 0
    old_limit = mha.mha_set_wait_limit_ns(20_000_000)   # 20 ms
    old_mode = mha.mha_set_fault_injection(1)
    try:
        mha.mha_fwd(Q, K, V, scale=x.scale, causal=True)
        status = mha.mha_get_device_status()
    finally:
        mha.mha_set_fault_injection(old_mode)
        mha.mha_set_wait_limit_ns(old_limit)
    assert status == MHA_ERR_TIMEOUT, mha.mha_status_string(status)
    # the error word was cleared by the read, and the context still works
    assert mha.mha_get_device_status() == 0
    O, L = mha.mha_fwd(Q, K, V, scale=x.scale, causal=True)
    assert mha.mha_get_device_status() == 0
    Or, Lr = oracle.attention(x.Q.values, x.K.values, x.V.values, x.scale, True)
    assert_bf16_close(O.float().cpu().numpy(), Or, L.cpu().numpy(), Lr)
