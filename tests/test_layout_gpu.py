"""O written as [B, S, H, D] (mha_fwd_ex) and the output projection reading it
as rows (mha_out_proj_ex), GPU only.

Both are properties that need no tolerance:
- Attention's O in [B, S, H, D] is the [B, H, S, D] result permuted, bit for
  bit (the same arithmetic, another store address), with the same LSE.
- The output projection of the permuted O equals the one through the 4-D
  view bit for bit: every output sums the same products in the same order,
  only the row tiling differs.
The [B, H, S, D] paths themselves are checked against the fp64 oracle in
test_parity_gpu.py and test_out_proj_gpu.py.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import dev_tensor

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


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,S,D,kl", [
    (2, 3, 300, 128, None), (3, 2, 257, 64, None), (1, 4, 1, 64, None),
    (3, 2, 520, 64, [131, 0, 520]), (2, 5, 640, 128, [640, 1]),
])
def test_fwd_o_bshd_is_the_permutation(B, H, S, D, kl, causal, dtype):
    x = si.prefill_inputs(B, H, S, D, seed=8100 + S + D, qk_std=2.0, dtype=dtype)
    t = TYPES[dtype]
    Q, K, V = dev_tensor(x.Q, t), dev_tensor(x.K, t), dev_tensor(x.V, t)
    KL = None if kl is None else torch.as_tensor(np.asarray(kl, np.int32)).cuda()
    O1, L1 = mha().mha_fwd_ex(Q, K, V, KL, scale=x.scale, causal=causal, o_layout="bhsd")
    O2, L2 = mha().mha_fwd_ex(Q, K, V, KL, scale=x.scale, causal=causal, o_layout="bshd")
    assert O2.shape == (B, S, H, D)
    assert same_bits(O2, O1.permute(0, 2, 1, 3))
    assert torch.equal(L1, L2)
    # the plain entry points give the same [B, H, S, D] result
    if kl is None:
        O3, L3 = (mha().mha_fwd_f16 if dtype == "f16" else mha().mha_fwd)(
            Q, K, V, scale=x.scale, causal=causal)
    else:
        O3, L3 = (mha().mha_fwd_varlen_f16 if dtype == "f16" else mha().mha_fwd_varlen)(
            Q, K, V, KL, scale=x.scale, causal=causal)
    assert same_bits(O1, O3) and torch.equal(L1, L3)


@pytest.mark.parametrize("B,H,S,D,N", [
    (1, 1, 100, 64, 32), (2, 3, 130, 128, 288), (1, 2, 1, 64, 64), (3, 5, 257, 64, 544),
    (2, 8, 1024, 128, 512),
])
def test_out_proj_rows_equal_the_4d_view(B, H, S, D, N):
    x = si.out_projection_inputs(B, H, S, D, N, seed=8200 + S + N)
    O = dev_tensor(x.O, torch.bfloat16)
    W = dev_tensor(x.W, torch.bfloat16)
    Y1 = mha().mha_out_proj(O, W)
    Y2 = mha().mha_out_proj(O.permute(0, 2, 1, 3).contiguous(), W, o_layout="bshd")
    assert Y2.shape == (B, S, N)
    assert same_bits(Y1, Y2)


def test_layer_pipeline_without_transposes():
    """X -> Q, K, V -> attention with O as [B, S, H, D] -> output projection
    reading it as rows: the same Y as through the [B, H, S, D] layout."""
    B, S, hid, H, D, N = 2, 300, 256, 4, 64, 256
    p = si.projection_inputs(B, S, hid, H, D, seed=91)
    w = si.out_projection_inputs(B, H, S, D, N, seed=92)
    t = torch.bfloat16
    Q, K, V = mha().mha_qkv_proj(dev_tensor(p.X, t), dev_tensor(p.W, t), H, D)
    Wo = dev_tensor(w.W, t)
    O1, _ = mha().mha_fwd_ex(Q, K, V, scale=D ** -0.5, causal=True, o_layout="bhsd")
    O2, _ = mha().mha_fwd_ex(Q, K, V, scale=D ** -0.5, causal=True, o_layout="bshd")
    Y1 = mha().mha_out_proj(O1, Wo)
    Y2 = mha().mha_out_proj(O2, Wo, o_layout="bshd")
    assert same_bits(Y1, Y2)
    assert torch.isfinite(Y2.float()).all()
