"""The C-ABI library builds, loads without a GPU and exports what mha.h declares.

Also checks the host-side argument validation, which returns before any CUDA
call (no compute call is made here: these tests run on machines without a GPU).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mha.h")

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3
FAKE = 0x10000  # an aligned address that is never dereferenced: validation fails first


@pytest.fixture(scope="module")
def lib():
    from causal_head_attention_mha_gb300 import build
    build.build()
    from causal_head_attention_mha_gb300 import binding
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mha_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("mha_fwd", "mha_fwd_f32", "mha_decode", "mha_get_device_status",
                     "mha_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_needs_no_driver_at_load_time(lib):
    from causal_head_attention_mha_gb300 import binding
    # loading a second handle with the dynamic loader directly must also work
    ctypes.CDLL(binding.library_path())


def fwd(lib, **kw):
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, LSE=None, B=1, H=2, S=128, D=64, scale=0.125,
             causal=1, stream=None)
    a.update(kw)
    return lib.mha_fwd(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["S"], a["D"],
                       a["scale"], a["causal"], a["stream"])


@pytest.mark.parametrize("kw,expected", [
    (dict(Q=None), INVALID), (dict(O=None), INVALID), (dict(B=0), INVALID), (dict(H=-1), INVALID),
    (dict(S=0), INVALID), (dict(D=0), INVALID), (dict(scale=0.0), INVALID),
    (dict(scale=-0.1), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID), (dict(causal=2), INVALID),
    (dict(B=1 << 12, H=1 << 12, S=1 << 12, D=64), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(D=256), UNSUPPORTED),
    (dict(Q=FAKE + 8), MISALIGNED), (dict(V=FAKE + 2), MISALIGNED), (dict(O=FAKE + 4), MISALIGNED),
    (dict(LSE=FAKE + 2), MISALIGNED),
])
def test_prefill_validation(lib, kw, expected):
    assert fwd(lib, **kw) == expected
    f32 = dict(kw)
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, LSE=None, B=1, H=2, S=128, D=64, scale=0.125,
             causal=1, stream=None)
    a.update(f32)
    assert lib.mha_fwd_f32(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["S"],
                           a["D"], a["scale"], a["causal"], a["stream"]) == expected


@pytest.mark.parametrize("kw,expected", [
    (dict(q=None), INVALID), (dict(seqlens=None), INVALID), (dict(B=0), INVALID),
    (dict(H=0), INVALID), (dict(scale=0.0), INVALID), (dict(D=32), UNSUPPORTED),
    (dict(Kc=FAKE + 8), MISALIGNED), (dict(seqlens=FAKE + 2), MISALIGNED),
])
def test_decode_validation(lib, kw, expected):
    a = dict(q=FAKE, Kc=FAKE, Vc=FAKE, seqlens=FAKE, O=FAKE, B=2, H=2, D=128, scale=0.1)
    a.update(kw)
    assert lib.mha_decode(a["q"], a["Kc"], a["Vc"], a["seqlens"], a["O"], a["B"], a["H"], a["D"],
                          a["scale"], None) == expected


def test_status_strings_and_wait_limit(lib):
    for s in range(6):
        assert lib.mha_status_string(s)
    assert b"unknown" in lib.mha_status_string(99)
    assert lib.mha_set_fault_injection(1) == 0
    assert lib.mha_set_fault_injection(7) == -1
    assert lib.mha_set_fault_injection(0) == 1
    old = lib.mha_set_wait_limit_ns(12345)
    assert old == 2_000_000_000
    assert lib.mha_set_wait_limit_ns(0) == 12345
    assert lib.mha_set_wait_limit_ns(0) == 2_000_000_000


@pytest.mark.parametrize("kw,expected", [
    (dict(Q=None), INVALID), (dict(B=0), INVALID), (dict(D=96), UNSUPPORTED),
    (dict(K=FAKE + 8), MISALIGNED), (dict(scale=0.0), INVALID),
])
def test_f16_and_varlen_prefill_validation(lib, kw, expected):
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, LSE=None, B=1, H=2, S=128, D=64, scale=0.125,
             causal=1)
    a.update(kw)
    args = (a["Q"], a["K"], a["V"], a["O"], a["LSE"])
    rest = (a["B"], a["H"], a["S"], a["D"], a["scale"], a["causal"], None)
    assert lib.mha_fwd_f16(*args, *rest) == expected
    assert lib.mha_fwd_varlen(*args, FAKE, *rest) == expected
    assert lib.mha_fwd_varlen_f16(*args, FAKE, *rest) == expected


def test_varlen_needs_aligned_lengths(lib):
    args = (FAKE, FAKE, FAKE, FAKE, None)
    rest = (1, 2, 128, 64, 0.125, 1, None)
    assert lib.mha_fwd_varlen(*args, None, *rest) == INVALID
    assert lib.mha_fwd_varlen(*args, FAKE + 2, *rest) == MISALIGNED


@pytest.mark.parametrize("kw,expected", [
    (dict(q=None), INVALID), (dict(D=32), UNSUPPORTED), (dict(Vc=FAKE + 8), MISALIGNED),
])
def test_f16_decode_validation(lib, kw, expected):
    a = dict(q=FAKE, Kc=FAKE, Vc=FAKE, seqlens=FAKE, O=FAKE, B=2, H=2, D=128, scale=0.1)
    a.update(kw)
    assert lib.mha_decode_f16(a["q"], a["Kc"], a["Vc"], a["seqlens"], a["O"], a["B"], a["H"],
                              a["D"], a["scale"], None) == expected


@pytest.mark.parametrize("kw,expected", [
    (dict(X=None), INVALID), (dict(V=None), INVALID), (dict(B=0), INVALID),
    (dict(hidden=0), INVALID), (dict(H=0), INVALID),
    (dict(B=1 << 12, S=1 << 12, hidden=4096), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(hidden=12), UNSUPPORTED),
    (dict(W=FAKE + 8), MISALIGNED), (dict(Q=FAKE + 4), MISALIGNED),
])
def test_qkv_proj_validation(lib, kw, expected):
    a = dict(X=FAKE, W=FAKE, Q=FAKE, K=FAKE, V=FAKE, B=1, S=128, hidden=256, H=2, D=64)
    a.update(kw)
    assert lib.mha_qkv_proj(a["X"], a["W"], a["Q"], a["K"], a["V"], a["B"], a["S"], a["hidden"],
                            a["H"], a["D"], None) == expected


@pytest.mark.parametrize("kw,expected", [
    (dict(O=None), INVALID), (dict(Y=None), INVALID), (dict(B=0), INVALID), (dict(S=0), INVALID),
    (dict(n_out=0), INVALID), (dict(B=1 << 12, S=1 << 12, H=64), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(n_out=48), UNSUPPORTED),
    (dict(W=FAKE + 8), MISALIGNED), (dict(Y=FAKE + 2), MISALIGNED),
])
def test_out_proj_validation(lib, kw, expected):
    a = dict(O=FAKE, W=FAKE, Y=FAKE, B=1, H=2, S=128, D=64, n_out=256)
    a.update(kw)
    assert lib.mha_out_proj(a["O"], a["W"], a["Y"], a["B"], a["H"], a["S"], a["D"], a["n_out"],
                            None) == expected


@pytest.mark.parametrize("kw,expected", [
    (dict(Q=None), INVALID), (dict(B=0), INVALID), (dict(D=96), UNSUPPORTED),
    (dict(dtype=2), UNSUPPORTED), (dict(o_layout=2), UNSUPPORTED), (dict(o_layout=-1), UNSUPPORTED),
    (dict(key_lens=FAKE + 2), MISALIGNED), (dict(O=FAKE + 8), MISALIGNED),
])
def test_fwd_ex_validation(lib, kw, expected):
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, LSE=None, key_lens=None, B=1, H=2, S=128, D=64,
             scale=0.125, causal=1, dtype=0, o_layout=1)
    a.update(kw)
    assert lib.mha_fwd_ex(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["key_lens"], a["B"], a["H"],
                          a["S"], a["D"], a["scale"], a["causal"], a["dtype"], a["o_layout"],
                          None) == expected


@pytest.mark.parametrize("kw,expected", [
    (dict(O=None), INVALID), (dict(o_layout=2), UNSUPPORTED), (dict(n_out=48), UNSUPPORTED),
    (dict(W=FAKE + 8), MISALIGNED),
])
def test_out_proj_ex_validation(lib, kw, expected):
    a = dict(O=FAKE, W=FAKE, Y=FAKE, B=1, H=2, S=128, D=64, n_out=256, o_layout=1)
    a.update(kw)
    assert lib.mha_out_proj_ex(a["O"], a["W"], a["Y"], a["B"], a["H"], a["S"], a["D"], a["n_out"],
                               a["o_layout"], None) == expected


# The prefill schedule choice (host arithmetic only; sm_count given, so no
# device is queried).  Each expectation is the group shape that measured
# faster on a GB300 for that shape.
@pytest.mark.parametrize("B,H,S,causal,wide", [
    (4, 32, 4096, 1, 0),    # the bench shape: narrow 6 % faster
    (4, 32, 4096, 0, 0),    # the same without the causal mask: narrow 6 % faster
    (2, 16, 16384, 1, 1),   # wide 10 % faster
    (2, 16, 16384, 0, 1),   # wide 32 % faster
    (1, 32, 8192, 0, 1),    # wide 38 % faster
])
def test_prefill_schedule_choice_d128(lib, B, H, S, causal, wide):
    assert lib.mha_prefill_wide_schedule(B, H, S, 128, causal, 0, 152) == wide


def test_prefill_schedule_choice_fixed_cases_and_errors(lib):
    # D = 64 and key padding always take the wide groups
    assert lib.mha_prefill_wide_schedule(4, 32, 4096, 64, 1, 0, 152) == 1
    assert lib.mha_prefill_wide_schedule(4, 32, 4096, 128, 1, 1, 152) == 1
    # a single item per CTA or less: both shapes deal the same items
    assert lib.mha_prefill_wide_schedule(1, 1, 256, 128, 1, 0, 152) in (0, 1)
    for bad in ((0, 32, 4096, 128), (4, 0, 4096, 128), (4, 32, 0, 128), (4, 32, 4096, 96)):
        assert lib.mha_prefill_wide_schedule(*bad, 1, 0, 152) == -INVALID


# ------------------------------------------------------------------ the prefill's item schedule
def _items(B, H, S, D, causal, key_padding, sm=152):
    """Every CTA's items through the binding: {cta: [(bh, qp), ...]}."""
    from causal_head_attention_mha_gb300 import binding
    n_qp = -(-S // 256)
    grid = min(B * H * n_qp, sm)
    return {c: binding.mha_prefill_schedule(B, H, S, D, causal, key_padding, sm, c)
            for c in range(grid)}, grid, n_qp


@pytest.mark.parametrize("B,H,S,D,causal,key_padding,bound", [
    (4, 32, 4096, 128, True, False, 1.03),    # narrow groups, causal (1.028)
    (4, 32, 4096, 128, False, False, 1.04),   # narrow groups: 2048 equal items (1.039)
    (1, 32, 2048, 128, True, False, 1.07),    # 256 items for 152 CTAs (1.062)
    (2, 16, 16384, 64, True, False, 1.01),    # D = 64: wide groups (1.002)
    (2, 16, 16384, 128, True, False, 1.01),   # wide, chosen by the load model (1.002)
    (2, 16, 16384, 128, False, False, 1.04),  # (1.039)
    (1, 32, 8192, 128, False, False, 1.04),   # (1.039)
    (8, 40, 600, 128, True, False, 1.16),     # ragged: the last block has one tile (1.154)
    (4, 32, 4096, 128, True, True, 1.01),     # key padding: wide groups (1.005)
    (3, 5, 77, 64, True, False, 1.0),         # fewer items than SMs: one each
    (64, 32, 4096, 128, True, False, 1.01),   # 32768 items, many groups (1.001)
])
def test_prefill_schedule_deals_every_item_once(lib, B, H, S, D, causal, key_padding, bound):
    per_cta, grid, n_qp = _items(B, H, S, D, causal, key_padding)
    seen = {}
    for c, items in per_cta.items():
        for it in items:
            assert it not in seen, f"item {it} dealt to CTAs {seen[it]} and {c}"
            seen[it] = c
    assert set(seen) == {(bh, qp) for bh in range(B * H) for qp in range(n_qp)}
    # no CTA past the grid, and every CTA of the grid has work
    from causal_head_attention_mha_gb300 import binding
    assert binding.mha_prefill_schedule(B, H, S, D, causal, key_padding, 152, grid) == []
    assert all(per_cta[c] for c in range(grid))
    # the busiest CTA's load (key tiles of its items plus two per item) against
    # the average, as the host's load model computes it when it picks the
    # group shape (the figure in brackets)
    def load(bh, qp):
        n_kt = -(-S // 128)
        nA = min(2 * qp + 1, n_kt) if causal else n_kt
        hasB = (2 * qp + 1) * 128 < S
        nB = (min(2 * qp + 2, n_kt) if causal else n_kt) if hasB else 0
        return nA + nB + 2
    loads = [sum(load(*it) for it in per_cta[c]) for c in range(grid)]
    assert max(loads) * grid <= bound * sum(loads) + 1e-9


def test_prefill_schedule_takes_heavy_blocks_first(lib):
    """Causal: within a group of heads a CTA's blocks come in decreasing order
    (the later query blocks, with more key tiles, first)."""
    per_cta, grid, n_qp = _items(4, 32, 4096, 128, True, False)
    for c in range(grid):
        qps = [qp for _, qp in per_cta[c]]
        # narrow groups: two items per CTA per group, heavy then light
        for i in range(0, len(qps) - 1, 2):
            assert qps[i] >= qps[i + 1]


def test_prefill_schedule_errors(lib):
    from causal_head_attention_mha_gb300 import binding
    ip = ctypes.POINTER(ctypes.c_int)
    for bad in ((0, 32, 4096, 128), (4, 0, 4096, 128), (4, 32, 0, 128), (4, 32, 4096, 96),
                (1024, 1024, 4096, 128)):    # B*H*S*D >= 2^31
        assert lib.mha_prefill_schedule(*bad, 1, 0, 152, 0, None, None, 0) == -INVALID
    assert lib.mha_prefill_schedule(4, 32, 4096, 128, 1, 0, 152, 0, None, None, -1) == -INVALID
    assert lib.mha_prefill_schedule(4, 32, 4096, 128, 1, 0, 152, 0, None, None, 4) == -INVALID
    # a capacity below the count writes only that many and still returns the count
    n = lib.mha_prefill_schedule(4, 32, 4096, 128, 1, 0, 152, 3, None, None, 0)
    assert n > 2
    bh = (ctypes.c_int * 3)(-1, -1, -1)
    qp = (ctypes.c_int * 3)(-1, -1, -1)
    assert lib.mha_prefill_schedule(4, 32, 4096, 128, 1, 0, 152, 3, bh, qp, 2) == n
    full = binding.mha_prefill_schedule(4, 32, 4096, 128, True, False, 152, 3)
    assert [(bh[0], qp[0]), (bh[1], qp[1])] == full[:2] and bh[2] == -1 and qp[2] == -1
    assert lib.mha_prefill_schedule(4, 32, 4096, 128, 1, 0, 152, -1, None, None, 0) == 0


def test_prefill_schedule_binding_raises(lib):
    from causal_head_attention_mha_gb300 import binding
    with pytest.raises(binding.MHAError):
        binding.mha_prefill_schedule(4, 32, 4096, 96, True, False, 152, 0)
    with pytest.raises(binding.MHAError):
        binding.mha_prefill_schedule(0, 32, 4096, 128, True, False, 152, 0)
    # one CTA per item when there are fewer items than SMs
    assert binding.mha_prefill_schedule(1, 1, 256, 128, True, False, 152, 0) == [(0, 0)]
    assert binding.mha_prefill_schedule(1, 1, 256, 128, True, False, 152, 1) == []
