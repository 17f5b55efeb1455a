"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module draws random numbers and stores them; it holds none of the
attention arithmetic.  Both sides get the same values: the CUDA path takes
the raw 16-bit patterns (bf16 or f16; float32 values for the fp32 path), the
oracle takes the float32 values that those bit patterns represent exactly.

Recipe (no public dataset or benchmark suite is involved anywhere; every
tensor is i.i.d. Gaussian from a fixed seed):
  * one numpy PCG64 stream per tensor, seeded with the pair (seed, stream id),
    stream ids 0 = Q/q, 1 = K, 2 = V, 3 = sequence lengths;
  * float32 standard normals times the requested standard deviation;
  * for bf16 or f16 tensors, round-to-nearest-even to that type (ties to even
    mantissa);
  * decode sequence lengths uniform on the integers [len_lo, len_hi].
"""
from __future__ import annotations

from dataclasses import dataclass
import math

import numpy as np

STREAM_Q, STREAM_K, STREAM_V, STREAM_LEN = 0, 1, 2, 3


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def normal_f32(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    x = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """The float32 value each bf16 bit pattern represents (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to IEEE half (nearest, ties to even); returns uint16 bit patterns."""
    with np.errstate(over="ignore"):  # beyond 65504 rounds to infinity, as IEEE says
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_to_f32(bits: np.ndarray) -> np.ndarray:
    """The float32 value each f16 bit pattern represents (exact)."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


@dataclass
class Tensor:
    """One input tensor: float32 values and, for 16-bit tensors, their bit patterns."""
    values: np.ndarray          # float32, exactly the value the kernel sees
    bits: np.ndarray | None     # uint16 bf16 or f16 patterns, or None for an fp32 tensor

    @property
    def shape(self):
        return self.values.shape


def make_tensor(seed: int, stream: int, shape, std: float, dtype: str) -> Tensor:
    x = normal_f32(seed, stream, shape, std)
    if dtype == "f32":
        return Tensor(x, None)
    if dtype == "bf16":
        bits = bf16_bits(x)
        return Tensor(bf16_to_f32(bits), bits)
    if dtype == "f16":
        bits = f16_bits(x)
        return Tensor(f16_to_f32(bits), bits)
    raise ValueError(dtype)


@dataclass
class PrefillInputs:
    Q: Tensor
    K: Tensor
    V: Tensor
    B: int
    H: int
    S: int
    D: int
    scale: float
    dtype: str
    key_lens: np.ndarray | None = None  # int32 [B] valid keys per sequence (key padding)


def prefill_key_lens(B: int, seed: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence key lengths, uniform on the integers [lo, hi]."""
    return np.ascontiguousarray(_rng(seed, STREAM_LEN).integers(lo, hi + 1, size=B), np.int32)


def prefill_inputs(B: int, H: int, S: int, D: int, seed: int, qk_std: float = 1.0,
                   v_std: float = 1.0, dtype: str = "bf16", scale: float | None = None) -> PrefillInputs:
    """Q, K, V of shape [B, H, S, D]; scale defaults to 1/sqrt(D)."""
    shape = (B, H, S, D)
    return PrefillInputs(
        make_tensor(seed, STREAM_Q, shape, qk_std, dtype),
        make_tensor(seed, STREAM_K, shape, qk_std, dtype),
        make_tensor(seed, STREAM_V, shape, v_std, dtype),
        B, H, S, D, (1.0 / math.sqrt(D)) if scale is None else float(scale), dtype)


@dataclass
class DecodeInputs:
    q: Tensor
    Kc: Tensor
    Vc: Tensor
    seqlens: np.ndarray   # int32 [B]
    B: int
    H: int
    D: int
    scale: float


def decode_inputs(B: int, H: int, D: int, seed: int, len_lo: int = 512, len_hi: int = 8192,
                  seqlens=None, std: float = 1.0, scale: float | None = None,
                  dtype: str = "bf16") -> DecodeInputs:
    """One query per (sequence, head) and a packed ragged cache (bf16 or f16).

    The cache holds the sequences back to back: token t of sequence b, head h
    is row (sum_{b'<b} L_b' + t) * H + h of a [sum L, H, D] array.
    """
    if seqlens is None:
        seqlens = _rng(seed, STREAM_LEN).integers(len_lo, len_hi + 1, size=B)
    seqlens = np.ascontiguousarray(seqlens, dtype=np.int32)
    total = int(seqlens.sum())
    return DecodeInputs(
        make_tensor(seed, STREAM_Q, (B, H, D), std, dtype),
        make_tensor(seed, STREAM_K, (total, H, D), std, dtype),
        make_tensor(seed, STREAM_V, (total, H, D), std, dtype),
        seqlens, B, H, D, (1.0 / math.sqrt(D)) if scale is None else float(scale))


@dataclass
class ProjectionInputs:
    X: Tensor   # [B, S, hidden]
    W: Tensor   # [hidden, 3*H*D] = [W_Q | W_K | W_V]
    B: int
    S: int
    hidden: int
    H: int
    D: int


def projection_inputs(B: int, S: int, hidden: int, H: int, D: int, seed: int) -> ProjectionInputs:
    """X ~ N(0, 1) and W ~ N(0, 1/hidden) (outputs of order one), bf16."""
    return ProjectionInputs(
        make_tensor(seed, STREAM_Q, (B, S, hidden), 1.0, "bf16"),
        make_tensor(seed, STREAM_K, (hidden, 3 * H * D), 1.0 / math.sqrt(hidden), "bf16"),
        B, S, hidden, H, D)


@dataclass
class OutProjectionInputs:
    O: Tensor   # [B, H, S, D], attention output layout
    W: Tensor   # [H*D, n_out] = W_O
    B: int
    H: int
    S: int
    D: int
    n_out: int


def out_projection_inputs(B: int, H: int, S: int, D: int, n_out: int,
                          seed: int) -> OutProjectionInputs:
    """O ~ N(0, 1) and W ~ N(0, 1/(H*D)) (outputs of order one), bf16."""
    return OutProjectionInputs(
        make_tensor(seed, STREAM_Q, (B, H, S, D), 1.0, "bf16"),
        make_tensor(seed, STREAM_V, (H * D, n_out), 1.0 / math.sqrt(H * D), "bf16"),
        B, H, S, D, n_out)


# The five synthetic workloads (shapes, distributions and seeds), then the
# same bench shapes on f16 data.
WORKLOADS = {
    "prefill_f32_b1h2s128d64": dict(kind="prefill", B=1, H=2, S=128, D=64, dtype="f32",
                                    qk_std=1.0, seed=1001, causal=(True,)),
    "prefill_bf16_b1h32s2048d128": dict(kind="prefill", B=1, H=32, S=2048, D=128, dtype="bf16",
                                        qk_std=1.0, seed=1002, causal=(True,)),
    "prefill_bf16_b4h32s4096d128_qk3": dict(kind="prefill", B=4, H=32, S=4096, D=128, dtype="bf16",
                                            qk_std=3.0, seed=1003, causal=(True, False)),
    "decode_bf16_b16h32d128_len512_8192": dict(kind="decode", B=16, H=32, D=128, seed=1004,
                                                len_lo=512, len_hi=8192),
    "prefill_bf16_b2h16s16384d64": dict(kind="prefill", B=2, H=16, S=16384, D=64, dtype="bf16",
                                        qk_std=1.0, seed=1005, causal=(True,)),
    "prefill_f16_b4h32s4096d128_qk3": dict(kind="prefill", B=4, H=32, S=4096, D=128, dtype="f16",
                                           qk_std=3.0, seed=1006, causal=(True, False)),
    "decode_f16_b16h32d128_len512_8192": dict(kind="decode", B=16, H=32, D=128, seed=1007,
                                               len_lo=512, len_hi=8192, dtype="f16"),
    # the fused Q/K/V projection feeding the bench's attention shape (LLaMA-7B
    # layer: hidden 4096 = 32 heads x 128)
    "qkv_bf16_b4s4096hid4096_h32d128": dict(kind="projection", B=4, S=4096, hidden=4096, H=32,
                                            D=128, seed=1009),
    # the output projection after the bench's attention shape (concatenated
    # 32 x 128 heads times W_O [4096, 4096])
    "outproj_bf16_b4h32s4096d128_n4096": dict(kind="out_projection", B=4, H=32, S=4096, D=128,
                                              n_out=4096, seed=1010),
    # key padding: the bench shape with per-sequence key lengths U{1024..4096}
    "prefill_varlen_bf16_b4h32s4096d128": dict(kind="prefill", B=4, H=32, S=4096, D=128,
                                               dtype="bf16", qk_std=1.0, seed=1008,
                                               causal=(True, False), key_len_lo=1024,
                                               key_len_hi=4096),
}


def workload_inputs(name: str):
    w = WORKLOADS[name]
    if w["kind"] == "out_projection":
        return out_projection_inputs(w["B"], w["H"], w["S"], w["D"], w["n_out"], w["seed"])
    if w["kind"] == "projection":
        return projection_inputs(w["B"], w["S"], w["hidden"], w["H"], w["D"], w["seed"])
    if w["kind"] == "prefill":
        x = prefill_inputs(w["B"], w["H"], w["S"], w["D"], w["seed"], qk_std=w["qk_std"],
                           dtype=w["dtype"])
        if "key_len_lo" in w:
            x.key_lens = prefill_key_lens(w["B"], w["seed"], w["key_len_lo"], w["key_len_hi"])
        return x
    return decode_inputs(w["B"], w["H"], w["D"], w["seed"], w["len_lo"], w["len_hi"],
                         dtype=w.get("dtype", "bf16"))
