"""fp64 CPU oracle for causal multi-head attention — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and it imports nothing from the product.

The arithmetic lives in ``attention_ref.c`` (plain C, double precision,
pthreads across rows); this module compiles it with gcc and marshals numpy
arrays to it.  What it computes is the definition on the page "Hand-written
masked multi-head attention CUDA kernel: underlying logic and practice",
section 2 (A = softmax(QK^T/sqrt(d_k) + M), O = A V with M = -inf above the
diagonal), with the valid-key rule j <= i of its section 2.2.  The fused
Q, K, V projection (``qkv_projection``) is one fp64 numpy matrix product and
a reshape, the definition of section 2 (Q = X W_Q, ...); the output
projection (``out_projection``) is the same over the concatenated heads.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force at high precision, closed forms, invariants, a library softmax)
and by ``tests/test_oracle_mutants.py`` (planted mistakes must fail a pin).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_ref.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# gcc flags: no fast-math and no FMA contraction, so the double arithmetic is
# the plain IEEE sequence written in the source on x86-64 and aarch64 alike.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared library and return its path."""
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", out + ".tmp", src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def _declare(lib):
    f64p = ctypes.POINTER(ctypes.c_double)
    f32p = ctypes.POINTER(ctypes.c_float)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    intp = ctypes.POINTER(ctypes.c_int)
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = [
        f32p, f32p, f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, ctypes.c_int, i64p, ctypes.c_int64, f64p, f64p, ctypes.c_int, intp]
    lib.oracle_attention_rows_kl.restype = ctypes.c_int
    lib.oracle_attention_rows_kl.argtypes = [
        f32p, f32p, f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, ctypes.c_int, i32p, i64p, ctypes.c_int64, f64p, f64p, ctypes.c_int, intp]
    lib.oracle_decode.restype = ctypes.c_int
    lib.oracle_decode.argtypes = [
        f32p, f32p, f32p, i32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, f64p, f64p, ctypes.c_int, intp]
    return lib


def load_library(path: str | None = None):
    """Load (building first when missing or stale) the oracle library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(_LIB_PATH)
                     or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
            if stale:
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


class OracleResult(tuple):
    """(O, LSE) plus the number of host threads the evaluation used."""
    threads: int


def attention(Q, K, V, scale: float, causal: bool, rows=None, nthreads: int = 0, lib=None,
              key_lens=None):
    """Prefill attention in fp64.

    Q, K, V: float arrays [B, H, S, D] (bf16 inputs are passed as the float32
    values they represent exactly).  ``rows``: optional flat row ids
    (b*H + h)*S + i.  ``key_lens``: optional int [B], each in [0, S]: only keys
    j < key_lens[b] of sequence b exist (a row without a valid key gets O = 0,
    LSE = -inf).  Returns (O, LSE): O [B,H,S,D] and LSE [B,H,S] in float64
    when ``rows`` is None, else O [len(rows), D] and LSE [len(rows)].
    """
    lib = lib or load_library()
    Q, qp = _f32(Q)
    K, kp = _f32(K)
    V, vp = _f32(V)
    B, H, S, D = Q.shape
    assert K.shape == Q.shape and V.shape == Q.shape
    if rows is None:
        n = B * H * S
        rows_arr, rp = None, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.size
        rp = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    O = np.empty((n, D), dtype=np.float64)
    LSE = np.empty((n,), dtype=np.float64)
    used = ctypes.c_int(0)
    if key_lens is not None:
        kl = np.ascontiguousarray(key_lens, dtype=np.int32)
        assert kl.shape == (B,)
        klp = kl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    else:
        klp = None
    rc = lib.oracle_attention_rows_kl(
        qp, kp, vp, B, H, S, D, float(scale), int(bool(causal)), klp, rp, n,
        O.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        LSE.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(nthreads), ctypes.byref(used))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed with status {rc}")
    if rows is None:
        O = O.reshape(B, H, S, D)
        LSE = LSE.reshape(B, H, S)
    res = OracleResult((O, LSE))
    res.threads = used.value
    return res


def decode(q, Kc, Vc, seqlens, scale: float, nthreads: int = 0, lib=None):
    """Single-query decode in fp64.

    q: [B, H, D]; Kc, Vc: packed [sum(seqlens), H, D]; seqlens: int [B].
    Returns (O [B,H,D], LSE [B,H]) in float64.
    """
    lib = lib or load_library()
    q, qp = _f32(q)
    Kc, kp = _f32(Kc)
    Vc, vp = _f32(Vc)
    B, H, D = q.shape
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    assert sl.shape == (B,)
    assert Kc.shape == (int(sl.sum()), H, D) and Vc.shape == Kc.shape
    O = np.empty((B, H, D), dtype=np.float64)
    LSE = np.empty((B, H), dtype=np.float64)
    used = ctypes.c_int(0)
    rc = lib.oracle_decode(
        qp, kp, vp, sl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, H, D, float(scale),
        O.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        LSE.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(nthreads), ctypes.byref(used))
    if rc != 0:
        raise RuntimeError(f"oracle_decode failed with status {rc}")
    res = OracleResult((O, LSE))
    res.threads = used.value
    return res


def qkv_projection(X, W, H: int, D: int):
    """The fused Q, K, V projection in fp64 (test infrastructure, like the rest
    of this module).

    Page "Hand-written masked multi-head attention CUDA kernel" section 2:
    Q = X W_Q, K = X W_K, V = X W_V, with (section 2.1) X of shape (batch,
    seq_len, hidden) and each W of shape (hidden, heads * head_dim); page
    "Week 4 CUDA notes" section 2.1 fuses the three products into one GEMM,
    so W here is [W_Q | W_K | W_V], shape (hidden, 3 * H * D).

    X: float [B, S, hidden]; W: float [hidden, 3*H*D] (16-bit inputs are passed
    as the float32 values they represent exactly).  Returns (Q, K, V), each
    float64 [B, H, S, D]: column n = c*H*D + h*D + d of X W is head h, feature
    d of Q (c = 0), K (c = 1) or V (c = 2).
    """
    X = np.asarray(X, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    B, S, hidden = X.shape
    assert W.shape == (hidden, 3 * H * D)
    Y = np.matmul(X.reshape(B * S, hidden), W)          # one product, fp64
    Y = Y.reshape(B, S, 3, H, D).transpose(2, 0, 3, 1, 4)  # [3, B, H, S, D]
    return Y[0].copy(), Y[1].copy(), Y[2].copy()


def out_projection(O, W):
    """The output projection in fp64 (test infrastructure).

    Page "Week 4 CUDA notes" section 2.1 lists it after attention as one more
    GEMM: the heads of O are concatenated (feature h*D + d of a row is head h,
    feature d) and multiplied by W_O, Y = concat_h(O_h) W_O; the same sum per
    head, Y = sum_h O_h W_O[h*D:(h+1)*D], is the grouped form.

    O: float [B, H, S, D]; W: float [H*D, N].  Returns Y, float64 [B, S, N].
    """
    O = np.asarray(O, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    B, H, S, D = O.shape
    assert W.shape[0] == H * D
    A = O.transpose(0, 2, 1, 3).reshape(B * S, H * D)   # rows (b, s), columns h*D + d
    return np.matmul(A, W).reshape(B, S, W.shape[1])
