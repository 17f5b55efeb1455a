"""ctypes binding of libmha.so: argument marshalling only.

Every function here checks the torch tensors it is given (device, dtype,
shape, contiguity), passes their device pointers and the current CUDA stream
to the C entry point of the same name, and raises :class:`MHAError` on a
non-zero status.  All arithmetic happens in the library's CUDA kernels;
there is no fallback of any kind: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libmha.so")
_lib = None
_lock = threading.Lock()

MHA_OK = 0
STATUS_NAMES = {0: "MHA_OK", 1: "MHA_ERR_INVALID_ARG", 2: "MHA_ERR_UNSUPPORTED",
                3: "MHA_ERR_MISALIGNED", 4: "MHA_ERR_CUDA", 5: "MHA_ERR_TIMEOUT"}


class MHAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        text = _load().mha_status_string(status).decode()
        extra = ""
        if status == 4:
            extra = f" (cudaError {_load().mha_last_cuda_error()})"
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {text}{extra}")


def library_path() -> str:
    return _LIB_PATH


def _declare(lib):
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.mha_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.mha_fwd.restype = i
    lib.mha_fwd_f16.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.mha_fwd_f16.restype = i
    lib.mha_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.mha_fwd_varlen.restype = i
    lib.mha_fwd_varlen_f16.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.mha_fwd_varlen_f16.restype = i
    lib.mha_fwd_f32.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.mha_fwd_f32.restype = i
    lib.mha_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, f, vp]
    lib.mha_decode.restype = i
    lib.mha_decode_f16.argtypes = [vp, vp, vp, vp, vp, i, i, i, f, vp]
    lib.mha_decode_f16.restype = i
    lib.mha_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, f, vp]
    lib.mha_decode_noalloc.restype = i
    lib.mha_decode_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, f, i, i, vp]
    lib.mha_decode_ex.restype = i
    lib.mha_qkv_proj.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.mha_qkv_proj.restype = i
    lib.mha_out_proj.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    lib.mha_out_proj.restype = i
    lib.mha_out_proj_ex.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp]
    lib.mha_out_proj_ex.restype = i
    lib.mha_fwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp]
    lib.mha_fwd_ex.restype = i
    lib.mha_decode_num_splits.argtypes = [i, i]
    lib.mha_decode_num_splits.restype = i
    lib.mha_prefill_wide_schedule.argtypes = [i, i, i, i, i, i, i]
    lib.mha_prefill_wide_schedule.restype = i
    ip = ctypes.POINTER(ctypes.c_int)
    lib.mha_prefill_schedule.argtypes = [i, i, i, i, i, i, i, i, ip, ip, i]
    lib.mha_prefill_schedule.restype = i
    lib.mha_get_device_status.argtypes = [vp]
    lib.mha_get_device_status.restype = i
    lib.mha_status_string.argtypes = [i]
    lib.mha_status_string.restype = ctypes.c_char_p
    lib.mha_last_cuda_error.argtypes = []
    lib.mha_last_cuda_error.restype = i
    lib.mha_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.mha_set_wait_limit_ns.restype = ctypes.c_uint64
    lib.mha_set_fault_injection.argtypes = [i]
    lib.mha_set_fault_injection.restype = i
    return lib


def load_library(path: str | None = None):
    """Load libmha.so; raises if it has not been built."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


_load = load_library


def _stream_ptr(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device or t.device.type != "cuda":
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _prefill(entry, dtype, Q, K, V, O, LSE, scale, causal, stream, want_lse, key_lens=None):
    if Q.dim() != 4:
        raise ValueError("Q must be [B, H, S, D]")
    B, H, S, D = Q.shape
    dev = Q.device
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        _check(t, name, dtype, (B, H, S, D), dev)
    if O is None:
        O = torch.empty_like(Q)
    _check(O, "O", dtype, (B, H, S, D), dev)
    if LSE is None and want_lse:
        LSE = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    if LSE is not None:
        _check(LSE, "LSE", torch.float32, (B, H, S), dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ptrs = [Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
            LSE.data_ptr() if LSE is not None else None]
    if key_lens is not None:
        _check(key_lens, "key_lens", torch.int32, (B,), dev)
        ptrs.append(key_lens.data_ptr())
    st = getattr(_load(), entry)(*ptrs, B, H, S, D, float(scale), int(bool(causal)),
                                 _stream_ptr(stream, dev))
    if st != MHA_OK:
        raise MHAError(st, entry)
    return O, LSE


def mha_fwd(Q, K, V, O=None, LSE=None, scale=None, causal=True, stream=None, want_lse=True):
    """bf16 [B,H,S,D] prefill; returns (O, LSE).  See include/mha.h: mha_fwd."""
    return _prefill("mha_fwd", torch.bfloat16, Q, K, V, O, LSE, scale, causal, stream, want_lse)


def mha_fwd_f16(Q, K, V, O=None, LSE=None, scale=None, causal=True, stream=None, want_lse=True):
    """f16 [B,H,S,D] prefill; returns (O, LSE).  See include/mha.h: mha_fwd_f16."""
    return _prefill("mha_fwd_f16", torch.float16, Q, K, V, O, LSE, scale, causal, stream,
                    want_lse)


def mha_fwd_varlen(Q, K, V, key_lens, O=None, LSE=None, scale=None, causal=True, stream=None,
                   want_lse=True):
    """bf16 prefill with key padding: key_lens int32 [B] on the device (keys
    j >= key_lens[b] are excluded).  See include/mha.h: mha_fwd_varlen."""
    return _prefill("mha_fwd_varlen", torch.bfloat16, Q, K, V, O, LSE, scale, causal, stream,
                    want_lse, key_lens=key_lens)


def mha_fwd_varlen_f16(Q, K, V, key_lens, O=None, LSE=None, scale=None, causal=True, stream=None,
                       want_lse=True):
    """f16 prefill with key padding.  See include/mha.h: mha_fwd_varlen_f16."""
    return _prefill("mha_fwd_varlen_f16", torch.float16, Q, K, V, O, LSE, scale, causal, stream,
                    want_lse, key_lens=key_lens)


def mha_fwd_ex(Q, K, V, key_lens=None, O=None, LSE=None, scale=None, causal=True,
               o_layout="bhsd", stream=None, want_lse=True):
    """bf16 or f16 prefill (from Q's dtype), optional key padding, and O either
    [B, H, S, D] (o_layout "bhsd") or [B, S, H, D] ("bshd", the concatenated
    heads an output projection reads as rows).  Returns (O, LSE).  See
    include/mha.h: mha_fwd_ex."""
    if Q.dim() != 4:
        raise ValueError("Q must be [B, H, S, D]")
    if Q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("Q must be bf16 or f16")
    if o_layout not in ("bhsd", "bshd"):
        raise ValueError("o_layout must be 'bhsd' or 'bshd'")
    B, H, S, D = Q.shape
    dev = Q.device
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        _check(t, name, Q.dtype, (B, H, S, D), dev)
    oshape = (B, H, S, D) if o_layout == "bhsd" else (B, S, H, D)
    if O is None:
        O = torch.empty(oshape, dtype=Q.dtype, device=dev)
    _check(O, "O", Q.dtype, oshape, dev)
    if LSE is None and want_lse:
        LSE = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    if LSE is not None:
        _check(LSE, "LSE", torch.float32, (B, H, S), dev)
    if key_lens is not None:
        _check(key_lens, "key_lens", torch.int32, (B,), dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = _load().mha_fwd_ex(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                            LSE.data_ptr() if LSE is not None else None,
                            key_lens.data_ptr() if key_lens is not None else None,
                            B, H, S, D, float(scale), int(bool(causal)),
                            1 if Q.dtype == torch.float16 else 0,
                            0 if o_layout == "bhsd" else 1, _stream_ptr(stream, dev))
    if st != MHA_OK:
        raise MHAError(st, "mha_fwd_ex")
    return O, LSE


def mha_fwd_f32(Q, K, V, O=None, LSE=None, scale=None, causal=True, stream=None, want_lse=True):
    """float32 [B,H,S,D] prefill; returns (O, LSE).  See include/mha.h: mha_fwd_f32."""
    return _prefill("mha_fwd_f32", torch.float32, Q, K, V, O, LSE, scale, causal, stream,
                    want_lse)


def _decode(entry, dtype, q, Kcache, Vcache, seqlens, O, scale, stream, extra=()):
    if q.dim() != 3:
        raise ValueError("q must be [B, H, D]")
    B, H, D = q.shape
    dev = q.device
    _check(q, "q", dtype, (B, H, D), dev)
    if Kcache.dim() != 3 or Kcache.shape[1:] != (H, D):
        raise ValueError("Kcache must be [total_tokens, H, D]")
    _check(Kcache, "Kcache", dtype, tuple(Kcache.shape), dev)
    _check(Vcache, "Vcache", dtype, tuple(Kcache.shape), dev)
    _check(seqlens, "seqlens", torch.int32, (B,), dev)
    if O is None:
        O = torch.empty_like(q)
    _check(O, "O", dtype, (B, H, D), dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = getattr(_load(), entry)(q.data_ptr(), Kcache.data_ptr(), Vcache.data_ptr(),
                                 seqlens.data_ptr(), O.data_ptr(), B, H, D, float(scale),
                                 *extra, _stream_ptr(stream, dev))
    if st != MHA_OK:
        raise MHAError(st, entry)
    return O


def mha_decode(q, Kcache, Vcache, seqlens, O=None, scale=None, stream=None):
    """bf16 single-query decode over a packed cache; returns O [B,H,D].

    q: [B,H,D]; Kcache, Vcache: [sum(seqlens), H, D]; seqlens: int32 [B] on the device.
    """
    return _decode("mha_decode", torch.bfloat16, q, Kcache, Vcache, seqlens, O, scale, stream)


def mha_decode_f16(q, Kcache, Vcache, seqlens, O=None, scale=None, stream=None):
    """mha_decode on f16 q, cache and O.  See include/mha.h: mha_decode_f16."""
    return _decode("mha_decode_f16", torch.float16, q, Kcache, Vcache, seqlens, O, scale, stream)


def mha_decode_ex(q, Kcache, Vcache, seqlens, O=None, scale=None, nsplit=0, stream=None):
    """mha_decode / mha_decode_f16 (by q's dtype) with the number of key splits
    chosen by the caller: 0 = automatic, 1..64 = that many.  See include/mha.h:
    mha_decode_ex."""
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("q must be bf16 or f16")
    dtype_code = 1 if q.dtype == torch.float16 else 0
    return _decode("mha_decode_ex", q.dtype, q, Kcache, Vcache, seqlens, O, scale, stream,
                   extra=(int(nsplit), dtype_code))


def mha_decode_noalloc(q, Kcache, Vcache, seqlens, O, scale=None, stream=None):
    """mha_decode with its scratch in the library's fixed device array.

    Allocates nothing: the caller passes O as well.  See include/mha.h:
    mha_decode_noalloc (size limit, first call before stream capture,
    overlapping calls race).
    """
    if q.dim() != 3:
        raise ValueError("q must be [B, H, D]")
    B, H, D = q.shape
    dev = q.device
    _check(q, "q", torch.bfloat16, (B, H, D), dev)
    if Kcache.dim() != 3 or Kcache.shape[1:] != (H, D):
        raise ValueError("Kcache must be [total_tokens, H, D]")
    _check(Kcache, "Kcache", torch.bfloat16, tuple(Kcache.shape), dev)
    _check(Vcache, "Vcache", torch.bfloat16, tuple(Kcache.shape), dev)
    _check(seqlens, "seqlens", torch.int32, (B,), dev)
    _check(O, "O", torch.bfloat16, (B, H, D), dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = _load().mha_decode_noalloc(q.data_ptr(), Kcache.data_ptr(), Vcache.data_ptr(),
                                    seqlens.data_ptr(), O.data_ptr(), B, H, D, float(scale),
                                    _stream_ptr(stream, dev))
    if st != MHA_OK:
        raise MHAError(st, "mha_decode_noalloc")
    return O


def mha_qkv_proj(X, W, H: int, D: int, Q=None, K=None, V=None, stream=None):
    """Fused projection [Q | K | V] = X [W_Q | W_K | W_V], bf16; returns (Q, K, V),
    each [B, H, S, D].  X: [B, S, hidden]; W: [hidden, 3*H*D].  See include/mha.h:
    mha_qkv_proj."""
    if X.dim() != 3:
        raise ValueError("X must be [B, S, hidden]")
    B, S, hidden = X.shape
    dev = X.device
    _check(X, "X", torch.bfloat16, (B, S, hidden), dev)
    _check(W, "W", torch.bfloat16, (hidden, 3 * H * D), dev)
    out = []
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t is None:
            t = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev)
        _check(t, name, torch.bfloat16, (B, H, S, D), dev)
        out.append(t)
    st = _load().mha_qkv_proj(X.data_ptr(), W.data_ptr(), out[0].data_ptr(), out[1].data_ptr(),
                              out[2].data_ptr(), B, S, hidden, int(H), int(D),
                              _stream_ptr(stream, dev))
    if st != MHA_OK:
        raise MHAError(st, "mha_qkv_proj")
    return tuple(out)


def mha_out_proj(O, W, Y=None, stream=None, o_layout="bhsd"):
    """Output projection Y = concat_h(O_h) W_O, bf16; O [B, H, S, D] (o_layout
    "bhsd") or [B, S, H, D] ("bshd"), W [H*D, n_out]; returns Y [B, S, n_out].
    See include/mha.h: mha_out_proj, mha_out_proj_ex."""
    if O.dim() != 4:
        raise ValueError("O must be 4-D")
    if o_layout == "bhsd":
        B, H, S, D = O.shape
    elif o_layout == "bshd":
        B, S, H, D = O.shape
    else:
        raise ValueError("o_layout must be 'bhsd' or 'bshd'")
    dev = O.device
    _check(O, "O", torch.bfloat16, tuple(O.shape), dev)
    if W.dim() != 2 or W.shape[0] != H * D:
        raise ValueError("W must be [H*D, n_out]")
    n_out = W.shape[1]
    _check(W, "W", torch.bfloat16, (H * D, n_out), dev)
    if Y is None:
        Y = torch.empty((B, S, n_out), dtype=torch.bfloat16, device=dev)
    _check(Y, "Y", torch.bfloat16, (B, S, n_out), dev)
    st = _load().mha_out_proj_ex(O.data_ptr(), W.data_ptr(), Y.data_ptr(), B, H, S, D, n_out,
                                 0 if o_layout == "bhsd" else 1, _stream_ptr(stream, dev))
    if st != MHA_OK:
        raise MHAError(st, "mha_out_proj")
    return Y


def mha_decode_num_splits(B: int, H: int) -> int:
    """Key splits (partials merged by a second kernel) mha_decode uses on this device."""
    n = _load().mha_decode_num_splits(int(B), int(H))
    if n <= 0:
        raise MHAError(4, "mha_decode_num_splits")
    return n


def mha_prefill_wide_schedule(B: int, H: int, S: int, D: int, causal: bool = True,
                              key_padding: bool = False, sm_count: int = 0) -> bool:
    """Whether a prefill of this shape deals its query blocks in the wide groups (host only)."""
    n = _load().mha_prefill_wide_schedule(int(B), int(H), int(S), int(D), int(bool(causal)),
                                          int(bool(key_padding)), int(sm_count))
    if n < 0:
        raise MHAError(-n, "mha_prefill_wide_schedule")
    return n == 1


def mha_prefill_schedule(B: int, H: int, S: int, D: int, causal: bool = True,
                         key_padding: bool = False, sm_count: int = 0,
                         cta: int = 0) -> list[tuple[int, int]]:
    """The (b*H + h, 256-row query block) items CTA `cta` of a prefill launch
    of this shape works on, in its order (host only)."""
    lib = _load()
    args = (int(B), int(H), int(S), int(D), int(bool(causal)), int(bool(key_padding)),
            int(sm_count), int(cta))
    n = lib.mha_prefill_schedule(*args, None, None, 0)
    if n < 0:
        raise MHAError(-n, "mha_prefill_schedule")
    bh = (ctypes.c_int * max(n, 1))()
    qp = (ctypes.c_int * max(n, 1))()
    m = lib.mha_prefill_schedule(*args, bh, qp, n)
    if m != n:
        raise MHAError(1 if m >= 0 else -m, "mha_prefill_schedule")
    return list(zip(bh[:n], qp[:n]))


def mha_get_device_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device wait status."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return _load().mha_get_device_status(_stream_ptr(stream, dev))


def mha_status_string(status: int) -> str:
    return _load().mha_status_string(int(status)).decode()


def mha_set_wait_limit_ns(limit_ns: int) -> int:
    return int(_load().mha_set_wait_limit_ns(int(limit_ns)))


def mha_set_fault_injection(mode: int) -> int:
    """Failure-detection hook (see include/mha.h); returns the previous mode."""
    return int(_load().mha_set_fault_injection(int(mode)))
