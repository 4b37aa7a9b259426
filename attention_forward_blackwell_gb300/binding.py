"""ctypes binding of libfa_gb300.so (argument marshalling only).

Every function here checks tensor shapes/dtypes/devices, allocates outputs with
torch when the caller does not pass them, and calls the C ABI declared in
``include/fa.h`` on the current torch CUDA stream.  All arithmetic runs in the
library's CUDA kernels; there is no fallback path.  If the library has not
been built, loading it raises.
"""
from __future__ import annotations

import collections
import ctypes
import math
import os
import threading

import torch

from .build import LIB_PATH

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED, FA_ERR_CUDA, \
    FA_ERR_TIMEOUT = range(6)
FA_DECODE_MAX_SQ = 16

# name -> (restype, argtypes); must match include/fa.h
_VP, _I, _F, _LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
_FWD = [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _I, _F, _I]
SIGNATURES = {
    "fa_fwd_prefill": (_I, _FWD + [_VP]),
    "fa_fwd_prefill_ex": (_I, _FWD + [_I, _VP, _VP]),
    "fa_fwd_decode_ex": (_I, _FWD + [_I, _VP, _VP]),
    "fa_fwd_prefill_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _I, _I, _I,
                                  _I, _F, _I, _VP]),
    "fa_fwd_decode_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _I, _I, _I,
                                 _I, _F, _I, _VP]),
    "fa_fwd_prefill_varlen": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I,
                                   _I, _F, _I, _I, _VP, _VP]),
    "fa_fwd_prefill_varlen_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I,
                                         _I, _I, _I, _I, _I, _F, _I, _I, _VP, _VP]),
    "fa_fwd_decode": (_I, _FWD + [_VP]),
    "fa_fwd_decode_splits": (_I, _FWD + [_I, _VP]),
    "fa_fwd_decode_noalloc": (_I, _FWD + [_VP]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_get_device_error": (_I, [_VP]),
    "fa_get_device_error_word": (_I, [_VP, ctypes.POINTER(ctypes.c_uint)]),
    "fa_selftest_wait_timeout": (_I, [_LL, _VP]),
    "fa_selftest_tmem_roundtrip": (_I, [_VP, _VP, _VP]),
    "fa_selftest_mma_tile": (_I, [_VP, _VP, _VP, _I, _I, _VP]),
    "fa_debug_prefill_trace": (_I, [_VP, _I]),
    "fa_selftest_exp2_poly": (_I, [_VP, _VP, _I, _VP]),
    "fa_debug_prefill_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _VP]),
    "fa_debug_prefill_plan_ex": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "fa_debug_prefill_plan_gqa": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "fa_version": (_I, []),
}

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def lib(path: str | None = None):
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build it with attention_forward_blackwell_gb300."
                    "build.build() (there is no CPU fallback)")
            handle = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def version() -> int:
    return lib().fa_version()


def _stream_ptr(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check_inputs(q, k, v, seqlens_k):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor")
    B, Hq, Sq, d = q.shape
    Bk, Hkv, Sk, dk = k.shape
    if v.shape != k.shape or Bk != B or dk != d:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if seqlens_k is not None:
        if seqlens_k.dtype != torch.int32 or not seqlens_k.is_cuda or seqlens_k.shape != (B,):
            raise ValueError("seqlens_k must be a CUDA int32 tensor of shape [B]")
        seqlens_k = seqlens_k.contiguous()
    return B, Hq, Hkv, Sq, Sk, d, seqlens_k


def _outputs(q, out, lse):
    B, Hq, Sq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, Hq, Sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor of shape [B, Hq, Sq]")
    return out, lse


def _check_sinks(sinks, hq):
    if sinks is None:
        return None
    if sinks.dtype != torch.float32 or sinks.shape != (hq,) or not sinks.is_cuda:
        raise ValueError("sinks must be a CUDA fp32 tensor of shape [Hq]")
    return sinks.contiguous()


def prefill(q, k, v, scale=None, causal=False, seqlens_k=None, out=None, lse=None,
            stream=None, window=0, sinks=None):
    """Attention forward through ``fa_fwd_prefill`` (``fa_fwd_prefill_ex`` with
    a sliding ``window`` > 0 or per-head ``sinks``); returns (o, lse)."""
    B, Hq, Hkv, Sq, Sk, d, seqlens_k = _check_inputs(q, k, v, seqlens_k)
    out, lse = _outputs(q, out, lse)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    sinks = _check_sinks(sinks, q.shape[1])
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk,
            _ptr(seqlens_k), d, scale, int(bool(causal)))
    if (window and window > 0) or sinks is not None:
        st = lib().fa_fwd_prefill_ex(*args, int(window or 0), _ptr(sinks), _stream_ptr(stream))
    else:
        st = lib().fa_fwd_prefill(*args, _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_prefill")
    return out, lse


def decode(q, k, v, scale=None, causal=False, seqlens_k=None, num_splits=0, out=None,
           lse=None, stream=None, window=0, sinks=None):
    """Split-KV attention forward through ``fa_fwd_decode_splits``
    (num_splits <= 0 lets the library choose, as ``fa_fwd_decode`` does), or
    ``fa_fwd_decode_ex`` with a sliding ``window`` > 0 or per-head ``sinks``."""
    B, Hq, Hkv, Sq, Sk, d, seqlens_k = _check_inputs(q, k, v, seqlens_k)
    out, lse = _outputs(q, out, lse)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    sinks = _check_sinks(sinks, q.shape[1])
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk,
            _ptr(seqlens_k), d, scale, int(bool(causal)))
    if (window and window > 0) or sinks is not None:
        if num_splits and num_splits > 0:
            raise ValueError("num_splits cannot be combined with window or sinks")
        st = lib().fa_fwd_decode_ex(*args, int(window or 0), _ptr(sinks), _stream_ptr(stream))
    elif num_splits and num_splits > 0:
        st = lib().fa_fwd_decode_splits(*args, int(num_splits), _stream_ptr(stream))
    else:
        st = lib().fa_fwd_decode(*args, _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_decode")
    return out, lse


def _paged(name, q, k_cache, v_cache, block_table, seqlens_k, scale, causal, out, lse, stream):
    if not (q.is_cuda and k_cache.is_cuda and v_cache.is_cuda):
        raise ValueError("q and the caches must be CUDA tensors")
    if q.dtype != torch.bfloat16 or k_cache.dtype != torch.bfloat16 or v_cache.dtype != torch.bfloat16:
        raise ValueError("q and the caches must be bf16")
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4:
        raise ValueError("caches must share a shape [num_pages, Hkv, page_size, d]")
    B, Hq, Sq, d = q.shape
    num_pages, Hkv, page_size, dk = k_cache.shape
    if dk != d:
        raise ValueError("head dims differ")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be int32 [B, max_pages]")
    if seqlens_k is None or seqlens_k.dtype != torch.int32 or seqlens_k.shape != (B,):
        raise ValueError("seqlens_k must be int32 [B]")
    q, k_cache, v_cache = q.contiguous(), k_cache.contiguous(), v_cache.contiguous()
    block_table, seqlens_k = block_table.contiguous(), seqlens_k.contiguous()
    out, lse = _outputs(q, out, lse)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = getattr(lib(), name)(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B, Hq,
                              Hkv, Sq, _ptr(seqlens_k), _ptr(block_table), block_table.shape[1],
                              page_size, num_pages, d, scale, int(bool(causal)),
                              _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, name)
    return out, lse


def prefill_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale=None,
                   causal=False, window=0, sinks=None, out=None, lse=None, stream=None):
    """Prefill over packed sequences through ``fa_fwd_prefill_varlen``:
    q [total_q, Hq, d], k and v [total_k, Hkv, d] bf16, int32 offsets
    cu_seqlens_q / cu_seqlens_k [B + 1]; returns o [total_q, Hq, d] and
    lse [Hq, total_q]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 3:
            raise ValueError(f"{n} must be a CUDA bf16 tensor [tokens, heads, d]")
    total_q, Hq, d = q.shape
    total_k, Hkv, dk = k.shape
    if v.shape != k.shape or dk != d:
        raise ValueError("k and v must be [total_k, Hkv, d] with q's d")
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        if not t.is_cuda or t.dtype != torch.int32 or t.dim() != 1:
            raise ValueError(f"{n} must be a CUDA int32 vector [B + 1]")
    if cu_seqlens_q.shape != cu_seqlens_k.shape or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both be [B + 1]")
    B = cu_seqlens_q.numel() - 1
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    cu_seqlens_q, cu_seqlens_k = cu_seqlens_q.contiguous(), cu_seqlens_k.contiguous()
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, total_q, device=q.device, dtype=torch.float32)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (Hq, total_q) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [Hq, total_q]")
    sinks = _check_sinks(sinks, Hq)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().fa_fwd_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                     _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, int(max_seqlen_q),
                                     int(max_seqlen_k), total_q, total_k, Hq, Hkv, d, scale,
                                     int(bool(causal)), int(window), _ptr(sinks),
                                     _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_prefill_varlen")
    return out, lse


def prefill_varlen_paged(q, k_cache, v_cache, cu_seqlens_q, max_seqlen_q, block_table, seqlens_k,
                         scale=None, causal=False, window=0, sinks=None, out=None, lse=None,
                         stream=None):
    """Packed queries q [total_q, Hq, d] (offsets cu_seqlens_q [B + 1]) over
    paged caches [num_pages, Hkv, page_size, d] (block_table [B, max_pages],
    seqlens_k [B]) through ``fa_fwd_prefill_varlen_paged``; returns
    o [total_q, Hq, d] and lse [Hq, total_q]."""
    if not q.is_cuda or q.dtype != torch.bfloat16 or q.dim() != 3:
        raise ValueError("q must be a CUDA bf16 tensor [tokens, heads, d]")
    if (k_cache.shape != v_cache.shape or k_cache.dim() != 4 or not k_cache.is_cuda
            or k_cache.dtype != torch.bfloat16 or v_cache.dtype != torch.bfloat16):
        raise ValueError("caches must be CUDA bf16 tensors [num_pages, Hkv, page_size, d]")
    total_q, Hq, d = q.shape
    num_pages, Hkv, page_size, dk = k_cache.shape
    if dk != d:
        raise ValueError("head dims differ")
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (seqlens_k, "seqlens_k")):
        if not t.is_cuda or t.dtype != torch.int32 or t.dim() != 1:
            raise ValueError(f"{n} must be a CUDA int32 vector")
    B = cu_seqlens_q.numel() - 1
    if seqlens_k.shape != (B,):
        raise ValueError("seqlens_k must be [B] with B + 1 query offsets")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be int32 [B, max_pages]")
    q, k_cache, v_cache = q.contiguous(), k_cache.contiguous(), v_cache.contiguous()
    cu_seqlens_q, seqlens_k = cu_seqlens_q.contiguous(), seqlens_k.contiguous()
    block_table = block_table.contiguous()
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, total_q, device=q.device, dtype=torch.float32)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (Hq, total_q) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [Hq, total_q]")
    sinks = _check_sinks(sinks, Hq)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().fa_fwd_prefill_varlen_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
        _ptr(seqlens_k), _ptr(block_table), block_table.shape[1], page_size, num_pages, B,
        int(max_seqlen_q), total_q, Hq, Hkv, d, scale, int(bool(causal)), int(window),
        _ptr(sinks), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_prefill_varlen_paged")
    return out, lse


def prefill_paged(q, k_cache, v_cache, block_table, seqlens_k, scale=None, causal=False,
                  out=None, lse=None, stream=None):
    """Prefill over paged caches [num_pages, Hkv, page_size, d] through
    ``fa_fwd_prefill_paged`` (page_size a multiple of 128); returns (o, lse)."""
    return _paged("fa_fwd_prefill_paged", q, k_cache, v_cache, block_table, seqlens_k, scale,
                  causal, out, lse, stream)


def decode_paged(q, k_cache, v_cache, block_table, seqlens_k, scale=None, causal=False,
                 out=None, lse=None, stream=None):
    """Decode over paged caches through ``fa_fwd_decode_paged``; returns (o, lse)."""
    return _paged("fa_fwd_decode_paged", q, k_cache, v_cache, block_table, seqlens_k, scale,
                  causal, out, lse, stream)


def get_device_error(stream=None) -> int:
    """Synchronise the stream and read/clear the device error word."""
    return lib().fa_get_device_error(_stream_ptr(stream))


def get_device_error_word(stream=None):
    """(status, raw error word) after synchronising the stream; clears it."""
    w = ctypes.c_uint(0)
    st = lib().fa_get_device_error_word(_stream_ptr(stream), ctypes.byref(w))
    return st, w.value


def selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return lib().fa_selftest_wait_timeout(int(limit_ns), _stream_ptr(stream))


def selftest_tmem_roundtrip(x, stream=None):
    """x: CUDA fp32 [128, 64]; returns the tensor-memory round trip of x."""
    if x.dtype != torch.float32 or x.shape != (128, 64) or not x.is_cuda:
        raise ValueError("x must be a CUDA fp32 tensor of shape [128, 64]")
    x = x.contiguous()
    out = torch.empty_like(x)
    st = lib().fa_selftest_tmem_roundtrip(_ptr(x), _ptr(out), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_selftest_tmem_roundtrip")
    return out


def selftest_mma_tile(a, b, mode, stream=None):
    """One 128x128 tile through the prefill kernel's MMA path (see fa.h)."""
    a, b = a.contiguous(), b.contiguous()
    d = torch.empty(128, 128, dtype=torch.float32, device=a.device)
    st = lib().fa_selftest_mma_tile(_ptr(a), _ptr(b), _ptr(d), int(mode), int(a.shape[1]),
                                    _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_selftest_mma_tile")
    return d


def debug_prefill_trace(buf=None, block=0):
    """Install (or with buf=None remove) a prefill trace buffer: a CUDA
    uint64/int64 tensor of at least 5 * 4096 elements (see fa.h)."""
    if buf is not None and (buf.numel() < 5 * 4096 or buf.element_size() != 8 or not buf.is_cuda):
        raise ValueError("trace buffer must be a CUDA 64-bit tensor of >= 20480 elements")
    st = lib().fa_debug_prefill_trace(_ptr(buf), int(block))
    if st != FA_OK:
        raise FaError(st, "fa_debug_prefill_trace")


def debug_prefill_plan(batch, hq, sq, sk, head_dim, causal, num_sms):
    """The prefill work split (host only, see fa.h): (n_full, n_tail, split)."""
    out = (ctypes.c_int * 3)()
    st = lib().fa_debug_prefill_plan(int(batch), int(hq), int(sq), int(sk), int(head_dim),
                                     int(bool(causal)), int(num_sms), ctypes.addressof(out))
    if st != FA_OK:
        raise FaError(st, "fa_debug_prefill_plan")
    return tuple(out)


PrefillPlan = collections.namedtuple(
    "PrefillPlan", "n_full n_tail split rows_per_unit keys_per_block persistent")


def debug_prefill_plan_ex(batch, hq, sq, sk, head_dim, causal, num_sms, *, window=0,
                          paged=False, packed=False):
    """The prefill work split of any launch kind (host only, see fa.h)."""
    out = (ctypes.c_int * 6)()
    st = lib().fa_debug_prefill_plan_ex(int(batch), int(hq), int(sq), int(sk), int(head_dim),
                                        int(bool(causal)), int(window), int(bool(paged)),
                                        int(bool(packed)), int(num_sms), ctypes.addressof(out))
    if st != FA_OK:
        raise FaError(st, "fa_debug_prefill_plan_ex")
    return PrefillPlan(*out[:5], bool(out[5]))


PrefillPlanGqa = collections.namedtuple(
    "PrefillPlanGqa", "n_full n_tail split rows_per_unit keys_per_block persistent pack")


def debug_prefill_plan_gqa(batch, hq, hkv, sq, sk, head_dim, causal, num_sms, *, window=0,
                           paged=False, packed=False):
    """The prefill work split with the kv head count: pack = query heads per
    unit of the 256-key kernel (host only, see fa.h)."""
    out = (ctypes.c_int * 7)()
    st = lib().fa_debug_prefill_plan_gqa(int(batch), int(hq), int(hkv), int(sq), int(sk),
                                         int(head_dim), int(bool(causal)), int(window),
                                         int(bool(paged)), int(bool(packed)), int(num_sms),
                                         ctypes.addressof(out))
    if st != FA_OK:
        raise FaError(st, "fa_debug_prefill_plan_gqa")
    return PrefillPlanGqa(*out[:5], bool(out[5]), out[6])


def selftest_exp2_poly(x, stream=None):
    """The prefill softmax's polynomial 2^x on a CUDA fp32 tensor."""
    if x.dtype != torch.float32 or not x.is_cuda:
        raise ValueError("x must be a CUDA fp32 tensor")
    x = x.contiguous()
    y = torch.empty_like(x)
    st = lib().fa_selftest_exp2_poly(_ptr(x), _ptr(y), x.numel(), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_selftest_exp2_poly")
    return y
