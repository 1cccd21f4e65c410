"""Quantized-KV decode attention for GB300: Python binding of libtq.so.

Argument marshalling only.  Every step of the path (encode/append, decode,
split combine, inverse rotation) runs in the CUDA kernels of ``libtq.so``; the
functions here turn torch tensors into device pointers and call the C ABI of
``include/tq.h`` under the same names.  There is no CPU fallback: if the
library cannot be loaded every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtq.so")

TQ_OK = 0
TQ_ERR_INVALID_ARG = -1
TQ_ERR_UNSUPPORTED = -2
TQ_ERR_CAPACITY = -3
TQ_ERR_CUDA = -4
TQ_ERR_NOMEM = -5

TQ_TURBO4_ASYM = 0
TQ_TURBO3 = 1
TQ_TURBO4 = 2
TQ_TURBO3_ASYM = 3
TQ_TURBO4K_3V = 4
TQ_TURBO3_TABLE = 5
MODES = {"turbo4_asym": TQ_TURBO4_ASYM, "turbo3": TQ_TURBO3, "turbo4": TQ_TURBO4,
         "turbo3_asym": TQ_TURBO3_ASYM, "turbo4k_3v": TQ_TURBO4K_3V,
         "turbo3_table": TQ_TURBO3_TABLE}
MODE_BITS = {TQ_TURBO4_ASYM: (16, 4), TQ_TURBO3: (3, 3), TQ_TURBO4: (4, 4),
             TQ_TURBO3_ASYM: (16, 3), TQ_TURBO4K_3V: (4, 3), TQ_TURBO3_TABLE: (3, 3)}
# modes whose 64-byte records carry the centroid x norm table (no norm arrays)
TABLE_MODES = {TQ_TURBO3_TABLE}
TABLE_RECORD_BYTES = 64

TQ_STATUS_CAPACITY = 1
TQ_STATUS_NORM_OVERFLOW = 2
TQ_STATUS_SHORT_CONTEXT = 4
TQ_STATUS_PIPELINE_STALL = 8

# every entry point declared in include/tq.h: name -> (restype, argtypes)
_c = ctypes
_SIGS = {
    "tq_encode_append": (_c.c_int, [_c.POINTER(_c.c_void_p), _c.c_void_p, _c.c_void_p,
                                    _c.c_void_p, _c.c_int32, _c.c_void_p]),
    "tq_decode_attention": (_c.c_int, [_c.POINTER(_c.c_void_p), _c.c_void_p, _c.c_void_p,
                                       _c.c_int32, _c.c_int32, _c.c_int32, _c.c_float,
                                       _c.c_void_p, _c.c_void_p]),
    "tq_prefill_attention": (_c.c_int, [_c.POINTER(_c.c_void_p), _c.c_void_p, _c.c_void_p,
                                        _c.c_int32, _c.c_int32, _c.c_int32, _c.c_float,
                                        _c.c_void_p, _c.c_void_p]),
    "tq_decode_attention_sparse_v": (_c.c_int, [_c.POINTER(_c.c_void_p), _c.c_void_p,
                                                _c.c_void_p, _c.c_int32, _c.c_int32, _c.c_int32,
                                                _c.c_float, _c.c_float, _c.c_void_p,
                                                _c.c_void_p]),
    "tq_decode_attention_noalloc": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int32,
                                               _c.c_int32, _c.c_float, _c.c_void_p, _c.c_void_p,
                                               _c.c_void_p]),
    "tq_selftest_bounded_wait": (_c.c_int, [_c.POINTER(_c.c_void_p), _c.c_int32, _c.c_void_p]),
    "tq_free": (None, [_c.c_void_p]),
    "tq_get_status": (_c.c_int, [_c.c_void_p, _c.POINTER(_c.c_uint32)]),
    "tq_lloyd_max_codebook": (_c.c_int, [_c.c_int32, _c.POINTER(_c.c_float)]),
    "tq_record_bytes": (_c.c_int, [_c.c_int32]),
    "tq_plan_splits": (_c.c_int, [_c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                  _c.POINTER(_c.c_int32), _c.POINTER(_c.c_int32)]),
    "tq_get_sparse_v_tiles": (_c.c_int, [_c.c_void_p, _c.POINTER(_c.c_uint64),
                                         _c.POINTER(_c.c_uint64)]),
    "tq_set_kernel_timing": (_c.c_int, [_c.c_void_p, _c.c_int32]),
    "tq_get_kernel_time": (_c.c_int, [_c.c_void_p, _c.POINTER(_c.c_float),
                                      _c.POINTER(_c.c_int32)]),
    "tq_error_string": (_c.c_char_p, [_c.c_int32]),
}


class TqError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} ({code})")


class tq_cache(ctypes.Structure):
    """Mirror of ``tq_cache`` in include/tq.h."""

    _fields_ = [
        ("mode", _c.c_int32), ("batch", _c.c_int32), ("num_kv_heads", _c.c_int32),
        ("head_dim", _c.c_int32), ("capacity", _c.c_int32),
        ("k_data", _c.c_void_p), ("k_norm", _c.c_void_p),
        ("v_data", _c.c_void_p), ("v_norm", _c.c_void_p),
        ("lengths", _c.c_void_p),
        ("codebook_k", _c.POINTER(_c.c_float)), ("codebook_k_size", _c.c_int32),
        ("codebook_v", _c.POINTER(_c.c_float)), ("codebook_v_size", _c.c_int32),
        ("rot_seed", _c.c_uint64), ("v_rescale", _c.c_float),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libtq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m quantized_kv_cache_flash_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


def error_string(code: int) -> str:
    return lib().tq_error_string(code).decode()


def _check(code: int, where: str) -> None:
    if code != TQ_OK:
        raise TqError(code, where)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


class Context:
    """Owner of a ``tq_ctx*`` (created lazily by the first call)."""

    def __init__(self):
        self.ptr = ctypes.c_void_p(None)

    def free(self) -> None:
        if self.ptr.value:
            tq_free(self)
            self.ptr = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def tq_lloyd_max_codebook(bits: int):
    """The library's Lloyd-Max codebook of N(0, 1/128) (list of fp32 floats)."""
    n = 1 << bits
    buf = (ctypes.c_float * n)()
    _check(lib().tq_lloyd_max_codebook(bits, buf), "tq_lloyd_max_codebook")
    return [float(v) for v in buf]


def tq_record_bytes(bits: int) -> int:
    r = lib().tq_record_bytes(bits)
    if r < 0:
        raise TqError(r, "tq_record_bytes")
    return r


def tq_plan_splits(mode: int, batch: int, num_kv_heads: int, rows_per_kv_head: int,
                   max_len_hint: int):
    st, ns = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().tq_plan_splits(mode, batch, num_kv_heads, rows_per_kv_head, max_len_hint,
                                ctypes.byref(st), ctypes.byref(ns)), "tq_plan_splits")
    return st.value, ns.value


class Cache:
    """Device tensors of one packed cache plus the ``tq_cache`` struct that
    points at them.  Allocation is torch's; layout is the library's."""

    def __init__(self, mode: int, batch: int, num_kv_heads: int, capacity: int, device,
                 codebook_k=None, codebook_v=None, rot_seed: int = 42, v_rescale: float = 1.0):
        import torch
        kb, vb = MODE_BITS[mode]
        self.mode, self.batch, self.num_kv_heads, self.capacity = mode, batch, num_kv_heads, capacity
        table = mode in TABLE_MODES
        if kb == 16:
            self.k_data = torch.zeros(batch, num_kv_heads, capacity, 128, dtype=torch.float16,
                                      device=device)
            self.k_norm = None
        elif table:
            self.k_data = torch.zeros(batch, num_kv_heads, capacity, TABLE_RECORD_BYTES,
                                      dtype=torch.uint8, device=device)
            self.k_norm = None
        else:
            self.k_data = torch.zeros(batch, num_kv_heads, capacity, tq_record_bytes(kb),
                                      dtype=torch.uint8, device=device)
            self.k_norm = torch.zeros(batch, num_kv_heads, capacity, dtype=torch.float16,
                                      device=device)
        self.v_data = torch.zeros(batch, num_kv_heads, capacity,
                                  TABLE_RECORD_BYTES if table else tq_record_bytes(vb),
                                  dtype=torch.uint8, device=device)
        self.v_norm = None if table else torch.zeros(batch, num_kv_heads, capacity,
                                                     dtype=torch.float16, device=device)
        self.lengths = torch.zeros(batch, dtype=torch.int32, device=device)
        cbk = codebook_k if codebook_k is not None else (
            tq_lloyd_max_codebook(kb) if kb != 16 else [])
        cbv = codebook_v if codebook_v is not None else tq_lloyd_max_codebook(vb)
        self._cbk = (ctypes.c_float * max(len(cbk), 1))(*cbk)
        self._cbv = (ctypes.c_float * len(cbv))(*cbv)
        self.codebook_k = list(cbk)
        self.codebook_v = list(cbv)
        self.struct = tq_cache(
            mode, batch, num_kv_heads, 128, capacity,
            _ptr(self.k_data), _ptr(self.k_norm), _ptr(self.v_data), _ptr(self.v_norm),
            _ptr(self.lengths),
            ctypes.cast(self._cbk, ctypes.POINTER(ctypes.c_float)), len(cbk),
            ctypes.cast(self._cbv, ctypes.POINTER(ctypes.c_float)), len(cbv),
            rot_seed, v_rescale)

    def set_v_rescale(self, v: float) -> None:
        self.struct.v_rescale = v


def tq_encode_append(ctx: Context, cache: Cache, k_new, v_new, stream=None) -> None:
    """Append k_new/v_new fp16 [B, Hkv, T, 128] at lengths[b]; lengths += T (on device)."""
    import torch
    for t in (k_new, v_new):
        if t.dtype != torch.float16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("k_new/v_new must be contiguous fp16 [B, Hkv, T, 128]")
    t_new = int(k_new.shape[2])
    _check(lib().tq_encode_append(ctypes.byref(ctx.ptr), ctypes.byref(cache.struct),
                                  _ptr(k_new), _ptr(v_new), t_new, _stream(stream)),
           "tq_encode_append")


def tq_decode_attention(ctx: Context, cache: Cache, q, out, max_len_hint: int,
                        scale: float = 0.0, stream=None) -> None:
    """out[B, Hq, Tq, 128] = decode attention of q[B, Hq, Tq, 128] over the cache."""
    import torch
    if q.dtype != torch.float16 or not q.is_contiguous() or q.dim() != 4:
        raise ValueError("q must be contiguous fp16 [B, Hq, Tq, 128]")
    if out.dtype != torch.float16 or not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous fp16 shaped like q")
    _check(lib().tq_decode_attention(ctypes.byref(ctx.ptr), ctypes.byref(cache.struct),
                                     _ptr(q), int(q.shape[1]), int(q.shape[2]),
                                     int(max_len_hint), float(scale), _ptr(out),
                                     _stream(stream)), "tq_decode_attention")


def tq_prefill_attention(ctx: Context, cache: Cache, q, out, max_len_hint: int,
                         scale: float = 0.0, stream=None) -> None:
    """Attention of a block of many queries q[B, Hq, Tq, 128] (a prefill chunk
    already appended to the cache) on the tcgen05 tensor cores."""
    import torch
    if q.dtype != torch.float16 or not q.is_contiguous() or q.dim() != 4:
        raise ValueError("q must be contiguous fp16 [B, Hq, Tq, 128]")
    if out.dtype != torch.float16 or not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous fp16 shaped like q")
    _check(lib().tq_prefill_attention(ctypes.byref(ctx.ptr), ctypes.byref(cache.struct),
                                      _ptr(q), int(q.shape[1]), int(q.shape[2]),
                                      int(max_len_hint), float(scale), _ptr(out),
                                      _stream(stream)), "tq_prefill_attention")


def tq_decode_attention_sparse_v(ctx: Context, cache: Cache, q, out, max_len_hint: int,
                                 tau: float, scale: float = 0.0, stream=None) -> None:
    """Decode with the V of tokens whose softmax weight is below `tau` skipped."""
    import torch
    if q.dtype != torch.float16 or not q.is_contiguous() or q.dim() != 4:
        raise ValueError("q must be contiguous fp16 [B, Hq, Tq, 128]")
    if out.dtype != torch.float16 or not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous fp16 shaped like q")
    _check(lib().tq_decode_attention_sparse_v(ctypes.byref(ctx.ptr), ctypes.byref(cache.struct),
                                              _ptr(q), int(q.shape[1]), int(q.shape[2]),
                                              int(max_len_hint), float(scale), float(tau),
                                              _ptr(out), _stream(stream)),
           "tq_decode_attention_sparse_v")


def tq_decode_attention_noalloc(cache: Cache, q, out, max_len_hint: int, scale: float = 0.0,
                                status=None, stream=None) -> None:
    """Decode without a context and without any device allocation: the split-K
    scratch is the library's fixed device array (shared by all calls; serialise
    calls that could overlap on the GPU).  `status` is an optional int32/uint32
    device tensor of one element that the kernels OR status bits into."""
    import torch
    if q.dtype != torch.float16 or not q.is_contiguous() or q.dim() != 4:
        raise ValueError("q must be contiguous fp16 [B, Hq, Tq, 128]")
    if out.dtype != torch.float16 or not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous fp16 shaped like q")
    _check(lib().tq_decode_attention_noalloc(ctypes.byref(cache.struct), _ptr(q), int(q.shape[1]),
                                             int(q.shape[2]), int(max_len_hint), float(scale),
                                             _ptr(out), _ptr(status), _stream(stream)),
           "tq_decode_attention_noalloc")


def tq_selftest_bounded_wait(ctx: Context, limit_us: int, stream=None) -> None:
    """Make one bounded in-kernel wait run out (failure-path self-test)."""
    _check(lib().tq_selftest_bounded_wait(ctypes.byref(ctx.ptr), int(limit_us), _stream(stream)),
           "tq_selftest_bounded_wait")


def tq_free(ctx: Context) -> None:
    lib().tq_free(ctx.ptr)


def tq_get_status(ctx: Context) -> int:
    """Return and clear the device status bits (waits for the context's latest stream)."""
    s = ctypes.c_uint32()
    _check(lib().tq_get_status(ctx.ptr, ctypes.byref(s)), "tq_get_status")
    return s.value


def tq_get_sparse_v_tiles(ctx: Context):
    """(skipped, judged) 16-token tiles of the sparse-V decode since the last read."""
    a, b = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib().tq_get_sparse_v_tiles(ctx.ptr, ctypes.byref(a), ctypes.byref(b)),
           "tq_get_sparse_v_tiles")
    return a.value, b.value


def tq_set_kernel_timing(ctx: Context, enable: bool) -> None:
    _check(lib().tq_set_kernel_timing(ctx.ptr, 1 if enable else 0), "tq_set_kernel_timing")


def tq_get_kernel_time(ctx: Context):
    ms, n = ctypes.c_float(), ctypes.c_int32()
    _check(lib().tq_get_kernel_time(ctx.ptr, ctypes.byref(ms), ctypes.byref(n)),
           "tq_get_kernel_time")
    return ms.value, n.value
