"""Host-side tests of libtq.so (no GPU): it loads, exports every entry point of
include/tq.h, its host utilities agree with the oracle, and every argument
error is caught on the host before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

import quantized_kv_cache_flash_gb300 as tqf
from quantized_kv_cache_flash_gb300 import build as tqbuild
from oracle import tq_oracle as o
from tests.helpers import decode_records

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    tqbuild.build()
    return tqf.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(tq_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "tq_encode_append" in names and "tq_decode_attention" in names and "tq_free" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in tqf._SIGS, f"{n} has no binding"


def test_codebook_matches_oracle_bitwise(lib):
    for bits in (1, 2, 3, 4):
        got = np.array(tqf.tq_lloyd_max_codebook(bits), np.float32)
        want = o.codebook(bits)
        assert np.array_equal(got, want), (bits, got, want)


def test_record_bytes(lib):
    assert tqf.tq_record_bytes(3) == 48
    assert tqf.tq_record_bytes(4) == 64
    assert tqf.tq_record_bytes(16) == 256
    with pytest.raises(tqf.TqError):
        tqf.tq_record_bytes(5)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("B,Hkv,rows,L", [(1, 2, 2, 256), (1, 4, 7, 8192), (1, 4, 7, 16384),
                                          (32, 8, 4, 32768), (4, 8, 16, 131072), (2, 2, 64, 777),
                                          (1, 1, 1, 1)])
def test_decode_grid_covers_context(lib, mode, B, Hkv, rows, L):
    st, ctas = tqf.tq_plan_splits(mode, B, Hkv, rows, L)
    units = B * Hkv * -(-rows // (8 if rows <= 8 else 16))
    chunks = units * -(-L // 32)
    waves = 1 if rows > 8 else 3                      # 16-row groups: one wave; smaller: two or three
    assert 1 <= ctas <= waves * 152 * 4
    assert st % 32 == 0 and ctas * st >= chunks * 32  # the CTAs cover every chunk
    assert st == -(-chunks // ctas) * 32              # the largest share, in tokens
    assert chunks >= ctas                             # every CTA has work
    assert ctas == 1 or st >= 8 * 32                  # at least two chunks per warp


def test_decode_grid_waves(lib):
    """The split grid's waves of resident CTAs (4 per SM for 4- and 8-row
    groups of quantized K, 3 for 16-row groups, 2 for fp16 K): two waves, a
    third when every CTA would still stream at least 96 chunks, one wave for
    16-row groups, fewer CTAs when a warp would get under two chunks."""
    assert tqf.tq_plan_splits(2, 32, 8, 4, 32768 + 128)[1] == 3 * 152 * 4   # the batched step
    assert tqf.tq_plan_splits(2, 16, 8, 4, 32768 + 128)[1] == 2 * 152 * 4   # half of it: two waves
    assert tqf.tq_plan_splits(1, 4, 8, 16, 131072)[1] == 1 * 152 * 3        # 16 rows: one wave
    assert tqf.tq_plan_splits(0, 1, 4, 7, 16384)[1] == 16384 * 4 // 32 // 8  # small: two chunks a warp
    assert tqf.tq_plan_splits(1, 1, 4, 7, 8192)[1] == 8192 * 4 // 32 // 8


def test_decode_records_helper_reads_the_format():
    rng = np.random.default_rng(0)
    for bits in (3, 4):
        idx = rng.integers(0, 1 << bits, (9, 128)).astype(np.uint8)
        assert np.array_equal(decode_records(o.pack_codes(idx, bits), bits), idx)


# ---------------------------------------------------------------------------
# argument errors: all detected on the host before any CUDA call, so they run
# without a GPU.  Device pointers are fake aligned addresses (never touched).
# ---------------------------------------------------------------------------
FAKE = 1 << 20


def _cache(mode=1, batch=2, hkv=2, head_dim=128, cap=64, cb=None, **kw):
    kb, vb = tqf.MODE_BITS.get(mode, (3, 3))
    cbv = cb if cb is not None else tqf.tq_lloyd_max_codebook(vb)
    cbk = cb if cb is not None else (tqf.tq_lloyd_max_codebook(kb) if kb != 16 else [])
    keep = [(ctypes.c_float * max(len(cbk), 1))(*cbk), (ctypes.c_float * len(cbv))(*cbv)]
    f = dict(mode=mode, batch=batch, num_kv_heads=hkv, head_dim=head_dim, capacity=cap,
             k_data=FAKE, k_norm=FAKE + 4096, v_data=FAKE + 8192, v_norm=FAKE + 16384,
             lengths=FAKE + 32768,
             codebook_k=ctypes.cast(keep[0], ctypes.POINTER(ctypes.c_float)),
             codebook_k_size=len(cbk),
             codebook_v=ctypes.cast(keep[1], ctypes.POINTER(ctypes.c_float)),
             codebook_v_size=len(cbv), rot_seed=42, v_rescale=1.0)
    f.update(kw)
    c = tqf.tq_cache(**f)
    c._keep = keep
    return c


def _decode(lib, c, hq=4, tq=1, max_len=32, scale=0.0, q=FAKE + 65536, out=FAKE + 131072):
    ctx = ctypes.c_void_p(None)
    r = lib.tq_decode_attention(ctypes.byref(ctx), ctypes.byref(c), q, hq, tq, max_len, scale,
                                out, None)
    assert ctx.value is None          # no context is created for a rejected call
    return r


def _append(lib, c, t_new=1, k=FAKE + 65536, v=FAKE + 131072):
    ctx = ctypes.c_void_p(None)
    r = lib.tq_encode_append(ctypes.byref(ctx), ctypes.byref(c), k, v, t_new, None)
    assert ctx.value is None
    return r


def test_errors_unsupported_head_dim_and_mode(lib):
    assert _decode(lib, _cache(head_dim=64)) == tqf.TQ_ERR_UNSUPPORTED
    assert _decode(lib, _cache(head_dim=96)) == tqf.TQ_ERR_UNSUPPORTED
    assert _append(lib, _cache(head_dim=256)) == tqf.TQ_ERR_UNSUPPORTED
    assert _decode(lib, _cache(mode=7)) == tqf.TQ_ERR_UNSUPPORTED
    assert _decode(lib, _cache(mode=6)) == tqf.TQ_ERR_UNSUPPORTED


def test_errors_gqa_and_shapes(lib):
    assert _decode(lib, _cache(hkv=2), hq=3) == tqf.TQ_ERR_INVALID_ARG      # Hq % Hkv != 0
    assert _decode(lib, _cache(hkv=2), hq=0) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(cap=60)) == tqf.TQ_ERR_INVALID_ARG            # capacity % 16
    assert _decode(lib, _cache(), tq=0) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(), tq=40, max_len=32) == tqf.TQ_ERR_INVALID_ARG  # Tq > context
    assert _decode(lib, _cache(cap=64), max_len=80) == tqf.TQ_ERR_INVALID_ARG   # hint > capacity
    assert _decode(lib, _cache(batch=0)) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(), scale=-1.0) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(hkv=1), hq=512) == tqf.TQ_ERR_UNSUPPORTED     # > 256 rows


def test_errors_pointers(lib):
    assert _decode(lib, _cache(k_data=None)) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(lengths=None)) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(k_norm=None)) == tqf.TQ_ERR_INVALID_ARG       # quantized K needs norms
    assert _decode(lib, _cache(v_data=FAKE + 8)) == tqf.TQ_ERR_INVALID_ARG   # misaligned
    assert _decode(lib, _cache(), q=None) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(), out=FAKE + 4) == tqf.TQ_ERR_INVALID_ARG
    assert _append(lib, _cache(), k=None) == tqf.TQ_ERR_INVALID_ARG
    # fp16-K modes take no K norms
    assert _decode(lib, _cache(mode=0, k_norm=None), q=None) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(mode=3, k_norm=None), q=None) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(mode=4, k_norm=None)) == tqf.TQ_ERR_INVALID_ARG   # 4-bit K needs them
    assert _decode(lib, _cache(mode=1, v_norm=None)) == tqf.TQ_ERR_INVALID_ARG   # turbo3 needs V norms
    # table records carry their norms: NULL norm arrays pass (rejected here only for q)
    assert _decode(lib, _cache(mode=5, k_norm=None, v_norm=None), q=None) == tqf.TQ_ERR_INVALID_ARG
    assert _append(lib, _cache(mode=5, k_norm=None, v_norm=None), k=None) == tqf.TQ_ERR_INVALID_ARG


def test_errors_sparse_v_threshold(lib):
    for tau in (-1e-6, float("nan"), float("inf")):
        ctx = ctypes.c_void_p(None)
        r = lib.tq_decode_attention_sparse_v(ctypes.byref(ctx), ctypes.byref(_cache()), FAKE + 65536,
                                             4, 1, 32, 0.0, tau, FAKE + 131072, None)
        assert r == tqf.TQ_ERR_INVALID_ARG and ctx.value is None


def test_errors_codebook(lib):
    cb = tqf.tq_lloyd_max_codebook(3)
    asym = list(cb); asym[0] -= 1e-3
    assert _decode(lib, _cache(cb=asym)) == tqf.TQ_ERR_INVALID_ARG
    unsorted = list(cb); unsorted[3], unsorted[4] = unsorted[4], unsorted[3]
    assert _decode(lib, _cache(cb=unsorted)) == tqf.TQ_ERR_INVALID_ARG
    assert _decode(lib, _cache(cb=cb[:4])) == tqf.TQ_ERR_INVALID_ARG          # wrong size
    nan = list(cb); nan[0] = float("nan")
    assert _decode(lib, _cache(cb=nan)) == tqf.TQ_ERR_INVALID_ARG


def test_errors_capacity_and_noop_append(lib):
    assert _append(lib, _cache(cap=64), t_new=65) == tqf.TQ_ERR_CAPACITY
    assert _append(lib, _cache(), t_new=-1) == tqf.TQ_ERR_INVALID_ARG
    assert _append(lib, _cache(), t_new=0) == tqf.TQ_OK                      # no-op, no launch


def test_null_context_calls(lib):
    lib.tq_free(None)
    s = ctypes.c_uint32(7)
    assert lib.tq_get_status(None, ctypes.byref(s)) == tqf.TQ_OK and s.value == 0
    assert lib.tq_set_kernel_timing(None, 1) == tqf.TQ_ERR_INVALID_ARG
    assert lib.tq_error_string(tqf.TQ_ERR_CUDA) == b"CUDA error"


def test_binding_raises_on_injected_cuda_error(monkeypatch):
    """A CUDA failure reported by the library surfaces as TqError with the
    library's message (the error is injected on the host)."""
    class FakeLib:
        def tq_record_bytes(self, bits):
            return tqf.TQ_ERR_CUDA

        def tq_error_string(self, code):
            return b"CUDA error"
    monkeypatch.setattr(tqf, "lib", lambda: FakeLib())
    with pytest.raises(tqf.TqError) as e:
        tqf.tq_record_bytes(3)
    assert e.value.code == tqf.TQ_ERR_CUDA


def test_selftest_rejects_bad_limits(lib):
    ctx = ctypes.c_void_p(None)
    assert lib.tq_selftest_bounded_wait(ctypes.byref(ctx), 0, None) == tqf.TQ_ERR_INVALID_ARG
    assert lib.tq_selftest_bounded_wait(ctypes.byref(ctx), 2000000, None) == tqf.TQ_ERR_INVALID_ARG
    assert lib.tq_selftest_bounded_wait(None, 100, None) == tqf.TQ_ERR_INVALID_ARG
    assert ctx.value is None
