"""GPU parity of sparse-V decode (V skipped for softmax weights below tau).

The kernel may skip any token whose normalised weight is below tau (it never
skips others), so its output must lie within the oracle's bound of what the
skipped tokens can add; the bound is taken at 2 tau to cover the rounding of
the kernel's own weights.  Sharp queries (q scaled up) make most weights tiny,
so most tiles are skipped; the full decode of the same queries is checked
against the oracle at every sharpness (the score path keeps the rotated
query's and the centroids' low-order parts).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import quantized_kv_cache_flash_gb300 as tqf
from quantized_kv_cache_flash_gb300 import workloads as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu

DEV = None


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    global DEV
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_kv_cache_flash_gb300 import build
    build.build()
    DEV = torch.device("cuda", 0)
    yield


CASES = [
    # mode, B, Hq, Hkv, lengths, Tq, cap, q scale, tau
    ("turbo4", 2, 32, 8, [3000, 1777], 1, 3008, 4.0, 1e-6),
    ("turbo3", 1, 32, 8, [2600], 4, 2608, 4.0, 1e-6),             # Tq 4: 16 rows, causal block
    ("turbo4_asym", 1, 28, 4, [4100], 1, 4112, 4.0, 1e-6),
    ("turbo3_asym", 1, 8, 2, [900], 1, 912, 4.0, 0.05),           # large tau: skips are visible
    ("turbo4k_3v", 2, 12, 4, [700, 1500], 2, 1504, 4.0, 0.05),
    ("turbo4", 2, 32, 8, [3000, 1777], 1, 3008, 32.0, 1e-6),      # very sharp
    ("turbo3", 1, 32, 8, [2600], 4, 2608, 32.0, 1e-6),
]


def _ulp_close(sparse, full, bound, rms):
    """sparse and full are the same kernel run with and without the skip: they
    differ by the skipped tokens' share (within bound) and the fp16 rounding
    of each output."""
    tol = bound + 2.0 ** -10 * np.maximum(np.abs(sparse), np.abs(full)) + 1e-6 * rms
    return np.abs(sparse - full) <= tol


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-q{c[7]:g}-tau{c[8]:g}")
def test_sparse_v_within_bound_of_full_decode(case):
    mode, B, Hq, Hkv, lengths, Tq, cap, qs, tau = case
    key = 9100 + sum(lengths) + Hq
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, key)
    q_np = (wl.random_fp16(key + 3, (B, Hq, Tq, 128)).astype(np.float32) * qs).astype(np.float16)
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, DEV, v_rescale=0.75)
    ctx = tqf.Context()
    q = H.upload(q_np, DEV)
    sparse = torch.empty_like(q)
    full = torch.empty_like(q)
    tqf.tq_decode_attention_sparse_v(ctx, cache, q, sparse, max(lengths), tau)
    tqf.tq_decode_attention(ctx, cache, q, full, max(lengths))
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == 0
    units = {(b, h): H.oracle_unit_from_records(mode, kd, kn, vd, vn, b, h, lengths[b])
             for b in range(B) for h in range(Hkv)}
    sc = 1 / math.sqrt(128)
    want_full = H.oracle_decode(mode, q_np, units, lengths, Hkv, Tq, sc, 0.75)
    _, bound = H.oracle_decode_sparse_v(mode, q_np, units, lengths, Hkv, Tq, sc, 0.75, 2 * tau)
    got = sparse.float().cpu().numpy()
    got_full = full.float().cpu().numpy()
    rms = math.sqrt(float(np.mean(want_full ** 2)))
    assert np.all(_ulp_close(got, got_full, bound, rms)), case
    H.assert_attention_close(got_full, want_full, f"{case} full")
    H.assert_within_skip_bound(got, want_full, bound, str(case))
    if tau >= 0.01:
        # the skip really happened: dropped weights of this size show in fp16
        assert float(np.abs(got - got_full).max()) > 1e-3 * rms


@pytest.mark.parametrize("mode,Tq", [("turbo3", 4), ("turbo4_asym", 1)])
def test_sparse_v_skips_tiles_after_a_dominant_token(mode, Tq):
    """The first token of every 32-token chunk is planted along the sum of the
    group's query rows, so it dominates every row's softmax: the second tile of
    each chunk is then below tau for all rows and must be skipped."""
    from oracle import tq_oracle as o
    B, Hq, Hkv, L, cap, tau = 1, 16, 4, 1200, 1216, 0.05
    G = Hq // Hkv
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 4242)
    q_np = (wl.random_fp16(4243, (B, Hq, Tq, 128)).astype(np.float32) * 4).astype(np.float16)
    kb, _ = H.MODE_BITS[mode]
    for h in range(Hkv):
        d = q_np[0, h * G:(h + 1) * G].astype(np.float64).reshape(-1, 128).sum(0)
        k_star = (0.3 * d).astype(np.float16)   # a score some 50 above the others: every row
        if kb == 16:
            kd[0, h, 0:L:32] = k_star
        else:
            idx, n16, _, _ = o.encode(k_star[None], o.codebook(kb), o.sign_vector(42))
            kd[0, h, 0:L:32] = o.pack_codes(idx, kb)[0]
            kn[0, h, 0:L:32] = n16[0]
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, [L], kd, kn, vd, vn, DEV)
    ctx = tqf.Context()
    q = H.upload(q_np, DEV)
    sparse, full = torch.empty_like(q), torch.empty_like(q)
    tqf.tq_decode_attention_sparse_v(ctx, cache, q, sparse, L, tau)
    tqf.tq_decode_attention(ctx, cache, q, full, L)
    torch.cuda.synchronize()
    # the tile counters: every tile of every unit judged once, the second tile
    # of (nearly) every chunk skipped; the plain decode counts nothing
    skipped, judged = tqf.tq_get_sparse_v_tiles(ctx)
    assert judged == Hkv * ((L + 15) // 16)     # one row group per kv head here
    assert 0.3 * judged <= skipped < judged, (skipped, judged)
    assert tqf.tq_get_sparse_v_tiles(ctx) == (0, 0)
    units = {(0, h): H.oracle_unit_from_records(mode, kd, kn, vd, vn, 0, h, L) for h in range(Hkv)}
    sc = 1 / math.sqrt(128)
    want_full = H.oracle_decode(mode, q_np, units, [L], Hkv, Tq, sc, 1.0)
    _, bound = H.oracle_decode_sparse_v(mode, q_np, units, [L], Hkv, Tq, sc, 1.0, 2 * tau)
    got, got_full = sparse.float().cpu().numpy(), full.float().cpu().numpy()
    rms = math.sqrt(float(np.mean(want_full ** 2)))
    assert np.all(_ulp_close(got, got_full, bound, rms))
    H.assert_within_skip_bound(got, want_full, bound, mode)


def test_sparse_v_zero_threshold_is_the_plain_decode():
    mode, B, Hq, Hkv, L, cap = "turbo4", 1, 16, 4, 1234, 1248
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 77)
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, [L], kd, kn, vd, vn, DEV)
    q = H.upload(wl.random_fp16(78, (B, Hq, 1, 128)), DEV)
    a, b = torch.empty_like(q), torch.empty_like(q)
    ctx = tqf.Context()
    tqf.tq_decode_attention_sparse_v(ctx, cache, q, a, L, 0.0)
    tqf.tq_decode_attention(ctx, cache, q, b, L)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
