"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bounds (from the benchmark definition): packed indices bit-exact except
elements whose fp64 u lies within 1e-5 of a decision midpoint (fewer than
1e-4 of the elements); norms bit-exact; attention max-abs error <= 1e-2 x RMS
and RMS error <= 2e-3 x RMS of the oracle output, over the whole tensor.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import quantized_kv_cache_flash_gb300 as tqf
from quantized_kv_cache_flash_gb300 import workloads as wl
from oracle import tq_oracle as o
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


def _run_decode(cache, q_np, tq_rows, max_len, scale=0.0, ctx=None):
    ctx = ctx or tqf.Context()
    q = H.upload(q_np, DEV)
    out = torch.empty_like(q)
    tqf.tq_decode_attention(ctx, cache, q, out, max_len, scale)
    torch.cuda.synchronize()
    status = tqf.tq_get_status(ctx)
    return out.float().cpu().numpy(), status, ctx


# ---------------------------------------------------------------------------
# decode on the same packed cache (random records from the input generator)
# ---------------------------------------------------------------------------
DECODE_CASES = [
    # mode, B, Hq, Hkv, lengths, Tq, cap, scale, v_rescale
    ("turbo3", 1, 4, 1, [1], 1, 16, 0.0, 1.0),                  # context 1
    ("turbo3", 2, 8, 2, [37, 300], 1, 320, 0.0, 1.0),           # ragged, tails
    ("turbo4", 3, 12, 4, [100, 513, 1000], 2, 1024, 0.0, 1.0),  # Tq 2, G 3
    ("turbo4_asym", 1, 4, 2, [256], 1, 256, 0.0, 1.0),          # tiny Turbo4Asym shape
    ("turbo4_asym", 2, 28, 4, [2049, 700], 1, 2064, 0.0, 0.5),  # v_rescale
    ("turbo3", 1, 32, 2, [777], 4, 784, 0.0, 1.0),              # 64 rows: 4 row groups
    ("turbo4", 2, 8, 8, [5000, 1], 1, 5008, 0.0, 1.0),          # many splits + a 1-token seq
    ("turbo3", 1, 4, 1, [40], 4, 48, 0.05, 1.0),                # causal block, custom scale
    ("turbo4", 1, 16, 2, [16], 8, 16, 0.0, 1.0),                # Tq 8 x G 8 = 64 rows, L = Tq*2
    ("turbo3", 2, 28, 4, [8192, 8191], 1, 8192, 0.0, 1.0),      # Qwen2.5-7B shape, min=max-1
    ("turbo3_asym", 1, 4, 2, [256], 1, 256, 0.0, 1.0),          # fp16 K + 3-bit V
    ("turbo3_asym", 2, 28, 4, [3001, 77], 2, 3008, 0.0, 0.5),   # ragged, Tq 2, v_rescale
    ("turbo3_asym", 1, 32, 2, [900], 4, 912, 0.0, 1.0),         # 64 rows
    ("turbo4k_3v", 1, 4, 1, [1], 1, 16, 0.0, 1.0),              # 4-bit K + 3-bit V, context 1
    ("turbo4k_3v", 3, 12, 4, [100, 513, 4000], 1, 4000, 0.0, 1.0),
    ("turbo4k_3v", 1, 32, 2, [777], 4, 784, 0.05, 1.0),         # 64 rows, custom scale
    ("turbo4", 40, 8, 2, [(37 * i) % 290 + 1 for i in range(40)], 1, 304, 0.0, 1.0),  # > 32 sequences
    ("turbo3_table", 2, 8, 2, [37, 1300], 1, 1312, 0.0, 1.0),  # centroid x norm table records
    ("turbo3_table", 1, 32, 8, [2049], 4, 2064, 0.0, 0.5),     # 16 rows, causal block
    ("turbo4", 1, 4, 1, [40000], 1, 40000, 0.0, 1.0),          # > 128 partials for one row
    # one long sequence among short ones: the merge runs with 4 warps (few CTAs
    # per unit on average) but the long sequence's units have ~118 partials
    # each, merged in several passes
    ("turbo4", 8, 8, 2, [30000] + [64] * 7, 1, 30016, 0.0, 1.0),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: f"{c[0]}-B{c[1]}-Hq{c[2]}-L{max(c[4])}-Tq{c[5]}")
def test_decode_same_cache(case):
    mode, B, Hq, Hkv, lengths, Tq, cap, scale, vr = case
    key = 7000 + sum(lengths) + 31 * Hq + Tq
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, key)
    q = wl.random_fp16(key + 5, (B, Hq, Tq, 128))
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, DEV, v_rescale=vr)
    got, status, _ = _run_decode(cache, q, Tq, max(lengths), scale)
    assert status == 0
    units = {(b, h): H.oracle_unit_from_records(mode, kd, kn, vd, vn, b, h, lengths[b])
             for b in range(B) for h in range(Hkv)}
    sc = scale if scale else 1 / math.sqrt(128)
    want = H.oracle_decode(mode, q, units, lengths, Hkv, Tq, sc, vr)
    H.assert_attention_close(got, want, str(case))


# Peaked softmax: q scaled by 8 .. 32 puts the leading scores at 20 .. 100
# (natural log units), where a relative score error of 2^-11 (one fp16
# rounding of the rotated query or of a centroid) would already move the
# dominant weights by a per cent.  Every row-group size (4, 8 and 16 rows per
# KV head) and every mode, against the oracle.
SHARP_CASES = [
    # mode, B, Hq, Hkv, lengths, Tq, cap, q scale
    ("turbo4", 2, 32, 8, [3000, 1777], 1, 3008, 8.0),            # 4 rows: q_lo in the pair columns
    ("turbo4", 2, 32, 8, [3000, 1777], 1, 3008, 32.0),
    ("turbo4", 1, 8, 4, [2000], 1, 2000, 16.0),                  # 2 rows
    ("turbo3", 1, 32, 8, [2600], 4, 2608, 8.0),                  # 16 rows, causal block
    ("turbo3", 1, 32, 8, [2600], 4, 2608, 32.0),
    ("turbo3", 1, 28, 4, [4100], 1, 4112, 32.0),                 # 7 rows (8-row group)
    ("turbo4k_3v", 2, 12, 4, [700, 1500], 2, 1504, 32.0),        # 6 rows
    ("turbo4k_3v", 1, 16, 4, [1100], 1, 1104, 24.0),             # 4 rows, 3-bit V
    ("turbo4_asym", 1, 28, 4, [4100], 1, 4112, 32.0),
    ("turbo3_asym", 1, 8, 2, [900], 1, 912, 32.0),
    ("turbo3_table", 1, 32, 8, [2049], 4, 2064, 32.0),
    ("turbo3_table", 2, 8, 2, [1300, 37], 1, 1312, 16.0),
]


# Codebooks whose entries are not fp16 values (the Lloyd-Max levels rounded
# to fp32) take the decode path that adds each score's centroid rounding
# residual through an fp8 product: the same peaked cases with those.
EXACT_CB_CASES = [c for c in SHARP_CASES if c[0] in ("turbo4", "turbo3", "turbo4k_3v")]


def _peaked(case, exact_cb):
    mode, B, Hq, Hkv, lengths, Tq, cap, qs = case
    key = 8800 + sum(lengths) + Hq + int(qs)
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, key)
    q = (wl.random_fp16(key + 3, (B, Hq, Tq, 128)).astype(np.float32) * qs).astype(np.float16)
    kb, vb = H.MODE_BITS[mode]
    cbk = H.exact_lloyd_max(kb) if exact_cb and kb != 16 else None
    cbv = H.exact_lloyd_max(vb) if exact_cb else None
    if exact_cb:
        assert not np.array_equal(cbk, cbk.astype(np.float16).astype(np.float32))
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, DEV, v_rescale=0.75,
                                     codebook_k=cbk, codebook_v=cbv)
    got, status, _ = _run_decode(cache, q, Tq, max(lengths))
    assert status == 0
    units = {(b, h): H.oracle_unit_from_records(mode, kd, kn, vd, vn, b, h, lengths[b])
             for b in range(B) for h in range(Hkv)}
    want = H.oracle_decode(mode, q, units, lengths, Hkv, Tq, 1 / math.sqrt(128), 0.75, cbk=cbk, cbv=cbv)
    H.assert_attention_close(got, want, f"{case} exact codebook {exact_cb}")


@pytest.mark.parametrize("case", SHARP_CASES, ids=lambda c: f"{c[0]}-Hq{c[2]}-Tq{c[5]}-q{c[7]:g}")
def test_decode_peaked_softmax(case):
    _peaked(case, False)


@pytest.mark.parametrize("case", EXACT_CB_CASES, ids=lambda c: f"{c[0]}-Hq{c[2]}-Tq{c[5]}-q{c[7]:g}")
def test_decode_peaked_softmax_fp32_codebook(case):
    _peaked(case, True)


@pytest.mark.parametrize("mode,B,Hq,Hkv,L,Tq,qs", [
    ("turbo4", 2, 32, 8, 1500, 1, 8.0), ("turbo4", 2, 32, 8, 1500, 1, 32.0),
    ("turbo3", 1, 32, 8, 1200, 4, 32.0), ("turbo3", 1, 28, 4, 2000, 1, 16.0),
    ("turbo4_asym", 1, 28, 4, 2000, 1, 32.0),
])
def test_end_to_end_peaked_softmax(mode, B, Hq, Hkv, L, Tq, qs):
    """Gaussian K with outlier channels and V, encoded by each side, queries
    scaled up: the encoded-cache path of the same regime."""
    _e2e(mode, B, Hq, Hkv, L, Tq, (L + 15) // 16 * 16, 600 + L + int(qs), q_scale=qs)


@pytest.mark.parametrize("mode,Hq,Tq,scale_v", [("turbo4", 8, 1, 1000.0), ("turbo3", 32, 1, 3000.0),
                                               ("turbo4k_3v", 8, 2, 1000.0), ("turbo4_asym", 4, 1, 2000.0)])
def test_decode_large_v_norms(mode, Hq, Tq, scale_v):
    # V norms ~ 6e3..5e4: p * n_v would overflow fp16 for p up to 16, so these
    # chunks scale the dequantised V values instead; chunk 0 of the second
    # sequence keeps ordinary norms (both paths in one launch)
    B, Hkv, cap = 2, 2, 3008
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 321)
    vn = (vn.astype(np.float32) * scale_v).astype(np.float16)
    vn[1, :, :32] = (vn[1, :, :32].astype(np.float32) / scale_v).astype(np.float16)
    assert np.isfinite(vn).all()
    q = wl.random_fp16(322, (B, Hq, Tq, 128))
    lengths = [3000, 1700]
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, DEV)
    got, status, _ = _run_decode(cache, q, Tq, 3000)
    assert status == 0
    units = {(b, h): H.oracle_unit_from_records(mode, kd, kn, vd, vn, b, h, lengths[b])
             for b in range(B) for h in range(Hkv)}
    want = H.oracle_decode(mode, q, units, lengths, Hkv, Tq, 1 / math.sqrt(128), 1.0)
    H.assert_attention_close(got, want, mode)


def test_decode_short_context_rows_are_zero_and_flagged():
    # lengths 2 with a 4-query block: rows j = 0, 1 see no token
    mode, B, Hq, Hkv, cap = "turbo3", 1, 2, 1, 16
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 99)
    q = wl.random_fp16(100, (B, Hq, 4, 128))
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, [2], kd, kn, vd, vn, DEV)
    got, status, _ = _run_decode(cache, q, 4, 16)
    assert status & tqf.TQ_STATUS_SHORT_CONTEXT
    assert np.all(got[:, :, :2] == 0)
    units = {(0, 0): H.oracle_unit_from_records(mode, kd, kn, vd, vn, 0, 0, 2)}
    want = H.oracle_decode(mode, q, units, [2], Hkv, 4, 1 / math.sqrt(128), 1.0)
    H.assert_attention_close(got[:, :, 2:], want[:, :, 2:])


def test_decode_empty_sequences_in_a_large_batch():
    # 45 sequences, some of length 0: their rows are 0 and flagged, the rest exact
    mode, B, Hq, Hkv, cap = "turbo3", 45, 4, 1, 96
    lengths = [0 if i % 7 == 3 else (11 * i) % 96 + 1 for i in range(B)]
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 123)
    q = wl.random_fp16(124, (B, Hq, 1, 128))
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, DEV)
    got, status, _ = _run_decode(cache, q, 1, cap)
    assert status & tqf.TQ_STATUS_SHORT_CONTEXT
    live = [b for b in range(B) if lengths[b] > 0]
    assert np.all(got[[b for b in range(B) if lengths[b] == 0]] == 0)
    units = {(b, 0): H.oracle_unit_from_records(mode, kd, kn, vd, vn, b, 0, lengths[b]) for b in live}
    want = H.oracle_decode(mode, q, units, lengths, Hkv, 1, 1 / math.sqrt(128), 1.0)
    H.assert_attention_close(got[live], want[live])


def test_decode_hint_far_above_lengths():
    # the grid is planned for 4096 tokens per sequence but the sequences hold
    # 5..70: most CTAs get no chunk, units span CTAs with empty shares
    mode, B, Hq, Hkv, cap = "turbo4", 3, 8, 2, 4096
    lengths = [5, 70, 33]
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 321)
    q = wl.random_fp16(322, (B, Hq, 1, 128))
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, DEV)
    ctx = tqf.Context()
    for _ in range(3):   # repeated calls reuse the arrival counters
        got, status, _ = _run_decode(cache, q, 1, cap, ctx=ctx)
        assert status == 0
        units = {(b, h): H.oracle_unit_from_records(mode, kd, kn, vd, vn, b, h, lengths[b])
                 for b in range(B) for h in range(Hkv)}
        want = H.oracle_decode(mode, q, units, lengths, Hkv, 1, 1 / math.sqrt(128), 1.0)
        H.assert_attention_close(got, want)


def test_decode_lengths_beyond_hint_are_clamped():
    # tokens past max_len_hint are not read: equals the oracle on the first 64
    mode = "turbo4"
    kd, kn, vd, vn = H.random_cache(mode, 1, 1, 128, 55)
    q = wl.random_fp16(56, (1, 2, 1, 128))
    cache = H.gpu_cache_from_records(mode, 1, 1, 128, [100], kd, kn, vd, vn, DEV)
    got, _, _ = _run_decode(cache, q, 1, 64)
    units = {(0, 0): H.oracle_unit_from_records(mode, kd, kn, vd, vn, 0, 0, 64)}
    # causal position is the true length (100) but only 64 tokens are visible
    want = H.oracle_decode(mode, q, units, [64], 1, 1, 1 / math.sqrt(128), 1.0)
    H.assert_attention_close(got, want)


# ---------------------------------------------------------------------------
# encode / append: bit-exact codes and norms
# ---------------------------------------------------------------------------
def _crafted_vectors():
    v = [np.zeros(128, np.float16)]
    x = np.zeros(128, np.float16); x[:3] = [2048, 64, 1]; v.append(x)         # norm tie -> even
    x = np.zeros(128, np.float16); x[:4] = [2050, 64, 2, 1]; v.append(x)      # norm tie -> up
    x = np.zeros(128, np.float16); x[0] = 1.0; v.append(x)                    # basis vector
    x = np.zeros(128, np.float16); x[5] = -3.0; x[77] = 3.0; v.append(x)      # exact zeros in u
    v.append(np.full(128, 5000, np.float16))                                  # norm 56568
    v.append(np.full(128, 6e-8, np.float16))                                  # subnormals
    v.append(np.full(128, -65504, np.float16))                                # overflow (inf norm)
    v.append(np.linspace(-8, 8, 128).astype(np.float16))
    return np.stack(v)


# T = 300 runs the warp-per-vector kernel (small appends), T = 700 and 1029
# the tensor-core kernel (more than 4096 vectors per stream; 1029 leaves a
# ragged last tile of vectors)
@pytest.mark.parametrize("T", [300, 700, 1029])
@pytest.mark.parametrize("mode", ["turbo3", "turbo4", "turbo4_asym", "turbo3_asym", "turbo4k_3v",
                                  "turbo3_table"])
def test_encode_append_bit_exact(mode, T):
    kb, vb = H.MODE_BITS[mode]
    B, Hkv = 2, 3
    cap = (T + 5 + 15) // 16 * 16
    rng = np.random.default_rng(3)
    k = wl.random_fp16(11, (B, Hkv, T, 128))
    v = wl.random_fp16(12, (B, Hkv, T, 128), scale=3.0)
    crafted = _crafted_vectors()
    k[0, 0, :len(crafted)] = crafted
    v[1, 2, :len(crafted)] = crafted
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.MODES[mode], B, Hkv, cap, DEV)
    cache.lengths.copy_(torch.tensor([5, 0], dtype=torch.int32))
    tqf.tq_encode_append(ctx, cache, H.upload(k, DEV), H.upload(v, DEV))
    torch.cuda.synchronize()
    status = tqf.tq_get_status(ctx)
    assert status == tqf.TQ_STATUS_NORM_OVERFLOW          # the -65504 vectors
    assert cache.lengths.cpu().tolist() == [5 + T, T]
    s = o.sign_vector(42)
    total = near = bad = 0
    for which, bits, x, data, norm in (("k", kb, k, cache.k_data, cache.k_norm),
                                       ("v", vb, v, cache.v_data, cache.v_norm)):
        for b, L0 in ((0, 5), (1, 0)):
            got_rec = data[b, :, L0:L0 + T].cpu().numpy()
            if bits == 16:
                assert np.array_equal(got_rec.view(np.float16), x[b])
                continue
            idx, n16, u, ov = o.encode(x[b], o.codebook(bits), s)
            if mode in H.TABLE_MODES:
                # the record's table replaces the norm: bit-exact fp16 c_j * n16
                want_t = o.centroid_norm_table(n16, o.codebook(bits))
                got_t = np.ascontiguousarray(got_rec[..., 48:64]).view("<u2")
                assert np.array_equal(got_t, want_t.view(np.uint16)), (which, b)
                got_rec = np.ascontiguousarray(got_rec[..., :48])
            else:
                got_n = norm[b, :, L0:L0 + T].cpu().numpy()
                assert np.array_equal(got_n.view(np.uint16), n16.view(np.uint16)), (which, b)
            got_idx = H.decode_records(got_rec, bits)
            dist = o.boundary_distance(u, o.codebook(bits))
            finite = ~ov[..., None] & np.ones_like(got_idx, bool)
            diff = (got_idx != idx) & finite
            total += int(finite.sum())
            near += int((diff & (dist < H.BOUNDARY)).sum())
            bad += int((diff & (dist >= H.BOUNDARY)).sum())
            # records with no element near a midpoint must match the oracle's bytes
            clean = ~np.any(dist < H.BOUNDARY, axis=-1) & ~ov
            want_rec = o.pack_codes(idx, bits)
            assert np.array_equal(got_rec[clean], want_rec[clean]), (which, b)
    assert bad == 0
    assert near <= max(1, H.BOUNDARY_FRACTION * total), (near, total)


def test_encode_capacity_overflow_is_flagged_and_skipped():
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.TQ_TURBO3, 2, 1, 16, DEV)
    cache.lengths.copy_(torch.tensor([10, 2], dtype=torch.int32))
    k = H.upload(wl.random_fp16(1, (2, 1, 8, 128)), DEV)
    tqf.tq_encode_append(ctx, cache, k, k)
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == tqf.TQ_STATUS_CAPACITY
    assert cache.lengths.cpu().tolist() == [10, 10]
    assert not cache.k_data[0].any().item()              # sequence 0 untouched


# A large append whose tiles do not fill the grid's last pass: 1 x 8 x 5664
# vectors per stream = 354 tiles of K and 354 of V, on 304 CTAs of two encode
# groups (608 groups), so 100 tiles are left for the groups that finish their
# first pass first.  Every record checked.
@pytest.mark.parametrize("mode", ["turbo3", "turbo4", "turbo4k_3v"])
def test_encode_large_append_partial_last_pass(mode):
    kb, vb = H.MODE_BITS[mode]
    B, Hkv, T = 1, 8, 5664
    cap = T + 16
    assert 2 * (B * Hkv * T // 128) % 608 == 100
    k = wl.random_fp16(41, (B, Hkv, T, 128))
    v = wl.random_fp16(42, (B, Hkv, T, 128), scale=2.0)
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.MODES[mode], B, Hkv, cap, DEV)
    tqf.tq_encode_append(ctx, cache, H.upload(k, DEV), H.upload(v, DEV))
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == 0
    assert cache.lengths.cpu().tolist() == [T]
    s = o.sign_vector(42)
    for which, bits, x, data, norm in (("k", kb, k, cache.k_data, cache.k_norm),
                                       ("v", vb, v, cache.v_data, cache.v_norm)):
        idx, n16, u, ov = o.encode(x[0], o.codebook(bits), s)
        assert not ov.any()
        got_n = norm[0, :, :T].cpu().numpy()
        assert np.array_equal(got_n.view(np.uint16), n16.view(np.uint16)), which
        got_idx = H.decode_records(data[0, :, :T].cpu().numpy(), bits)
        dist = o.boundary_distance(u, o.codebook(bits))
        diff = got_idx != idx
        assert not (diff & (dist >= H.BOUNDARY)).any(), which
        assert diff.sum() < 1e-4 * diff.size, which


@pytest.mark.parametrize("mode", ["turbo3", "turbo4_asym", "turbo4k_3v"])
def test_encode_large_append_capacity_overflow(mode):
    """The tensor-core encode (4800 vectors per stream): the sequence that
    would overflow is flagged and left untouched, the other is encoded."""
    kb, vb = H.MODE_BITS[mode]
    B, Hkv, T, cap = 2, 8, 300, 400
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.MODES[mode], B, Hkv, cap, DEV)
    cache.lengths.copy_(torch.tensor([10, 200], dtype=torch.int32))
    k = wl.random_fp16(21, (B, Hkv, T, 128))
    v = wl.random_fp16(22, (B, Hkv, T, 128))
    tqf.tq_encode_append(ctx, cache, H.upload(k, DEV), H.upload(v, DEV))
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == tqf.TQ_STATUS_CAPACITY
    assert cache.lengths.cpu().tolist() == [10 + T, 200]
    assert not cache.v_data[1].any().item()              # sequence 1 untouched
    assert not cache.k_data[1].any().item()
    # sequence 0: the oracle's codes (but the boundary band)
    s = o.sign_vector(42)
    got = H.decode_records(cache.v_data[0, :, 10:10 + T].cpu().numpy(), vb)
    idx, n16, u, _ = o.encode(v[0], o.codebook(vb), s)
    diff = got != idx
    assert np.all(o.boundary_distance(u[diff], o.codebook(vb)) < H.BOUNDARY)
    assert np.array_equal(cache.v_norm[0, :, 10:10 + T].cpu().numpy().view(np.uint16), n16.view(np.uint16))
    if kb == 16:
        assert np.array_equal(cache.k_data[0, :, 10:10 + T].cpu().numpy().view(np.float16), k[0])


# ---------------------------------------------------------------------------
# end to end: each side encodes on its own, then decodes
# ---------------------------------------------------------------------------
def _e2e(mode, B, Hq, Hkv, L, Tq, cap, outliers_key, q_scale=1.0):
    w = wl.Workload(0, "test", mode, B, Hq, Hkv, L, tq=Tq)
    k = np.stack([np.stack([wl.random_fp16(outliers_key + 10 * b + h, (L, 128))
                            for h in range(Hkv)]) for b in range(B)])
    k[..., [3, 50, 77, 120]] = (k[..., [3, 50, 77, 120]].astype(np.float32) * 8).astype(np.float16)
    v = np.stack([np.stack([wl.random_fp16(outliers_key + 1000 + 10 * b + h, (L, 128))
                            for h in range(Hkv)]) for b in range(B)])
    q = wl.random_fp16(outliers_key + 77, (B, Hq, Tq, 128), scale=q_scale)
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.MODES[mode], B, Hkv, cap, DEV)
    tqf.tq_encode_append(ctx, cache, H.upload(k, DEV), H.upload(v, DEV))
    got, status, _ = _run_decode(cache, q, Tq, L, ctx=ctx)
    assert status == 0
    kb, vb = H.MODE_BITS[mode]
    s = o.sign_vector(42)
    units = {}
    for b in range(B):
        for h in range(Hkv):
            vi, vn, _, _ = o.encode(v[b, h], o.codebook(vb), s)
            u = {"v_idx": vi, "v_norm": vn}
            if mode in H.TABLE_MODES:
                ki, kn, _, _ = o.encode(k[b, h], o.codebook(kb), s)
                u = {"k_idx": ki, "k_table": o.centroid_norm_table(kn, o.codebook(kb)),
                     "v_idx": vi, "v_table": o.centroid_norm_table(vn, o.codebook(vb))}
            elif kb == 16:
                u["k"] = k[b, h]
            else:
                ki, kn, _, _ = o.encode(k[b, h], o.codebook(kb), s)
                u["k_idx"], u["k_norm"] = ki, kn
            units[(b, h)] = u
    want = H.oracle_decode(mode, q, units, [L] * B, Hkv, Tq, 1 / math.sqrt(128), 1.0)
    return H.assert_attention_close(got, want, f"e2e {mode}")


@pytest.mark.parametrize("mode,B,Hq,Hkv,L,Tq,cap", [
    ("turbo4_asym", 1, 4, 2, 256, 1, 256),
    ("turbo3", 1, 28, 4, 1000, 1, 1024),
    ("turbo4", 2, 32, 8, 700, 1, 704),
    ("turbo3", 1, 32, 8, 600, 4, 608),
    ("turbo3_asym", 1, 28, 4, 900, 1, 912),
    ("turbo4k_3v", 2, 32, 8, 500, 2, 512),
    ("turbo3_table", 1, 28, 4, 700, 1, 704),
])
def test_end_to_end_own_encodings(mode, B, Hq, Hkv, L, Tq, cap):
    _e2e(mode, B, Hq, Hkv, L, Tq, cap, 400 + L)


def test_multistep_append_decode_lockstep():
    """16 append+decode steps on the tiny Turbo4Asym shape (GQA 4/2), as in the
    mlxcel parity test: the lengths stay in lockstep and every step is within
    the bounds."""
    w = wl.by_number(1)
    B, Hq, Hkv, cap = w.batch, w.num_q_heads, w.num_kv_heads, 272
    L0 = 240
    s = o.sign_vector(w.rot_seed)
    cbv = o.codebook(4)
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.TQ_TURBO4_ASYM, B, Hkv, cap, DEV)
    oc = {"mode": "turbo4_asym", "capacity": cap, "lengths": np.zeros(B, np.int32),
          "k": np.zeros((B, Hkv, cap, 128), np.float16),
          "v_data": np.zeros((B, Hkv, cap, 64), np.uint8),
          "v_norm": np.zeros((B, Hkv, cap), np.float16)}
    kall = np.stack([wl.keys(w, 0, h, 0, L0 + 16) for h in range(Hkv)])[None]
    vall = np.stack([wl.values(w, 0, h, 0, L0 + 16) for h in range(Hkv)])[None]
    tqf.tq_encode_append(ctx, cache, H.upload(kall[:, :, :L0], DEV), H.upload(vall[:, :, :L0], DEV))
    o.encode_append(oc, kall[:, :, :L0], vall[:, :, :L0], None, cbv, s)
    for step in range(16):
        kn = np.ascontiguousarray(kall[:, :, L0 + step:L0 + step + 1])
        vn = np.ascontiguousarray(vall[:, :, L0 + step:L0 + step + 1])
        tqf.tq_encode_append(ctx, cache, H.upload(kn, DEV), H.upload(vn, DEV))
        o.encode_append(oc, kn, vn, None, cbv, s)
        L = int(oc["lengths"][0])
        assert cache.lengths.cpu().tolist() == oc["lengths"].tolist()
        q = wl.random_fp16(5000 + step, (B, Hq, 1, 128))
        got, status, _ = _run_decode(cache, q, 1, L, ctx=ctx)
        assert status == 0
        units = {(0, h): {"k": oc["k"][0, h, :L], "v_idx": o.unpack_codes(oc["v_data"][0, h, :L], 4),
                          "v_norm": oc["v_norm"][0, h, :L]} for h in range(Hkv)}
        want = H.oracle_decode("turbo4_asym", q, units, [L], Hkv, 1, 1 / math.sqrt(128), 1.0)
        H.assert_attention_close(got, want, f"step {step}")
