"""Pins for the fp64 oracle against facts fixed outside of it (CPU only).

Each test checks the oracle against something it does not compute itself:
published test vectors, a textbook table, closed forms, a library routine,
brute force over small inputs, or an algebraic identity.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import torch

from oracle import tq_oracle as o


# --------------------------------------------------------------------------
# sign vector
# --------------------------------------------------------------------------
def test_splitmix64_published_vectors(golden_dir):
    rows = [l.split() for l in open(os.path.join(golden_dir, "splitmix64.txt"))
            if l.strip() and not l.startswith("#")]
    for seed, i, val in rows:
        assert o.splitmix64(int(seed), int(i) + 1)[int(i)] == int(val)


def test_sign_vector_is_top_bit():
    s = o.sign_vector(0, 4)
    # top bits of the seed-0 outputs: e220..., 6e78..., 06c4..., f88b...
    assert list(s) == [-1.0, 1.0, 1.0, -1.0]
    s42 = o.sign_vector(42)
    assert s42.shape == (128,) and set(np.unique(s42)) <= {-1.0, 1.0}
    # roughly balanced (a fixed seed: 128 fair bits)
    assert 40 < np.sum(s42 > 0) < 88


# --------------------------------------------------------------------------
# rotation
# --------------------------------------------------------------------------
def test_hadamard_matches_scipy_sylvester():
    for d in (2, 8, 128):
        assert np.array_equal(o.hadamard(d), scipy.linalg.hadamard(d).astype(np.float64))


def test_hadamard_orthogonality_exact():
    H = o.hadamard(128)
    assert np.array_equal(H @ H.T, 128.0 * np.eye(128))


def test_normalised_hadamard_involution():
    Hn = o.hadamard(128) / math.sqrt(128)
    assert np.max(np.abs(Hn @ Hn - np.eye(128))) < 1e-14


def test_rotation_inverse_and_norm():
    rng = np.random.default_rng(0)
    s = o.sign_vector(42)
    x = rng.standard_normal((50, 128))
    y = o.rotate(x, s)
    assert np.max(np.abs(o.rotate_inv(y, s) - x)) < 1e-12
    assert np.max(np.abs(np.linalg.norm(y, axis=1) - np.linalg.norm(x, axis=1))) < 1e-12
    # Rot is linear and orthogonal: inner products preserved
    assert abs(float(y[0] @ y[1]) - float(x[0] @ x[1])) < 1e-12


def test_rotation_closed_forms():
    ones = np.ones(128)
    e0 = np.zeros(128); e0[0] = 1.0
    # with no sign flips, Rot(e_0) is the constant vector 1/sqrt(128)
    assert np.max(np.abs(o.rotate(e0, ones) - 1 / math.sqrt(128))) < 1e-15
    # Rot(e_k) = s_k * (column k of H) / sqrt(128)
    s = o.sign_vector(7)
    H = scipy.linalg.hadamard(128)
    for k in (0, 5, 127):
        ek = np.zeros(128); ek[k] = 1.0
        assert np.max(np.abs(o.rotate(ek, s) - s[k] * H[:, k] / math.sqrt(128))) < 1e-15
    # Rot^-1 applies the signs after the transform: Rot^-1(e_0) = s / sqrt(128)
    assert np.max(np.abs(o.rotate_inv(e0, s) - s / math.sqrt(128))) < 1e-15


# --------------------------------------------------------------------------
# codebook
# --------------------------------------------------------------------------
def test_lloyd_max_two_levels_closed_form():
    # the 1-bit optimum for N(0, s^2) is +-s*sqrt(2/pi) (the half-normal mean)
    c, _, _ = o.lloyd_max(2)
    sig = 1 / math.sqrt(128)
    assert np.max(np.abs(c - np.array([-1, 1]) * sig * math.sqrt(2 / math.pi))) < 1e-15


@pytest.mark.parametrize("levels", [4, 8, 16])
def test_lloyd_max_fixed_point_and_symmetry(levels):
    c, it, delta = o.lloyd_max(levels)
    assert delta < 1e-15
    assert np.all(np.diff(c) > 0)
    assert np.max(np.abs(c + c[::-1])) < 1e-15
    c32 = o.codebook(int(math.log2(levels)))
    assert np.array_equal(c32, -c32[::-1])        # exactly symmetric after rounding


@pytest.mark.parametrize("levels", [4, 8, 16])
def test_lloyd_max_centroid_condition_by_quadrature(levels):
    # each level is the conditional mean of its cell, integrated numerically
    c, _, _ = o.lloyd_max(levels, sigma=1.0)
    t = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
    pdf = lambda x: math.exp(-x * x / 2) / math.sqrt(2 * math.pi)
    for j in range(levels):
        m = scipy.integrate.quad(lambda x: x * pdf(x), t[j], t[j + 1], epsabs=1e-14)[0]
        p = scipy.integrate.quad(pdf, t[j], t[j + 1], epsabs=1e-14)[0]
        assert abs(m / p - c[j]) < 1e-9


def test_lloyd_max_matches_max_1960_table(golden_dir):
    pdf = lambda x: math.exp(-x * x / 2) / math.sqrt(2 * math.pi)
    for line in open(os.path.join(golden_dir, "lloyd_max_gaussian_max1960.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        n, mse, lv = int(f[0]), float(f[1]), np.array([float(v) for v in f[2:]])
        c, _, _ = o.lloyd_max(n, sigma=1.0)
        # four significant digits as printed, plus one unit of slack in the last
        assert np.all(np.abs(c[n // 2:] - lv) <= 5e-4 * lv + 1e-4)
        t = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
        d = sum(scipy.integrate.quad(lambda x: (x - c[j]) ** 2 * pdf(x), t[j], t[j + 1])[0]
                for j in range(n))
        assert abs(d - mse) < 1e-3 * mse     # four printed digits, last one loose


def test_codebook_is_scaled_unit_gaussian_quantiser():
    for bits in (3, 4):
        c1, _, _ = o.lloyd_max(1 << bits, sigma=1.0)
        c64, _, _ = o.lloyd_max(1 << bits)
        assert np.max(np.abs(c64 * math.sqrt(128) - c1)) < 1e-12


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_levels_are_the_nearest_fp16_values(bits):
    """Each standard level is the fp16 value nearest the fp64 Lloyd-Max level,
    found by exact rational comparison against every finite fp16 value of the
    same sign (ties would go to the even one: there are none here)."""
    c64, _, _ = o.lloyd_max(1 << bits)
    cb = o.codebook(bits)
    assert cb.dtype == np.float32
    allf = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    for x, got in zip(c64, cb):
        a = Fraction(abs(float(x)))
        near = [i for i in range(len(allf)) if a / 2 <= allf[i] <= 2 * a]
        d = {i: abs(Fraction(allf[i]) - a) for i in near}
        best = min(near, key=lambda i: (d[i], i % 2))   # bit pattern i: even = even mantissa
        assert sorted(d.values())[0] < sorted(d.values())[1]   # no tie
        assert float(got) == math.copysign(allf[best], x)
    # the rounding moves each level by at most 2^-11 of itself (half an fp16 ulp)
    assert np.all(np.abs(cb - c64) <= 2.0 ** -11 * np.abs(c64))


# --------------------------------------------------------------------------
# encode: norm, nearest centroid, packing
# --------------------------------------------------------------------------
def _sqrt_fraction_rne(S: int) -> float:
    """Brute-force reference: fp16 RNE of sqrt(S) * 2^-24 by exact rational bisection."""
    if S == 0:
        return 0.0
    # the fp16 candidate is the nearest grid point; compare squares exactly
    allf = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    target2 = Fraction(S, 2 ** 48)
    if target2 >= Fraction(65520) ** 2:
        return math.inf
    lo, hi = 0, len(allf) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if Fraction(allf[mid]) ** 2 <= target2:
            lo = mid
        else:
            hi = mid
    if Fraction(allf[hi]) ** 2 <= target2:
        lo = hi
        if lo == len(allf) - 1:
            m = (Fraction(allf[lo]) + 65536) / 2
            return float(allf[lo]) if target2 < m * m else math.inf
        hi = lo + 1
    m = (Fraction(allf[lo]) + Fraction(allf[hi])) / 2
    if target2 < m * m:
        return float(allf[lo])
    if target2 > m * m:
        return float(allf[hi])
    return float(allf[lo]) if lo % 2 == 0 else float(allf[hi])


def test_fp16_norm_closed_forms_and_ties():
    assert float(o.fp16_norm(np.array([3, 4], np.float16))) == 5.0
    # 2048^2 + 64^2 + 1^2 = 2049^2: exactly the midpoint of 2048 and 2050 -> even (2048)
    assert float(o.fp16_norm(np.array([2048, 64, 1], np.float16))) == 2048.0
    # 2050^2 + 64^2 + 2^2 ... check a tie that goes up: 2051^2 = 2050^2 + 4101
    # (2051 is the midpoint of 2050 and 2052; 2050 has an odd mantissa -> 2052)
    x = np.zeros(128, np.float16); x[0] = 2050; x[1] = 64; x[2] = 2; x[3] = 1
    # 2050^2 + 64^2 + 2^2 + 1 = 4202500 + 4096 + 4 + 1 = 4206601 = 2051^2
    assert 2050 ** 2 + 64 ** 2 + 4 + 1 == 2051 ** 2
    assert float(o.fp16_norm(x)) == 2052.0
    assert float(o.fp16_norm(np.zeros(128, np.float16))) == 0.0
    assert math.isinf(float(o.fp16_norm(np.full(128, 6000, np.float16))))
    # smallest subnormal: norm 2^-24
    assert float(o.fp16_norm(np.array([2.0 ** -24], np.float16))) == 2.0 ** -24


def test_fp16_norm_matches_bruteforce_rounding():
    rng = np.random.default_rng(1)
    cases = [rng.standard_normal(128).astype(np.float16) for _ in range(40)]
    cases += [(rng.standard_normal(128) * 1e-3).astype(np.float16) for _ in range(10)]
    cases += [(rng.standard_normal(128) * 3000).astype(np.float16) for _ in range(10)]
    cases += [(rng.standard_normal(128) * 1e-6).astype(np.float16) for _ in range(5)]
    for x in cases:
        S = sum(int(Fraction(float(v)) * 2 ** 24) ** 2 for v in x)
        assert float(o.fp16_norm(x)) == _sqrt_fraction_rne(S)


def _argmin_exact(u: float, cb32: np.ndarray) -> int:
    """Nearest codebook entry by exact rational distances, ties to the lower index."""
    uf = Fraction(float(u))
    d = [abs(uf - Fraction(float(c))) for c in cb32]
    return min(range(len(d)), key=lambda j: (d[j], j))


@pytest.mark.parametrize("bits", [3, 4])
def test_nearest_index_bruteforce_near_every_threshold(bits):
    cb = o.codebook(bits)
    us = [0.0, -0.0, 1e-30, -1e-30, 0.5, -0.5, 10.0, -10.0]
    c = cb.astype(np.float64)
    for j in range(len(cb) - 1):
        mid = np.float32(0.5 * (c[j] + c[j + 1]))
        v = mid
        for _ in range(6):
            v = np.nextafter(v, np.float32(-np.inf))
        for _ in range(13):
            us.append(float(v))
            v = np.nextafter(v, np.float32(np.inf))
    rng = np.random.default_rng(3)
    us += list((rng.standard_normal(300) * 0.1).astype(np.float32))
    u32 = np.array(us, np.float32)
    got = o.nearest_index(u32, cb)
    for u, g in zip(u32, got):
        assert int(g) == _argmin_exact(u, cb), u


def _boundary_distance_exact(u: float, cb32: np.ndarray) -> Fraction:
    """Distance from u to the nearest decision midpoint (c_j + c_{j+1}) / 2,
    in exact rationals over the fp64 value of u and the fp32 levels."""
    uf = Fraction(float(u))
    cs = [Fraction(float(c)) for c in cb32]
    return min(abs(uf - (cs[j] + cs[j + 1]) / 2) for j in range(len(cs) - 1))


@pytest.mark.parametrize("bits", [3, 4])
def test_boundary_distance_bruteforce_and_closed_forms(bits):
    """The distance that exempts encode mismatches near a decision boundary.

    Pinned by exact rational brute force over fp64 u values placed a few fp64
    steps and a few fp32 steps around every midpoint (so taking the distance
    from the fp32-rounded u, or from the levels instead of the midpoints,
    fails), at every level and far outside the codebook."""
    cb = o.codebook(bits)
    c = [Fraction(float(x)) for x in cb]
    us = []
    for j in range(len(cb) - 1):
        mid = float((c[j] + c[j + 1]) / 2)
        assert Fraction(mid) == (c[j] + c[j + 1]) / 2     # fp64 holds the midpoint exactly
        for k in (-3, -1, 0, 1, 2):
            us.append(mid + k * 2.0 ** -52 * abs(mid))      # fp64 steps: far below fp32 resolution
            us.append(float(np.float32(mid)) + k * float(np.spacing(np.float32(mid))))
        us.append(mid + 3e-6)
        us.append(mid - 7e-6)
    us += [float(x) for x in cb] + [0.0, -0.0, 5.0, -5.0]
    rng = np.random.default_rng(bits + 40)
    us += list(rng.standard_normal(200) * 0.12)
    u = np.array(us, np.float64)
    got = o.boundary_distance(u, cb)
    for ui, g in zip(us, got):
        want = _boundary_distance_exact(ui, cb)
        assert abs(Fraction(float(g)) - want) <= Fraction(2.0 ** -50) * (abs(Fraction(ui)) + 1), ui
    # closed forms: a midpoint is at distance 0, a level at half the gap to its
    # nearer neighbour, and a value beyond the codebook at its distance to the
    # outermost midpoint
    for j in range(len(cb) - 1):
        mid = float((c[j] + c[j + 1]) / 2)
        assert o.boundary_distance(np.array([mid]), cb)[0] == 0.0
    for j in range(len(cb)):
        gaps = [c[j] - c[j - 1]] if j > 0 else []
        gaps += [c[j + 1] - c[j]] if j + 1 < len(cb) else []
        assert math.isclose(o.boundary_distance(np.array([float(c[j])]), cb)[0],
                            float(min(gaps) / 2), rel_tol=1e-14)
    top_mid = (c[-2] + c[-1]) / 2
    assert math.isclose(o.boundary_distance(np.array([5.0]), cb)[0], float(5 - top_mid),
                        rel_tol=1e-14)
    # an element 1e-12 past a midpoint (the same fp32 value as the midpoint)
    # is 1e-12 from it, not 0
    mid0 = float((c[0] + c[1]) / 2)
    assert math.isclose(o.boundary_distance(np.array([mid0 + 1e-12]), cb)[0], 1e-12, rel_tol=1e-3)


def test_zero_vector_encodes_to_lower_middle_index():
    for bits in (3, 4):
        idx, n16, _, ov = o.encode(np.zeros((2, 128), np.float16), o.codebook(bits),
                                   o.sign_vector(42))
        assert float(n16[0]) == 0.0 and not ov.any()
        assert np.all(idx == (1 << (bits - 1)) - 1)


def test_encode_basis_vector_closed_form():
    # x = e_0: n = 1, u = Rot(e_0) = s_0/sqrt(128) everywhere = +-0.0884; for 3 bits
    # the nearest levels are +-0.0668 (rank 1, between the 0.0442 and 0.0928 midpoints)
    s = o.sign_vector(42)
    x = np.zeros((1, 128), np.float16); x[0, 0] = 1.0
    cb = o.codebook(3)
    idx, n16, u, _ = o.encode(x, cb, s)
    assert float(n16[0]) == 1.0
    assert np.allclose(u[0], s[0] / math.sqrt(128))
    want = 5 if s[0] > 0 else 2
    assert np.all(idx[0] == want)


@pytest.mark.parametrize("bits", [3, 4])
def test_pack_roundtrip(bits):
    rng = np.random.default_rng(bits)
    idx = rng.integers(0, 1 << bits, size=(37, 128)).astype(np.uint8)
    p = o.pack_codes(idx, bits)
    assert p.shape == (37, 16 * bits) and p.dtype == np.uint8
    assert np.array_equal(o.unpack_codes(p, bits), idx)


def test_code_mapping_sign_magnitude():
    # 3 bits: ascending 0..7 = -m3,-m2,-m1,-m0,+m0,+m1,+m2,+m3
    assert list(o.to_code(np.arange(8), 3)) == [7, 6, 5, 4, 0, 1, 2, 3]
    assert list(o.to_code(np.arange(16), 4)) == [15, 14, 13, 12, 11, 10, 9, 8,
                                                  0, 1, 2, 3, 4, 5, 6, 7]


def test_pack_hand_computed_bytes():
    # 3-bit, every index 3 (-m0): code 4 = 0b100 in every nibble -> words 0 and 1
    # are 0x44444444; word 2 also carries bit 2 of the dims-24..31 codes -> 0xCCCCCCCC
    idx = np.full((1, 128), 3, np.uint8)
    p = o.pack_codes(idx, 3)[0]
    want = bytes([0x44] * 4 + [0x44] * 4 + [0xCC] * 4) * 4
    assert bytes(p) == want
    # 3-bit one-hots on a background of index 4 (+m0, code 0):
    idx = np.full((1, 128), 4, np.uint8)
    idx[0, 25] = 7   # +m3, code 3 -> spare bit of nibble 1 (bit 7) in words 0 and 1
    idx[0, 42] = 0   # -m3, code 7 -> quarter 1, word 1, nibble 2 -> byte 16+4+1 = 0x07
    p = o.pack_codes(idx, 3)[0]
    want = bytearray(48)
    want[0] = 0x80; want[4] = 0x80; want[17] = 0x07
    assert bytes(p) == bytes(want)
    # 4-bit, background index 8 (+m0: sign 0, rank 0).  dim 5 = index 15 (+m7):
    # rank 7 in bits 20-22 -> byte 2 = 0x70.  dim 6 = index 0 (-m7): rank 7 in
    # bits 24-26 -> byte 3 = 0x07, sign at bit 8*2+3 = 19 -> byte 2 |= 0x08.
    # dim 1 = index 7 (-m0): rank 0, sign at bit 8*1+7 = 15 -> byte 1 = 0x80.
    # dim 8 (word 1) = index 9 (+m1): rank 1 in bits 32-34 -> byte 4 = 0x01.
    idx = np.full((1, 128), 8, np.uint8)
    idx[0, 5] = 15; idx[0, 6] = 0; idx[0, 1] = 7; idx[0, 8] = 9
    p = o.pack_codes(idx, 4)[0]
    want = bytearray(64); want[1] = 0x80; want[2] = 0x78; want[3] = 0x07; want[4] = 0x01
    assert bytes(p) == bytes(want)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def _naive_attention(q, K, V, scale):
    """Loop-by-loop softmax attention (no numpy vector ops on the softmax)."""
    out = np.zeros((q.shape[0], V.shape[1]))
    for r in range(q.shape[0]):
        sc = [scale * sum(q[r, d] * K[t, d] for d in range(q.shape[1]))
              for t in range(K.shape[0])]
        m = max(sc)
        w = [math.exp(v - m) for v in sc]
        z = sum(w)
        for t in range(K.shape[0]):
            out[r] += (w[t] / z) * V[t]
    return out


def test_unquantised_attention_equals_naive_loop_and_torch_sdpa():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, 16)); K = rng.standard_normal((9, 16))
    V = rng.standard_normal((9, 16))
    got = o.softmax_attention(q, K, V, 0.25, np.array([9, 9, 9]))
    assert np.max(np.abs(got - _naive_attention(q, K, V, 0.25))) < 1e-12
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None], torch.tensor(K)[None], torch.tensor(V)[None], scale=0.25)[0]
    assert np.max(np.abs(got - ref.numpy())) < 1e-12


def test_causal_block_equals_truncated_single_query():
    rng = np.random.default_rng(6)
    L, tq = 20, 4
    q = rng.standard_normal((tq, 8)); K = rng.standard_normal((L, 8))
    V = rng.standard_normal((L, 8))
    blk = o.softmax_attention(q, K, V, 0.3, o.visible_counts(L, tq))
    for j in range(tq):
        n = L - tq + j + 1
        one = o.softmax_attention(q[j:j + 1], K[:n], V[:n], 0.3, np.array([n]))
        assert np.max(np.abs(blk[j] - one[0])) < 1e-14
    # tq = 1 is plain decode over all L tokens
    assert list(o.visible_counts(L, 1)) == [L]


def _random_unit(rng, mode, L, cbk, cbv):
    kb, vb = o.MODES[mode]
    unit = {"v_idx": rng.integers(0, 1 << vb, (L, 128)).astype(np.uint8),
            "v_norm": (rng.random(L) * 12 + 1).astype(np.float16)}
    if mode in o.TABLE_MODES:
        unit["k_idx"] = rng.integers(0, 1 << kb, (L, 128)).astype(np.uint8)
        unit["k_table"] = o.centroid_norm_table((rng.random(L) * 12 + 1).astype(np.float16), cbk)
        unit["v_table"] = o.centroid_norm_table(unit.pop("v_norm"), cbv)
        return unit
    if kb is None:
        unit["k"] = rng.standard_normal((L, 128)).astype(np.float16)
    else:
        unit["k_idx"] = rng.integers(0, 1 << kb, (L, 128)).astype(np.uint8)
        unit["k_norm"] = (rng.random(L) * 12 + 1).astype(np.float16)
    return unit


@pytest.mark.parametrize("mode", ["turbo4_asym", "turbo3", "turbo4", "turbo3_asym", "turbo4k_3v",
                                  "turbo3_table"])
def test_rotated_basis_identity(mode):
    """rotate(SDPA(q,k,v)) == SDPA(q,k,rotate(v)): the shortcut equals full dequant."""
    rng = np.random.default_rng(11)
    kb, vb = o.MODES[mode]
    cbk = o.codebook(kb) if kb else None
    cbv = o.codebook(vb)
    s = o.sign_vector(42)
    L, G, tq = 50, 3, 2
    unit = _random_unit(rng, mode, L, cbk, cbv)
    q = rng.standard_normal((G, tq, 128)).astype(np.float16)
    a = o.decode_unit(mode, q, unit, L, tq, G, cbk, cbv, s, 1 / math.sqrt(128), 0.75)
    b = o.decode_rotated_unit(mode, q, unit, L, tq, G, cbk, cbv, s, 1 / math.sqrt(128), 0.75)
    assert np.max(np.abs(a - b)) < 1e-12


def test_symmetric_scores_invariant_under_rotation():
    rng = np.random.default_rng(12)
    s = o.sign_vector(99)
    q = rng.standard_normal(128); k = rng.standard_normal(128)
    assert abs(o.rotate(q, s) @ o.rotate(k, s) - q @ k) < 1e-12


def test_gqa_head_map():
    """q head h reads kv head h // G: distinct KV heads give per-head answers."""
    rng = np.random.default_rng(13)
    cbv = o.codebook(4); s = o.sign_vector(42)
    L, G = 16, 2
    units = [_random_unit(rng, "turbo4_asym", L, None, cbv) for _ in range(2)]
    q = rng.standard_normal((2 * G, 1, 128)).astype(np.float16)
    for h in range(2 * G):
        u = units[h // G]
        got = o.decode_unit("turbo4_asym", q[h:h + 1], u, L, 1, 1, None, cbv, s,
                            0.1, 1.0)[0, 0]
        K = np.asarray(u["k"], np.float64)
        V = o.dequant_full(u["v_idx"], u["v_norm"], cbv, s)
        assert np.max(np.abs(got - _naive_attention(q[h].astype(np.float64), K, V, 0.1)[0])) < 1e-12


def test_quantisation_error_is_at_the_codebook_mse_level():
    """Informational sanity: 4-bit dequant of Gaussian vectors has the Lloyd-Max MSE."""
    rng = np.random.default_rng(14)
    x = rng.standard_normal((400, 128)).astype(np.float16)
    s = o.sign_vector(42)
    cb = o.codebook(4)
    idx, n16, _, _ = o.encode(x, cb, s)
    xr = o.dequant_full(idx, n16, cb, s)
    rel = np.sum((xr - x.astype(np.float64)) ** 2) / np.sum(x.astype(np.float64) ** 2)
    assert 0.006 < rel < 0.013      # Max's 16-level MSE is 0.0095 of the variance


def test_encode_append_semantics_and_capacity():
    s = o.sign_vector(42); cb = o.codebook(3)
    cache = {"mode": "turbo3", "capacity": 5, "lengths": np.array([2, 4], np.int32),
             "k_data": np.zeros((2, 1, 5, 48), np.uint8), "k_norm": np.zeros((2, 1, 5), np.float16),
             "v_data": np.zeros((2, 1, 5, 48), np.uint8), "v_norm": np.zeros((2, 1, 5), np.float16)}
    rng = np.random.default_rng(15)
    k = rng.standard_normal((2, 1, 2, 128)).astype(np.float16)
    v = rng.standard_normal((2, 1, 2, 128)).astype(np.float16)
    err = o.encode_append(cache, k, v, cb, cb, s)
    assert list(err) == [0, 1]                  # sequence 1 would pass capacity 5
    assert list(cache["lengths"]) == [4, 4]
    idx, n16, _, _ = o.encode(k[0, 0], cb, s)
    assert np.array_equal(cache["k_data"][0, 0, 2:4], o.pack_codes(idx, 3))
    assert np.array_equal(cache["k_norm"][0, 0, 2:4], n16)
    assert not cache["k_data"][1].any()


def test_v_rescale_is_a_plain_output_scale():
    rng = np.random.default_rng(16)
    cbv = o.codebook(3); s = o.sign_vector(42)
    unit = _random_unit(rng, "turbo3", 12, cbv, cbv)
    q = rng.standard_normal((2, 1, 128)).astype(np.float16)
    a = o.decode_unit("turbo3", q, unit, 12, 1, 2, cbv, cbv, s, 0.1, 1.0)
    b = o.decode_unit("turbo3", q, unit, 12, 1, 2, cbv, cbv, s, 0.1, 2.5)
    assert np.max(np.abs(b - 2.5 * a)) < 1e-12


def test_symmetric_decode_is_attention_over_dequantised_cache():
    rng = np.random.default_rng(17)
    cb = o.codebook(4); s = o.sign_vector(5)
    unit = _random_unit(rng, "turbo4", 10, cb, cb)
    q = rng.standard_normal((1, 1, 128)).astype(np.float16)
    got = o.decode_unit("turbo4", q, unit, 10, 1, 1, cb, cb, s, 0.2, 1.0)[0, 0]
    K = o.dequant_full(unit["k_idx"], unit["k_norm"], cb, s)
    V = o.dequant_full(unit["v_idx"], unit["v_norm"], cb, s)
    assert np.max(np.abs(got - _naive_attention(q[0].astype(np.float64), K, V, 0.2)[0])) < 1e-12


def test_dequant_reconstructs_encoded_vector():
    rng = np.random.default_rng(18)
    s = o.sign_vector(42); cb = o.codebook(4)
    x = rng.standard_normal((20, 128)).astype(np.float16)
    idx, n16, u, _ = o.encode(x, cb, s)
    # rotated-basis coordinates are n * u; dequant replaces u by its centroid
    xr = o.dequant_rotated(idx, n16, cb)
    assert np.allclose(xr / n16.astype(np.float64)[:, None], cb.astype(np.float64)[idx])
    # every coordinate lands on its nearest centroid: error below half the local gap
    c = cb.astype(np.float64)
    near = c[idx]
    assert np.all(np.abs(u - near) <= np.abs(u[..., None] - c).min(-1) + 1e-12)


# --------------------------------------------------------------------------
# sparse-V (V skipped for softmax weights below tau)
# --------------------------------------------------------------------------
def test_sparse_v_two_token_closed_form():
    # scores 0 and -20 (scale 1): p1 = e^-20 / (1 + e^-20) ~ 2.06e-9
    q = np.zeros((1, 4)); q[0, 0] = 1.0
    K = np.zeros((2, 4)); K[1, 0] = -20.0
    V = np.array([[1.0, 2.0, 0.0, -3.0], [1000.0, -1000.0, 5.0, 0.0]])
    p1 = math.exp(-20.0) / (1.0 + math.exp(-20.0))
    p0 = 1.0 / (1.0 + math.exp(-20.0))
    out, bound = o.softmax_attention_sparse_v(q, K, V, 1.0, np.array([2]), 1e-6)
    assert np.allclose(out[0], p0 * V[0], rtol=1e-15, atol=0)
    assert np.allclose(bound[0], p1 * np.abs(V[1]), rtol=1e-15, atol=0)
    # below the smaller weight nothing is skipped
    out, bound = o.softmax_attention_sparse_v(q, K, V, 1.0, np.array([2]), 1e-10)
    assert np.allclose(out[0], p0 * V[0] + p1 * V[1], rtol=1e-15, atol=0)
    assert not bound.any()


def test_sparse_v_degenerate_thresholds():
    rng = np.random.default_rng(21)
    q = rng.standard_normal((3, 16)) * 4; K = rng.standard_normal((40, 16))
    V = rng.standard_normal((40, 16)); vis = np.array([40, 17, 1])
    full = o.softmax_attention(q, K, V, 0.5, vis)
    out, bound = o.softmax_attention_sparse_v(q, K, V, 0.5, vis, 0.0)
    assert np.array_equal(out, full) and not bound.any()
    # every weight is <= 1, so tau > 1 skips everything
    out, bound = o.softmax_attention_sparse_v(q, K, V, 0.5, vis, 1.5)
    assert not out.any()
    assert np.allclose(bound, o.softmax_attention(q, K, np.abs(V), 0.5, vis), rtol=1e-14)


def test_sparse_v_equals_naive_skip_loop_and_stays_within_bound():
    rng = np.random.default_rng(22)
    q = rng.standard_normal((4, 8)) * 6; K = rng.standard_normal((30, 8))
    V = rng.standard_normal((30, 8)); tau = 1e-6
    out, bound = o.softmax_attention_sparse_v(q, K, V, 1.0, np.full(4, 30), tau)
    skipped = 0
    for r in range(4):
        sc = [sum(q[r, d] * K[t, d] for d in range(8)) for t in range(30)]
        m = max(sc)
        w = [math.exp(v - m) for v in sc]
        z = sum(w)
        want = np.zeros(8)
        for t in range(30):
            if w[t] / z >= tau:
                want += (w[t] / z) * V[t]
            else:
                skipped += 1
        assert np.max(np.abs(out[r] - want)) < 1e-12
    assert skipped > 0      # sharp queries: the threshold is not vacuous here
    full = o.softmax_attention(q, K, V, 1.0, np.full(4, 30))
    assert np.all(np.abs(out - full) <= bound + 1e-15)


def test_sparse_v_decode_unit_reduces_to_decode_unit_at_zero_tau():
    rng = np.random.default_rng(23)
    s = o.sign_vector(42); cb = o.codebook(3)
    unit = _random_unit(rng, "turbo3", 33, cb, cb)
    q = rng.standard_normal((2, 3, 128)).astype(np.float16)
    want = o.decode_unit("turbo3", q, unit, 33, 3, 2, cb, cb, s, 0.1, -0.5)
    got, bound = o.decode_unit_sparse_v("turbo3", q, unit, 33, 3, 2, cb, cb, s, 0.1, -0.5, 0.0)
    assert np.array_equal(got, want) and not bound.any()
    got, bound = o.decode_unit_sparse_v("turbo3", q, unit, 33, 3, 2, cb, cb, s, 0.1, -0.5, 2.0)
    assert not got.any() and np.all(bound >= np.abs(want) - 1e-12)


# --------------------------------------------------------------------------
# centroid x norm table records (format B)
# --------------------------------------------------------------------------
def _fp16_rne_fraction(x: Fraction) -> float:
    """Round an exact rational to fp16 (normal range), ties to even, by brute
    force over the binade's grid."""
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = 0
    while a >= 2:
        a /= 2; e += 1
    while a < 1:
        a *= 2; e -= 1
    step = Fraction(1, 1024)
    lo = (a // step) * step
    hi = lo + step
    d_lo, d_hi = a - lo, hi - a
    if d_lo < d_hi or (d_lo == d_hi and (lo / step) % 2 == 0):
        r = lo
    else:
        r = hi
    return sign * float(r * Fraction(2) ** e)


def test_centroid_norm_table_is_one_rounding_of_the_exact_product():
    rng = np.random.default_rng(31)
    cb = o.codebook(3)
    n16 = (rng.random(50) * 30 + 0.5).astype(np.float16)
    tab = o.centroid_norm_table(n16, cb)
    for i in range(50):
        for j in range(8):
            exact = Fraction(float(n16[i])) * Fraction(float(cb[j]))
            assert float(tab[i, j]) == _fp16_rne_fraction(exact), (i, j)
    # a zero norm gives an all-zero table; symmetry of the codebook carries over
    assert not o.centroid_norm_table(np.float16(0), cb).astype(np.float64).any()
    assert np.array_equal(tab[:, :4].astype(np.float64), -tab[:, ::-1][:, :4].astype(np.float64))


def test_table_record_bytes_and_roundtrip():
    cb = o.codebook(3)
    idx = np.zeros((1, 128), np.uint8)
    idx[0, 0] = 7
    n16 = np.array([2.0], np.float16)
    rec = o.pack_table_records(idx, o.centroid_norm_table(n16, cb))
    assert rec.shape == (1, 64)
    assert np.array_equal(rec[0, :48], o.pack_codes(idx, 3)[0])
    # bytes 48..63: fp16 little-endian 2*c_0 .. 2*c_7
    want = (2.0 * cb.astype(np.float64)).astype(np.float16).astype("<f2").view(np.uint8)
    assert np.array_equal(rec[0, 48:], want)
    rng = np.random.default_rng(32)
    idx = rng.integers(0, 8, (9, 128)).astype(np.uint8)
    tab = o.centroid_norm_table((rng.random(9) * 5).astype(np.float16), cb)
    i2, t2 = o.unpack_table_records(o.pack_table_records(idx, tab))
    assert np.array_equal(i2, idx) and np.array_equal(t2.view(np.uint16), tab.view(np.uint16))


def test_table_dequant_is_the_fp16_rounding_of_the_norm_format():
    rng = np.random.default_rng(33)
    cb = o.codebook(3)
    idx = rng.integers(0, 8, (20, 128)).astype(np.uint8)
    n16 = (rng.random(20) * 9 + 1).astype(np.float16)
    a = o.dequant_rotated(idx, n16, cb)
    b = o.dequant_table(idx, o.centroid_norm_table(n16, cb))
    assert np.all(np.abs(a - b) <= np.abs(a) * 2.0 ** -11)
    assert np.any(a != b)


def test_table_mode_append_matches_encode():
    s = o.sign_vector(42); cb = o.codebook(3)
    rng = np.random.default_rng(34)
    x = rng.standard_normal((1, 2, 5, 128)).astype(np.float16)
    cache = {"mode": "turbo3_table", "capacity": 16, "lengths": np.array([3], np.int32),
             "k_data": np.zeros((1, 2, 16, 64), np.uint8), "v_data": np.zeros((1, 2, 16, 64), np.uint8)}
    assert not o.encode_append(cache, x, -x, cb, cb, s).any()
    assert cache["lengths"][0] == 8
    idx, tab = o.unpack_table_records(cache["k_data"][0, 1, 3:8])
    ei, en, _, _ = o.encode(x[0, 1], cb, s)
    assert np.array_equal(idx, ei)
    assert np.array_equal(tab.view(np.uint16), o.centroid_norm_table(en, cb).view(np.uint16))
