"""fp64 CPU oracle for TurboQuant-style quantized-KV decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import or run this module.
The product (the CUDA library and its Python binding) never calls it, and it
shares no code, table or constant generator with the CUDA path.

What it computes (plain, slow, obviously correct; float64 unless stated):

* Sign vector: splitmix64 seeded with ``rot_seed``; s_i = -1 iff the top bit of
  output i is set.  The pages call for a seeded sign flip but name no
  generator (mlxcel PR #369 "route Turbo4Asym decode through dequant-SDPA",
  Change), so this is a format reading.
* Rotation: Rot(x) = H (s * x) / sqrt(D), Rot^-1(y) = s * (H y) / sqrt(D), H the
  Sylvester Hadamard matrix H[i][j] = (-1)^popcount(i & j), D = 128 -- the
  Walsh-Hadamard rotated basis of mlxcel PR #369 (Change), over the 128-element
  rotation group of turboquant_plus smem-dequant-experiment.md (Hypothesis 1).
* Codebook: Lloyd-Max quantiser of N(0, 1/128) with 2^b levels, iterated in
  fp64 to a fixed point and rounded to fp16 (the half-precision centroid
  tables of the pages); those values, carried as fp32, are the standard
  codebook both sides use (any symmetric fp32 codebook can be given instead).  The 3-bit codebook is a sign and four magnitudes (the
  four-magnitude lookup table of smem-dequant-experiment.md); the 4-bit one is
  the V codec of mlxcel PR #369 (Result).
* Encode: n16 = fp16 round-to-nearest-even of the exact L2 norm of the fp16
  input; u = Rot(x) / n (unrounded fp64 n), rounded to fp32; idx = the nearest
  codebook entry to that fp32 u in exact arithmetic, ties to the lower index.
* Packing: sign-magnitude codes in the 4-bit / 3-bit layouts spelled out in
  ``pack_codes``.  Format choice; the pages give no byte layout (the 56-byte
  turbo3 block of smem-dequant-experiment.md, Hypothesis 1, is not broken down).
* Dequant: rotated basis n16 * c[idx]; original basis Rot^-1 of that.
* Attention (the definition the fast path must reproduce): full dequant of K
  and V to the original basis, then softmax(q K^T * scale) V with the GQA map
  kv_head = q_head // G, query j of a Tq block seeing tokens [0, L - Tq + j],
  times the scalar v_rescale -- the exact attention over the fully dequantised
  cache that the mlxcel parity test compares against (PR #369, Result).
* The rotated-basis shortcut rotate(SDPA(q,k,v)) == SDPA(q,k,rotate(v))
  (PR #369, Change) is computed separately in ``decode_rotated_unit`` and checked
  against the definition by the tests; it is never used to produce the
  reference output.
"""
from __future__ import annotations

import math
import numpy as np

D = 128
MASK64 = (1 << 64) - 1
MODES = {"turbo4_asym": (None, 4), "turbo3": (3, 3), "turbo4": (4, 4),
         "turbo3_asym": (None, 3), "turbo4k_3v": (4, 3), "turbo3_table": (3, 3)}
# modes whose records carry the centroid x norm table instead of a norm
TABLE_MODES = {"turbo3_table"}


# --------------------------------------------------------------------------
# sign vector (format reading: splitmix64, Steele/Lea/Flood 2014, the
# finaliser of Vigna's public splitmix64.c)
# --------------------------------------------------------------------------
def splitmix64(seed: int, n: int) -> list:
    out = []
    state = seed & MASK64
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        out.append(z ^ (z >> 31))
    return out


def sign_vector(rot_seed: int, d: int = D) -> np.ndarray:
    """s in {+1, -1}^d: s_i = -1 iff bit 63 of the i-th splitmix64 output is set."""
    return np.array([-1.0 if (v >> 63) & 1 else 1.0 for v in splitmix64(rot_seed, d)])


# --------------------------------------------------------------------------
# rotation (mlxcel PR #369, Change: the Walsh-Hadamard rotated basis; sign flip
# then normalised WHT)
# --------------------------------------------------------------------------
def hadamard(d: int = D) -> np.ndarray:
    """Sylvester Hadamard matrix, H[i][j] = (-1)^popcount(i & j), as float64."""
    i = np.arange(d)
    bits = i[:, None] & i[None, :]
    parity = np.zeros_like(bits)
    for k in range(int(math.log2(d)) + 1):
        parity ^= (bits >> k) & 1
    return np.where(parity == 0, 1.0, -1.0)


def rotate(x: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Rot(x) = H (s * x) / sqrt(D) along the last axis (row vectors)."""
    d = x.shape[-1]
    return (np.asarray(x, np.float64) * s) @ hadamard(d).T / math.sqrt(d)


def rotate_inv(y: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Rot^-1(y) = s * (H y) / sqrt(D) along the last axis."""
    d = y.shape[-1]
    return (np.asarray(y, np.float64) @ hadamard(d).T / math.sqrt(d)) * s


# --------------------------------------------------------------------------
# Lloyd-Max codebook for N(0, sigma^2), sigma = 1/sqrt(D)
# --------------------------------------------------------------------------
def _phi(a):
    return np.exp(-0.5 * a * a) / math.sqrt(2.0 * math.pi)


def _Phi(a):
    return 0.5 * np.vectorize(math.erfc)(-np.asarray(a, np.float64) / math.sqrt(2.0))


def lloyd_max(levels: int, sigma: float = 1.0 / math.sqrt(D), tol: float = 1e-15,
              max_iter: int = 200000):
    """Lloyd-Max fixed point for a zero-mean Gaussian, in fp64.

    Alternates the two optimality conditions: thresholds at the midpoints of
    neighbouring levels, each level at the conditional mean of its cell,
    E[X | a <= X < b] = sigma^2 (phi_s(a) - phi_s(b)) / (Phi_s(b) - Phi_s(a)).
    Returns (levels fp64 ascending, iterations, final max |delta|).
    """
    c = sigma * np.linspace(-2.0, 2.0, levels)
    delta = np.inf
    it = 0
    for it in range(1, max_iter + 1):
        t = 0.5 * (c[:-1] + c[1:])
        a = np.concatenate([[-np.inf], t / sigma, [np.inf]])
        num = _phi(a[:-1]) - _phi(a[1:])
        den = _Phi(a[1:]) - _Phi(a[:-1])
        new = sigma * num / den
        delta = float(np.max(np.abs(new - c)))
        c = new
        if delta < tol:
            break
    return c, it, delta


def codebook(bits: int) -> np.ndarray:
    """The standard codebook (2^bits entries, ascending) both sides quantise
    with: the Lloyd-Max levels rounded to the nearest fp16 value (ties to
    even), carried as fp32 (every fp16 value is one).  The pages' centroid
    lookup tables and dequantized caches are half precision (the turbo3
    dequant into a half4 buffer and the fp16 centroid x norm table of the
    smem-dequant experiment, the FP16 dequantized V of mlxcel PR #369), so
    the levels are fp16 values; the rounding moves each level by at most
    2^-12 of itself.  Any other symmetric fp32 codebook may be passed to
    both sides instead."""
    c64, _, _ = lloyd_max(1 << bits)
    return c64.astype(np.float16).astype(np.float32)


# --------------------------------------------------------------------------
# encode
# --------------------------------------------------------------------------
def _fp16_grid_floor(x: float) -> np.float16:
    """Largest fp16 value <= x (x >= 0, finite, below 65520)."""
    h = np.float16(x)
    if float(h) > x:
        h = np.nextafter(h, np.float16(-np.inf))
    return h


def fp16_sqrt_rne(S: int) -> np.float16:
    """fp16 round-to-nearest-even of sqrt(S) * 2^-24, exactly (S a non-negative int).

    In units of 2^-25 every fp16 value is an even integer and every midpoint
    between neighbouring fp16 values is an integer, and the target is
    w = sqrt(S) * 2^-24 * 2^25 = sqrt(4 S).  So every comparison with a
    midpoint m is the integer comparison 4 S <=> m^2.  The overflow point is
    65520 (midpoint of 65504 and 2^16; the tie goes to the even 2^16 = inf).
    """
    if S == 0:
        return np.float16(0.0)
    W2 = 4 * S
    if W2 >= (65520 * 2 ** 25) ** 2:
        return np.float16(np.inf)
    k = math.isqrt(W2)                      # floor(w)
    f = _fp16_grid_floor(k / 2.0 ** 25)     # largest fp16 <= w (grid points are integers)
    fi = int(float(f) * 2 ** 25)
    if float(f) == 65504.0:
        g, gi = np.float16(np.inf), 65536 * 2 ** 25
    else:
        g = np.nextafter(f, np.float16(np.inf))
        gi = int(float(g) * 2 ** 25)
    m = (fi + gi) // 2
    if W2 < m * m:
        return f
    if W2 > m * m:
        return g
    return f if int(np.array(f, np.float16).view(np.uint16)) % 2 == 0 else g


def exact_sum_squares(x16: np.ndarray):
    """Row-wise sum of squares of fp16 values times 2^48, as exact Python ints.

    Every fp16 value is an integer multiple of 2^-24, so M = x * 2^24 is an
    exact integer (|M| < 2^40) and sum(M^2) is exact in Python integers.
    """
    x = np.asarray(x16, np.float16)
    M = (x.astype(np.float64) * 2.0 ** 24).astype(np.int64).astype(object)
    return np.sum(M * M, axis=-1)


def fp16_norm(x16: np.ndarray) -> np.float16:
    """fp16 (RNE) of the exact L2 norm of one fp16 vector."""
    return fp16_sqrt_rne(int(exact_sum_squares(np.asarray(x16).reshape(1, -1))[0]))


def nearest_index(u32: np.ndarray, cb32: np.ndarray) -> np.ndarray:
    """Index of the codebook entry nearest to each fp32 u, exactly; ties -> lower.

    A tie means u is exactly the midpoint of two neighbouring entries; the
    midpoint of two fp32 numbers is exact in fp64, so "u > midpoint" is an
    exact test and the count of midpoints strictly below u is the index.
    """
    c = cb32.astype(np.float64)
    mids = 0.5 * (c[:-1] + c[1:])
    u = np.asarray(u32, np.float32).astype(np.float64)
    return np.sum(u[..., None] > mids, axis=-1).astype(np.uint8)


def encode(x16: np.ndarray, cb32: np.ndarray, s: np.ndarray):
    """Encode fp16 vectors [..., 128].

    Returns (idx uint8 [..., 128], n16 fp16 [...], u fp64 [..., 128],
    overflow bool [...]).  u is kept for the boundary-distance bookkeeping of
    the parity tests.
    """
    x16 = np.asarray(x16, np.float16)
    shp = x16.shape[:-1]
    flat = x16.reshape(-1, x16.shape[-1])
    n16 = np.empty(flat.shape[0], np.float16)
    n64 = np.empty(flat.shape[0], np.float64)
    sums = exact_sum_squares(flat)
    for r in range(flat.shape[0]):
        S = int(sums[r])
        n16[r] = fp16_sqrt_rne(S)
        n64[r] = math.sqrt(S) / 2.0 ** 24
    y = rotate(flat.astype(np.float64), s)
    with np.errstate(invalid="ignore", divide="ignore"):
        u = np.where(n64[:, None] > 0, y / np.where(n64 > 0, n64, 1.0)[:, None], 0.0)
    idx = nearest_index(u.astype(np.float32), cb32)
    overflow = ~np.isfinite(n16.astype(np.float64))
    return (idx.reshape(*shp, -1), n16.reshape(shp), u.reshape(*shp, -1),
            overflow.reshape(shp))


def boundary_distance(u: np.ndarray, cb32: np.ndarray) -> np.ndarray:
    """|u - nearest decision midpoint| per element (fp64)."""
    c = cb32.astype(np.float64)
    mids = 0.5 * (c[:-1] + c[1:])
    return np.min(np.abs(np.asarray(u, np.float64)[..., None] - mids), axis=-1)


# --------------------------------------------------------------------------
# packing (format choice)
# --------------------------------------------------------------------------
def to_code(idx: np.ndarray, bits: int) -> np.ndarray:
    """Ascending index -> sign-magnitude code kappa = (sign << (b-1)) | rank.

    sign = 1 for the negative half; rank 0 is the entry nearest zero.  With
    h = 2^(b-1): idx >= h -> kappa = idx - h; idx < h -> kappa = h | (h-1-idx).
    """
    h = 1 << (bits - 1)
    idx = np.asarray(idx, np.int64)
    return np.where(idx >= h, idx - h, h | (h - 1 - idx)).astype(np.uint8)


def from_code(kappa: np.ndarray, bits: int) -> np.ndarray:
    h = 1 << (bits - 1)
    k = np.asarray(kappa, np.int64)
    sign = (k >> (bits - 1)) & 1
    rank = k & (h - 1)
    return np.where(sign == 0, h + rank, h - 1 - rank).astype(np.uint8)


def record_bytes(bits: int) -> int:
    return D * bits // 8


def pack_codes(idx: np.ndarray, bits: int) -> np.ndarray:
    """Pack [..., 128] ascending indices into [..., 16*bits] bytes.

    4-bit: eight 32-bit little-endian words, word k = dimensions 8k .. 8k+7.
    Bits 4j .. 4j+2 hold the magnitude rank of dimension 8k+j (j = 0..7); the
    sign bits sit in the nibbles' top bits: bit 8j+7 = sign of dim 8k+j and
    bit 8j+3 = sign of dim 8k+4+j (j = 0..3).
    3-bit: four 12-byte quarters; quarter q holds dimensions 32q .. 32q+31 as
    three little-endian 32-bit words w0, w1, w2 (bytes 12q + 4k).  In word k,
    bits 4j .. 4j+2 hold the code of dimension 32q + 8k + j (j = 0..7) and bit
    4j+3 holds bit k of the code of dimension 32q + 24 + j.
    """
    kap = to_code(idx, bits).astype(np.uint32)
    shp = kap.shape[:-1]
    kap = kap.reshape(-1, D)
    n = kap.shape[0]
    if bits == 4:
        rank, sign = kap & 7, kap >> 3
        words = np.zeros((n, 16), np.uint32)
        for k in range(16):
            w = np.zeros(n, np.uint32)
            for j in range(8):
                w |= rank[:, 8 * k + j] << (4 * j)
            for j in range(4):
                w |= sign[:, 8 * k + j] << (8 * j + 7)
                w |= sign[:, 8 * k + 4 + j] << (8 * j + 3)
            words[:, k] = w
        return words.astype("<u4").view(np.uint8).reshape(*shp, 64)
    if bits != 3:
        raise ValueError("bits must be 3 or 4")
    words = np.zeros((n, 12), np.uint32)
    for q in range(4):
        for k in range(3):
            w = np.zeros(n, np.uint32)
            for j in range(8):
                w |= (kap[:, 32 * q + 8 * k + j] & 7) << (4 * j)
                w |= ((kap[:, 32 * q + 24 + j] >> k) & 1) << (4 * j + 3)
            words[:, 3 * q + k] = w
    return words.astype("<u4").view(np.uint8).reshape(*shp, 48)


def unpack_codes(packed: np.ndarray, bits: int) -> np.ndarray:
    """Inverse of pack_codes: bytes [..., 16*bits] -> ascending indices [..., 128]."""
    packed = np.ascontiguousarray(packed, np.uint8)
    shp = packed.shape[:-1]
    p = packed.reshape(-1, packed.shape[-1])
    n = p.shape[0]
    kap = np.zeros((n, D), np.uint32)
    if bits == 4:
        words = p.view("<u4").astype(np.uint32)
        for k in range(16):
            w = words[:, k]
            for j in range(8):
                kap[:, 8 * k + j] = (w >> (4 * j)) & 7
            for j in range(4):
                kap[:, 8 * k + j] |= ((w >> (8 * j + 7)) & 1) << 3
                kap[:, 8 * k + 4 + j] |= ((w >> (8 * j + 3)) & 1) << 3
    elif bits == 3:
        words = p.view("<u4").astype(np.uint32)
        for q in range(4):
            for k in range(3):
                w = words[:, 3 * q + k]
                for j in range(8):
                    kap[:, 32 * q + 8 * k + j] = (w >> (4 * j)) & 7
                    kap[:, 32 * q + 24 + j] |= ((w >> (4 * j + 3)) & 1) << k
    else:
        raise ValueError("bits must be 3 or 4")
    return from_code(kap, bits).reshape(*shp, D)


# --------------------------------------------------------------------------
# dequant
# --------------------------------------------------------------------------
def dequant_rotated(idx: np.ndarray, n16: np.ndarray, cb32: np.ndarray) -> np.ndarray:
    """n16 * c[idx] in the rotated basis (fp64)."""
    return np.asarray(n16, np.float64)[..., None] * cb32.astype(np.float64)[idx]


def centroid_norm_table(n16: np.ndarray, cb32: np.ndarray) -> np.ndarray:
    """fp16 [..., 2^b]: entry j = fp16 round-to-nearest-even of c_j * n16.

    The record format of turboquant_plus smem-dequant-experiment.md, "What
    Would Actually Work" item 1: the pre-multiplied centroid x norm values of
    each 128-element group stored with its block.  c_j (fp32) times n16 (fp16)
    is exact in fp64, so this is one rounding of the exact product.
    """
    prod = np.asarray(n16, np.float16).astype(np.float64)[..., None] * cb32.astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return prod.astype(np.float16)


def pack_table_records(idx: np.ndarray, table16: np.ndarray) -> np.ndarray:
    """3-bit codes (the 48-byte layout of pack_codes) followed by the 8-entry
    fp16 table in ascending index order, little-endian: 64 bytes per record."""
    codes = pack_codes(idx, 3)
    tab = np.ascontiguousarray(np.asarray(table16, np.float16)).astype("<f2").view(np.uint8)
    return np.concatenate([codes, tab.reshape(*codes.shape[:-1], 16)], axis=-1)


def unpack_table_records(rec: np.ndarray):
    """Inverse of pack_table_records: (ascending indices [..., 128], fp16 table [..., 8])."""
    rec = np.ascontiguousarray(rec, np.uint8)
    idx = unpack_codes(rec[..., :48], 3)
    tab = np.ascontiguousarray(rec[..., 48:64]).view("<f2").astype(np.float16)
    return idx, tab


def dequant_table(idx: np.ndarray, table16: np.ndarray) -> np.ndarray:
    """table[idx] in the rotated basis (fp64): the whole dequant of the table format."""
    t = np.asarray(table16, np.float16).astype(np.float64)
    return np.take_along_axis(t, np.asarray(idx, np.int64), axis=-1)


def dequant_full(idx, n16, cb32, s) -> np.ndarray:
    """Rot^-1(n16 * c[idx]): the vector back in the original basis."""
    return rotate_inv(dequant_rotated(idx, n16, cb32), s)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                      visible: np.ndarray) -> np.ndarray:
    """Direct attention for one KV head.

    q [R, D], K/V [L, D] (fp64), visible[r] = number of leading tokens row r
    sees.  Rows that see nothing return 0.
    """
    R = q.shape[0]
    out = np.zeros((R, V.shape[1]))
    scores = (np.asarray(q, np.float64) @ np.asarray(K, np.float64).T) * scale
    for r in range(R):
        n = int(visible[r])
        if n <= 0:
            continue
        sr = scores[r, :n]
        p = np.exp(sr - sr.max())
        p /= p.sum()
        out[r] = p @ V[:n]
    return out


def softmax_attention_sparse_v(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                               visible: np.ndarray, tau: float):
    """Sparse-V attention for one KV head: the V skip of turboquant_plus
    (smem-dequant-experiment.md, "What Would Actually Work" item 2: V dequant
    is skipped for negligible weights) at the threshold the mlxcel ADR 0002
    commit calls exact (tau = 1e-6).

    The softmax weights p are the ordinary ones, normalised over every visible
    token; a token whose weight is below tau adds nothing to the weighted sum
    of V (the denominator keeps it).  Returns (out, bound) with
    bound[r, i] = sum over the skipped tokens of p_t * |V[t, i]|: the most any
    subset of the skipped tokens can add to out[r, i].
    """
    R = q.shape[0]
    out = np.zeros((R, V.shape[1]))
    bound = np.zeros((R, V.shape[1]))
    scores = (np.asarray(q, np.float64) @ np.asarray(K, np.float64).T) * scale
    for r in range(R):
        n = int(visible[r])
        if n <= 0:
            continue
        sr = scores[r, :n]
        p = np.exp(sr - sr.max())
        p /= p.sum()
        skip = p < tau
        out[r] = np.where(skip, 0.0, p) @ V[:n]
        bound[r] = np.where(skip, p, 0.0) @ np.abs(V[:n])
    return out, bound


def visible_counts(L: int, tq: int) -> np.ndarray:
    """Query j of a Tq block at the end of an L-token context sees L - Tq + j + 1 tokens."""
    return np.array([L - tq + j + 1 for j in range(tq)])


def unit_kv_full(mode: str, unit: dict, cbk, cbv, s):
    """Original-basis K and V (fp64) for one (b, kv-head) from its cache record.

    unit keys: 'k' (fp16 [L,128], asym only) or 'k_idx','k_norm'; 'v_idx','v_norm';
    the table modes: 'k_idx','k_table','v_idx','v_table' (fp16 [L, 8] tables).
    """
    if mode in TABLE_MODES:
        return (rotate_inv(dequant_table(unit["k_idx"], unit["k_table"]), s),
                rotate_inv(dequant_table(unit["v_idx"], unit["v_table"]), s))
    if MODES[mode][0] is None:
        K = np.asarray(unit["k"], np.float64)
    else:
        K = dequant_full(unit["k_idx"], unit["k_norm"], cbk, s)
    V = dequant_full(unit["v_idx"], unit["v_norm"], cbv, s)
    return K, V


def decode_unit(mode: str, q_rows: np.ndarray, unit: dict, L: int, tq: int, G: int,
                cbk, cbv, s, scale: float, v_rescale: float) -> np.ndarray:
    """Reference decode for one (b, kv-head): q_rows fp16 [G, Tq, 128] -> fp64 [G, Tq, 128].

    Definition: full dequant, then direct softmax attention, then v_rescale.
    """
    K, V = unit_kv_full(mode, unit, cbk, cbv, s)
    K, V = K[:L], V[:L] * v_rescale
    q = np.asarray(q_rows, np.float64).reshape(G * tq, D)
    vis = np.tile(visible_counts(L, tq), G)
    return softmax_attention(q, K, V, scale, vis).reshape(G, tq, D)


def decode_unit_sparse_v(mode: str, q_rows: np.ndarray, unit: dict, L: int, tq: int, G: int,
                         cbk, cbv, s, scale: float, v_rescale: float, tau: float):
    """Sparse-V decode for one (b, kv-head): (out, bound), both fp64 [G, Tq, 128].

    Full dequant, then ``softmax_attention_sparse_v``, then v_rescale (|v_rescale|
    for the bound).
    """
    K, V = unit_kv_full(mode, unit, cbk, cbv, s)
    K, V = K[:L], V[:L] * v_rescale
    q = np.asarray(q_rows, np.float64).reshape(G * tq, D)
    vis = np.tile(visible_counts(L, tq), G)
    out, bound = softmax_attention_sparse_v(q, K, V, scale, vis, tau)
    return out.reshape(G, tq, D), bound.reshape(G, tq, D)


def decode_rotated_unit(mode: str, q_rows, unit: dict, L: int, tq: int, G: int,
                        cbk, cbv, s, scale: float, v_rescale: float) -> np.ndarray:
    """Rotated-basis shortcut for one unit (for the identity check only).

    Symmetric modes: scores from Rot(q) against n*c[idx]; asym: q against fp16 K.
    V stays rotated; only the output is inverse-rotated.
    """
    q = np.asarray(q_rows, np.float64).reshape(G * tq, D)
    if mode in TABLE_MODES:
        qk, K = rotate(q, s), dequant_table(unit["k_idx"], unit["k_table"])
        Vr = dequant_table(unit["v_idx"], unit["v_table"])
    elif MODES[mode][0] is None:
        qk, K = q, np.asarray(unit["k"], np.float64)
        Vr = dequant_rotated(unit["v_idx"], unit["v_norm"], cbv)
    else:
        qk, K = rotate(q, s), dequant_rotated(unit["k_idx"], unit["k_norm"], cbk)
        Vr = dequant_rotated(unit["v_idx"], unit["v_norm"], cbv)
    vis = np.tile(visible_counts(L, tq), G)
    o_rot = softmax_attention(qk, K[:L], Vr[:L], scale, vis)
    return (rotate_inv(o_rot, s) * v_rescale).reshape(G, tq, D)


# --------------------------------------------------------------------------
# cache append (decode-step semantics: append, then attend)
# --------------------------------------------------------------------------
def encode_append(cache: dict, k_new: np.ndarray, v_new: np.ndarray, cbk, cbv, s
                  ) -> np.ndarray:
    """Append fp16 k_new/v_new [B, Hkv, T, 128] at position lengths[b] of each sequence.

    cache (numpy, modified in place): 'mode', 'lengths' int32 [B], 'capacity',
    'k' fp16 [B,Hkv,C,128] (asym) or 'k_data' uint8 [B,Hkv,C,RB] + 'k_norm' fp16
    [B,Hkv,C]; 'v_data', 'v_norm' (the table modes: 'k_data', 'v_data' with
    64-byte records and no norms).  A sequence whose append would pass the
    capacity is left untouched.  Returns per-sequence error flags
    (bit 0 = capacity, bit 1 = norm overflow).
    """
    mode = cache["mode"]
    kb, vb = MODES[mode]
    B, H, T, _ = k_new.shape
    err = np.zeros(B, np.int32)
    for b in range(B):
        L = int(cache["lengths"][b])
        if L + T > cache["capacity"]:
            err[b] |= 1
            continue
        for h in range(H):
            if mode in TABLE_MODES:
                for x, cb, key in ((k_new, cbk, "k_data"), (v_new, cbv, "v_data")):
                    idx, n16, _, ov = encode(x[b, h], cb, s)
                    cache[key][b, h, L:L + T] = pack_table_records(
                        idx, centroid_norm_table(n16, cb))
                    if ov.any():
                        err[b] |= 2
                continue
            if kb is None:
                cache["k"][b, h, L:L + T] = k_new[b, h]
            else:
                idx, n16, _, ov = encode(k_new[b, h], cbk, s)
                cache["k_data"][b, h, L:L + T] = pack_codes(idx, kb)
                cache["k_norm"][b, h, L:L + T] = n16
                if ov.any():
                    err[b] |= 2
            idx, n16, _, ov = encode(v_new[b, h], cbv, s)
            cache["v_data"][b, h, L:L + T] = pack_codes(idx, vb)
            cache["v_norm"][b, h, L:L + T] = n16
            if ov.any():
                err[b] |= 2
        cache["lengths"][b] = L + T
    return err
