"""Shared test helpers: GPU-side cache setup through the C ABI, the format
decoder used to read GPU output, and the parity bounds."""
import math

import numpy as np

from oracle import tq_oracle as o
from quantized_kv_cache_flash_gb300 import workloads as wl

# attention parity bounds (relative to the RMS of the oracle output)
MAX_ABS_REL = 1e-2
RMS_REL = 2e-3
# encode: elements whose fp64 u is this close to a decision midpoint may differ
BOUNDARY = 1e-5
BOUNDARY_FRACTION = 1e-4

MODE_BITS = {"turbo4_asym": (16, 4), "turbo3": (3, 3), "turbo4": (4, 4),
             "turbo3_asym": (16, 3), "turbo4k_3v": (4, 3), "turbo3_table": (3, 3)}
TABLE_MODES = {"turbo3_table"}


def attention_errors(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    rms = math.sqrt(float(np.mean(want * want)))
    err = got - want
    return rms, float(np.max(np.abs(err))), math.sqrt(float(np.mean(err * err)))


def assert_attention_close(got, want, what=""):
    rms, mx, rmse = attention_errors(got, want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert rms > 0, f"{what}: degenerate reference"
    assert mx <= MAX_ABS_REL * rms, f"{what}: max-abs {mx:.3e} > {MAX_ABS_REL} x rms {rms:.3e}"
    assert rmse <= RMS_REL * rms, f"{what}: rms err {rmse:.3e} > {RMS_REL} x rms {rms:.3e}"
    return rms, mx, rmse


def decode_records(packed: np.ndarray, bits: int) -> np.ndarray:
    """Read ascending codebook indices back from packed records (GPU output).

    Written separately from the oracle's unpacker: sign-magnitude code kappa
    -> index h + rank (sign 0) or h - 1 - rank (sign 1).
    """
    p = np.ascontiguousarray(packed, np.uint8).reshape(-1, packed.shape[-1])
    n = p.shape[0]
    if bits == 4:
        w = p.view("<u4").astype(np.int64).reshape(n, 16)       # [vec, word]
        j = np.arange(8)
        rank = (w[:, :, None] >> (4 * j)) & 7                   # dims 8k + j
        s_lo = (w[:, :, None] >> (8 * j[:4] + 7)) & 1           # sign of dims 8k + 0..3
        s_hi = (w[:, :, None] >> (8 * j[:4] + 3)) & 1           # sign of dims 8k + 4..7
        kappa = (rank | (np.concatenate([s_lo, s_hi], axis=2) << 3)).reshape(n, 128)
    else:
        w = p.view("<u4").astype(np.int64).reshape(n, 4, 3)     # [vec, quarter, word]
        j = np.arange(8)
        nib = (w[:, :, :, None] >> (4 * j)) & 0xF               # [vec, q, k, j]
        low = nib & 7                                           # dims 8k + j
        spare = (nib >> 3) & 1                                  # bit k of dim 24 + j
        kappa = np.empty((n, 4, 32), np.int64)
        kappa[:, :, :24] = low.reshape(n, 4, 24)
        kappa[:, :, 24:] = spare[:, :, 0] | (spare[:, :, 1] << 1) | (spare[:, :, 2] << 2)
        kappa = kappa.reshape(n, 128)
    h = 1 << (bits - 1)
    sign = kappa >> (bits - 1)
    rank = kappa & (h - 1)
    idx = np.where(sign == 0, h + rank, h - 1 - rank)
    return idx.astype(np.uint8).reshape(*packed.shape[:-1], 128)


def torch_device():
    import torch
    return torch.device("cuda", 0)


def upload(x, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def gpu_cache_from_records(mode, B, Hkv, cap, lengths, kdata, knorm, vdata, vnorm, device,
                           v_rescale=1.0, rot_seed=42, codebook_k=None, codebook_v=None):
    """A library Cache whose buffers hold the given records (numpy, [B,Hkv,cap,...]);
    the standard codebooks unless others are given."""
    import torch
    import quantized_kv_cache_flash_gb300 as tqf
    c = tqf.Cache(tqf.MODES[mode], B, Hkv, cap, device, rot_seed=rot_seed, v_rescale=v_rescale,
                  codebook_k=None if codebook_k is None else [float(x) for x in codebook_k],
                  codebook_v=None if codebook_v is None else [float(x) for x in codebook_v])
    c.k_data.copy_(upload(kdata, device))
    if c.k_norm is not None:
        c.k_norm.copy_(upload(knorm, device))
    c.v_data.copy_(upload(vdata, device))
    if c.v_norm is not None:
        c.v_norm.copy_(upload(vnorm, device))
    c.lengths.copy_(torch.from_numpy(np.asarray(lengths, np.int32)))
    return c


def random_cache(mode, B, Hkv, cap, key):
    """Random packed records straight from the input generator (numpy)."""
    kb, vb = MODE_BITS[mode]
    rows = B * Hkv * cap
    if mode in TABLE_MODES:
        # random 3-bit codes and tables built from random norms (the table is
        # format data: values drawn from the generator, not computed by the kernels)
        kcodes = wl.random_codes(key, rows, 48).reshape(B, Hkv, cap, 48)
        vcodes = wl.random_codes(key + 1, rows, 48).reshape(B, Hkv, cap, 48)
        cb = o.codebook(3)
        kt = o.centroid_norm_table(wl.random_norms(key, rows).reshape(B, Hkv, cap), cb)
        vt = o.centroid_norm_table(wl.random_norms(key + 1, rows).reshape(B, Hkv, cap), cb)
        kdata = np.concatenate([kcodes, kt.astype("<f2").view(np.uint8)], axis=-1)
        vdata = np.concatenate([vcodes, vt.astype("<f2").view(np.uint8)], axis=-1)
        return kdata, None, vdata, None
    if kb == 16:
        kdata = wl.random_fp16(key, (B, Hkv, cap, 128))
        knorm = None
    else:
        kdata = wl.random_codes(key, rows, 16 * kb).reshape(B, Hkv, cap, 16 * kb)
        knorm = wl.random_norms(key, rows).reshape(B, Hkv, cap)
    vdata = wl.random_codes(key + 1, rows, 16 * vb).reshape(B, Hkv, cap, 16 * vb)
    vnorm = wl.random_norms(key + 1, rows).reshape(B, Hkv, cap)
    return kdata, knorm, vdata, vnorm


def oracle_unit_from_records(mode, kdata, knorm, vdata, vnorm, b, h, L):
    """Oracle view of unit (b, h) of a record cache (the oracle unpacks the bytes)."""
    kb, vb = MODE_BITS[mode]
    if mode in TABLE_MODES:
        ki, kt = o.unpack_table_records(kdata[b, h, :L])
        vi, vt = o.unpack_table_records(vdata[b, h, :L])
        return {"k_idx": ki, "k_table": kt, "v_idx": vi, "v_table": vt}
    unit = {"v_idx": o.unpack_codes(vdata[b, h, :L], vb), "v_norm": vnorm[b, h, :L]}
    if kb == 16:
        unit["k"] = kdata[b, h, :L]
    else:
        unit["k_idx"] = o.unpack_codes(kdata[b, h, :L], kb)
        unit["k_norm"] = knorm[b, h, :L]
    return unit


def exact_lloyd_max(bits):
    """The Lloyd-Max levels rounded to fp32 instead of fp16: a codebook whose
    entries are not fp16 values (the decode path with the residual product)."""
    return o.lloyd_max(1 << bits)[0].astype(np.float32)


def oracle_decode(mode, q, units, lengths, Hkv, tq, scale, v_rescale, rot_seed=42, cbk=None, cbv=None):
    """Oracle output [B, Hq, Tq, 128] (fp64) from per-unit dicts units[(b, h)]
    (the standard codebooks unless others are given)."""
    kb, vb = MODE_BITS[mode]
    if cbk is None:
        cbk = o.codebook(kb) if kb != 16 else None
    if cbv is None:
        cbv = o.codebook(vb)
    s = o.sign_vector(rot_seed)
    B, Hq = q.shape[0], q.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, tq, 128))
    for (b, h), unit in units.items():
        out[b, h * G:(h + 1) * G] = o.decode_unit(mode, q[b, h * G:(h + 1) * G], unit,
                                                  int(lengths[b]), tq, G, cbk, cbv, s, scale,
                                                  v_rescale)
    return out


def oracle_decode_sparse_v(mode, q, units, lengths, Hkv, tq, scale, v_rescale, tau, rot_seed=42):
    """Oracle sparse-V output and bound, both fp64 [B, Hq, Tq, 128]."""
    kb, vb = MODE_BITS[mode]
    cbk = o.codebook(kb) if kb != 16 else None
    cbv = o.codebook(vb)
    s = o.sign_vector(rot_seed)
    B, Hq = q.shape[0], q.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, tq, 128))
    bound = np.zeros((B, Hq, tq, 128))
    for (b, h), unit in units.items():
        sl = slice(h * G, (h + 1) * G)
        out[b, sl], bound[b, sl] = o.decode_unit_sparse_v(mode, q[b, sl], unit, int(lengths[b]), tq,
                                                          G, cbk, cbv, s, scale, v_rescale, tau)
    return out, bound


def assert_within_skip_bound(got, full, bound, what=""):
    """got may drop any subset of the tokens covered by `bound`: the error left
    after taking `bound` off must meet the ordinary attention bounds."""
    got = np.asarray(got, np.float64)
    rms = math.sqrt(float(np.mean(full * full)))
    excess = np.maximum(np.abs(got - full) - bound, 0.0)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert float(excess.max()) <= MAX_ABS_REL * rms, f"{what}: max excess {excess.max():.3e}"
    assert math.sqrt(float(np.mean(excess * excess))) <= RMS_REL * rms, f"{what}: rms excess"


def assert_attention_close_rows(got, want, what=""):
    """The attention bounds applied to each output row (last axis) against that
    row's own RMS, plus the RMS-error bound over the whole tensor.  For a
    causal prefill block, whose rows range from a single visible token (an
    output about as large as one V vector) to the whole context (an average,
    an order of magnitude smaller), so that one tensor-wide RMS would be set
    by the small rows alone."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    g = got.reshape(-1, got.shape[-1])
    w = want.reshape(-1, want.shape[-1])
    rms_row = np.sqrt(np.mean(w * w, axis=1))
    err = np.abs(g - w)
    zero = rms_row == 0
    assert np.all(g[zero] == 0), f"{what}: rows without visible tokens must be 0"
    live = ~zero
    mx = err[live].max(axis=1) / rms_row[live]
    rm = np.sqrt(np.mean(err[live] ** 2, axis=1)) / rms_row[live]
    assert mx.max() <= MAX_ABS_REL, f"{what}: row max-abs {mx.max():.3e} x its rms"
    assert rm.max() <= RMS_REL, f"{what}: row rms err {rm.max():.3e} x its rms"
    rms = math.sqrt(float(np.mean(w * w)))
    assert math.sqrt(float(np.mean(err * err))) <= RMS_REL * rms, f"{what}: rms err over the tensor"
