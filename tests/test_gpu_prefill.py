"""GPU parity of chunked-prefill attention (tcgen05) against the fp64 oracle.

Query j of a Tq block sees tokens [0, L - Tq + j]; the cases cover a prompt
prefilled into an empty cache (L = Tq), a chunk appended behind an existing
context, group sizes 1, 2, 4, 7 and 8 (7 leaves padding rows in the 128-row
tiles), every mode with its own record format, a hint below the lengths, and
Tq = 1 (which must agree with the decode kernel).  The attention bounds are
applied per output row against that row's RMS (a causal block's rows range
from one visible token to the whole context), plus the RMS-error bound over
the whole tensor.
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


CASES = [
    # mode, B, Hq, Hkv, lengths, Tq, cap, max_len hint (None = max length), q scale
    ("turbo4", 1, 8, 2, [300], 300, 304, None, 1.0),            # prompt into an empty cache, G 4
    ("turbo3", 2, 28, 4, [700, 450], 200, 704, None, 1.0),      # chunk behind a context, G 7, ragged
    ("turbo4_asym", 1, 4, 2, [513], 513, 528, None, 1.0),       # fp16 K through the tensor map, G 2
    ("turbo3_asym", 1, 8, 8, [260], 130, 272, None, 1.0),       # G 1: 128 positions per tile
    ("turbo4k_3v", 1, 16, 2, [1000], 64, 1008, None, 1.0),      # G 8
    ("turbo4", 2, 8, 2, [100, 37], 1, 112, None, 1.0),          # Tq 1
    ("turbo3", 1, 8, 2, [600], 300, 608, 450, 1.0),             # hint below the length
    ("turbo3", 1, 8, 2, [200], 200, 208, None, 1.0),            # two K/V tiles: no copy past the prologue's
    ("turbo4", 1, 8, 2, [128], 128, 128, None, 1.0),            # one full K/V tile
    ("turbo4_asym", 1, 8, 2, [256], 256, 256, None, 1.0),       # fp16 K, two full tiles
    ("turbo4", 2, 16, 2, [1300, 1290], 1290, 1312, None, 1.0),  # eleven tiles: slot phases wrap several times
    # peaked softmax: scores of 20 .. 100, where one fp16 rounding of the
    # rotated query would move the dominant weights by a per cent
    ("turbo4", 1, 8, 2, [300], 300, 304, None, 8.0),
    ("turbo3", 2, 28, 4, [700, 450], 200, 704, None, 32.0),
    ("turbo4_asym", 1, 4, 2, [513], 513, 528, None, 32.0),
    ("turbo4k_3v", 1, 16, 2, [1000], 64, 1008, None, 16.0),
    ("turbo3_asym", 1, 8, 8, [260], 130, 272, None, 32.0),
]


@pytest.mark.parametrize("case", CASES,
                         ids=lambda c: f"{c[0]}-Hq{c[2]}-Hkv{c[3]}-L{max(c[4])}-Tq{c[5]}-q{c[8]:g}")
def test_prefill_same_cache(case):
    mode, B, Hq, Hkv, lengths, Tq, cap, hint, qs = case
    hint = hint or max(lengths)
    key = 12000 + sum(lengths) + Tq
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, key)
    q = wl.random_fp16(key + 5, (B, Hq, Tq, 128), scale=qs)
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, DEV, v_rescale=0.5)
    ctx = tqf.Context()
    qd = H.upload(q, DEV)
    out = torch.full_like(qd, float("nan"))
    tqf.tq_prefill_attention(ctx, cache, qd, out, hint)
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == 0
    got = out.float().cpu().numpy()
    vis = [min(L, hint) for L in lengths]
    units = {(b, h): H.oracle_unit_from_records(mode, kd, kn, vd, vn, b, h, vis[b])
             for b in range(B) for h in range(Hkv)}
    # the causal position is the true length; tokens past the hint are not read
    want = np.zeros((B, Hq, Tq, 128))
    G = Hq // Hkv
    kb, vb = H.MODE_BITS[mode]
    s = o.sign_vector(42)
    cbk = o.codebook(kb) if kb != 16 else None
    cbv = o.codebook(vb)
    for (b, h), u in units.items():
        K, V = o.unit_kv_full(mode, u, cbk, cbv, s)
        qq = q[b, h * G:(h + 1) * G].astype(np.float64).reshape(G * Tq, 128)
        visible = np.tile([min(lengths[b] - Tq + j + 1, vis[b]) for j in range(Tq)], G)
        want[b, h * G:(h + 1) * G] = (o.softmax_attention(qq, K, V * 0.5, 1 / math.sqrt(128), visible)
                                      .reshape(G, Tq, 128))
    H.assert_attention_close_rows(got, want, str(case))


def test_prefill_tq1_matches_decode_kernel():
    mode, B, Hq, Hkv, cap = "turbo4", 3, 32, 8, 2048
    lengths = [2000, 517, 1]
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 777)
    q = H.upload(wl.random_fp16(778, (B, Hq, 1, 128)), DEV)
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, DEV)
    ctx = tqf.Context()
    a, d = torch.empty_like(q), torch.empty_like(q)
    tqf.tq_prefill_attention(ctx, cache, q, a, 2000)
    tqf.tq_decode_attention(ctx, cache, q, d, 2000)
    torch.cuda.synchronize()
    H.assert_attention_close(a.float().cpu().numpy(), d.float().cpu().numpy(), "prefill vs decode")


def test_prefill_rejects_a_codebook_of_non_fp16_levels():
    mode, B, Hq, Hkv, cap = "turbo4", 1, 8, 2, 64
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 31)
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, [40], kd, kn, vd, vn, DEV,
                                     codebook_k=H.exact_lloyd_max(4))
    q = H.upload(wl.random_fp16(32, (B, Hq, 8, 128)), DEV)
    out = torch.empty_like(q)
    with pytest.raises(tqf.TqError) as e:
        tqf.tq_prefill_attention(tqf.Context(), cache, q, out, 40)
    assert e.value.code == tqf.TQ_ERR_UNSUPPORTED


def test_prefill_after_own_append_end_to_end():
    # a 384-token prompt: encode_append into an empty cache, then prefill attention
    mode, B, Hq, Hkv, T, cap = "turbo3", 1, 28, 4, 384, 400
    k = np.stack([wl.random_fp16(600 + h, (T, 128)) for h in range(Hkv)])[None]
    k[..., [5, 60, 90, 111]] = (k[..., [5, 60, 90, 111]].astype(np.float32) * 8).astype(np.float16)
    v = np.stack([wl.random_fp16(700 + h, (T, 128)) for h in range(Hkv)])[None]
    q = wl.random_fp16(801, (B, Hq, T, 128))
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.MODES[mode], B, Hkv, cap, DEV)
    tqf.tq_encode_append(ctx, cache, H.upload(k, DEV), H.upload(v, DEV))
    qd = H.upload(q, DEV)
    out = torch.empty_like(qd)
    tqf.tq_prefill_attention(ctx, cache, qd, out, T)
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == 0
    s = o.sign_vector(42)
    cb = o.codebook(3)
    units = {}
    for h in range(Hkv):
        ki, kn_, _, _ = o.encode(k[0, h], cb, s)
        vi, vn_, _, _ = o.encode(v[0, h], cb, s)
        units[(0, h)] = {"k_idx": ki, "k_norm": kn_, "v_idx": vi, "v_norm": vn_}
    want = H.oracle_decode(mode, q, units, [T], Hkv, T, 1 / math.sqrt(128), 1.0)
    H.assert_attention_close_rows(out.float().cpu().numpy(), want, "prefill e2e")
