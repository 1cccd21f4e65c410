"""The five benchmark configurations at their own shape and data, against the
oracle (GPU).

Each configuration is built the way its decode step runs: the cache is filled
through tq_encode_append from the seeded workload generators (outlier K
channels, ragged lengths), the step's own append follows (one token per
sequence for the batched turbo4 configuration, a 4096-token prefill chunk for
the long-context one), then tq_decode_attention runs over the whole grown
cache.  A seeded sample of (batch, kv head) units, at least four per
configuration where there are that many, is checked against the oracle over
its full visible context: the oracle encodes the same fp16 inputs itself, so
the comparison is end to end.

Per configuration the test checks and reports (set TQ_CONFIG_REPORT to a file
path to get them as JSON):
  * max-abs error / RMS and RMS error / RMS of the sampled units' outputs
    (bounds 1e-2 and 2e-3);
  * the encoded records of those units against the oracle's: elements that
    differ, all of them within 1e-5 of a decision midpoint, fewer than 1e-4
    of the elements (the boundary count);
  * for information, the relative RMS difference between attention over the
    quantized cache and over the unquantized fp16 inputs (the quantisation
    error, not a parity bound).
"""
import json
import math
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import quantized_kv_cache_flash_gb300 as tqf
from quantized_kv_cache_flash_gb300 import workloads as wl
from oracle import tq_oracle as o
from tests import helpers as H

pytestmark = pytest.mark.gpu

DEV = None
_REPORT = {}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    global DEV
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_kv_cache_flash_gb300 import build
    build.build()
    DEV = torch.device("cuda", 0)
    yield
    path = os.environ.get("TQ_CONFIG_REPORT")
    if path and _REPORT:
        with open(path, "w") as f:
            json.dump(_REPORT, f, indent=1, sort_keys=True)


def _chunk(w, b_lens, t0, t1):
    """fp16 K and V [B, Hkv, t1 - t0, 128] of tokens [t0, t1) of every unit
    (the workload's seeded streams)."""
    B, Hkv = w.batch, w.num_kv_heads
    k = np.empty((B, Hkv, t1 - t0, 128), np.float16)
    v = np.empty_like(k)
    for b in range(B):
        for h in range(Hkv):
            k[b, h] = wl.keys(w, b, h, t0, t1)
            v[b, h] = wl.values(w, b, h, t0, t1)
    return k, v


def _build(w):
    """The decode step's cache, filled through the library; returns
    (ctx, cache, lengths at the decode)."""
    lens = wl.lengths(w).astype(np.int64)
    B, Hkv = w.batch, w.num_kv_heads
    cap = int(math.ceil(int(lens.max()) / 16) * 16)
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.MODES[w.mode], B, Hkv, cap, DEV, rot_seed=w.rot_seed)
    # the tokens before the step's own append
    tail = max(w.append, w.prefill_chunk, 0)
    pre = int(lens.max()) - tail
    CH = 4096
    t = 0
    while t < pre:
        n = min(CH, pre - t)
        k, v = _chunk(w, lens, t, t + n)
        tqf.tq_encode_append(ctx, cache, H.upload(k, DEV), H.upload(v, DEV))
        t += n
    # ragged sequences: trim to their own length before the step's append
    cache.lengths.copy_(torch.from_numpy((lens - tail).astype(np.int32)))
    if tail:
        k = np.empty((B, Hkv, tail, 128), np.float16)
        v = np.empty_like(k)
        for b in range(B):
            s0 = int(lens[b]) - tail
            for h in range(Hkv):
                k[b, h] = wl.keys(w, b, h, s0, s0 + tail)
                v[b, h] = wl.values(w, b, h, s0, s0 + tail)
        tqf.tq_encode_append(ctx, cache, H.upload(k, DEV), H.upload(v, DEV))
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == 0
    assert cache.lengths.cpu().numpy().tolist() == lens.tolist()
    return ctx, cache, lens


def _sample_units(w, lens, n):
    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    if len(units) <= n:
        return units
    rng = np.random.default_rng(w.seed + 77)
    pick = set()
    # the longest and the shortest sequence, then seeded others
    pick.add((int(np.argmax(lens)), int(rng.integers(w.num_kv_heads))))
    pick.add((int(np.argmin(lens)), int(rng.integers(w.num_kv_heads))))
    while len(pick) < n:
        pick.add(units[int(rng.integers(len(units)))])
    return sorted(pick)


@pytest.mark.parametrize("number", [1, 2, 3, 4, 5])
def test_configuration_matches_oracle(number):
    w = wl.by_number(number)
    ctx, cache, lens = _build(w)
    q = wl.query_all(w)
    qd = H.upload(q, DEV)
    out = torch.empty_like(qd)
    tqf.tq_decode_attention(ctx, cache, qd, out, int(lens.max()))
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == 0
    got = out.float().cpu().numpy()

    kb, vb = H.MODE_BITS[w.mode]
    cbk = o.codebook(kb) if kb != 16 else None
    cbv = o.codebook(vb)
    s = o.sign_vector(w.rot_seed)
    G, Tq = w.group, w.tq
    sc = 1 / math.sqrt(128)
    g_all, w_all, unq_err, unq_ref = [], [], [], []
    elems = near = bad = 0
    for b, h in _sample_units(w, lens, 4):
        L = int(lens[b])
        k = wl.keys(w, b, h, 0, L)
        v = wl.values(w, b, h, 0, L)
        unit = {}
        recs = []
        vi, vn, vu, vov = o.encode(v, cbv, s)
        unit["v_idx"], unit["v_norm"] = vi, vn
        recs.append((cache.v_data, cache.v_norm, vb, vi, vn, vu, vov))
        if kb == 16:
            unit["k"] = k
            assert np.array_equal(cache.k_data[b, h, :L].cpu().numpy(), k)
        else:
            ki, kn, ku, kov = o.encode(k, cbk, s)
            unit["k_idx"], unit["k_norm"] = ki, kn
            recs.append((cache.k_data, cache.k_norm, kb, ki, kn, ku, kov))
        # encode: norms bit-exact, codes bit-exact but for the boundary band
        for data, norm, bits, idx, n16, u, ov in recs:
            assert not ov.any()
            got_n = norm[b, h, :L].cpu().numpy()
            assert np.array_equal(got_n.view(np.uint16), n16.view(np.uint16))
            got_idx = H.decode_records(data[b, h, :L].cpu().numpy(), bits)
            diff = got_idx != idx
            dist = o.boundary_distance(u[diff], o.codebook(bits))  # only where they differ
            elems += diff.size
            near += int((dist < H.BOUNDARY).sum())
            bad += int((dist >= H.BOUNDARY).sum())
        rows = q[b, h * G:(h + 1) * G]
        want = o.decode_unit(w.mode, rows, unit, L, Tq, G, cbk, cbv, s, sc, 1.0)
        g_all.append(got[b, h * G:(h + 1) * G])
        w_all.append(want)
        # the quantisation error (information): the same attention over the raw fp16 K, V
        raw = o.softmax_attention(rows.astype(np.float64).reshape(G * Tq, 128), k.astype(np.float64),
                                  v.astype(np.float64), sc, np.tile(o.visible_counts(L, Tq), G))
        unq_err.append((want.reshape(G * Tq, 128) - raw).ravel())
        unq_ref.append(raw.ravel())
    rms, mx, rmse = H.attention_errors(np.concatenate([x.ravel() for x in g_all]),
                                       np.concatenate([x.ravel() for x in w_all]))
    qerr = math.sqrt(float(np.mean(np.concatenate(unq_err) ** 2)) /
                     float(np.mean(np.concatenate(unq_ref) ** 2)))
    _REPORT[w.name] = {"units": len(g_all), "max_abs_over_rms": mx / rms, "rms_err_over_rms": rmse / rms,
                       "code_elements": elems, "boundary_mismatches": near,
                       "boundary_fraction": near / max(elems, 1), "mismatches_outside_band": bad,
                       "quantisation_rel_rms": qerr}
    print(w.name, json.dumps(_REPORT[w.name]))
    assert bad == 0
    assert near <= max(1, H.BOUNDARY_FRACTION * elems), (near, elems)
    assert mx <= H.MAX_ABS_REL * rms, (mx / rms)
    assert rmse <= H.RMS_REL * rms, (rmse / rms)


def test_prompt_prefill_configuration_matches_oracle_on_sampled_rows():
    """The 8192-token prompt prefill at its own shape and data (Qwen2.5-7B
    attention shape, turbo3, outlier K channels): the prompt appended to an
    empty cache through tq_encode_append (the tensor-core encode), then the
    causal attention of all 8192 queries (tcgen05 prefill).  For two seeded
    kv heads: their records against the oracle's encoding (norms bit-exact,
    codes but for the boundary band); then sampled rows -- every q head of
    those kv heads at positions spanning the first token, both sides of a
    128-token tile boundary, the middle and the last token -- against the
    oracle on the same packed records (per-row bounds) and, end to end,
    against the oracle's own encoding (the bounds over the sampled rows)."""
    w = wl.by_number(6)
    B, Hq, Hkv, T = w.batch, w.num_q_heads, w.num_kv_heads, w.tq
    G = Hq // Hkv
    ctx = tqf.Context()
    cache = tqf.Cache(tqf.MODES[w.mode], B, Hkv, T, DEV, rot_seed=w.rot_seed)
    k, v = _chunk(w, None, 0, T)
    tqf.tq_encode_append(ctx, cache, H.upload(k, DEV), H.upload(v, DEV))
    q = wl.query_all(w)
    qd = H.upload(q, DEV)
    out = torch.full_like(qd, float("nan"))
    tqf.tq_prefill_attention(ctx, cache, qd, out, T)
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == 0
    assert cache.lengths.cpu().tolist() == [T]

    rng = np.random.default_rng(w.seed + 66)
    heads = sorted(set(int(x) for x in rng.choice(Hkv, size=2, replace=False)))
    pos = sorted({0, 1, 127, 128, T // 2, T - 1} | {int(x) for x in rng.integers(2, T - 1, size=2)})
    s = o.sign_vector(w.rot_seed)
    cb = o.codebook(3)
    sc = 1 / math.sqrt(128)
    kd, kn = cache.k_data.cpu().numpy(), cache.k_norm.cpu().numpy()
    vd, vn = cache.v_data.cpu().numpy(), cache.v_norm.cpu().numpy()
    got, same, e2e = [], [], []
    elems = near = bad = 0
    for h in heads:
        ki, kn_, ku, kov = o.encode(k[0, h], cb, s)
        vi, vn_, vu, vov = o.encode(v[0, h], cb, s)
        for data, norm, idx, n16, u, ov in ((kd, kn, ki, kn_, ku, kov), (vd, vn, vi, vn_, vu, vov)):
            assert not ov.any()
            assert np.array_equal(norm[0, h].view(np.uint16), n16.view(np.uint16))
            diff = H.decode_records(data[0, h], 3) != idx
            dist = o.boundary_distance(u[diff], cb)
            elems += diff.size
            near += int((dist < H.BOUNDARY).sum())
            bad += int((dist >= H.BOUNDARY).sum())
        Ks, Vs = o.unit_kv_full(w.mode, H.oracle_unit_from_records(w.mode, kd, kn, vd, vn, 0, h, T), cb, cb, s)
        Ko, Vo = o.unit_kv_full(w.mode, {"k_idx": ki, "k_norm": kn_, "v_idx": vi, "v_norm": vn_}, cb, cb, s)
        for j in pos:
            qq = q[0, h * G:(h + 1) * G, j].astype(np.float64)
            vis = np.full(G, j + 1)
            got.append(out[0, h * G:(h + 1) * G, j].float().cpu().numpy())
            same.append(o.softmax_attention(qq, Ks[:j + 1], Vs[:j + 1], sc, vis))
            e2e.append(o.softmax_attention(qq, Ko[:j + 1], Vo[:j + 1], sc, vis))
    assert bad == 0
    assert near <= max(1, H.BOUNDARY_FRACTION * elems), (near, elems)
    got = np.stack(got)
    H.assert_attention_close_rows(got, np.stack(same), "prompt prefill, sampled rows, same records")
    H.assert_attention_close(got, np.stack(e2e), "prompt prefill, sampled rows, end to end")
