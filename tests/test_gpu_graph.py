"""A decode step (append one token per sequence, then attend) captured into a
CUDA graph and replayed (GPU).

After one eager call has sized the context's workspace, the step's kernels
can be captured: the encode's tensor maps are built on the host at capture
time, its tile and ticket counters and the status word live in device memory
and are back at zero after every launch, and the decode's grid is fixed by the
length hint given at capture (so the hint covers the lengths of every
replay).  Each replay appends the next token and decodes over the grown
context; the outputs must be bit-identical to the same steps run eagerly on
an identical cache.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import quantized_kv_cache_flash_gb300 as tqf
from quantized_kv_cache_flash_gb300 import workloads as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_kv_cache_flash_gb300 import build
    build.build()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("mode,B,Hq,Hkv,t_new", [
    ("turbo4", 4, 32, 8, 1),       # a decode step's append (a warp per vector)
    ("turbo3", 2, 28, 4, 640),     # a chunk append: 5120 vectors per stream (tensor-core encode)
    ("turbo4_asym", 2, 28, 4, 1),
])
def test_step_replayed_from_a_graph_matches_eager(dev, mode, B, Hq, Hkv, t_new):
    L0, cap, steps = 1500, 4096, 3
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 500 + t_new)
    lens = [L0, L0 - 77][:B] + [L0 - 13] * max(0, B - 2)
    caches = [H.gpu_cache_from_records(mode, B, Hkv, cap, lens, kd, kn, vd, vn, dev) for _ in range(2)]
    ctxs = [tqf.Context(), tqf.Context()]
    hint = cap
    k_in = torch.empty(B, Hkv, t_new, 128, dtype=torch.float16, device=dev)
    v_in = torch.empty_like(k_in)
    q_in = torch.empty(B, Hq, 1, 128, dtype=torch.float16, device=dev)
    out_g = torch.empty_like(q_in)

    def data(i):
        return (H.upload(wl.random_fp16(900 + 3 * i, (B, Hkv, t_new, 128)), dev),
                H.upload(wl.random_fp16(901 + 3 * i, (B, Hkv, t_new, 128)), dev),
                H.upload(wl.random_fp16(902 + 3 * i, (B, Hq, 1, 128)), dev))

    # warm-up on the graph's cache (sizes the workspace), step 0
    k, v, q = data(0)
    k_in.copy_(k); v_in.copy_(v); q_in.copy_(q)
    tqf.tq_encode_append(ctxs[0], caches[0], k_in, v_in)
    tqf.tq_decode_attention(ctxs[0], caches[0], q_in, out_g, hint)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            tqf.tq_encode_append(ctxs[0], caches[0], k_in, v_in)
            tqf.tq_decode_attention(ctxs[0], caches[0], q_in, out_g, hint)
    torch.cuda.synchronize()

    # eager reference: the same steps (0 .. steps) on the second cache
    want = []
    for i in range(steps + 1):
        k, v, q = data(i)
        o = torch.empty_like(q)
        tqf.tq_encode_append(ctxs[1], caches[1], k, v)
        tqf.tq_decode_attention(ctxs[1], caches[1], q, o, hint)
        want.append(o)
    torch.cuda.synchronize()
    assert torch.equal(out_g, want[0])
    for i in range(1, steps + 1):
        k, v, q = data(i)
        k_in.copy_(k); v_in.copy_(v); q_in.copy_(q)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, want[i]), f"replay {i}"
    assert caches[0].lengths.cpu().tolist() == caches[1].lengths.cpu().tolist()
    assert caches[0].lengths.cpu().tolist() == [n + (steps + 1) * t_new for n in lens]
    assert tqf.tq_get_status(ctxs[0]) == 0 and tqf.tq_get_status(ctxs[1]) == 0
    assert torch.equal(caches[0].v_data, caches[1].v_data)
    assert torch.equal(caches[0].k_data, caches[1].k_data)
