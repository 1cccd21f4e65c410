"""tq_decode_attention_noalloc against tq_decode_attention (GPU).

The no-allocation entry point serves callers that may not allocate device
memory while decoding (servers that own all device memory through their own
pools, processes under a hard memory budget): it keeps its split-K scratch in
the library's fixed device array instead of a context workspace.  It must give
the same answer as the regular entry point, call after call, although every
call reuses (and leaves behind) the same scratch.
"""
import ctypes

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


CASES = [
    ("turbo4", 2, 8, 2, [3000, 777], 1, 3008),
    ("turbo4_asym", 1, 28, 4, [5000], 1, 5008),
    ("turbo3", 1, 32, 8, [4100], 4, 4112),
    ("turbo3_table", 2, 16, 4, [2049, 300], 1, 2064),   # records carrying their centroid x norm tables
    # 67 x 30 = 2010 (batch, kv head) units of a 2016-slot array: the decode
    # grid is cut to the 6 slots left
    ("turbo4k_3v", 67, 60, 30, [((37 * i) % 60) + 4 for i in range(67)], 1, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}")
def test_noalloc_matches_regular_decode_on_two_calls(dev, case):
    mode, B, Hq, Hkv, lengths, Tq, cap = case
    key = 31000 + sum(lengths)
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, key)
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, lengths, kd, kn, vd, vn, dev)
    ctx = tqf.Context()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        q = H.upload(wl.random_fp16(key + 7 * call, (B, Hq, Tq, 128)), dev)
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        tqf.tq_decode_attention(ctx, cache, q, ref, max(lengths))
        rc = tqf.lib().tq_decode_attention_noalloc(
            ctypes.byref(cache.struct), q.data_ptr(), Hq, Tq, max(lengths), 0.0,
            got.data_ptr(), status.data_ptr(), stream)
        assert rc == tqf.TQ_OK
        torch.cuda.synchronize()
        H.assert_attention_close(got.float().cpu().numpy(), ref.float().cpu().numpy(),
                                 f"{mode} call {call}")
    assert int(status.item()) == 0
    assert tqf.tq_get_status(ctx) == 0


def test_noalloc_rejects_problems_beyond_its_scratch(dev):
    # 64 x 32 (batch x kv heads) unit slots of 8320 bytes exceed the 16 MiB array
    cache = tqf.Cache(tqf.TQ_TURBO4, 64, 32, 16, dev)
    q = torch.zeros(64, 32, 1, 128, dtype=torch.float16, device=dev)
    out = torch.empty_like(q)
    rc = tqf.lib().tq_decode_attention_noalloc(
        ctypes.byref(cache.struct), q.data_ptr(), 32, 1, 16, 0.0, out.data_ptr(), None,
        torch.cuda.current_stream().cuda_stream)
    assert rc == tqf.TQ_ERR_CAPACITY
