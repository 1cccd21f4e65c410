"""Failure path on the GPU without a fault: a bounded in-kernel wait that
nothing satisfies gives up after its limit, the status word reports it, and
the same context keeps working (a decode right after matches the oracle)."""
import math
import time

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


def test_bounded_wait_gives_up_and_the_context_stays_usable(dev):
    ctx = tqf.Context()
    t0 = time.perf_counter()
    tqf.tq_selftest_bounded_wait(ctx, 2000)   # 2 ms limit
    status = tqf.tq_get_status(ctx)
    dt = time.perf_counter() - t0
    assert status == tqf.TQ_STATUS_PIPELINE_STALL
    assert dt < 1.0
    assert tqf.tq_get_status(ctx) == 0         # read clears it
    mode, B, Hq, Hkv, L, cap = "turbo4", 1, 8, 2, 300, 304
    kd, kn, vd, vn = H.random_cache(mode, B, Hkv, cap, 4321)
    cache = H.gpu_cache_from_records(mode, B, Hkv, cap, [L], kd, kn, vd, vn, dev)
    q = wl.random_fp16(4322, (B, Hq, 1, 128))
    out = torch.empty((B, Hq, 1, 128), dtype=torch.float16, device=dev)
    tqf.tq_decode_attention(ctx, cache, H.upload(q, dev), out, L)
    assert tqf.tq_get_status(ctx) == 0
    units = {(0, h): H.oracle_unit_from_records(mode, kd, kn, vd, vn, 0, h, L) for h in range(Hkv)}
    want = H.oracle_decode(mode, q, units, [L], Hkv, 1, 1 / math.sqrt(128), 1.0)
    H.assert_attention_close(out.float().cpu().numpy(), want)
