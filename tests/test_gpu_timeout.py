"""The failure path of the decode's bounded waits, on the GPU, without faulting or hanging it.

Under the test switch kvq_debug_stall_decode the 3-bit nuq tensor-core decode runs with its
copy-issuing warp idle and its waits bounded at about 1 ms, so no stage ever lands (a flag that
nothing sets): every wait must run out, the status word must read KVQ_ERR_TIMEOUT, the output must
be NaN (never a merge of stale partials), and the call must return. With the switch off and the
status cleared, the next decode of the same cache must be correct (the context stays usable).
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    yield


def test_decode_wait_timeout_is_reported_and_recoverable():
    import time
    import torch
    import bit_kv_cache_block_gb300 as K
    w = WL.WORKLOADS[2].scaled(batch=1, n_kv_heads=2, n_q_heads=2, ctx=6 * 128)
    cache = U.new_cache(w, layout="mma")   # nuq3, pre-RoPE keys, one query head per KV head
    Kx, Vx = WL.blocks(w, 0, w.n_blocks)
    cache.append(U.to_device(Kx, w.dtype), U.to_device(Vx, w.dtype))
    q = WL.query(w)
    qd = U.to_device(q, w.dtype)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    K.kvq_debug_stall_decode(True)
    try:
        t0 = time.time()
        out = cache.decode(qd)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        K.kvq_debug_stall_decode(False)
    assert cache.device_status() == K._lib.KVQ_ERR_TIMEOUT
    assert torch.isnan(out).all()
    assert elapsed < 5.0, f"the stalled decode took {elapsed:.2f} s"
    cache.status.zero_()
    out = cache.decode(qd)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    oc = O.OracleCache.for_workload(w, codebook=U.codebook_for(w)[0], layout=O.LAYOUT_MMA)
    oc.append(Kx, Vx)
    err = np.max(np.abs(out.cpu().numpy().astype(np.float64) - oc.decode(q)))
    assert err <= 2e-3, f"decode after the timeout: max abs err {err:.3e}"
