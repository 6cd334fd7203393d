"""The long-context streaming workload (LLaMA-7B-shaped MHA layer, batch 1, 2-bit RTN keys per
channel / values per token, up to 1,048,576 tokens) built the way a server grows its cache: one
block, then a bulk append, then one 128-token block per kvq_append_block call, with decodes at
growing fp tails in between, all through the C ABI in the benchmark's code layout.

Two sampled KV heads carry the seeded test inputs and the oracle follows them block by block; the
other heads hold seeded device noise. At contexts of 128, 131072, 524288 and 1048576 cached
tokens (and with tails of 0 to 127 tokens) the decode outputs of the sampled heads must lie
within max-abs 2e-3 of the oracle's fp64 attention and their records of the newest block must
equal the oracle's bit for bit; every decode in between must leave the status word clear and
give finite outputs.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
TOL = 2e-3
SAMPLED = (0, 17)   # KV heads carrying the seeded inputs (batch 0)
CHUNK = 512         # blocks generated per device-noise chunk


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    yield


def test_config5_streaming_append_and_decode():
    import torch
    w = WL.WORKLOADS[5]
    nb_total = w.n_blocks
    assert nb_total * 128 == 1048576 and w.method == "rtn" and w.bits == 2
    cache = U.new_cache(w, layout="mma")
    w1 = w.scaled(batch=1, n_kv_heads=1, n_q_heads=1)
    ocs = {h: O.OracleCache.for_workload(w1, layout=O.LAYOUT_MMA) for h in SAMPLED}
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4242)
    dt = torch.float16

    def inputs(first, n):
        """Device K, V [1][32][n*128][128] (noise, the sampled heads seeded) and the oracle's tiles."""
        shape = (1, w.n_kv_heads, n * 128, 128)
        Kd = torch.randn(shape, generator=gen, device="cuda", dtype=dt)
        Vd = torch.randn(shape, generator=gen, device="cuda", dtype=dt)
        host = {}
        for h in SAMPLED:
            Kh = np.concatenate([WL.tile(w, 0, h, first + i, WL.KIND_K) for i in range(n)])
            Vh = np.concatenate([WL.tile(w, 0, h, first + i, WL.KIND_V) for i in range(n)])
            Kd[0, h] = U.to_device(Kh, w.dtype)
            Vd[0, h] = U.to_device(Vh, w.dtype)
            host[h] = (Kh, Vh)
        return Kd, Vd, host

    def append(first, n):
        Kd, Vd, host = inputs(first, n)
        cache.append(Kd, Vd)
        for h in SAMPLED:
            ocs[h].append(host[h][0][None, None], host[h][1][None, None])

    def decode(step, n_tail, check):
        q = WL.query(w, step)
        tk, tv = WL.tail(w, n_tail, step)
        out = cache.decode(U.to_device(q, w.dtype), U.to_device(tk, w.dtype) if n_tail else None,
                           U.to_device(tv, w.dtype) if n_tail else None)
        torch.cuda.synchronize()
        assert cache.device_status() == 0, f"status after decode at {cache.n_blocks} blocks"
        out = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(out))
        if check:
            L = cache.n_blocks * 128
            for h in SAMPLED:
                ref = ocs[h].decode(q[:, h:h + 1], tk[:, h:h + 1] if n_tail else None,
                                    tv[:, h:h + 1] if n_tail else None)
                err = np.max(np.abs(out[0, h] - ref[0, 0]))
                assert err <= TOL, f"L={L} tail={n_tail} head {h}: max abs err {err:.3e}"
            recs = cache.record_view()
            last = cache.n_blocks - 1
            for h in SAMPLED:
                rec = recs[0, h, last].cpu().numpy()
                for kind in (0, 1):
                    got = U.tile_fields(rec, cache.layout, kind, "rtn", 2, "mma")
                    exp = ocs[h].recs[(0, 0, last, kind)]
                    assert np.array_equal(got["words"], exp["words"]), f"L={L} head {h} kind {kind} words"
                    assert np.array_equal(U.f16_bits(got["s16"]), U.f16_bits(exp["s16"])), f"L={L} h {h} s"
                    assert np.array_equal(U.f16_bits(got["z16"]), U.f16_bits(exp["z16"])), f"L={L} h {h} z"

    step = 0
    append(0, 1)                      # L = 128
    for n_tail in (0, 5):
        decode(step, n_tail, True)
        step += 1
    append(1, 1023)                   # one bulk call: L = 131072
    decode(step, 77, True)
    step += 1
    blk = 1024
    for stop, checks in ((4096, (100,)), (nb_total, (0, 127))):
        while blk < stop:             # one block per call, decodes at growing tails in between
            n = min(CHUNK, stop - blk)
            Kd, Vd, host = inputs(blk, n)
            for i in range(n):
                cache.append(Kd[:, :, i * 128:(i + 1) * 128].contiguous(), Vd[:, :, i * 128:(i + 1) * 128].contiguous())
            for h in SAMPLED:
                ocs[h].append(host[h][0][None, None], host[h][1][None, None])
            blk += n
            if blk < stop:
                decode(step, (37 * step) % 128, False)
                step += 1
        for n_tail in checks:         # L = 524288, then 1048576
            decode(step, n_tail, True)
            step += 1
    assert cache.n_blocks == nb_total
