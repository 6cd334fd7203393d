"""KVQuant's offline-calibrated keys and attention sink on the GPU, against the oracle.

- The calibration table (tau fp32, s and zp fp16 per (KV head, channel)) written by
  kvq_calibrate_keys equals the oracle's calibrate_keys bit for bit (fp16 and bf16 keys; no
  outliers, 1% and 5%).
- Appended records of calibrated caches are bit-exact: key tiles take the table's statistics
  and the entries over tau (capped at the tile's capacity; the CSR's unused capacity is zero),
  value tiles stay per token. With the sink, block 0 holds zeros for the first token and its K
  and V rows are kept as given.
- Decode (with and without an fp tail) is within max-abs 2e-3 of the oracle, on the tensor-core
  nuq kernel and on the CUDA-core kernel (token-row layout; GQA).
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
TOL = 2e-3
N_CAL_BLOCKS = 3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    yield


def _calib_keys(w):
    """Calibration keys [H_kv][N_CAL_BLOCKS*128][128]: the workload's key distribution, another seed."""
    return np.stack([np.concatenate([WL.tile(w, 0, h, blk, WL.KIND_K, seed=99) for blk in range(N_CAL_BLOCKS)])
                     for h in range(w.n_kv_heads)])


def _cache(w, layout, key_calib, sink, paged=False):
    import torch
    import bit_kv_cache_block_gb300 as K
    cb = U.codebook_for(w)
    n_pages = w.batch * w.n_blocks + 3 if paged else 0
    cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, in_dtype=w.dtype,
                        pre_rope=w.pre_rope, rope_theta=w.rope_theta, outlier_frac=w.outlier_frac, layout=layout,
                        n_pages=n_pages, key_calib=key_calib, sink=sink)
    table = None
    if paged:
        table = torch.from_numpy(np.random.default_rng(3).permutation(n_pages)[:w.batch * w.n_blocks]
                                 .reshape(w.batch, w.n_blocks).astype(np.int32))
    return K.KVCache(cfg, torch.from_numpy(cb), block_table=table)


def _device_table(cache, H):
    lay = cache.layout
    raw = cache.base[int(lay.calib_off):int(lay.calib_off + lay.calib_bytes)].cpu().numpy()
    tau = raw[:H * 128 * 4].view(np.float32).reshape(H, 128)
    s16 = raw[H * 128 * 4:H * 128 * 6].view(np.uint16).reshape(H, 128)
    zp16 = raw[H * 128 * 6:].view(np.uint16).reshape(H, 128)
    return tau, s16, zp16


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("frac", [0.0, 0.01, 0.05])
def test_calibration_table_matches_oracle(dtype, frac):
    import torch
    w = WL.WORKLOADS[2].scaled(batch=1, n_kv_heads=3, n_q_heads=3, ctx=2 * 128, dtype=dtype, outlier_frac=frac)
    cache = _cache(w, "mma", True, False)
    kc = _calib_keys(w)
    cache.calibrate_keys(U.to_device(kc, w.dtype))
    torch.cuda.synchronize()
    tau, s16, zp16 = _device_table(cache, w.n_kv_heads)
    for h in range(w.n_kv_heads):
        et, es, ez = O.calibrate_keys(kc[h], frac)
        assert np.array_equal(tau[h], et), f"tau h={h}"
        assert np.array_equal(s16[h], U.f16_bits(es)) and np.array_equal(zp16[h], U.f16_bits(ez)), f"s/zp h={h}"


CASES = [
    ("mma_calib_sink", "mma", dict(batch=2, n_kv_heads=2, n_q_heads=2, ctx=5 * 128), True, True),
    ("mma_sink", "mma", dict(batch=1, n_kv_heads=3, n_q_heads=3, ctx=4 * 128), False, True),
    ("mma_calib_5pct", "mma", dict(batch=1, n_kv_heads=2, n_q_heads=2, ctx=4 * 128, outlier_frac=0.05), True, False),
    ("rows_calib_sink", "rows", dict(batch=2, n_kv_heads=2, n_q_heads=2, ctx=3 * 128), True, True),
    ("gqa_norope_calib_sink", "mma", dict(batch=1, n_kv_heads=2, n_q_heads=8, ctx=3 * 128, pre_rope=False), True, True),
]


@pytest.mark.parametrize("name,layout,kw,key_calib,sink", CASES, ids=[c[0] for c in CASES])
def test_calibrated_sink_records_and_decode(name, layout, kw, key_calib, sink):
    import torch
    w = WL.WORKLOADS[2].scaled(**kw)
    nb = w.n_blocks
    cache = _cache(w, layout, key_calib, sink)
    calib = None
    if key_calib:
        kc = _calib_keys(w)
        cache.calibrate_keys(U.to_device(kc, w.dtype))
        parts = [O.calibrate_keys(kc[h], w.outlier_frac) for h in range(w.n_kv_heads)]
        calib = tuple(np.stack([p[i] for p in parts]) for i in range(3))
    Kx, Vx = WL.blocks(w, 0, nb)
    cache.append(U.to_device(Kx[:, :, :128], w.dtype), U.to_device(Vx[:, :, :128], w.dtype))
    cache.append(U.to_device(Kx[:, :, 128:], w.dtype), U.to_device(Vx[:, :, 128:], w.dtype))
    oc = O.OracleCache.for_workload(w, codebook=U.codebook_for(w)[0], layout=U.oracle_layout(layout),
                                    key_calib=calib, sink=sink)
    oc.append(Kx, Vx)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    recs = U.records_np(cache)
    n_cap = int(cache.layout.n_outliers)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            for blk in range(nb):
                for kind in (0, 1):
                    got = U.tile_fields(recs[b, h, blk], cache.layout, kind, "nuq", 3, layout)
                    exp = oc.recs[(b, h, blk, kind)]
                    where = f"{name} b={b} h={h} blk={blk} kind={kind}"
                    assert np.array_equal(got["words"], exp["words"]), where + " code words"
                    assert np.array_equal(U.f16_bits(got["s16"]), U.f16_bits(exp["s16"])), where + " s"
                    assert np.array_equal(U.f16_bits(got["zp16"]), U.f16_bits(exp["zp16"])), where + " zp"
                    if n_cap:
                        n = len(exp["col"])
                        assert np.array_equal(got["row_ptr"], exp["row_ptr"]), where + " row_ptr"
                        assert np.array_equal(got["val"][:n], exp["val"]) and not got["val"][n:].any(), where + " val"
                        assert np.array_equal(got["col"][:n], exp["col"]) and not got["col"][n:].any(), where + " col"
    if sink:
        lay = cache.layout
        kept = cache.base[int(lay.sink_off):int(lay.sink_off + lay.sink_bytes)].cpu().numpy().view(np.uint16)
        kept = kept.reshape(w.batch, w.n_kv_heads, 2, 128)
        assert np.array_equal(kept[:, :, 0], WL.to_storage(Kx[:, :, 0], w.dtype))
        assert np.array_equal(kept[:, :, 1], WL.to_storage(Vx[:, :, 0], w.dtype))
    for step, n_tail in ((0, 0), (1, 55)):
        q = WL.query(w, step)
        tk, tv = WL.tail(w, n_tail, step)
        out = cache.decode(U.to_device(q, w.dtype), U.to_device(tk, w.dtype) if n_tail else None,
                           U.to_device(tv, w.dtype) if n_tail else None).cpu().numpy().astype(np.float64)
        ref = oc.decode(q, tk if n_tail else None, tv if n_tail else None)
        err = np.max(np.abs(out - ref))
        assert err <= TOL, f"{name} tail={n_tail}: max abs err {err:.3e}"
    torch.cuda.synchronize()
    assert cache.device_status() == 0


def test_paged_sink_equals_contiguous():
    w = WL.WORKLOADS[2].scaled(batch=2, n_kv_heads=2, n_q_heads=2, ctx=4 * 128)
    flat, paged = _cache(w, "mma", True, True), _cache(w, "mma", True, True, paged=True)
    kc = U.to_device(_calib_keys(w), w.dtype)
    Kx, Vx = WL.blocks(w, 0, w.n_blocks)
    for c in (flat, paged):
        c.calibrate_keys(kc)
        c.append(U.to_device(Kx, w.dtype), U.to_device(Vx, w.dtype))
    q = U.to_device(WL.query(w), w.dtype)
    tk, tv = WL.tail(w, 9)
    a = flat.decode(q, U.to_device(tk, w.dtype), U.to_device(tv, w.dtype)).cpu().numpy()
    b = paged.decode(q, U.to_device(tk, w.dtype), U.to_device(tv, w.dtype)).cpu().numpy()
    assert np.array_equal(a, b)
