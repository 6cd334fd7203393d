"""Value outliers stored by column (CSC, [KVQ] §3.4 "by column") on the GPU.

- Append: every record bit-exact against the oracle's CSC value tiles (keys stay CSR), both
  code layouts, 1% and 5% outliers, 2/3/4 bits, with and without pre-RoPE keys.
- Decode (the CUDA-core kernel and the tensor-core nuq kernel), dequant and the error
  statistics of a CSC cache are bitwise those of the same cache with CSR value tiles: the
  outlier set is the same, the per-channel sums run in the same token order, and the
  tensor-core kernel's outlier sums are exact integers. Decode also within 2e-3 of the oracle.
- Calibrated keys with an attention sink and a CSC value tile; a paged CSC cache.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U
from tests.test_gpu_parity import _compare_exact, _oracle_cache

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    yield


CASES = [
    ("nuq3_rope", dict(batch=1, n_kv_heads=2, n_q_heads=2, ctx=3 * 128)),
    ("nuq3_5pct_gqa", dict(outlier_frac=0.05, batch=2, n_kv_heads=2, n_q_heads=4, ctx=2 * 128)),
    ("nuq3_5pct_mha", dict(outlier_frac=0.05, batch=1, n_kv_heads=2, n_q_heads=2, ctx=2 * 128)),
    ("nuq2", dict(bits=2, batch=1, n_kv_heads=1, n_q_heads=1, ctx=2 * 128)),
    ("nuq4_norope", dict(bits=4, pre_rope=False, batch=1, n_kv_heads=2, n_q_heads=2, ctx=2 * 128)),
]


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("layout", ["rows", "mma"])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_csc_records_and_equal_to_csr(name, kw, layout):
    import torch
    w = WL.WORKLOADS[2].scaled(**kw)
    Kx, Vx = WL.blocks(w, 0, w.n_blocks)
    Kd, Vd = U.to_device(Kx, w.dtype), U.to_device(Vx, w.dtype)
    csc = U.new_cache(w, layout=layout, v_csc=True)
    csr = U.new_cache(w, layout=layout)
    csc.append(Kd, Vd)
    csr.append(Kd, Vd)
    oc = _oracle_cache(w, layout, v_csc=True)
    oc.append(Kx, Vx)
    torch.cuda.synchronize()
    assert csc.device_status() == 0 and csr.device_status() == 0
    _compare_exact(csc, oc, w, w.n_blocks, layout)
    for n_tail in (0, 37):
        q = WL.query(w, 1)
        tk, tv = WL.tail(w, n_tail, 1)
        args = (U.to_device(q, w.dtype), U.to_device(tk, w.dtype) if n_tail else None,
                U.to_device(tv, w.dtype) if n_tail else None)
        a, b = csc.decode(*args), csr.decode(*args)
        assert np.array_equal(_bits(a.float()), _bits(b.float())), f"{name} {layout} tail={n_tail}: CSC != CSR"
        ref = oc.decode(q, tk if n_tail else None, tv if n_tail else None)
        err = np.max(np.abs(a.cpu().numpy().astype(np.float64) - ref))
        assert err <= TOL, f"{name} {layout} tail={n_tail}: max abs err {err:.3e}"
    for x, y in zip(csc.dequant(0, w.n_blocks), csr.dequant(0, w.n_blocks)):
        assert np.array_equal(_bits(x), _bits(y))
    for x, y in zip(csc.error_stats(Kd, Vd), csr.error_stats(Kd, Vd)):
        assert np.array_equal(_bits(x), _bits(y))
    torch.cuda.synchronize()
    assert csc.device_status() == 0


@pytest.mark.parametrize("layout", ["rows", "mma"])
def test_csc_with_calibrated_keys_sink_and_pages(layout):
    """CSC value tiles next to calibrated keys and a kept first token, on a shuffled page pool:
    records exact against the oracle, decode equal to the CSR cache's."""
    import torch
    import bit_kv_cache_block_gb300 as K
    w = WL.WORKLOADS[2].scaled(batch=2, n_kv_heads=2, n_q_heads=2, ctx=3 * 128)
    Kx, Vx = WL.blocks(w, 0, w.n_blocks)
    calib = np.stack([np.concatenate([WL.tile(w, 0, h, blk, WL.KIND_K, seed=99) for blk in range(3)])
                      for h in range(w.n_kv_heads)])   # calibration keys [H_kv][384][128], another seed
    cb = U.codebook_for(w)
    rng = np.random.default_rng(3)
    n_pages = w.batch * w.n_blocks + 3
    table = rng.permutation(n_pages)[:w.batch * w.n_blocks].reshape(w.batch, w.n_blocks).astype(np.int32)
    outs = []
    for csc in (True, False):
        cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, w.dtype, w.pre_rope,
                            w.rope_theta, w.outlier_frac, layout=layout, key_calib=True, sink=True, v_csc=csc,
                            n_pages=n_pages)
        cache = K.KVCache(cfg, torch.from_numpy(cb), block_table=torch.from_numpy(table))
        cache.calibrate_keys(U.to_device(calib, w.dtype))
        cache.append(U.to_device(Kx, w.dtype), U.to_device(Vx, w.dtype))
        q = WL.query(w, 2)
        tk, tv = WL.tail(w, 11, 2)
        outs.append(cache.decode(U.to_device(q, w.dtype), U.to_device(tk, w.dtype), U.to_device(tv, w.dtype)))
        torch.cuda.synchronize()
        assert cache.device_status() == 0
        if csc:
            parts = [O.calibrate_keys(calib[h], w.outlier_frac) for h in range(w.n_kv_heads)]
            table_o = tuple(np.stack([p[i] for p in parts]) for i in range(3))
            oc = O.OracleCache.for_workload(w, codebook=cb[0], layout=U.oracle_layout(layout),
                                            key_calib=table_o, sink=True, v_csc=True)
            oc.append(Kx, Vx)
            recs = U.records_np(cache)   # [n_pages][H_kv][record bytes]: page of (b, blk) is table[b][blk]
            for b in range(w.batch):
                for h in range(w.n_kv_heads):
                    for blk in range(w.n_blocks):
                        got = U.tile_fields(recs[table[b, blk], h], cache.layout, 1, "nuq", w.bits, layout)
                        ptr, idx, val = U.sparse_parts(oc.recs[(b, h, blk, 1)])
                        assert np.array_equal(got["row_ptr"], ptr) and np.array_equal(got["col"], idx)
                        assert np.array_equal(got["val"], val)
            err = np.max(np.abs(outs[0].cpu().numpy().astype(np.float64) - oc.decode(q, tk, tv)))
            assert err <= TOL, f"max abs err {err:.3e}"
    assert np.array_equal(_bits(outs[0].float()), _bits(outs[1].float()))
