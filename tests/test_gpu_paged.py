"""Paged caches: the records of each 128-token block live on a page of a shared pool, found
through a caller block table (the vLLM-style paged KV cache of the KVQuant and TurboQuant
pages' serving sections). Paging changes where a record sits, not what it holds, so a paged
cache must reproduce the contiguous one exactly: on the same inputs and a shuffled block table
with spare pages, every record of (b, h, block) is byte-identical to the contiguous record,
decode outputs (with fp tails) and dequantised tiles are bitwise equal, and both match the
oracle. Covered per decode kernel: the tensor-core kernels (nuq3 pre-RoPE; RTN2; KVarN2; int4)
and the CUDA-core kernel (token-row layout). An out-of-range table entry is reported in the
status word and never addresses memory outside the pool."""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
TOL = 2e-3

CASES = [
    ("nuq3_rope_mma", WL.WORKLOADS[2], dict(batch=3, n_kv_heads=2, n_q_heads=2, ctx=9 * 128), "mma"),
    ("rtn2_mha_mma", WL.WORKLOADS[5], dict(batch=2, n_kv_heads=3, n_q_heads=3, ctx=7 * 128), "mma"),
    ("varn2_gqa_mma", WL.WORKLOADS[3], dict(batch=2, n_kv_heads=2, n_q_heads=8, ctx=5 * 128), "mma"),
    ("int4_gqa_mma", WL.WORKLOADS[4], dict(batch=3, n_kv_heads=2, n_q_heads=8, ctx=6 * 128), "mma"),
    ("nuq3_rope_rows", WL.WORKLOADS[2], dict(batch=2, n_kv_heads=2, n_q_heads=2, ctx=5 * 128), "rows"),
    ("rtn4_gqa_rows", WL.WORKLOADS[5], dict(bits=4, batch=2, n_kv_heads=2, n_q_heads=4, ctx=6 * 128), "rows"),
]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    yield


def _paged_cache(w, layout, n_pages, table):
    import torch
    import bit_kv_cache_block_gb300 as K
    cb = U.codebook_for(w)
    cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, in_dtype=w.dtype,
                        pre_rope=w.pre_rope, rope_theta=w.rope_theta, outlier_frac=w.outlier_frac,
                        varn_iters=w.varn_iters, hadamard=True, layout=layout, n_pages=n_pages)
    return K.KVCache(cfg, None if cb is None else torch.from_numpy(cb), block_table=torch.from_numpy(table))


def _append_in_chunks(cache, w, K, V, edges):
    for a, b in zip(edges[:-1], edges[1:]):
        cache.append(U.to_device(K[:, :, a * 128:b * 128], w.dtype), U.to_device(V[:, :, a * 128:b * 128], w.dtype))


@pytest.mark.parametrize("name,base,kw,layout", CASES, ids=[c[0] for c in CASES])
def test_paged_equals_contiguous(name, base, kw, layout):
    import torch
    w = base.scaled(**kw)
    nb = w.n_blocks
    rng = np.random.default_rng(11)
    n_pages = w.batch * nb + 5                        # spare pages stay unused
    table = rng.permutation(n_pages)[:w.batch * nb].reshape(w.batch, nb).astype(np.int32)
    flat = U.new_cache(w, layout=layout)
    paged = _paged_cache(w, layout, n_pages, table)
    K, V = WL.blocks(w, 0, nb)
    edges = [0, 1, nb // 2, nb]
    _append_in_chunks(flat, w, K, V, edges)
    _append_in_chunks(paged, w, K, V, edges)
    fr, pr = U.records_np(flat), U.records_np(paged)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            for blk in range(nb):
                assert np.array_equal(pr[table[b, blk], h], fr[b, h, blk]), f"{name} record ({b}, {h}, {blk})"
    oc = O.OracleCache.for_workload(w, codebook=U.codebook_for(w)[0] if w.method == "nuq" else None,
                                    layout=U.oracle_layout(layout))
    oc.append(K, V)
    for step, n_tail in ((0, 0), (1, 33)):
        q = WL.query(w, step)
        tk, tv = WL.tail(w, n_tail, step)
        args = (U.to_device(q, w.dtype), U.to_device(tk, w.dtype) if n_tail else None,
                U.to_device(tv, w.dtype) if n_tail else None)
        of, op = flat.decode(*args).cpu().numpy(), paged.decode(*args).cpu().numpy()
        assert np.array_equal(of, op), f"{name} tail={n_tail}: paged decode differs from contiguous"
        ref = oc.decode(q, tk if n_tail else None, tv if n_tail else None)
        assert np.max(np.abs(op.astype(np.float64) - ref)) <= TOL
    dk_f, dv_f = flat.dequant(0, nb, 1)
    dk_p, dv_p = paged.dequant(0, nb, 1)
    assert torch.equal(dk_f, dk_p) and torch.equal(dv_f, dv_p)
    torch.cuda.synchronize()
    assert flat.device_status() == 0 and paged.device_status() == 0


def test_out_of_range_page_is_reported():
    import torch
    import bit_kv_cache_block_gb300 as K
    w = WL.WORKLOADS[2].scaled(batch=2, n_kv_heads=2, n_q_heads=2, ctx=3 * 128)
    nb = w.n_blocks
    n_pages = w.batch * nb
    table = np.arange(n_pages, dtype=np.int32).reshape(w.batch, nb)
    paged = _paged_cache(w, "mma", n_pages, table)
    Kx, Vx = WL.blocks(w, 0, nb)
    paged.append(U.to_device(Kx, w.dtype), U.to_device(Vx, w.dtype))
    torch.cuda.synchronize()
    assert paged.device_status() == 0
    bad = table.copy()
    bad[1, 2] = n_pages                                # one past the pool
    paged.set_block_table(torch.from_numpy(bad))
    out = paged.decode(U.to_device(WL.query(w), w.dtype))
    torch.cuda.synchronize()
    assert paged.device_status() == K._lib.KVQ_ERR_PAGE
    assert torch.isfinite(out).all()
