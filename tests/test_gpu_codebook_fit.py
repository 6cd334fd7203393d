"""Sensitivity-weighted nuq codebook fitting ([KVQ] Algorithm 2) on the GPU: the codebook of
every head equals the oracle's bit for bit (its sums are exact 64-bit fixed point, so thread
order cannot matter), for 1..4 bits, one to several heads, sample counts that are not multiples
of the CTA size, zero weights, out-of-range inputs (clamped), iteration caps that stop before
convergence, and samples so close together that the fitted centres are nearly equal (the
kernels' plain-argmin path). A fitted codebook then drives a nuq cache whose decode matches the oracle."""
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


def _samples(H, n, seed, kind):
    rng = np.random.default_rng(seed)
    if kind == "normal":      # normalised like the nuq tiles: values over the tile's half-range
        a = np.tanh(0.8 * rng.standard_normal((H, n)))
    elif kind == "wide":      # includes values outside [-1, 1] (clamped)
        a = 1.3 * rng.standard_normal((H, n))
    elif kind == "tiny":      # all within 1e-7 of 0: the fitted centres end up closer than 2^-21,
        a = 5e-8 * rng.standard_normal((H, n))  # where the kernels fall back to the plain argmin
    else:                     # uniform
        a = rng.uniform(-1, 1, (H, n))
    w = rng.uniform(0, 1, (H, n)) ** 2
    w[:, ::7] = 0.0           # zero weights
    if kind == "wide":
        w[:, 1::11] = 1.7     # weights above 1 (clamped)
    return a.astype(np.float32), w.astype(np.float32)


@pytest.mark.parametrize("H,n,bits,max_iter,kind", [
    (1, 1, 3, 5, "normal"), (1, 300, 1, 20, "uniform"), (2, 5000, 2, 30, "normal"), (3, 20011, 3, 50, "wide"),
    (4, 65536, 4, 40, "normal"), (2, 100003, 3, 3, "normal"), (8, 4096, 3, 200, "uniform"),
    (1, 5000, 2, 30, "tiny"), (2, 3001, 3, 30, "tiny")])
def test_fit_codebook_matches_oracle(H, n, bits, max_iter, kind):
    import torch
    import bit_kv_cache_block_gb300 as K
    a, w = _samples(H, n, H * 1000 + n, kind)
    got = K.fit_codebook(torch.from_numpy(a).cuda(), torch.from_numpy(w).cuda(), bits, max_iter).cpu().numpy()
    for h in range(H):
        exp, _ = O.fit_codebook(a[h], w[h], bits, max_iter)
        assert np.array_equal(got[h].view(np.uint32), exp.view(np.uint32)), (h, got[h], exp)
    again = K.fit_codebook(torch.from_numpy(a).cuda(), torch.from_numpy(w).cuda(), bits, max_iter).cpu().numpy()
    assert np.array_equal(got, again)


def test_fitted_codebook_drives_a_cache():
    import torch
    import bit_kv_cache_block_gb300 as K
    w_ = WL.WORKLOADS[2].scaled(batch=1, n_kv_heads=2, n_q_heads=2, ctx=3 * 128)
    a, wt = _samples(2, 30000, 7, "normal")
    cb = K.fit_codebook(torch.from_numpy(a).cuda(), torch.from_numpy(wt).cuda(), 3, 60)
    cache = K.KVCache(U.cfg_for(w_, layout="mma"), cb)
    Kx, Vx = WL.blocks(w_, 0, w_.n_blocks)
    cache.append(U.to_device(Kx, w_.dtype), U.to_device(Vx, w_.dtype))
    cbn = cb.cpu().numpy()
    oc = O.OracleCache.for_workload(w_, codebook=cbn, layout=O.LAYOUT_MMA)
    oc.append(Kx, Vx)
    q = WL.query(w_)
    out = cache.decode(U.to_device(q, w_.dtype)).cpu().numpy()
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    assert np.max(np.abs(out - oc.decode(q))) <= 2e-3
