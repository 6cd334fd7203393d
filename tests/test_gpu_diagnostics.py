"""Error diagnostics on the GPU ([KVN] key innovation, Figures 1a/1b), against the oracle.

- kvq_error_stats: per token (|x|, |x_dq| - |x|, E_T, E_D) for every method and layout. The
  oracle reads the same inputs and the cache's own records (each record format is checked bit
  for bit against the oracle's quantiser elsewhere; KVarN codes carry documented +-1 exemptions),
  dequantises them in fp64 and applies the definitions: the kernel is checked on what it adds
  (dequantisation in fp32 plus the sums), within tolerances derived from fp32 rounding.
  The kept first token of a sink cache has zero error exactly.
- kvq_error_topk: k exact and the fp64 sums of E_T, E_M, E_D within 1e-10 relative of the
  oracle's over the same rows (sums in another order), on real statistics and on rows built
  with many equal errors, where only the lower-row-first rule gives the oracle's sums.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
FRACS = [0.001, 0.01, 0.05, 0.1, 0.5, 1.0]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    yield


CASES = [
    ("rtn2_rows", 5, dict(batch=2, n_kv_heads=2, n_q_heads=2, ctx=3 * 128), "rows", {}),
    ("rtn2_mma", 5, dict(batch=1, n_kv_heads=3, n_q_heads=3, ctx=3 * 128), "mma", {}),
    ("varn2_mma", 3, dict(batch=2, n_kv_heads=2, n_q_heads=8, ctx=3 * 128), "mma", {}),
    ("varn2_rows", 3, dict(batch=1, n_kv_heads=2, n_q_heads=4, ctx=2 * 128), "rows", {}),
    ("int4_bf16_mma", 4, dict(batch=2, n_kv_heads=2, n_q_heads=8, ctx=3 * 128), "mma", {}),
    ("nuq3_mma", 2, dict(batch=1, n_kv_heads=3, n_q_heads=3, ctx=3 * 128), "mma", {}),
    ("nuq3_rows", 2, dict(batch=2, n_kv_heads=2, n_q_heads=2, ctx=2 * 128), "rows", {}),
    ("nuq3_calib_sink", 2, dict(batch=2, n_kv_heads=2, n_q_heads=2, ctx=3 * 128), "mma",
     dict(key_calib=True, sink=True)),
    ("int8_g64_rows", 4, dict(bits=8, scale_group=64, batch=1, n_kv_heads=2, n_q_heads=2, ctx=2 * 128), "rows", {}),
]


def _build(w, layout, key_calib=False, sink=False):
    import torch
    import bit_kv_cache_block_gb300 as K
    cb = U.codebook_for(w)
    cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, in_dtype=w.dtype,
                        pre_rope=w.pre_rope, rope_theta=w.rope_theta, outlier_frac=w.outlier_frac,
                        varn_iters=w.varn_iters, hadamard=True, layout=layout, key_calib=key_calib, sink=sink,
                        scale_group=w.scale_group)
    cache = K.KVCache(cfg, None if cb is None else torch.from_numpy(cb))
    if key_calib:
        kc = np.stack([np.concatenate([WL.tile(w, 0, h, blk, WL.KIND_K, seed=99) for blk in range(3)])
                       for h in range(w.n_kv_heads)])
        cache.calibrate_keys(U.to_device(kc, w.dtype))
    return cache, cb


def _oracle_stats(w, cache, cb, layout, X, kind, sink):
    """fp64 stats of every token of X [B][H][n*128][128] against the cache's records."""
    oc = O.OracleCache.for_workload(w, codebook=None if cb is None else cb[0], layout=U.oracle_layout(layout))
    recs = U.records_np(cache)
    out = np.zeros(X.shape[:3] + (4,))
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            for blk in range(w.n_blocks):
                f = U.tile_fields(recs[b, h, blk], cache.layout, kind, w.method, w.bits, layout)
                xq = oc.dequant_tile(f, kind, h, blk, "input")
                x = X[b, h, blk * 128:(blk + 1) * 128].astype(np.float64)
                if sink and blk == 0:
                    xq = xq.copy()
                    xq[0] = x[0]
                out[b, h, blk * 128:(blk + 1) * 128] = O.token_error_stats(x, xq)
    return out


def _check_stats(got, exp, where):
    got = got.astype(np.float64)
    nx = exp[..., 0]
    assert np.allclose(got[..., 0], nx, rtol=1e-5, atol=1e-30), where + " |x|"
    assert np.all(np.abs(got[..., 1] - exp[..., 1]) <= 1e-5 * nx + 1e-7), where + " norm deviation"
    for col, name in ((2, "E_T"), (3, "E_D")):
        err = np.abs(got[..., col] - exp[..., col])
        assert np.all(err <= 1e-4 * np.abs(exp[..., col]) + 2e-6 * nx ** 2 + 1e-9), where + " " + name
    # the split closes: E_T = E_M + E_D within the same rounding
    em = got[..., 1] ** 2
    assert np.all(np.abs(em + got[..., 3] - got[..., 2]) <= 1e-4 * got[..., 2] + 4e-6 * nx ** 2 + 1e-9), where


@pytest.mark.parametrize("name,cfg_id,kw,layout,extra", CASES, ids=[c[0] for c in CASES])
def test_error_stats_match_oracle(name, cfg_id, kw, layout, extra):
    import torch
    w = WL.WORKLOADS[cfg_id].scaled(**kw)
    sink = extra.get("sink", False)
    cache, cb = _build(w, layout, **extra)
    Kx, Vx = WL.blocks(w, 0, w.n_blocks)
    Kd, Vd = U.to_device(Kx, w.dtype), U.to_device(Vx, w.dtype)
    cache.append(Kd, Vd)
    sk, sv = cache.error_stats(Kd, Vd)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    for kind, X, S in ((0, Kx, sk), (1, Vx, sv)):
        exp = _oracle_stats(w, cache, cb, layout, X, kind, sink)
        got = S.cpu().numpy()
        _check_stats(got, exp, f"{name} kind={kind}")
        if sink:
            assert np.all(got[:, :, 0, 1:] == 0.0), "kept first token: no error"
    # a sub-range (blocks 1..) and one kind only
    sk1, sv1 = cache.error_stats(Kd[:, :, 128:].contiguous(), None, first_block=1)
    torch.cuda.synchronize()
    assert sv1 is None
    assert np.array_equal(sk1.cpu().numpy(), sk.cpu().numpy()[:, :, 128:])


def _topk_check(stats_np, got, fracs):
    exp = O.topk_error_share(stats_np, fracs)
    assert np.array_equal(got[:, 0], exp[:, 0]), (got[:, 0], exp[:, 0])
    assert np.allclose(got[:, 1:], exp[:, 1:], rtol=1e-10, atol=0), (got, exp)


def test_topk_share_on_real_stats():
    import torch
    import bit_kv_cache_block_gb300 as K
    w = WL.WORKLOADS[3].scaled(batch=2, n_kv_heads=2, n_q_heads=8, ctx=4 * 128)
    cache, _ = _build(w, "mma")
    Kx, Vx = WL.blocks(w, 0, w.n_blocks)
    Kd, Vd = U.to_device(Kx, w.dtype), U.to_device(Vx, w.dtype)
    cache.append(Kd, Vd)
    sk, sv = cache.error_stats(Kd, Vd)
    for S in (sk, sv):
        got = K.error_topk(S, FRACS).cpu().numpy()
        _topk_check(S.cpu().numpy(), got, FRACS)


@pytest.mark.parametrize("n", [1, 7, 255, 256, 1000, 3 * 2 ** 20 + 17])
def test_topk_share_ties_and_sizes(n):
    import torch
    import bit_kv_cache_block_gb300 as K
    rng = np.random.default_rng(n)
    st = np.zeros((n, 4), np.float32)
    st[:, 0] = 1.0
    st[:, 1] = rng.standard_normal(n).astype(np.float32)           # distinct E_M per row
    st[:, 2] = (rng.integers(0, 5, n) / 4.0).astype(np.float32)    # five error values: ties everywhere
    st[:, 3] = rng.random(n).astype(np.float32)
    if n > 3:
        st[n // 2, 2] = np.float32(-0.0)
    d = torch.from_numpy(st).cuda()
    fracs = [1e-6, 0.001, 0.013, 0.25, 0.5, 0.999, 1.0]
    got = K.error_topk(d, fracs).cpu().numpy()
    _topk_check(st, got, fracs)
    again = K.error_topk(d, fracs).cpu().numpy()
    assert np.array_equal(got, again), "bitwise reproducible"
