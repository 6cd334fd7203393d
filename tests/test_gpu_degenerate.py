"""Degenerate inputs on the GPU against the oracle: blocks that are all zero, constant, full of
equal magnitudes (ties in the outlier choice), or near the fp16 range.

- Append records bit-exact for RTN, nuq (outliers, ties broken towards the lower flat index),
  absmax int4 / int8 / 64-channel scales; KVarN records exact on zero blocks (no variance to
  normalise: every scale 1).
- Decode within max-abs 2e-3 of the oracle on the zero, constant and tie blocks (next to normal
  blocks, with a tail); on the large-magnitude blocks every output is finite and the records
  are exact.
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


def _fill(w, kind_of_block, seed=0):
    """K, V [B][H][nb*128][128] (float32, exactly representable in w.dtype): block i filled by
    kind_of_block[i] in ("normal", "zero", "const", "ties", "large")."""
    rng = np.random.default_rng(seed)
    nb = len(kind_of_block)
    Kn, Vn = WL.blocks(w.scaled(ctx=nb * 128), 0, nb)
    K, V = Kn.copy(), Vn.copy()
    for i, kind in enumerate(kind_of_block):
        sl = slice(i * 128, (i + 1) * 128)
        shape = K[:, :, sl].shape
        if kind == "zero":
            K[:, :, sl] = 0.0
            V[:, :, sl] = 0.0
        elif kind == "const":
            K[:, :, sl] = 0.375
            V[:, :, sl] = -1.25
        elif kind == "ties":     # magnitudes 1 almost everywhere, a few 2s: outlier ties
            K[:, :, sl] = rng.choice([-1.0, 1.0], size=shape)
            V[:, :, sl] = rng.choice([-1.0, 1.0], size=shape)
            K[:, :, sl][..., ::37, 5] = 2.0
            V[:, :, sl][..., 3, ::11] = -2.0
        elif kind == "large":    # near the fp16 range, exactly representable
            K[:, :, sl] = np.round(rng.uniform(-1, 1, size=shape) * 64) * 512.0
            V[:, :, sl] = np.round(rng.uniform(-1, 1, size=shape) * 64) * 512.0
    return WL.round_dtype(K, w.dtype), WL.round_dtype(V, w.dtype)


CASES = [
    ("rtn2", 5, dict(batch=1, n_kv_heads=2, n_q_heads=2)),
    ("rtn4_gqa", 5, dict(bits=4, batch=1, n_kv_heads=2, n_q_heads=4)),
    ("nuq3_rope", 2, dict(batch=1, n_kv_heads=2, n_q_heads=2)),
    ("nuq3_5pct", 2, dict(batch=1, n_kv_heads=1, n_q_heads=1, outlier_frac=0.05)),
    ("int4_bf16", 4, dict(batch=1, n_kv_heads=2, n_q_heads=8)),
    ("int8_g64", 4, dict(bits=8, scale_group=64, batch=1, n_kv_heads=2, n_q_heads=2)),
]
PATTERN = ["normal", "zero", "const", "ties", "normal"]


@pytest.mark.parametrize("layout", ["rows", "mma"])
@pytest.mark.parametrize("name,cfg_id,kw", CASES, ids=[c[0] for c in CASES])
def test_degenerate_blocks(name, cfg_id, kw, layout):
    import torch
    w = WL.WORKLOADS[cfg_id].scaled(ctx=len(PATTERN) * 128, **kw)
    K, V = _fill(w, PATTERN)
    cache = U.new_cache(w, layout=layout)
    cache.append(U.to_device(K, w.dtype), U.to_device(V, w.dtype))
    oc = _oracle_cache(w, layout)
    oc.append(K, V)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    _compare_exact(cache, oc, w, w.n_blocks, layout)
    for n_tail in (0, 45):
        q = WL.query(w, 1)
        tk, tv = WL.tail(w, n_tail, 1)
        out = cache.decode(U.to_device(q, w.dtype), U.to_device(tk, w.dtype) if n_tail else None,
                           U.to_device(tv, w.dtype) if n_tail else None).cpu().numpy().astype(np.float64)
        ref = oc.decode(q, tk if n_tail else None, tv if n_tail else None)
        err = np.max(np.abs(out - ref))
        assert err <= TOL, f"{name} {layout} tail={n_tail}: max abs err {err:.3e}"


@pytest.mark.parametrize("layout", ["rows", "mma"])
def test_varn_zero_blocks_exact(layout):
    """KVarN on an all-zero block: nothing to normalise, every scale 1, every code 0."""
    import torch
    w = WL.WORKLOADS[3].scaled(batch=1, n_kv_heads=2, n_q_heads=8, ctx=2 * 128)
    K, V = _fill(w, ["zero", "zero"])
    cache = U.new_cache(w, layout=layout)
    cache.append(U.to_device(K, w.dtype), U.to_device(V, w.dtype))
    oc = _oracle_cache(w, layout)
    oc.append(K, V)
    torch.cuda.synchronize()
    recs = U.records_np(cache)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            for blk in range(w.n_blocks):
                for kind in (0, 1):
                    got = U.tile_fields(recs[b, h, blk], cache.layout, kind, "varn", 2, layout)
                    exp = oc.recs[(b, h, blk, kind)]
                    assert np.array_equal(got["words"], exp["words"])
                    for key in ("s16", "z16", "s1"):
                        assert np.array_equal(U.f16_bits(got[key]), U.f16_bits(exp[key])), key
    q = WL.query(w)
    out = cache.decode(U.to_device(q, w.dtype)).cpu().numpy()
    assert np.max(np.abs(out - oc.decode(q))) <= TOL


@pytest.mark.parametrize("name,cfg_id,kw", [c for c in CASES if c[0] != "nuq3_5pct"],
                         ids=[c[0] for c in CASES if c[0] != "nuq3_5pct"])
def test_large_magnitude_blocks(name, cfg_id, kw):
    import torch
    w = WL.WORKLOADS[cfg_id].scaled(ctx=2 * 128, **kw)
    K, V = _fill(w, ["large", "normal"], seed=3)
    cache = U.new_cache(w, layout="mma")
    cache.append(U.to_device(K, w.dtype), U.to_device(V, w.dtype))
    oc = _oracle_cache(w, "mma")
    oc.append(K, V)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    _compare_exact(cache, oc, w, w.n_blocks, "mma")
    out = cache.decode(U.to_device(WL.query(w), w.dtype)).cpu().numpy()
    assert np.all(np.isfinite(out))
