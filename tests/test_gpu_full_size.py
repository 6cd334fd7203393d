"""Parity at the full workload sizes, in the launch configuration the benchmark times.

For each of the five workloads the whole cache is built on the device in the tensor-core tile
format (the benchmark's) and decoded once, with a fp tail, through kvq_decode_attn with a
caller workspace, as the benchmark does. The oracle cannot quantize and attend every head of
these contexts in reasonable time, so it follows sampled (batch, KV head) pairs one by one:
their inputs come from the seeded generators of the parity tests, while the other heads hold
seeded device noise of the same shape (they do not enter the sampled outputs). Checked per
sampled pair: the decode outputs of all its query heads within max-abs 2e-3 of the oracle's
fp64 result over the whole context, and the code words, metadata and CSR of its first, middle
and last blocks bit-exact (KVarN: equal under the exemptions of kvq_testutil.varn_check_tile,
with the kernel's fp32 VarN scales read back from the bulk append). Every output of the launch must be finite and the status word clear.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
TOL = 2e-3
N_TAIL = 77
CHUNK = 512  # blocks per host->device copy of a sampled head

SAMPLES = {1: [(0, 0)], 2: [(0, 0), (0, 13), (0, 31)], 3: [(0, 0), (3, 5), (7, 7)], 4: [(0, 0), (17, 3), (31, 7)],
           5: [(0, 0), (0, 17)], "4-int8": [(0, 0), (31, 7)]}
# the absmax workload with 8-bit codes (the sensitive-layer precision), same shapes
VARIANTS = {"4-int8": (4, dict(bits=8))}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    yield


def _head_tiles(w, b, h, first, n):
    """K and V of one (b, h) for blocks [first, first + n): float32 [n*128][128] each."""
    K = np.empty((n * 128, 128), np.float32)
    V = np.empty_like(K)
    for i in range(n):
        K[i * 128:(i + 1) * 128] = WL.tile(w, b, h, first + i, WL.KIND_K)
        V[i * 128:(i + 1) * 128] = WL.tile(w, b, h, first + i, WL.KIND_V)
    return K, V


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, "4-int8"])
def test_full_size_sampled_heads(cfg):
    import torch
    w = WL.WORKLOADS[VARIANTS[cfg][0]].scaled(**VARIANTS[cfg][1]) if cfg in VARIANTS else WL.WORKLOADS[cfg]
    nb, G = w.n_blocks, w.group
    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    cache = U.new_cache(w, layout="mma")
    shape = (w.batch, w.n_kv_heads, nb * 128, 128)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7919 * (cfg if isinstance(cfg, int) else 11))
    Kd = torch.randn(shape, generator=gen, device="cuda", dtype=dt)
    Vd = torch.randn(shape, generator=gen, device="cuda", dtype=dt)
    heads = {}
    for (b, h) in SAMPLES[cfg]:
        Kh = np.empty((nb * 128, 128), np.float32)
        Vh = np.empty_like(Kh)
        for c0 in range(0, nb, CHUNK):
            n = min(CHUNK, nb - c0)
            k, v = _head_tiles(w, b, h, c0, n)
            Kh[c0 * 128:(c0 + n) * 128], Vh[c0 * 128:(c0 + n) * 128] = k, v
            Kd[b, h, c0 * 128:(c0 + n) * 128] = U.to_device(k, w.dtype)
            Vd[b, h, c0 * 128:(c0 + n) * 128] = U.to_device(v, w.dtype)
        heads[(b, h)] = (Kh, Vh)
    dbg = None
    if w.method == "varn":  # the fp32 VarN scales of every tile, for the exemption check
        dbg = torch.zeros((w.batch, w.n_kv_heads, nb, 2, 2, 128), dtype=torch.float32, device="cuda")
    cache.append(Kd, Vd, dbg_varn_scales=dbg)
    del Kd, Vd
    q = WL.query(w)
    tk, tv = WL.tail(w, N_TAIL)
    out = cache.decode(U.to_device(q, w.dtype), U.to_device(tk, w.dtype), U.to_device(tv, w.dtype))
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    out = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(out))
    recs = cache.record_view()
    cb = U.codebook_for(w)
    for (b, h), (Kh, Vh) in heads.items():
        w1 = w.scaled(batch=1, n_kv_heads=1, n_q_heads=G)
        oc = O.OracleCache.for_workload(w1, codebook=cb[h] if cb is not None else None, layout=O.LAYOUT_MMA)
        oc.append(Kh[None, None], Vh[None, None])
        ref = oc.decode(q[b:b + 1, h * G:(h + 1) * G], tk[b:b + 1, h:h + 1], tv[b:b + 1, h:h + 1])
        err = np.max(np.abs(out[b, h * G:(h + 1) * G] - ref[0]))
        assert err <= TOL, f"config {cfg} (b={b}, h={h}): max abs err {err:.3e}"
        for blk in sorted({0, nb // 2, nb - 1}):
            rec = recs[b, h, blk].cpu().numpy()
            for kind in (0, 1):
                got = U.tile_fields(rec, cache.layout, kind, w.method, w.bits, "mma")
                exp = oc.recs[(0, 0, blk, kind)]
                where = f"config {cfg} (b={b}, h={h}) blk={blk} kind={kind}"
                if w.method == "varn":
                    c = U.varn_check_tile(got, exp, kind, dbg[b, h, blk, kind].cpu().numpy(), "mma")
                    assert sum(c.values()) - c["derived_groups"] <= 0.001 * 16384 + 2, where + f" exemptions {c}"
                    continue
                assert np.array_equal(got["words"], exp["words"]), where + " code words"
                assert np.array_equal(U.f16_bits(got["s16"]), U.f16_bits(exp["s16"])), where + " s"
                for key in ("z16", "zp16"):
                    if key in exp:
                        assert np.array_equal(U.f16_bits(got[key]), U.f16_bits(exp[key])), where + " " + key
                if w.method == "nuq" and oc.n_out:
                    for key in ("val", "row_ptr", "col"):
                        assert np.array_equal(got[key], exp[key]), where + " csr " + key
