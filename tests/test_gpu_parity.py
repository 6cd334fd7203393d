"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on seeded inputs that
span several tiles, ragged tails and several sequence splits.

Bar: append records (code words, fp16 metadata, CSR) bit-exact for RTN, INT4 and NUQ; KVarN
records equal to the oracle's except the exemptions of kvq_testutil.varn_check_tile (VarN
scales within 1e-5 relative, fp16 metadata one ulp apart only next to an fp16 rounding
midpoint, codes +-1 only next to a rounding boundary, all judged against the oracle's own
metadata); decode outputs within max-abs 2e-3 of the oracle's fp64 result.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    yield


def _append_all(cache, w, K, V, chunks):
    edges = np.linspace(0, K.shape[2] // 128, chunks + 1).astype(int)
    for a, b in zip(edges[:-1], edges[1:]):
        if b > a:
            cache.append(U.to_device(K[:, :, a * 128:b * 128], w.dtype), U.to_device(V[:, :, a * 128:b * 128], w.dtype))


def _oracle_cache(w, layout, v_csc=False):
    return O.OracleCache.for_workload(w, codebook=U.codebook_for(w)[0] if w.method == "nuq" else None,
                                      layout=U.oracle_layout(layout), v_csc=v_csc)


def _compare_exact(cache, oc, w, nb, layout):
    recs = U.records_np(cache)
    lay = cache.layout
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            for blk in range(nb):
                for kind in (0, 1):
                    got = U.tile_fields(recs[b, h, blk], lay, kind, w.method, w.bits, layout)
                    exp = oc.recs[(b, h, blk, kind)]
                    where = f"b={b} h={h} blk={blk} kind={kind}"
                    assert np.array_equal(got["words"], exp["words"]), where + " code words"
                    assert np.array_equal(U.f16_bits(got["s16"]), U.f16_bits(exp["s16"])), where + " s"
                    if "z16" in exp:
                        assert np.array_equal(U.f16_bits(got["z16"]), U.f16_bits(exp["z16"])), where + " z"
                    if "zp16" in exp:
                        assert np.array_equal(U.f16_bits(got["zp16"]), U.f16_bits(exp["zp16"])), where + " zp"
                    if w.method == "nuq" and oc.n_out:
                        ptr, idx, val = U.sparse_parts(exp)  # CSR, or CSC for v_csc value tiles
                        assert np.array_equal(got["val"], val), where + " outlier val"
                        assert np.array_equal(got["row_ptr"], ptr), where + " outlier pointers"
                        assert np.array_equal(got["col"], idx), where + " outlier index"
                        assert not got["csr_pad"].any(), where + " outlier padding"


CASES_EXACT = [
    ("rtn4_cfg1_full", WL.WORKLOADS[1], {}),
    ("rtn2_mha", WL.WORKLOADS[5], dict(batch=2, n_kv_heads=3, n_q_heads=3, ctx=5 * 128)),
    ("rtn3_gqa", WL.WORKLOADS[5], dict(bits=3, batch=1, n_kv_heads=2, n_q_heads=8, ctx=3 * 128)),
    ("rtn4_gqa", WL.WORKLOADS[5], dict(bits=4, batch=2, n_kv_heads=2, n_q_heads=4, ctx=2 * 128)),
    ("int4_bf16", WL.WORKLOADS[4], dict(batch=2, n_kv_heads=2, n_q_heads=8, ctx=3 * 128)),
    ("int4_f16", WL.WORKLOADS[4], dict(dtype="f16", batch=1, n_kv_heads=1, n_q_heads=1, ctx=2 * 128)),
    ("nuq3_rope", WL.WORKLOADS[2], dict(batch=1, n_kv_heads=3, n_q_heads=3, ctx=4 * 128)),
    ("nuq3_gqa_norope", WL.WORKLOADS[2], dict(pre_rope=False, batch=2, n_kv_heads=2, n_q_heads=4, ctx=2 * 128)),
    ("nuq2_5pct", WL.WORKLOADS[2], dict(bits=2, outlier_frac=0.05, batch=1, n_kv_heads=1, n_q_heads=1, ctx=2 * 128)),
    ("nuq4_nooutl", WL.WORKLOADS[2], dict(bits=4, outlier_frac=0.0, batch=1, n_kv_heads=2, n_q_heads=2, ctx=2 * 128)),
    ("int8_bf16", WL.WORKLOADS[4], dict(bits=8, batch=2, n_kv_heads=2, n_q_heads=8, ctx=3 * 128)),
    ("int8_f16_g64", WL.WORKLOADS[4], dict(bits=8, scale_group=64, dtype="f16", batch=1, n_kv_heads=2, n_q_heads=2,
                                           ctx=2 * 128)),
    ("int4_g64", WL.WORKLOADS[4], dict(scale_group=64, batch=2, n_kv_heads=1, n_q_heads=4, ctx=2 * 128)),
]


@pytest.mark.parametrize("layout", ["rows", "mma"])
@pytest.mark.parametrize("name,base,kw", CASES_EXACT, ids=[c[0] for c in CASES_EXACT])
def test_append_records_bit_exact(name, base, kw, layout):
    w = base.scaled(**kw)
    nb = w.n_blocks
    cache = U.new_cache(w, layout=layout)
    K, V = WL.blocks(w, 0, nb)
    _append_all(cache, w, K, V, chunks=min(3, nb))
    oc = _oracle_cache(w, layout)
    oc.append(K, V)
    _compare_exact(cache, oc, w, nb, layout)
    assert cache.device_status() == 0


@pytest.mark.parametrize("layout", ["rows", "mma"])
def test_append_varn_exemptions(layout):
    import torch
    w = WL.WORKLOADS[3].scaled(batch=2, n_kv_heads=2, n_q_heads=8, ctx=3 * 128)
    nb = w.n_blocks
    cache = U.new_cache(w, layout=layout)
    K, V = WL.blocks(w, 0, nb)
    dbg = torch.zeros((w.batch, w.n_kv_heads, nb, 2, 2, 128), dtype=torch.float32, device="cuda")
    cache.append(U.to_device(K, w.dtype), U.to_device(V, w.dtype), dbg_varn_scales=dbg)
    oc = _oracle_cache(w, layout)
    oc.append(K, V)
    dbg = dbg.cpu().numpy()
    recs = U.records_np(cache)
    tot = {}
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            for blk in range(nb):
                for kind in (0, 1):
                    got = U.tile_fields(recs[b, h, blk], cache.layout, kind, "varn", 2, layout)
                    c = U.varn_check_tile(got, oc.recs[(b, h, blk, kind)], kind, dbg[b, h, blk, kind], layout)
                    for k, v in c.items():
                        tot[k] = tot.get(k, 0) + v
    # exemptions must stay rare: every exempted cell and code together under 0.1% of the codes
    n_codes = w.batch * w.n_kv_heads * nb * 2 * 16384
    assert sum(tot.values()) - tot["derived_groups"] <= 0.001 * n_codes, tot
    assert tot["derived_groups"] <= 0.001 * (w.batch * w.n_kv_heads * nb * 2 * 128), tot


def _run_decode(w, nb, n_tail, chunks=2, oracle_planes=False, step=0, layout="rows"):
    import torch
    cache = U.new_cache(w, max_blocks=max(nb, 1), layout=layout)
    K, V = WL.blocks(w, 0, nb) if nb else (None, None)
    oc = _oracle_cache(w, layout)
    if nb:
        _append_all(cache, w, K, V, chunks)
        oc.append(K, V)
    if oracle_planes and nb:
        recs = cache.record_view()
        host = recs.cpu().numpy()
        for (b, h, blk, kind), rec in oc.recs.items():
            U.serialize_tile(host[b, h, blk], cache.layout, kind, rec, w.method)
        recs.copy_(torch.from_numpy(host))
    q = WL.query(w, step)
    tk, tv = WL.tail(w, n_tail, step)
    out = cache.decode(U.to_device(q, w.dtype),
                       U.to_device(tk, w.dtype) if n_tail else None,
                       U.to_device(tv, w.dtype) if n_tail else None)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    ref = oc.decode(q, tk if n_tail else None, tv if n_tail else None)
    return out.cpu().numpy().astype(np.float64), ref


DECODE_CASES = [
    ("rtn4_cfg1", WL.WORKLOADS[1], {}, [0, 1, 127]),
    ("rtn2_mha", WL.WORKLOADS[5], dict(batch=1, n_kv_heads=4, n_q_heads=4, ctx=7 * 128), [0, 5]),
    ("rtn2_gqa_ragged_splits", WL.WORKLOADS[5], dict(batch=8, n_kv_heads=8, n_q_heads=32, ctx=45 * 128), [3]),
    ("rtn3_gqa", WL.WORKLOADS[5], dict(bits=3, batch=2, n_kv_heads=2, n_q_heads=8, ctx=3 * 128), [127]),
    ("int4_bf16", WL.WORKLOADS[4], dict(batch=2, n_kv_heads=2, n_q_heads=8, ctx=5 * 128), [0, 64]),
    ("nuq3_rope", WL.WORKLOADS[2], dict(batch=1, n_kv_heads=3, n_q_heads=3, ctx=6 * 128), [0, 1, 127]),
    ("nuq3_rope_ragged_ranges", WL.WORKLOADS[2], dict(batch=3, n_kv_heads=5, n_q_heads=5, ctx=37 * 128), [0, 77]),
    ("nuq3_rope_5pct", WL.WORKLOADS[2], dict(outlier_frac=0.05, batch=1, n_kv_heads=2, n_q_heads=2, ctx=9 * 128), [3]),
    # more (b, head) pairs than the nuq decode has CTAs: its tail warps loop over heads
    ("nuq3_rope_160_heads", WL.WORKLOADS[2], dict(batch=10, n_kv_heads=16, n_q_heads=16, ctx=2 * 128), [0, 50, 127]),
    ("nuq3_rope_no_outliers", WL.WORKLOADS[2], dict(outlier_frac=0.0, batch=2, n_kv_heads=2, n_q_heads=2, ctx=4 * 128), [0]),
    ("nuq3_norope_gqa", WL.WORKLOADS[2], dict(pre_rope=False, batch=2, n_kv_heads=2, n_q_heads=4, ctx=3 * 128), [9]),
    ("varn2_gqa", WL.WORKLOADS[3], dict(batch=2, n_kv_heads=2, n_q_heads=8, ctx=4 * 128), [0, 100]),
    ("varn2_g16", WL.WORKLOADS[3], dict(batch=1, n_kv_heads=1, n_q_heads=16, ctx=2 * 128), [1]),
    # one and two query heads per KV head with 2-bit codes: the e4m3 tensor-core kernel (K/V halves
    # for one head, whole records for two); heavy-tailed keys with outlier channels stress the
    # per-channel scale range its operand splits must carry
    ("varn2_mha", WL.WORKLOADS[3], dict(batch=1, n_kv_heads=3, n_q_heads=3, ctx=4 * 128), [0, 33]),
    ("varn2_g2", WL.WORKLOADS[3], dict(batch=2, n_kv_heads=2, n_q_heads=4, ctx=3 * 128), [5]),
    ("rtn2_g2", WL.WORKLOADS[5], dict(batch=2, n_kv_heads=3, n_q_heads=6, ctx=5 * 128), [0, 17]),
    ("rtn2_mha_heavy_keys", WL.WORKLOADS[3], dict(method="rtn", batch=1, n_kv_heads=2, n_q_heads=2, ctx=6 * 128),
     [0, 9]),
    ("int8_bf16", WL.WORKLOADS[4], dict(bits=8, batch=2, n_kv_heads=2, n_q_heads=8, ctx=5 * 128), [0, 64]),
    ("int8_g64_f16", WL.WORKLOADS[4], dict(bits=8, scale_group=64, dtype="f16", batch=1, n_kv_heads=3, n_q_heads=3,
                                           ctx=4 * 128), [127]),
    ("int4_g64_bf16", WL.WORKLOADS[4], dict(scale_group=64, batch=2, n_kv_heads=2, n_q_heads=4, ctx=3 * 128), [5]),
]


@pytest.mark.parametrize("layout", ["rows", "mma"])
@pytest.mark.parametrize("name,base,kw,tails", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_decode_parity(name, base, kw, tails, layout):
    w = base.scaled(**kw)
    for n_tail in tails:
        out, ref = _run_decode(w, w.n_blocks, n_tail, oracle_planes=(w.method == "varn"), layout=layout)
        err = np.max(np.abs(out - ref))
        assert err <= TOL, f"{name} tail={n_tail}: max abs err {err:.3e}"


def test_decode_shared_memory_sizes_in_any_order():
    """Decodes whose kernels need different dynamic shared memory (outlier fractions 1%, 5%, 0%,
    then 1% again, in one process) all launch: a smaller configuration must not leave the
    kernel's shared-memory limit below what a later, larger one needs."""
    for frac in (0.01, 0.05, 0.0, 0.01, 0.05):
        w = WL.WORKLOADS[2].scaled(outlier_frac=frac, batch=1, n_kv_heads=2, n_q_heads=2, ctx=3 * 128)
        out, ref = _run_decode(w, w.n_blocks, 0, layout="mma")
        assert np.max(np.abs(out - ref)) <= TOL, f"outlier_frac={frac}"


@pytest.mark.parametrize("layout", ["rows", "mma"])
def test_decode_varn_own_planes(layout):
    w = WL.WORKLOADS[3].scaled(batch=1, n_kv_heads=2, n_q_heads=8, ctx=3 * 128)
    out, ref = _run_decode(w, w.n_blocks, 17, oracle_planes=False, layout=layout)
    assert np.max(np.abs(out - ref)) <= TOL


@pytest.mark.parametrize("method", ["rtn", "nuq", "int4", "varn"])
def test_decode_tail_only(method):
    base = {"rtn": WL.WORKLOADS[1], "nuq": WL.WORKLOADS[2], "int4": WL.WORKLOADS[4], "varn": WL.WORKLOADS[3]}[method]
    w = base.scaled(batch=1, n_kv_heads=1, n_q_heads=base.group if base.group <= 4 else 4, ctx=128)
    out, ref = _run_decode(w, 0, 50)
    assert np.max(np.abs(out - ref)) <= TOL


@pytest.mark.parametrize("layout", ["rows", "mma"])
@pytest.mark.parametrize("name,base,kw", CASES_EXACT[1:8:2] + CASES_EXACT[11:12] +
                         [("varn", WL.WORKLOADS[3], dict(batch=1, n_kv_heads=2, n_q_heads=2, ctx=2 * 128))],
                         ids=[c[0] for c in CASES_EXACT[1:8:2] + CASES_EXACT[11:12]] + ["varn"])
def test_dequant_parity(name, base, kw, layout):
    w = base.scaled(**kw)
    nb = w.n_blocks
    cache = U.new_cache(w, layout=layout)
    K, V = WL.blocks(w, 0, nb)
    cache.append(U.to_device(K, w.dtype), U.to_device(V, w.dtype))
    oc = _oracle_cache(w, layout)
    oc.append(K, V)
    for domain in (0, 1):
        dk, dv = cache.dequant(0, nb, domain)
        dk, dv = dk.cpu().numpy(), dv.cpu().numpy()
        for b in range(w.batch):
            for h in range(w.n_kv_heads):
                for kind, got in ((0, dk), (1, dv)):
                    if w.method == "varn":   # compare the kernel's planes, dequantised by the oracle
                        recs = U.records_np(cache)
                        ref = np.concatenate([oc.dequant_tile(U.tile_fields(recs[b, h, blk], cache.layout, kind, "varn", 2, layout),
                                                              kind, h, blk, "input" if domain else "stored")
                                              for blk in range(nb)])
                        tol = 1e-5 * (1 + np.abs(ref))
                    else:
                        ref = oc.dequant(b, h, kind, "stored")
                        tol = 0.0 if w.method in ("rtn", "int4") else 1e-6 * (1 + np.abs(ref))
                    assert np.all(np.abs(got[b, h] - ref) <= tol), f"{name} domain={domain} kind={kind}"


def test_capacity_and_truncate():
    import torch
    import bit_kv_cache_block_gb300 as K
    w = WL.WORKLOADS[5].scaled(batch=1, n_kv_heads=1, n_q_heads=1, ctx=2 * 128)
    cache = U.new_cache(w)
    Kx, Vx = WL.blocks(w, 0, 2)
    cache.append(U.to_device(Kx, "f16"), U.to_device(Vx, "f16"))
    with pytest.raises(K.KVQError) as ei:
        cache.append(U.to_device(Kx[:, :, :128], "f16"), U.to_device(Vx[:, :, :128], "f16"))
    assert ei.value.status == K._lib.KVQ_ERR_CAPACITY
    cache.truncate(1)
    cache.append(U.to_device(Kx[:, :, 128:], "f16"), U.to_device(Vx[:, :, 128:], "f16"))
    torch.cuda.synchronize()
    assert cache.n_blocks == 2 and cache.device_status() == 0


DETERMINISM_CASES = [c for c in DECODE_CASES if c[0] in ("rtn2_mha", "rtn3_gqa", "int4_bf16", "nuq3_rope",
                                                         "nuq3_rope_5pct", "nuq3_norope_gqa", "varn2_gqa",
                                                         "int8_g64_f16", "int8_bf16")]


@pytest.mark.parametrize("layout", ["rows", "mma"])
@pytest.mark.parametrize("name,base,kw,tails", DETERMINISM_CASES, ids=[c[0] for c in DETERMINISM_CASES])
def test_decode_is_deterministic(name, base, kw, tails, layout):
    """Two decodes of the same cache and inputs give bitwise-equal outputs (no result depends on
    thread timing: outlier sums run in a fixed order)."""
    import torch
    w = base.scaled(**kw)
    cache = U.new_cache(w, layout=layout)
    K, V = WL.blocks(w, 0, w.n_blocks)
    cache.append(U.to_device(K, w.dtype), U.to_device(V, w.dtype))
    n_tail = tails[-1]
    tk, tv = WL.tail(w, n_tail)
    args = (U.to_device(WL.query(w), w.dtype), U.to_device(tk, w.dtype) if n_tail else None,
            U.to_device(tv, w.dtype) if n_tail else None)
    outs = [cache.decode(*args).cpu().numpy() for _ in range(3)]
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2]), name


@pytest.mark.parametrize("name,cfg_id,kw", [("nuq3_rope", 2, dict(batch=2, n_kv_heads=2, n_q_heads=2, ctx=3 * 128)),
                                            ("varn2_gqa", 3, dict(batch=2, n_kv_heads=2, n_q_heads=8, ctx=2 * 128))])
def test_decode_tail_capacity_buffers(name, cfg_id, kw):
    """kvq_decode_attn_ex over tail buffers of capacity 127 tokens (per-(b, h) rows, and token-major),
    n_tail of them in use, equals the decode over the same tokens packed contiguously, bit for bit."""
    import torch
    w = WL.WORKLOADS[cfg_id].scaled(**kw)
    cache = U.new_cache(w, layout="mma")
    K, V = WL.blocks(w, 0, w.n_blocks)
    cache.append(U.to_device(K, w.dtype), U.to_device(V, w.dtype))
    q = U.to_device(WL.query(w), w.dtype)
    tk, tv = WL.tail(w, 127)
    dk, dv = U.to_device(tk, w.dtype), U.to_device(tv, w.dtype)
    import bit_kv_cache_block_gb300 as K
    tok_k = dk.permute(2, 0, 1, 3).contiguous()  # token-major [127][B][H][128]
    tok_v = dv.permute(2, 0, 1, 3).contiguous()
    for n_tail in (1, 37, 127):
        a = cache.decode(q, dk, dv, n_tail=n_tail).cpu().numpy()
        b = cache.decode(q, dk[:, :, :n_tail].contiguous(), dv[:, :, :n_tail].contiguous()).cpu().numpy()
        assert np.array_equal(a, b), f"{name} n_tail={n_tail}"
        c = torch.empty(q.shape[0], q.shape[1], 128, dtype=torch.float32, device="cuda")
        K.kvq_decode_attn_ex(cache.cache, q, tok_k, tok_v, n_tail, 128, w.batch * w.n_kv_heads * 128, c,
                             cache.workspace)
        assert np.array_equal(a, c.cpu().numpy()), f"{name} token-major n_tail={n_tail}"
    torch.cuda.synchronize()
    assert cache.device_status() == 0
