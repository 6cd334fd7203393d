"""The C ABI without a GPU: the library loads, exports every entry point include/kvq.h
declares, the ctypes structs match the C layout, and the host-only logic (layouts, sizes,
argument checks) behaves as documented. No compute call runs here."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

import oracle as O
import workloads as WL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_block_gb300 as K
    return K


def _header_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(K):
    declared = _header_functions()
    assert set(declared) == set(K._lib.EXPORTS)
    lib = K._lib.lib()
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", K.lib_path()], capture_output=True, text=True).stdout
    for name in declared:
        assert re.search(rf"\bT {name}$", out, re.M), f"{name} not exported"


def test_struct_layout_matches_c(K, tmp_path):
    prog = tmp_path / "sizes.c"
    prog.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "kvq.h"
int main(void) {
  printf("%zu %zu %zu\n", sizeof(kvq_config), sizeof(kvq_layout_t), sizeof(kvq_cache));
  printf("%zu %zu %zu %zu\n", offsetof(kvq_config, rope_theta), offsetof(kvq_config, outlier_frac),
         offsetof(kvq_config, hadamard), offsetof(kvq_layout_t, total_bytes));
  printf("%zu %zu %zu %zu\n", offsetof(kvq_cache, lay), offsetof(kvq_cache, base), offsetof(kvq_cache, n_blocks),
         offsetof(kvq_cache, device));
  printf("%zu %zu %zu\n", offsetof(kvq_config, layout), offsetof(kvq_config, n_pages),
         offsetof(kvq_cache, block_table));
  printf("%zu %zu %zu %zu %zu\n", offsetof(kvq_config, key_calib), offsetof(kvq_config, sink),
         offsetof(kvq_layout_t, calib_off), offsetof(kvq_layout_t, sink_bytes), offsetof(kvq_cache, calibrated));
  printf("%zu %zu\n", offsetof(kvq_config, scale_group), offsetof(kvq_config, v_csc));
  return 0;
}
''')
    exe = tmp_path / "sizes"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include",
                    str(prog), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    L = K._lib
    py = [C.sizeof(L.kvq_config), C.sizeof(L.kvq_layout_t), C.sizeof(L.kvq_cache),
          L.kvq_config.rope_theta.offset, L.kvq_config.outlier_frac.offset, L.kvq_config.hadamard.offset,
          L.kvq_layout_t.total_bytes.offset, L.kvq_cache.lay.offset, L.kvq_cache.base.offset,
          L.kvq_cache.n_blocks.offset, L.kvq_cache.device.offset, L.kvq_config.layout.offset,
          L.kvq_config.n_pages.offset, L.kvq_cache.block_table.offset, L.kvq_config.key_calib.offset,
          L.kvq_config.sink.offset, L.kvq_layout_t.calib_off.offset, L.kvq_layout_t.sink_bytes.offset,
          L.kvq_cache.calibrated.offset, L.kvq_config.scale_group.offset, L.kvq_config.v_csc.offset]
    assert vals == py


def test_dense_kv_bytes_matches_oracle(K):
    for args in [(32, 32, 128, 2, 1, 131072), (32, 8, 128, 2, 16, 8192), (80, 8, 128, 2, 3, 12345)]:
        assert K.kvq_dense_kv_bytes(*args) == O.kv_cache_bytes(*args)


def _cfg(K, wid, **kw):
    w = WL.WORKLOADS[wid].scaled(**kw)
    return K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, w.dtype, w.pre_rope,
                         w.rope_theta, w.outlier_frac, w.varn_iters, True)


# algorithmic packed bytes per decode step at the full workloads (codes + fp16 metadata + CSR); the
# layouts differ only for 3-bit tiles (13-word rows vs 48-byte planes)
EXPECTED_DECODE_BYTES = {1: 278528, 2: 129728512, 3: 79691776, 4: 1107296256, 5: 2415919104}
EXPECTED_RECORD_BYTES = {1: 2 * (8192 + 512), 2: 2 * (6656 + 512 + 752), 3: 2 * (4096 + 768),
                         4: 2 * (8192 + 256), 5: 2 * (4096 + 512)}
EXPECTED_MMA = {2: (121339904, 2 * (6144 + 512 + 752))}


@pytest.mark.parametrize("layout", ["rows", "mma"])
@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_layout_and_decode_bytes(K, wid, layout):
    cfg = _cfg(K, wid)
    cfg.layout = K.LAYOUTS[layout]
    lay = K.kvq_layout(cfg)
    w = WL.WORKLOADS[wid]
    dec_bytes, rec_bytes = EXPECTED_DECODE_BYTES[wid], EXPECTED_RECORD_BYTES[wid]
    if layout == "mma" and wid in EXPECTED_MMA:
        dec_bytes, rec_bytes = EXPECTED_MMA[wid]
    assert lay.record_bytes == rec_bytes
    assert lay.words_per_row == (12 if w.bits == 3 and layout == "mma" else -(-128 // (32 // w.bits)))
    assert lay.format_version == 2
    for k in range(2):
        assert lay.codes_off[k] % 16 == 0 and lay.meta_off[k] % 16 == 0 and lay.csr_off[k] % 16 == 0
    assert lay.records_bytes == w.batch * w.n_kv_heads * w.n_blocks * lay.record_bytes
    assert lay.total_bytes >= lay.records_bytes
    if w.pre_rope:
        assert lay.rope_off % 128 == 0 and lay.rope_bytes == (w.n_blocks + 1 + 128) * 64 * 8
    if w.method == "nuq":
        assert lay.n_outliers == O.n_outliers(w.outlier_frac) == 164
    assert K.kvq_decode_bytes(cfg, w.n_blocks) == dec_bytes
    S = K.kvq_decode_splits(cfg, w.n_blocks)
    assert 1 <= S <= w.n_blocks
    # at least one partial (m, l, o[128]) per (batch, query head)
    assert K.kvq_decode_workspace_bytes(cfg, w.n_blocks) >= 4 * (w.batch * w.n_q_heads * 130)


def test_config_checks(K):
    L = K._lib
    bad = [dict(head_dim=64), dict(block=64), dict(bits=5), dict(bits=1), dict(n_q_heads=33),
           dict(n_q_heads=8 * 17), dict(max_blocks=0), dict(batch=0), dict(in_dtype=7), dict(method=9),
           dict(layout=2), dict(layout=-1)]
    for b in bad:
        cfg = _cfg(K, 4)
        for k, v in b.items():
            setattr(cfg, k, v)
        with pytest.raises(K.KVQError):
            K.kvq_layout(cfg)
    cfg = _cfg(K, 4)
    cfg.bits = 3                      # absmax is 4- or 8-bit only
    with pytest.raises(K.KVQError) as e:
        K.kvq_layout(cfg)
    assert e.value.status == L.KVQ_ERR_UNSUPPORTED
    cfg = _cfg(K, 1)
    cfg.pre_rope = 1                  # pre-RoPE keys only with nuq
    with pytest.raises(K.KVQError) as e:
        K.kvq_layout(cfg)
    assert e.value.status == L.KVQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("layout", ["rows", "mma"])
@pytest.mark.parametrize("group", [1, 4])
def test_outlier_fraction_limited_by_decode_shared_memory(K, layout, group):
    """A nuq cache whose records would not fit the CUDA-core decode's three-record ring in one
    CTA's 227 KB of shared memory is refused when its layout is computed, before any memory is
    bound or any append runs; fractions up to half of each tile still lay out."""
    L = K._lib
    for frac, ok in ((0.05, True), (0.5, True), (0.9, False), (1.0, False)):
        cfg = _cfg(K, 2, outlier_frac=frac, n_kv_heads=2, n_q_heads=2 * group, ctx=4 * 128)
        cfg.layout = K.LAYOUTS[layout]
        if ok:
            assert K.kvq_layout(cfg).n_outliers == O.n_outliers(frac)
        else:
            with pytest.raises(K.KVQError) as e:
                K.kvq_layout(cfg)
            assert e.value.status == L.KVQ_ERR_UNSUPPORTED


def test_host_argument_checks_launch_nothing(K):
    """Argument errors are caught on the host before any CUDA call (works without a GPU)."""
    L = K._lib
    lib = L.lib()
    cfg = _cfg(K, 1)
    lay = K.kvq_layout(cfg)
    cache = L.kvq_cache()
    # misaligned base / too small / missing status
    st = lib.kvq_cache_init(C.byref(cache), C.byref(cfg), C.c_void_p(0x1001), lay.total_bytes, None,
                            C.c_void_p(0x2000), None)
    assert st == L.KVQ_ERR_ALIGNMENT
    st = lib.kvq_cache_init(C.byref(cache), C.byref(cfg), C.c_void_p(0x1000), lay.total_bytes - 1, None,
                            C.c_void_p(0x2000), None)
    assert st == L.KVQ_ERR_CAPACITY
    st = lib.kvq_cache_init(C.byref(cache), C.byref(cfg), C.c_void_p(0x1000), lay.total_bytes, None, None, None)
    assert st == L.KVQ_ERR_INVALID_ARG
    ncfg = _cfg(K, 2)
    nlay = K.kvq_layout(ncfg)
    st = lib.kvq_cache_init(C.byref(cache), C.byref(ncfg), C.c_void_p(0x1000), nlay.total_bytes, None,
                            C.c_void_p(0x2000), None)
    assert st == L.KVQ_ERR_INVALID_ARG            # nuq needs a codebook
    # a hand-built (never initialised on a device) cache for the append/decode checks
    cache.cfg = cfg
    cache.lay = lay
    cache.base = 0x100000
    cache.n_blocks = cfg.max_blocks
    assert lib.kvq_append_block(C.byref(cache), C.c_void_p(0x1000), C.c_void_p(0x2000), 1, None, None) \
        == L.KVQ_ERR_CAPACITY
    cache.n_blocks = 0
    assert lib.kvq_append_block(C.byref(cache), C.c_void_p(0x1008), C.c_void_p(0x2000), 1, None, None) \
        == L.KVQ_ERR_ALIGNMENT
    assert lib.kvq_append_block(C.byref(cache), None, C.c_void_p(0x2000), 1, None, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_append_block(C.byref(cache), C.c_void_p(0x1000), C.c_void_p(0x2000), 0, None, None) \
        == L.KVQ_ERR_INVALID_ARG
    q, out, ws = C.c_void_p(0x1000), C.c_void_p(0x3000), C.c_void_p(0x5000)
    assert lib.kvq_decode_attn(C.byref(cache), q, None, None, 0, out, ws, 1 << 20, None) == L.KVQ_ERR_INVALID_ARG
    cache.n_blocks = 4
    assert lib.kvq_decode_attn(C.byref(cache), q, None, None, 128, out, ws, 1 << 20, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attn(C.byref(cache), q, None, None, 3, out, ws, 1 << 20, None) == L.KVQ_ERR_INVALID_ARG
    tk = C.c_void_p(0x9000)
    ex = lib.kvq_decode_attn_ex
    assert ex(C.byref(cache), q, tk, tk, 5, 640, 64, out, ws, 1 << 20, None) == L.KVQ_ERR_INVALID_ARG  # token < 128
    assert ex(C.byref(cache), q, tk, tk, 5, -128, 128, out, ws, 1 << 20, None) == L.KVQ_ERR_INVALID_ARG
    assert ex(C.byref(cache), q, tk, tk, 5, (1 << 40) + 8, 128, out, ws, 1 << 20, None) == L.KVQ_ERR_INVALID_ARG
    assert ex(C.byref(cache), q, tk, tk, 5, 644, 128, out, ws, 1 << 20, None) == L.KVQ_ERR_ALIGNMENT
    assert ex(C.byref(cache), q, tk, tk, 5, 640, 132, out, ws, 1 << 20, None) == L.KVQ_ERR_ALIGNMENT
    assert lib.kvq_decode_attn(C.byref(cache), q, None, None, 0, out, ws, 16, None) == L.KVQ_ERR_CAPACITY
    assert lib.kvq_decode_attn(C.byref(cache), C.c_void_p(0x1004), None, None, 0, out, ws, 1 << 20, None) \
        == L.KVQ_ERR_ALIGNMENT
    assert lib.kvq_dequant(C.byref(cache), 3, 2, 0, out, None, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_dequant(C.byref(cache), 0, 1, 2, out, None, None) == L.KVQ_ERR_INVALID_ARG
    # error statistics: range, pairing and alignment
    x, sx = C.c_void_p(0x1000), C.c_void_p(0x7000)
    assert lib.kvq_error_stats(C.byref(cache), x, None, 3, 2, sx, None, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_error_stats(C.byref(cache), x, None, 0, 1, None, None, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_error_stats(C.byref(cache), None, None, 0, 1, None, None, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_error_stats(C.byref(cache), x, None, 0, 1, C.c_void_p(0x7004), None, None) \
        == L.KVQ_ERR_ALIGNMENT
    # top-k shares: sizes, fractions, workspace
    wsb = lib.kvq_error_topk_workspace_bytes()
    assert wsb > 0
    fr = (C.c_double * 9)(*([0.5] * 9))
    bad = (C.c_double * 2)(0.0, 0.5)
    big = (C.c_double * 1)(1.5)
    topk = lib.kvq_error_topk
    assert topk(sx, 100, fr, 9, out, ws, wsb, None) == L.KVQ_ERR_INVALID_ARG          # > 8 fractions
    assert topk(sx, 100, fr, 0, out, ws, wsb, None) == L.KVQ_ERR_INVALID_ARG
    assert topk(sx, 0, fr, 1, out, ws, wsb, None) == L.KVQ_ERR_INVALID_ARG
    assert topk(sx, 1 << 32, fr, 1, out, ws, wsb, None) == L.KVQ_ERR_INVALID_ARG
    assert topk(sx, 100, bad, 2, out, ws, wsb, None) == L.KVQ_ERR_INVALID_ARG         # f = 0
    assert topk(sx, 100, big, 1, out, ws, wsb, None) == L.KVQ_ERR_INVALID_ARG         # f > 1
    assert topk(sx, 100, fr, 1, out, ws, wsb - 1, None) == L.KVQ_ERR_CAPACITY
    assert topk(C.c_void_p(0x7008), 100, fr, 1, out, ws, wsb, None) == L.KVQ_ERR_ALIGNMENT
    # codebook fitting: sizes, bits, iterations, workspace, alignment
    fit = lib.kvq_fit_codebook
    fws = lib.kvq_fit_codebook_workspace_bytes(2, 1000)
    assert fws == 2 * 272 and lib.kvq_fit_codebook_workspace_bytes(0, 1000) == 0
    av, wv, cbv, wsv = C.c_void_p(0x10000), C.c_void_p(0x20000), C.c_void_p(0x30000), C.c_void_p(0x40000)
    assert fit(av, wv, 2, 1000, 5, 10, cbv, wsv, fws, None) == L.KVQ_ERR_INVALID_ARG      # bits 5
    assert fit(av, wv, 2, 1000, 0, 10, cbv, wsv, fws, None) == L.KVQ_ERR_INVALID_ARG
    assert fit(av, wv, 2, 1000, 3, 0, cbv, wsv, fws, None) == L.KVQ_ERR_INVALID_ARG       # no iteration
    assert fit(av, wv, 2, 0, 3, 10, cbv, wsv, fws, None) == L.KVQ_ERR_INVALID_ARG
    assert fit(av, wv, 2, (1 << 30) + 1, 3, 10, cbv, wsv, fws, None) == L.KVQ_ERR_INVALID_ARG
    assert fit(av, wv, 2, 1000, 3, 10, cbv, wsv, fws - 1, None) == L.KVQ_ERR_CAPACITY
    assert fit(C.c_void_p(0x10002), wv, 2, 1000, 3, 10, cbv, wsv, fws, None) == L.KVQ_ERR_ALIGNMENT
    assert fit(None, wv, 2, 1000, 3, 10, cbv, wsv, fws, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_truncate(C.byref(cache), 5) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_truncate(C.byref(cache), 2) == L.KVQ_OK and cache.n_blocks == 2
    assert lib.kvq_reset(C.byref(cache)) == L.KVQ_OK and cache.n_blocks == 0
    assert K.kvq_status_str(L.KVQ_ERR_TIMEOUT) == "device wait timed out"
    assert K.kvq_status_str(L.KVQ_ERR_PAGE) == "block table entry out of range"


def test_paged_layout_and_checks(K):
    """A paged cache's record pool is n_pages pages of H_kv records; append, decode and dequant
    need its block table (non-null, 4-byte aligned) and refuse on the host without one."""
    L = K._lib
    lib = L.lib()
    w = WL.WORKLOADS[2].scaled(batch=3, n_kv_heads=4, n_q_heads=4, ctx=5 * 128)
    cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, w.dtype, w.pre_rope,
                        w.rope_theta, w.outlier_frac, layout="mma", n_pages=17)
    lay = K.kvq_layout(cfg)
    flat_cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, w.dtype,
                             w.pre_rope, w.rope_theta, w.outlier_frac, layout="mma")
    flat = K.kvq_layout(flat_cfg)
    assert lay.record_bytes == flat.record_bytes
    assert lay.records_bytes == 17 * 4 * lay.record_bytes
    assert flat.records_bytes == 3 * 4 * 5 * flat.record_bytes
    assert lay.rope_off % 128 == 0 and lay.rope_off >= lay.records_bytes
    assert K.kvq_decode_bytes(cfg, 5) == K.kvq_decode_bytes(flat_cfg, 5)
    bad = K.make_config("rtn", 2, 1, 1, 1, 4, n_pages=-1)
    out = L.kvq_layout_t()
    assert lib.kvq_layout(C.byref(bad), C.byref(out)) == L.KVQ_ERR_INVALID_ARG
    cache = L.kvq_cache()
    cache.cfg = cfg
    cache.lay = lay
    cache.base = 0x100000
    cache.codebook = 0x200000
    cache.n_blocks = 0
    k, v = C.c_void_p(0x1000), C.c_void_p(0x2000)
    assert lib.kvq_append_block(C.byref(cache), k, v, 1, None, None) == L.KVQ_ERR_INVALID_ARG  # no table
    cache.block_table = 0x3002
    assert lib.kvq_append_block(C.byref(cache), k, v, 1, None, None) == L.KVQ_ERR_ALIGNMENT
    cache.block_table = None
    cache.n_blocks = 2
    q, o, ws = C.c_void_p(0x1000), C.c_void_p(0x3000), C.c_void_p(0x5000)
    assert lib.kvq_decode_attn(C.byref(cache), q, None, None, 0, o, ws, 1 << 24, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attn_static(C.byref(cache), q, None, None, 0, o, None) == L.KVQ_ERR_INVALID_ARG
    assert lib.kvq_dequant(C.byref(cache), 0, 1, 0, o, None, None) == L.KVQ_ERR_INVALID_ARG


def test_absmax_variants_layout_and_checks(K):
    """8-bit absmax tiles hold 4 codes per word (32 words per row) and one fp16 scale per token;
    64-channel blocks double the scales. Both are INT4-only; other bit widths are refused."""
    L = K._lib
    mk = lambda **kw: K.make_config("int4", kw.pop("bits", 4), 2, 3, 6, 5, **kw)
    for layout in ("rows", "mma"):
        for bits in (4, 8):
            for sg in (128, 64):
                lay = K.kvq_layout(mk(bits=bits, scale_group=sg, layout=layout))
                W = 128 // (32 // bits)
                assert lay.words_per_row == W and lay.codes_bytes[0] == 128 * W * 4
                assert lay.meta_bytes[0] == lay.meta_bytes[1] == (128 // sg) * 256
                assert lay.record_bytes == 2 * (128 * W * 4 + (128 // sg) * 256)
                assert K.kvq_decode_bytes(mk(bits=bits, scale_group=sg, layout=layout), 3) == 2 * 3 * 3 * lay.record_bytes
    assert K.kvq_layout(mk(scale_group=0)).meta_bytes[0] == 256
    # CSC value outliers: nuq only, same layout as CSR
    nq = lambda **kw: K.make_config("nuq", 3, 1, 2, 2, 4, **kw)
    a, b = K.kvq_layout(nq()), K.kvq_layout(nq(v_csc=True))
    assert (a.record_bytes, a.csr_off[1], a.csr_bytes[1]) == (b.record_bytes, b.csr_off[1], b.csr_bytes[1])
    for m in ("rtn", "varn", "int4"):
        with pytest.raises(K.KVQError):
            K.kvq_layout(K.make_config(m, 4 if m == "int4" else 2, 1, 1, 1, 2, v_csc=True))
    for bad in (dict(bits=2), dict(bits=3), dict(bits=6), dict(bits=16)):
        with pytest.raises(K.KVQError):
            K.kvq_layout(mk(**bad))
    with pytest.raises(K.KVQError):
        K.kvq_layout(mk(scale_group=32))
    for m in ("rtn", "nuq", "varn"):
        with pytest.raises(K.KVQError):
            K.kvq_layout(K.make_config(m, 8, 1, 1, 1, 2))
        with pytest.raises(K.KVQError):
            K.kvq_layout(K.make_config(m, 2, 1, 1, 1, 2, scale_group=64))


def test_calibrated_keys_and_sink_layout_and_checks(K):
    """key_calib and sink are NUQ-only; they add a calibration table (tau fp32, s and zp fp16 per
    (KV head, channel)) and a sink region (the first token's K and V rows per (b, h)) after the
    records; append refuses a key_calib cache until kvq_calibrate_keys has run."""
    L = K._lib
    lib = L.lib()
    w = WL.WORKLOADS[2].scaled(batch=3, n_kv_heads=4, n_q_heads=4, ctx=5 * 128)
    mk = lambda **kw: K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, w.dtype,
                                    w.pre_rope, w.rope_theta, w.outlier_frac, layout="mma", **kw)
    plain, both = K.kvq_layout(mk()), K.kvq_layout(mk(key_calib=True, sink=True))
    assert plain.calib_bytes == 0 and plain.sink_bytes == 0 and plain.total_bytes < both.total_bytes
    assert both.records_bytes == plain.records_bytes
    assert both.calib_bytes == 4 * 128 * 8 and both.sink_bytes == 3 * 4 * 2 * 128 * 2
    assert both.calib_off % 128 == 0 and both.calib_off >= plain.rope_off + plain.rope_bytes
    assert both.sink_off % 128 == 0 and both.sink_off >= both.calib_off + both.calib_bytes
    assert both.total_bytes == both.sink_off + both.sink_bytes
    out = L.kvq_layout_t()
    for kw in (dict(key_calib=True), dict(sink=True)):
        assert lib.kvq_layout(C.byref(K.make_config("rtn", 2, 1, 1, 1, 4, **kw)), C.byref(out)) == L.KVQ_ERR_UNSUPPORTED
    bad = mk()
    bad.sink = 2
    assert lib.kvq_layout(C.byref(bad), C.byref(out)) == L.KVQ_ERR_INVALID_ARG
    cache = L.kvq_cache()
    cache.cfg = mk(key_calib=True)
    cache.lay = K.kvq_layout(cache.cfg)
    cache.base = 0x100000
    cache.codebook = 0x200000
    k, v = C.c_void_p(0x1000), C.c_void_p(0x2000)
    assert lib.kvq_append_block(C.byref(cache), k, v, 1, None, None) == L.KVQ_ERR_INVALID_ARG  # not calibrated
    assert lib.kvq_calibrate_keys(C.byref(cache), k, 1, None) == L.KVQ_ERR_INVALID_ARG        # < 2 tokens
    assert lib.kvq_calibrate_keys(C.byref(cache), C.c_void_p(0x1008), 64, None) == L.KVQ_ERR_ALIGNMENT
    cache.cfg = mk()
    assert lib.kvq_calibrate_keys(C.byref(cache), k, 64, None) == L.KVQ_ERR_INVALID_ARG        # no key_calib


def test_nuq_decode_workspace_holds_the_tail_row(K):
    """The 3-bit nuq pre-RoPE decode (tensor-core format) keeps, per (batch, query head), one
    partial row per consumer warp and range slot plus one row for the fp tail its idle warps
    attend. Without a device the plan assumes a 152-SM part with one CTA per SM."""
    w = WL.WORKLOADS[2]
    cfg = K.make_config(w.method, w.bits, w.batch, w.n_kv_heads, w.n_q_heads, w.n_blocks, w.dtype, w.pre_rope,
                        w.rope_theta, w.outlier_frac, layout="mma")
    for nb in (1, 3, 200, w.n_blocks):
        total = w.batch * w.n_kv_heads * nb
        ranges = min(152, total)
        slots = min((nb - 1) * ranges // total + 2, nb)
        rows = w.batch * w.n_q_heads * (slots * 8 + 1)   # 8 consumer warps per range, + the tail row
        assert K.kvq_decode_workspace_bytes(cfg, nb) == 4 * (2 * rows + 4 + rows * 128), nb
