"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each test ties an oracle function to something other than itself: a value the pages
print (tests/golden/*.json), a closed form, an invariant, a library routine, or brute
force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.stats

import oracle as O
import workloads as WL


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ KV-cache size formula

def test_kv_cache_size_formula_matches_printed_values(golden_dir):
    g = _golden(golden_dir, "kv_cache_sizes.json")
    for c in g["cases"]:
        got = O.kv_cache_bytes(c["layers"], c["heads"], c["head_dim"], c["elem_bytes"],
                               c["batch"], c["seq_len"])
        assert abs(got - c["printed_bytes"]) <= c["tolerance_rel"] * c["printed_bytes"] + 0.5, c["cite"]
    # LLaMA-7B at 128K is exactly 64 GiB
    assert O.kv_cache_bytes(32, 32, 128, 2, 1, 131072) == 64 * 2 ** 30


# ------------------------------------------------------------------ packing layout

def test_3bit_layout_printed_words(golden_dir):
    g = _golden(golden_dir, "kvquant_3bit_layout.json")
    assert O.codes_per_word(3) == g["codes_per_word"]
    for c in g["cases"]:
        row = np.zeros(128, np.uint8)
        row[:10] = c["codes"]
        words = O.pack_rows(row[None, :], 3)[0]
        assert int(words[0]) == c["word"], c["cite"]
        assert int(words[0]) >> 30 == 0
    assert 128 * 3 == g["bits_per_128_channel_key"]["value"]


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_roundtrip_and_unused_bits(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, size=(64, 128)).astype(np.uint8)
    words = O.pack_rows(codes, bits)
    n = 32 // bits
    assert words.shape == (64, -(-128 // n))
    assert np.array_equal(O.unpack_rows(words, bits), codes)
    used = n * bits
    if used < 32:
        assert np.all((words >> np.uint32(used)) == 0)
    # the last word of a 3-bit row holds codes 120..127 only
    if bits == 3:
        assert np.all((words[:, 12] >> np.uint32(24)) == 0)
    # field i of word w is code w*n + i: check one element by direct bit reading
    assert ((int(words[5, 1]) >> (bits * 2)) & ((1 << bits) - 1)) == codes[5, n + 2]


def test_tile3_size_bijection_and_roundtrip(golden_dir):
    g = _golden(golden_dir, "kvquant_3bit_layout.json")
    assert O.TILE3_WORDS * 4 == 128 * g["bytes_per_128_channel_key"]["value"]
    t, c = np.meshgrid(np.arange(128), np.arange(128), indexing="ij")
    rng = np.random.default_rng(3)
    for kind in (O.KIND_K, O.KIND_V):
        lw, ls, hw, hs = O.tile3_slot(kind, t.ravel(), c.ravel())
        assert np.all((ls & 1) == 0) and np.all(ls <= 30) and np.all(hs <= 31)
        bit_ids = np.concatenate([lw * 32 + ls, lw * 32 + ls + 1, hw * 32 + hs])
        # every one of the 49152 bits of the tile holds exactly one bit of one code
        assert np.array_equal(np.sort(bit_ids), np.arange(O.TILE3_WORDS * 32))
        codes = rng.integers(0, 8, size=(128, 128)).astype(np.uint8)
        words = O.pack_tile3(codes, kind)
        assert words.dtype == np.uint32 and words.shape == (O.TILE3_WORDS,)
        assert np.array_equal(O.unpack_tile3(words, kind), codes)
        # a single code 5 = 0b101: low bits 01 at its low-bit slot, high bit at its high slot
        one = np.zeros((128, 128), np.uint8)
        one[77, 101] = 5
        w = O.pack_tile3(one, kind)
        lw1, ls1, hw1, hs1 = (int(x) for x in O.tile3_slot(kind, 77, 101))
        exp = np.zeros(O.TILE3_WORDS, np.uint64)
        exp[lw1] |= 1 << ls1
        exp[hw1] |= 1 << hs1
        assert np.array_equal(w.astype(np.uint64), exp)


def test_tile3_slots_follow_the_documented_rule():
    """Hand-evaluated positions from the rule in the layout's description."""
    # key (t=9, c=13): segment 0, t%8=1, (t%16)//8=1, (c//2)%4=2, c//8=1, c%2=1
    #   group 4*1+2=6 (word base 36), nibble word 13//16=0, slot 4*1+2*1+1=7
    assert tuple(int(x) for x in O.tile3_slot(O.KIND_K, 9, 13)) == (36, 28, 40, 30)
    # key (t=50, c=100): segment 3, t%16=2 -> g=2, r=0,
    #   (c//2)%4=2, c//8=12, c%2=0: group 10 (base 3*192+60=636), nibble word 6, slot 0
    #   low bits: word 636+3, shift 0; high bit: word 636+4+1, shift (2,3,0,1)[2] = 0
    assert tuple(int(x) for x in O.tile3_slot(O.KIND_K, 50, 100)) == (639, 0, 641, 0)
    # value (t=23, c=45): segment 1, t%16=7 -> t%4=3, (t%16)//4=1; c%8=5, (c//8)%2=1, c//16=2
    #   group 4*5+3=23 (base 192+138=330), nibble word 2, slot 4*1+2*1+0=6
    #   low bits: word 330+1, shift 24; high bit: word 330+4, shift 24+(2,3,0,1)[2]=24
    assert tuple(int(x) for x in O.tile3_slot(O.KIND_V, 23, 45)) == (331, 24, 334, 24)


@pytest.mark.parametrize("kind", [0, 1])
def test_tile3_groups_hold_one_lanes_fragment_codes(kind):
    """Group l = 4g + tq of segment s holds: keys, tokens 16s+g and 16s+g+8 at the 32
    channels c with (c//2)%4 = tq; values, tokens 16s+tq+4v (v = 0..3) at the 16 channels
    16m+g and 16m+g+8."""
    t, c = np.meshgrid(np.arange(128), np.arange(128), indexing="ij")
    lw, _, hw, _ = O.tile3_slot(kind, t, c)
    grp = lw // 6
    assert np.array_equal(grp, hw // 6)
    for s in (0, 5):
        for g in range(8):
            for tq in range(4):
                sel = grp == s * 32 + 4 * g + tq
                if kind == O.KIND_K:
                    exp = np.zeros((128, 128), bool)
                    for r in (0, 1):
                        exp[16 * s + g + 8 * r, [ch for ch in range(128) if (ch // 2) % 4 == tq]] = True
                else:
                    exp = np.zeros((128, 128), bool)
                    for v in range(4):
                        for m in range(8):
                            exp[16 * s + tq + 4 * v, [16 * m + g, 16 * m + g + 8]] = True
                assert np.array_equal(sel, exp)


# ------------------------------------------------------------------ uniform RTN

def test_scale_examples_per_token_vs_per_channel(golden_dir):
    g = _golden(golden_dir, "kvquant_scale_examples.json")
    bits = g["per_token"]["bits"]
    rng = np.random.default_rng(0)
    x = rng.uniform(-1, 1, size=(128, 128)).astype(np.float32)
    x[0, :] = -1.0
    x[1, :] = 1.0                           # every channel spans exactly [-1, 1]
    oc, oc2 = 7, 8
    x[:, oc] = np.where(np.arange(128) % 2 == 0, 15.0, -15.0)   # |K_{t,c'}| = 15
    x[:, oc2] = -x[:, oc]                  # each token spans [-15, 15]: range 30 as on the page
    x = WL.round_f16(x)
    _, s_tok, _ = O.rtn_quantize(x, bits, axis=1)
    _, s_ch, _ = O.rtn_quantize(x, bits, axis=0)
    s_tok = s_tok.astype(np.float64)
    s_ch = s_ch.astype(np.float64)
    assert np.all(np.abs(s_tok - g["per_token"]["approx"]) <= g["per_token"]["tolerance_abs"])
    normal = np.delete(s_ch, [oc, oc2])
    assert np.all(np.abs(normal - g["per_channel_normal"]["approx"]) <= g["per_channel_normal"]["tolerance_abs"])
    for c in (oc, oc2):
        assert abs(s_ch[c] - g["per_channel_outlier"]["approx"]) <= g["per_channel_outlier"]["tolerance_abs"]


def _rtn_bound_check(x, codes, s16, z16, bits, axis):
    xh = O.rtn_dequant(codes, s16, z16, axis)
    s = s16.astype(np.float64)
    z = z16.astype(np.float64)
    if axis == 0:
        s, z = s[None, :], z[None, :]
        mn = x.min(axis=0)[None, :].astype(np.float64)
    else:
        s, z = s[:, None], z[:, None]
        mn = x.min(axis=1)[:, None].astype(np.float64)
    err = np.abs(x.astype(np.float64) - xh)
    t = x.astype(np.float64) / s - z
    eps = 2.0 ** -22 * (np.abs(x / s) + np.abs(z) + 1.0)
    unclamped = (np.rint(t) >= 0) & (np.rint(t) <= 2 ** bits - 1)
    # |x - x_dq| <= s/2 on every element that was not clamped (rounding of fp32 steps aside)
    sb = np.broadcast_to(s, x.shape)
    assert np.all(err[unclamped] <= sb[unclamped] * (0.5 + eps[unclamped]))
    # clamping only comes from fp16 rounding of the zero point: error <= s/2 + s*|z16 - min/s|
    zerr = np.abs(z - mn / s)
    bound = s * (0.5 + zerr + eps + 2.0 ** -10 * (2 ** bits))
    assert np.all(err <= bound)
    return unclamped


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("axis", [0, 1])
def test_rtn_error_bound(bits, axis):
    w = WL.WORKLOADS[5]
    for blk in range(3):
        x = WL.tile(w, 0, 3, blk, WL.KIND_K)       # includes x12 outlier channels
        codes, s16, z16 = O.rtn_quantize(x, bits, axis)
        assert codes.max() <= 2 ** bits - 1
        _rtn_bound_check(x, codes, s16, z16, bits, axis)
        # the extremes of each group are reproduced to within s/2
        xh = O.rtn_dequant(codes, s16, z16, axis)
        am = np.argmax(x, axis=axis)
        if axis == 0:
            assert np.all(np.abs(xh[am, np.arange(128)] - x[am, np.arange(128)]) <= s16.astype(float) * 0.5 + 1e-6)


def test_rtn_constant_group_is_exact():
    x = np.full((128, 128), 0.75, np.float32)
    codes, s16, z16 = O.rtn_quantize(x, 2, 0)
    assert np.all(s16 == 1.0) and np.all(codes == 0)
    assert np.array_equal(O.rtn_dequant(codes, s16, z16, 0), x.astype(np.float64))


def test_rtn_grid_inputs_are_lossless():
    # values on the grid {min + k*s}, s a power of two, are reproduced exactly
    rng = np.random.default_rng(1)
    q = rng.integers(0, 4, size=(128, 128))
    q[0, :], q[1, :] = 0, 3
    x = (q.astype(np.float32) - 2.0) * np.float32(0.25)
    codes, s16, z16 = O.rtn_quantize(x, 2, 0)
    assert np.array_equal(O.rtn_dequant(codes, s16, z16, 0), x.astype(np.float64))


# ------------------------------------------------------------------ int4 absmax

def test_int4_codes_range_and_bound():
    w = WL.WORKLOADS[4]
    for blk in range(3):
        x = WL.tile(w, 1, 2, blk, WL.KIND_V)
        q, s16 = O.int4_quantize(x)
        assert q.min() >= -7 and q.max() <= 7
        s = s16.astype(np.float64)
        a = np.abs(x).max(axis=1)
        # the element with |x| = absmax maps to +-7
        for t in range(128):
            j = int(np.argmax(np.abs(x[t])))
            assert abs(int(q[t, j])) == 7
        err = np.abs(x.astype(np.float64) - O.int4_dequant(q, s16))
        assert np.all(err <= (s * 0.5 * (1 + 2.0 ** -10))[:, None])
        # fp16 scale is absmax/7 rounded once
        assert np.all(np.abs(s - a / 7.0) <= np.abs(a / 7.0) * 2.0 ** -11)
        nib = O.int4_nibbles(q)
        assert nib.max() <= 15 and np.array_equal(O.int4_from_nibbles(nib), q)


def test_int4_zero_block_and_lossless_grid():
    x = np.zeros((128, 128), np.float32)
    q, s16 = O.int4_quantize(x)
    assert np.all(q == 0) and np.all(s16 == 0)
    rng = np.random.default_rng(2)
    q0 = rng.integers(-7, 8, size=(128, 128))
    q0[:, 5] = 7
    x = (q0 * 0.125).astype(np.float32)         # scale = 7*0.125/7 = 0.125 exactly
    q, s16 = O.int4_quantize(x)
    assert np.array_equal(q, q0) and np.all(s16 == 0.125)
    # two's complement nibble of -1 is 0xF, of -7 is 0x9
    assert O.int4_nibbles(np.array([-1, -7, 7, 0]))[:4].tolist() == [15, 9, 7, 0]


@pytest.mark.parametrize("bits,group", [(8, 128), (8, 64), (4, 64)])
def test_absmax_variants_codes_range_and_bound(bits, group):
    """8-bit and 64-channel blocks ([TQ] §5.1, §2.1): codes within +-(2^(b-1)-1), each block's
    largest element at the end of the range, |x - q*s| <= s/2 per block, s = absmax/(2^(b-1)-1)
    rounded once to fp16, codes round-trip through their two's complement form."""
    w = WL.WORKLOADS[4]
    qmax = 2 ** (bits - 1) - 1
    for blk in range(2):
        x = WL.tile(w, 1, 2, blk, WL.KIND_K)
        q, s16 = O.absmax_quantize(x, bits, group)
        assert s16.shape == (128 // group, 128)
        assert q.min() >= -qmax and q.max() <= qmax
        xg = x.astype(np.float64).reshape(128, 128 // group, group)
        a = np.abs(xg).max(axis=2)                       # [t][g]
        s = s16.T.astype(np.float64)                     # [t][g]
        assert np.all(np.abs(s - a / qmax) <= np.abs(a / qmax) * 2.0 ** -11)
        qg = q.reshape(128, 128 // group, group)
        for t in range(0, 128, 7):
            for g in range(128 // group):
                j = int(np.argmax(np.abs(xg[t, g])))
                assert abs(int(qg[t, g, j])) == qmax
        err = np.abs(xg - qg * s[:, :, None])
        assert np.all(err <= s[:, :, None] * 0.5 * (1 + 2.0 ** -10))
        assert np.allclose(O.absmax_dequant(q, s16), (qg * s[:, :, None]).reshape(128, 128), rtol=0, atol=0)
        codes = O.absmax_codes(q, bits)
        assert codes.max() < 2 ** bits and np.array_equal(O.absmax_from_codes(codes, bits), q)
    assert O.absmax_codes(np.array([-1, -127, 127, -128]), 8).tolist() == [255, 129, 127, 128]


@pytest.mark.parametrize("bits", [4, 8])
def test_absmax_group64_is_group128_on_each_half(bits):
    """A 64-channel block is a 128-channel block whose other half is zero."""
    x = WL.tile(WL.WORKLOADS[4], 0, 1, 1, WL.KIND_V)
    q, s16 = O.absmax_quantize(x, bits, 64)
    for g in range(2):
        pad = np.zeros_like(x)
        pad[:, :64] = x[:, 64 * g:64 * (g + 1)]
        q1, s1 = O.absmax_quantize(pad, bits, 128)
        assert np.array_equal(q[:, 64 * g:64 * (g + 1)], q1[:, :64]) and not q1[:, 64:].any()
        assert np.array_equal(s16[g], s1[0])


def test_absmax_int8_lossless_grid_and_zero_block():
    rng = np.random.default_rng(3)
    q0 = rng.integers(-127, 128, size=(128, 128))
    q0[:, 5], q0[:, 77] = 127, -127
    x = (q0 * 0.0078125).astype(np.float32)      # scale = 127/128/127 = 2^-7 exactly
    for group in (128, 64):
        q, s16 = O.absmax_quantize(x, 8, group)
        assert np.array_equal(q, q0) and np.all(s16 == 0.0078125)
    q, s16 = O.absmax_quantize(np.zeros((128, 128), np.float32), 8, 64)
    assert not q.any() and not s16.any()


# ------------------------------------------------------------------ nuq (KVQuant)

def test_worked_example_normalise_and_argmin(golden_dir):
    g = _golden(golden_dir, "kvquant_worked_example.json")
    cb = np.array(g["codebook_channel_15"]["values"], np.float32)
    for key in ("channel_15", "channel_0"):
        c = g[key]
        t = O.nuq_normalise(np.float32(c["k"]), np.float16(c["s"]), np.float16(c["z"]))
        assert abs(float(t) - c["k_norm"]) < 2e-3, c["cite"]
        assert int(O.nuq_encode(np.array([t]), cb)[0]) == c["index"], c["cite"]
    for key in ("outlier_channel_7", "channel_0_not_outlier"):
        c = g[key]
        dense, sparse = O.threshold_split(np.array([c["k"]]), np.array([c["tau"]]))
        assert (sparse[0] != 0) == c["is_outlier"], c["cite"]
        assert dense[0] == (0.0 if c["is_outlier"] else c["k"])


def test_codebook_is_scaled_normal_quantiles():
    cb = O.nuq_codebook(3).astype(np.float64)
    ref = scipy.stats.norm.ppf((np.arange(8) + 0.5) / 8)
    ref = ref / ref[-1]
    assert np.allclose(cb, ref, rtol=0, atol=1e-7)
    assert cb[0] == -1.0 and cb[-1] == 1.0
    assert np.all(np.diff(cb) > 0) and np.allclose(cb, -cb[::-1])


def test_nuq_argmin_equals_brute_force():
    rng = np.random.default_rng(3)
    cb = O.nuq_codebook(3)
    mids = (cb[:-1].astype(np.float64) + cb[1:]) / 2
    t = np.concatenate([rng.uniform(-1, 1, 500), mids, cb.astype(np.float64), [-1.0, 1.0, 0.0]]).astype(np.float32)
    got = O.nuq_encode(t, cb)
    for i, v in enumerate(t):
        best, bj = None, None
        for j, c in enumerate(cb):
            d = abs(np.float32(v) - np.float32(c))
            if best is None or d < best:
                best, bj = d, j
        assert got[i] == bj


def test_outlier_selection_planted_and_ties():
    rng = np.random.default_rng(4)
    x = rng.uniform(-1, 1, size=(128, 128)).astype(np.float32)
    flat = rng.choice(128 * 128, size=164, replace=False)
    x.ravel()[flat] = rng.uniform(5, 9, size=164) * rng.choice([-1, 1], size=164)
    x = WL.round_f16(x)
    m = O.outlier_mask(x, 164)
    assert set(np.flatnonzero(m)) == set(flat)
    # ties on |x|: 200 entries of equal magnitude -> the 164 with the lowest flat index
    y = np.zeros((128, 128), np.float32)
    pos = np.sort(rng.choice(128 * 128, size=200, replace=False))
    y.ravel()[pos] = np.where(rng.random(200) < 0.5, -3.0, 3.0)
    m = O.outlier_mask(y, 164)
    assert set(np.flatnonzero(m)) == set(pos[:164])


def test_nuq_quantize_csr_and_bound():
    w = WL.WORKLOADS[2]
    cb = O.nuq_codebook(3)
    for kind, axis in ((WL.KIND_K, 0), (WL.KIND_V, 1)):
        x = WL.tile(w, 0, 7, 3, kind)
        r = O.nuq_quantize(x, cb, axis, 164)
        rp, col, val = r["row_ptr"].astype(int), r["col"].astype(int), r["val"]
        assert rp[0] == 0 and rp[-1] == 164 and np.all(np.diff(rp) >= 0)
        for t in range(128):
            cs = col[rp[t]:rp[t + 1]]
            assert np.all(np.diff(cs) > 0)
            for j, c in enumerate(cs):
                assert r["mask"][t, c]
                assert val[rp[t] + j] == np.float16(x[t, c]).view(np.uint16)   # bit-exact fp16
        # the outliers are the 164 largest magnitudes
        thr = np.sort(np.abs(x).ravel())[-164]
        assert np.all(np.abs(x[r["mask"]]) >= thr) and np.all(np.abs(x[~r["mask"]]) <= thr)
        xh = O.nuq_dequant(r["codes"], r["s16"], r["zp16"], cb, axis, r["row_ptr"], r["col"], r["val"])
        s = r["s16"].astype(np.float64)
        s = s[None, :] if axis == 0 else s[:, None]
        gap = np.max(np.diff(cb.astype(np.float64))) / 2
        err = np.abs(xh - x)
        dense_ok = ~r["mask"]
        sb = np.broadcast_to(s, x.shape)
        assert np.all(err[dense_ok] <= (sb * (gap + 2.0 ** -9))[dense_ok])
        # at an outlier the error is the quantisation error of a dense zero
        t0 = O.nuq_normalise(np.zeros_like(x), r["s16"][None, :] if axis == 0 else r["s16"][:, None],
                             r["zp16"][None, :] if axis == 0 else r["zp16"][:, None])
        e0 = np.abs(t0.astype(np.float64) - cb.astype(np.float64)[O.nuq_encode(t0, cb)]) * sb
        zp = r["zp16"].astype(np.float64)
        zp = zp[None, :] if axis == 0 else zp[:, None]
        clampx = np.abs(np.broadcast_to(zp, x.shape)) - sb
        lim = e0 + np.maximum(clampx, 0) + 1e-6
        assert np.all(err[r["mask"]] <= lim[r["mask"]])


def test_csc_of_brute_force_and_same_entries_as_csr():
    """Value outliers by column ([KVQ] §3.4): column pointers and the per-entry token, built
    here by plain loops over channels then tokens, and the (token, channel, value) set equals
    the CSR's."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((O.T, O.D)).astype(np.float32)
    for frac in (0.0, 0.01, 0.05, 0.3):
        mask = rng.uniform(size=x.shape) < frac
        mask[5, :] = True   # a full row
        mask[:, 77] = True  # a full column
        col_ptr, row, val = O.csc_of(x, mask)
        cp, rr, vv = [0], [], []
        for c in range(O.D):
            for t in range(O.T):
                if mask[t, c]:
                    rr.append(t)
                    vv.append(np.float16(x[t, c]).view(np.uint16))
            cp.append(len(rr))
        assert col_ptr.tolist() == cp and row.tolist() == rr and val.tolist() == [int(v) for v in vv]
        row_ptr, col, val_r = O.csr_of(x, mask)
        csr_set = {(t, int(col[j]), int(val_r[j])) for t in range(O.T) for j in range(int(row_ptr[t]), int(row_ptr[t + 1]))}
        csc_set = {(int(row[j]), c, int(val[j])) for c in range(O.D) for j in range(int(col_ptr[c]), int(col_ptr[c + 1]))}
        assert csr_set == csc_set and len(csc_set) == int(mask.sum())


def test_csc_tiles_dequantise_and_decode_like_csr():
    """The storage order of the value outliers changes nothing: dequantised tiles and the cache's
    decode are identical for CSR and CSC value tiles, for 1% and 5% outliers."""
    for frac in (0.01, 0.05):
        w = WL.WORKLOADS[2].scaled(batch=1, n_kv_heads=2, n_q_heads=2, ctx=2 * 128, outlier_frac=frac)
        K, V = WL.blocks(w, 0, w.n_blocks)
        caches = []
        for csc in (False, True):
            oc = O.OracleCache.for_workload(w, v_csc=csc)
            oc.append(K, V)
            caches.append(oc)
        for key in caches[0].recs:
            a, b = caches[0].recs[key], caches[1].recs[key]
            if key[3] == O.KIND_V:
                assert "col_ptr" in b and "row_ptr" not in b
                assert int(b["col_ptr"][-1]) == int(a["row_ptr"][-1]) == O.n_outliers(frac)
            assert np.array_equal(caches[0].dequant_tile(a, key[3], key[1], key[2], "attn"),
                                  caches[1].dequant_tile(b, key[3], key[1], key[2], "attn"))
        q = WL.query(w)
        tk, tv = WL.tail(w, 9)
        assert np.array_equal(caches[0].decode(q, tk, tv), caches[1].decode(q, tk, tv))


def test_nuq_lossless_on_codebook_grid():
    cb = np.array([-1, -0.75, -0.5, -0.25, 0.25, 0.5, 0.75, 1.0], np.float32)
    rng = np.random.default_rng(5)
    q = rng.integers(0, 8, size=(128, 128))
    q[0, :], q[1, :] = 0, 7
    x = (cb[q] * 0.5 + 0.25).astype(np.float32)            # s = 0.5, zp = 0.25 per channel
    x[10, 20] = 40.0                                       # one planted outlier, stored exactly
    r = O.nuq_quantize(x, cb, 0, 1)
    xh = O.nuq_dequant(r["codes"], r["s16"], r["zp16"], cb, 0, r["row_ptr"], r["col"], r["val"])
    dense0 = cb[r["codes"][10, 20]] * 0.5 + 0.25          # dense zero quantised, then += 40
    assert xh[10, 20] == pytest.approx(40.0 + dense0)
    xh[10, 20] = x[10, 20]
    assert np.array_equal(xh, x.astype(np.float64))


# ------------------------------------------------------------------ RoPE

def test_rope_norm_identity_and_relative_position(golden_dir):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((300, 128))
    pos = rng.integers(0, 1 << 20, size=300)
    y = O.rope(x, pos)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12, atol=0)
    assert np.array_equal(O.rope(x[:5], np.zeros(5)), x[:5])
    # (R_m q) . (R_n k) = q . (R_{n-m} k)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for m, n in ((3, 10), (1000, 77), (123456, 654321)):
        lhs = O.rope(q[None], [m])[0] @ O.rope(k[None], [n])[0]
        rhs = q @ O.rope(k[None], [n - m])[0]
        assert lhs == pytest.approx(rhs, rel=1e-9, abs=1e-9)
    # orientation of the printed matrix: (1, 0) at angle phi goes to (cos phi, sin phi)
    e = np.zeros((1, 128))
    e[0, 0] = 1.0
    y = O.rope(e, [1])                    # theta_0 = 1 rad
    assert y[0, 0] == pytest.approx(math.cos(1.0)) and y[0, 1] == pytest.approx(math.sin(1.0))
    # lowest frequency pair i = 63: theta^(-126/128)
    e = np.zeros((1, 128))
    e[0, 126] = 1.0
    y = O.rope(e, [1000])
    ang = 1000 * 10000.0 ** (-126 / 128)
    assert y[0, 126] == pytest.approx(math.cos(ang)) and y[0, 127] == pytest.approx(math.sin(ang))


def test_rope_variance_example(golden_dir):
    g = _golden(golden_dir, "rope_variance_example.json")
    rng = np.random.default_rng(7)
    n = 200000
    x = np.zeros((n, 128))
    x[:, 0] = rng.standard_normal(n) * math.sqrt(g["var_channel0"])
    x[:, 1] = rng.standard_normal(n) * math.sqrt(g["var_channel1"])
    y = O.rope(x, rng.integers(0, 100000, size=n))
    v = y[:, 0].var()
    assert abs(v - g["post_rope_var"]) <= g["tolerance_rel"] * g["post_rope_var"]
    assert abs(math.sqrt(v) - g["post_rope_std_approx"]) < 0.2


# ------------------------------------------------------------------ KVarN

def test_hadamard_sylvester_and_orthogonality():
    H = O.hadamard(128)
    assert np.array_equal(H, scipy.linalg.hadamard(128))
    assert np.array_equal(H @ H.T, 128 * np.eye(128))
    x = np.random.default_rng(8).standard_normal((16, 128))
    assert np.allclose(O.fwht(O.fwht(x)), x, rtol=0, atol=1e-12)
    # integer inputs: H (H x) = 128 x exactly
    xi = np.random.default_rng(9).integers(-50, 50, size=(4, 128)).astype(np.float64)
    assert np.array_equal((xi @ H) @ H, 128 * xi)
    # unit vector e_0 spreads evenly: every output is 1/sqrt(128)
    e = np.zeros((1, 128))
    e[0, 0] = 1
    assert np.allclose(O.fwht(e), 1 / math.sqrt(128))


def test_varn_recomposition_and_stds():
    w = WL.WORKLOADS[3]
    x = O.fwht(WL.tile(w, 2, 1, 0, WL.KIND_K))
    Y, r, c = O.varn(x, 8)
    assert np.allclose(r[:, None] * Y * c[None, :], x, rtol=1e-12, atol=1e-12)
    assert np.allclose(Y.std(axis=1), 1.0, atol=1e-12)          # rows normalised last
    assert np.max(np.abs(Y.std(axis=0) - 1.0)) < 0.05           # columns near 1 after 8 rounds
    Y0, r0, c0 = O.varn(x, 0)
    assert np.array_equal(Y0, x) and np.all(r0 == 1) and np.all(c0 == 1)


@pytest.mark.parametrize("kind", [0, 1])
def test_varn_reduces_to_rtn_without_hadamard_and_iterations(kind):
    w = WL.WORKLOADS[3]
    x = WL.tile(w, 0, 0, 1, kind)
    v = O.varn_quantize(x, 2, kind, iters=0, use_hadamard=False)
    codes, s16, z16 = O.rtn_quantize(x, 2, 0 if kind == 0 else 1)
    assert np.array_equal(v["codes"], codes)
    assert np.array_equal(v["s16"], s16) and np.array_equal(v["z16"], z16)
    assert np.all(v["s1"] == 1)


@pytest.mark.parametrize("kind", [0, 1])
def test_varn_reconstruction_bound(kind):
    w = WL.WORKLOADS[3]
    x = WL.tile(w, 1, 5, 2, kind)
    v = O.varn_quantize(x, 2, kind, 8, True)
    xh_H = O.varn_dequant(v["codes"], v["s16"], v["z16"], v["s1"], kind)
    # Hadamard-domain error = s1 * RTN error on Z, plus the fp16 rounding of s1
    Z = v["Z"]
    zh = O.rtn_dequant(v["codes"], v["s16"], v["z16"], v["axis"])
    s = v["s16"].astype(np.float64)
    s = s[None, :] if kind == 0 else s[:, None]
    assert np.all(np.abs(Z - zh) <= s * (0.5 + 2e-3) + 1e-6)
    s1 = v["s1"].astype(np.float64)
    true_s1 = v["r"] if kind == 0 else v["c"]
    assert np.all(np.abs(s1 - true_s1) <= true_s1 * 2.0 ** -11)
    X = O.fwht(x)
    ref = (Z * true_s1[:, None]) if kind == 0 else (Z * true_s1[None, :])
    assert np.allclose(ref, X, rtol=1e-10, atol=1e-10)
    # norm/direction identity on the reconstruction
    xh = O.fwht(xh_H)
    em, ed = O.norm_direction_errors(x, xh)
    tot = ((x.astype(np.float64) - xh) ** 2).sum(axis=1)
    assert np.allclose(em + ed, tot, rtol=1e-9, atol=1e-12)


def test_norm_direction_decomposition_closed_forms():
    K = np.array([[3.0, 4.0]])
    assert O.norm_direction_errors(K, 2 * K)[0][0] == pytest.approx(25.0)   # scaled copy: norm error only
    assert O.norm_direction_errors(K, 2 * K)[1][0] == pytest.approx(0.0, abs=1e-12)
    e = O.norm_direction_errors(np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]]))
    assert e[0][0] == pytest.approx(0.0) and e[1][0] == pytest.approx(2.0)   # rotation: direction only


def test_token_error_stats_closed_forms():
    x = np.array([[3.0, 4.0, 0.0], [1.0, 0.0, 0.0], [0.0, 2.0, 0.0], [0.0, 0.0, 0.0], [1.0, 1.0, 1.0]])
    xq = np.array([[6.0, 8.0, 0.0],    # scaled copy: |dx| = |x|, all of it norm error
                   [0.0, 1.0, 0.0],    # same norm, orthogonal: all of it direction error, 2|x|^2
                   [0.0, 0.0, 0.0],    # reconstructed as zero: E_T = E_M = |x|^2, no direction
                   [0.0, 0.0, 1.0],    # input zero
                   [1.0, 1.0, 1.0]])   # exact
    s = O.token_error_stats(x, xq)
    assert np.allclose(s[0], [5.0, 5.0, 25.0, 0.0], atol=1e-12)
    assert np.allclose(s[1], [1.0, 0.0, 2.0, 2.0], atol=1e-12)
    assert np.allclose(s[2], [2.0, -2.0, 4.0, 0.0], atol=1e-12)
    assert np.allclose(s[3], [0.0, 1.0, 1.0, 0.0], atol=1e-12)
    assert np.allclose(s[4], [math.sqrt(3.0), 0.0, 0.0, 0.0], atol=1e-12)
    # antiparallel copy of equal norm: E_D = 4|x|^2, E_M = 0
    assert np.allclose(O.token_error_stats(x[:1], -x[:1])[0], [5.0, 0.0, 100.0, 100.0], atol=1e-9)


def test_token_error_stats_identity_on_reconstructions():
    """E_T = E_M + E_D on real reconstructions (RTN2 keys and values, int4), with the norm part
    the square of the norm deviation; and E_T equals the squared error summed directly."""
    w = WL.WORKLOADS[3]
    for kind in (0, 1):
        x = WL.tile(w, 0, 1, 3, kind)
        c, s16, z16 = O.rtn_quantize(x, 2, 0 if kind == 0 else 1)
        xq = O.rtn_dequant(c, s16, z16, 0 if kind == 0 else 1)
        st = O.token_error_stats(x, xq)
        em, ed = O.norm_direction_errors(x, xq)
        assert np.allclose(st[:, 1] ** 2, em, rtol=1e-9, atol=1e-12)
        assert np.allclose(st[:, 3], ed, rtol=1e-9, atol=1e-12)
        assert np.allclose(st[:, 1] ** 2 + st[:, 3], st[:, 2], rtol=1e-9, atol=1e-12)
        assert np.allclose(st[:, 2], [sum((float(a) - float(b)) ** 2 for a, b in zip(r, rq)) for r, rq in zip(x, xq)],
                           rtol=1e-12)
    q, s16 = O.int4_quantize(WL.tile(w, 0, 0, 0, 0))
    xq = O.int4_dequant(q, s16)
    st = O.token_error_stats(WL.tile(w, 0, 0, 0, 0), xq)
    assert np.allclose(st[:, 1] ** 2 + st[:, 3], st[:, 2], rtol=1e-9, atol=1e-12)


def test_topk_error_share_brute_force():
    rng = np.random.default_rng(5)
    n = 37
    st = np.zeros((n, 4))
    st[:, 0] = rng.random(n) + 1.0
    st[:, 1] = rng.standard_normal(n) * 0.1
    st[:, 2] = np.round(rng.random(n) * 8) / 8.0 + st[:, 1] ** 2  # several equal errors
    st[:, 3] = st[:, 2] - st[:, 1] ** 2
    st[[3, 17, 30], 2] = 7.0  # three-way tie at the top
    fracs = [1 / 37, 2 / 37, 0.1, 0.5, 1.0]
    got = O.topk_error_share(st, fracs)
    for f, row in zip(fracs, got):
        k = math.ceil(f * n)
        ranked = sorted(range(n), key=lambda i: (-st[i, 2], i))[:k]  # Python's own sort
        assert row[0] == k
        assert row[1] == pytest.approx(math.fsum(st[i, 2] for i in ranked), rel=1e-14)
        assert row[2] == pytest.approx(math.fsum(st[i, 1] ** 2 for i in ranked), rel=1e-14)
        assert row[3] == pytest.approx(math.fsum(st[i, 3] for i in ranked), rel=1e-14)
    assert got[0, 1] == 7.0 and got[0, 2] == st[3, 1] ** 2   # the tie goes to the lowest row
    assert got[1, 2] == pytest.approx(st[3, 1] ** 2 + st[17, 1] ** 2, rel=1e-14)


# ------------------------------------------------------------------ codebook fitting (KVQuant Algorithm 2)

def test_fit_codebook_uniform_density_gives_the_uniform_quantizer():
    """Lloyd's fixed point for a uniform density on [-1, 1] with equal weights is the uniform
    quantizer: centres at the midpoints (2j + 1)/k - 1 of k equal cells."""
    rng = np.random.default_rng(0)
    a = rng.uniform(-1, 1, 200_000).astype(np.float32)
    for bits in (2, 3):
        k = 2 ** bits
        c, it = O.fit_codebook(a, np.ones_like(a), bits, 200)
        assert it < 200
        assert np.allclose(c, (2 * np.arange(k) + 1) / k - 1, atol=0.01)


def test_fit_codebook_weighted_means_of_separated_groups():
    """Four well-separated groups: after convergence each centre is its group's weighted mean
    (Python's exact fsum of w*a over fsum of w), not the plain mean."""
    rng = np.random.default_rng(1)
    groups = [(-0.9, 0.03), (-0.3, 0.05), (0.25, 0.04), (0.85, 0.02)]
    a = np.concatenate([np.float32(m) + np.float32(sd) * rng.standard_normal(500).astype(np.float32) for m, sd in groups])
    w = rng.uniform(0.0, 1.0, a.size).astype(np.float32) ** 3
    c, _ = O.fit_codebook(a, w, 2, 100)
    for j, (m, _) in enumerate(groups):
        sel = slice(500 * j, 500 * (j + 1))
        exp = math.fsum(float(x) * float(y) for x, y in zip(a[sel], w[sel])) / math.fsum(float(y) for y in w[sel])
        assert abs(float(c[j]) - exp) <= 1e-6, (j, c[j], exp)
        plain = float(np.mean(a[sel].astype(np.float64)))
        assert abs(exp - plain) > 1e-4  # the weights matter in this fixture


def test_fit_codebook_converged_state_and_ties():
    rng = np.random.default_rng(2)
    a = np.tanh(rng.standard_normal(20_000)).astype(np.float32)
    w = rng.uniform(0, 1, a.size).astype(np.float32)
    c, it = O.fit_codebook(a, w, 3, 500)
    assert it < 500
    # every sample's nearest centre (brute force, first on ties) is the one it was averaged into
    d = np.abs(a[:, None] - c[None, :])
    assign = np.array([min(range(8), key=lambda j: (d[i, j], j)) for i in range(0, a.size, 97)])
    assert np.array_equal(assign, np.argmin(d[::97], axis=1))
    full = np.argmin(d, axis=1)
    for j in range(8):
        m = full == j
        exp = float(np.sum(w[m].astype(np.float64) * a[m]) / np.sum(w[m].astype(np.float64)))
        assert abs(float(c[j]) - exp) <= 1e-6
    # a sample equidistant from two centres joins the lower one: bits 1, centres start at -1, 1
    c, _ = O.fit_codebook(np.array([0.0, 0.5], np.float32), np.ones(2, np.float32), 1, 10)
    assert c.tolist() == [0.0, 0.5]
    # one-bit symmetric data: the centres are -+ the weighted mean magnitude
    x = np.array([-0.75, -0.25, 0.25, 0.75], np.float32)
    c, _ = O.fit_codebook(x, np.array([0.25, 0.75, 0.75, 0.25], np.float32), 1, 10)
    assert c.tolist() == [-0.375, 0.375]
    # weights are clamped to [0, 1] (and samples to [-1, 1]): 3 weighs as 1
    c, _ = O.fit_codebook(x, np.array([1, 3, 3, 1], np.float32), 1, 10)
    assert c.tolist() == [-0.5, 0.5]


# ------------------------------------------------------------------ attention

def _brute_attention(q, K, V):
    out = []
    for qi in q:
        s = [sum(float(qi[c]) * float(k[c]) for c in range(len(qi))) / math.sqrt(len(qi)) for k in K]
        m = max(s)
        e = [math.exp(v - m) for v in s]
        z = sum(e)
        out.append([sum(e[n] * float(V[n][c]) for n in range(len(K))) / z for c in range(len(qi))])
    return np.array(out)


@pytest.mark.parametrize("L", [1, 127, 128, 129, 255])
def test_attention_brute_force(L):
    rng = np.random.default_rng(L)
    q = rng.standard_normal((2, 16)) * 2
    K = rng.standard_normal((L, 16)) * 2
    V = rng.standard_normal((L, 16))
    assert np.allclose(O.attention(q, K, V), _brute_attention(q, K, V), rtol=1e-12, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((3, 128))
    V = rng.standard_normal((1, 128))
    assert np.array_equal(O.attention(q, rng.standard_normal((1, 128)), V), np.repeat(V, 3, axis=0))
    V = rng.standard_normal((50, 128))
    K = np.repeat(rng.standard_normal((1, 128)), 50, axis=0)
    assert np.allclose(O.attention(q, K, V), V.mean(axis=0)[None, :], rtol=0, atol=1e-12)


def _lossless_cache_inputs(method, B, H, n_blocks, rng, cb=None):
    """Inputs the quantizer reproduces exactly: every group (a key channel, a value token;
    a token for int4) lies on its own dyadic grid with its extremes present. Group scales
    differ, so grouping along the wrong axis would not be lossless."""
    K = np.empty((B, H, n_blocks * 128, 128), np.float32)
    V = np.empty_like(K)
    ch = (2.0 ** (np.arange(128) % 3 - 2))[None, :]           # per-channel scales 1/4, 1/2, 1
    tok = (2.0 ** (np.arange(128) % 4 - 3))[:, None]          # per-token scales 1/8 .. 1
    for b in range(B):
        for h in range(H):
            for blk in range(n_blocks):
                sl = slice(blk * 128, (blk + 1) * 128)
                if method == "rtn":            # 2-bit grid, per channel (K) / per token (V)
                    qk = rng.integers(0, 4, (128, 128)); qk[0], qk[1] = 0, 3
                    qv = rng.integers(0, 4, (128, 128)); qv[:, 0], qv[:, 1] = 0, 3
                    K[b, h, sl] = (qk - 1.5) * ch
                    V[b, h, sl] = (qv - 2.0) * tok
                elif method.startswith("int"):  # per token (per half-token for g64) for both
                    m = 127 if method.startswith("int8") else 7
                    qk = rng.integers(-m, m + 1, (128, 128)); qk[:, 3] = qk[:, 70] = -m
                    qv = rng.integers(-m, m + 1, (128, 128)); qv[:, 9] = qv[:, 100] = m
                    K[b, h, sl] = qk * 0.125 * tok
                    V[b, h, sl] = qv * 0.0625 * tok[::-1]
                    if method.endswith("g64"):  # the two halves of a token on different grids
                        K[b, h, sl, 64:] *= 2.0
                        V[b, h, sl, 64:] *= 0.5
                else:                          # nuq with a dyadic codebook, no outliers
                    qk = rng.integers(0, 8, (128, 128)); qk[0], qk[1] = 0, 7
                    qv = rng.integers(0, 8, (128, 128)); qv[:, 0], qv[:, 1] = 0, 7
                    K[b, h, sl] = cb[qk] * ch + 0.25 * ch
                    V[b, h, sl] = cb[qv] * tok - 0.5 * tok
    return K, V


@pytest.mark.parametrize("method,G,pre_rope", [("rtn", 1, False), ("rtn", 4, False),
                                               ("int4", 4, False), ("nuq", 1, True), ("nuq", 2, False),
                                               ("int8", 2, False), ("int4g64", 1, False), ("int8g64", 4, False)])
def test_cache_decode_equals_plain_attention_on_lossless_inputs(method, G, pre_rope):
    """On inputs the quantizer reproduces exactly, decode over the packed cache must equal
    plain fp64 attention over the raw K/V (RoPE at absolute positions for pre-RoPE keys),
    including the fp tail and the GQA head mapping."""
    rng = np.random.default_rng(12)
    B, H, nb = 2, 2, 3
    cb = np.array([-1, -0.75, -0.5, -0.25, 0.25, 0.5, 0.75, 1.0], np.float32)
    bits = {"rtn": 2, "int4": 4, "nuq": 3, "int8": 8, "int4g64": 4, "int8g64": 8}[method]
    group = 64 if method.endswith("g64") else 128
    cache = O.OracleCache("int4" if method.startswith("int") else method, bits, B, H, H * G, pre_rope=pre_rope,
                          outlier_frac=0.0, codebook=cb if method == "nuq" else None, scale_group=group)
    K, V = _lossless_cache_inputs(method, B, H, nb, rng, cb)
    cache.append(K[:, :, :256], V[:, :, :256])
    cache.append(K[:, :, 256:], V[:, :, 256:])
    q = rng.standard_normal((B, H * G, 128))
    tk = rng.standard_normal((B, H, 5, 128))
    tv = rng.standard_normal((B, H, 5, 128))
    got = cache.decode(q, tk, tv)
    for b in range(B):
        for j in range(H * G):
            h = j // G
            Kf = np.concatenate([K[b, h], tk[b, h]]).astype(np.float64)
            if pre_rope:
                Kf = O.rope(Kf, np.arange(Kf.shape[0]))
            Vf = np.concatenate([V[b, h], tv[b, h]]).astype(np.float64)
            ref = O.attention(q[b, j][None], Kf, Vf)[0]
            assert np.allclose(got[b, j], ref, rtol=1e-12, atol=1e-12)


def test_varn_cache_decode_matches_dequantised_attention():
    """KVarN decode works in the Hadamard domain (q -> Hq, o -> H o); the result equals
    attention over the input-domain reconstruction, because H/sqrt(128) is orthonormal."""
    w = WL.WORKLOADS[3].scaled(batch=1, n_kv_heads=2, n_q_heads=4, ctx=256)
    cache = O.OracleCache.for_workload(w)
    K, V = WL.blocks(w, 0, 2)
    cache.append(K, V)
    q = WL.query(w)
    tk, tv = WL.tail(w, 3)
    got = cache.decode(q, tk, tv)
    for j in range(4):
        h = j // 2
        Kd = np.concatenate([cache.dequant(0, h, 0, "input"), tk[0, h]])
        Vd = np.concatenate([cache.dequant(0, h, 1, "input"), tv[0, h]])
        assert np.allclose(got[0, j], O.attention(q[0, j][None], Kd, Vd)[0], rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_tile_layouts(golden_dir, bits):
    """Row layout: keys and values alike are token rows of the bit listing (13 words per 3-bit row).
    Tensor-core layout: 3-bit tiles are the 48-byte-per-vector planes, 2/4-bit value tiles are
    channel rows (the transpose), 2/4-bit key tiles are unchanged token rows."""
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, size=(128, 128)).astype(np.uint8)
    for kind in (O.KIND_K, O.KIND_V):
        rows = O.pack_tile(codes, bits, kind, O.LAYOUT_ROWS)
        assert rows.shape == (128, -(-128 // (32 // bits)))
        assert np.array_equal(rows, O.pack_rows(codes, bits))
        assert np.array_equal(O.unpack_tile(rows, bits, kind, O.LAYOUT_ROWS), codes)
        mma = O.pack_tile(codes, bits, kind, O.LAYOUT_MMA)
        assert np.array_equal(O.unpack_tile(mma, bits, kind, O.LAYOUT_MMA), codes)
        if bits == 3:
            assert rows.size * 4 == 128 * 52 and mma.size * 4 == 128 * 48
            assert np.array_equal(mma, O.pack_tile3(codes, kind))
        elif kind == O.KIND_V:
            # channel row c holds the codes of tokens 0..127 of channel c
            n = 32 // bits
            c, t = 37, 2 * n + 3
            assert (int(mma[c, t // n]) >> (bits * (t % n))) & (2 ** bits - 1) == codes[t, c]
        else:
            assert np.array_equal(mma, rows)


# ------------------------------------------------------------------ calibrated keys, attention sink

def test_calibrate_keys_brute_force():
    """tau_c is the ceil((1-f)M)-th smallest |K[t, c]| over tokens 1..N-1 (token 0, the sink,
    excluded); zp_c, s_c are the centre and half-range of the entries at or below tau_c."""
    rng = np.random.default_rng(21)
    N, f = 301, 0.02
    K = rng.standard_normal((N, 128)).astype(np.float16).astype(np.float32)
    tau, s16, zp16 = O.calibrate_keys(K, f)
    M = N - 1
    r = math.ceil((1 - float(np.float32(f))) * M)   # the fraction as the fp32 value a config holds
    for c in (0, 37, 127):
        col = [abs(float(K[t, c])) for t in range(1, N)]
        assert tau[c] == sorted(col)[r - 1]
        keep = [float(K[t, c]) for t in range(1, N) if abs(float(K[t, c])) <= tau[c]]
        assert len(keep) >= r
        assert float(zp16[c]) == float(np.float16((np.float32(max(keep)) + np.float32(min(keep))) / 2))
        assert float(s16[c]) == float(np.float16((np.float32(max(keep)) - np.float32(min(keep))) / 2))
    K2 = K.copy()
    K2[0] = 1000.0                                   # the first token does not enter
    for a, b in zip(O.calibrate_keys(K2, f), (tau, s16, zp16)):
        assert np.array_equal(a, b)
    t0, s0, z0 = O.calibrate_keys(K, 0.0)            # no outliers: the full range of tokens 1..
    assert np.all(np.isinf(t0))
    assert np.array_equal(s0, ((K[1:].max(0) - K[1:].min(0)) / 2).astype(np.float16))


def test_calibrated_quantizer_threshold_cap_and_grid():
    rng = np.random.default_rng(22)
    cb = np.array([-1, -0.75, -0.5, -0.25, 0.25, 0.5, 0.75, 1.0], np.float32)
    q = rng.integers(0, 8, size=(128, 128))
    x = (cb[q] * 0.5 + 0.25).astype(np.float32)     # on the grid of s = 0.5, zp = 0.25
    tau = np.full(128, 2.0, np.float32)
    s16, zp16 = np.full(128, 0.5, np.float16), np.full(128, 0.25, np.float16)
    planted = [(3, 4, 9.5), (3, 90, -7.25), (77, 4, 5.0)]
    for t, c, v in planted:
        x[t, c] = v
    r = O.nuq_quantize_calibrated(x, cb, tau, s16, zp16, n_out=10)
    dense, sparse = O.threshold_split(x, tau)       # the pages' threshold form
    assert np.array_equal(r["mask"], sparse != 0)
    assert int(r["row_ptr"][-1]) == len(planted)
    xh = O.nuq_dequant(r["codes"], r["s16"], r["zp16"], cb, 0, r["row_ptr"], r["col"], r["val"])
    for t, c, v in planted:                          # dense zero (code of -0.25 on this grid) + v
        assert xh[t, c] == pytest.approx(v + 0.0)
        xh[t, c] = x[t, c]
    assert np.array_equal(xh, x.astype(np.float64))
    capped = O.nuq_quantize_calibrated(x, cb, tau, s16, zp16, n_out=2)
    assert capped["mask"].sum() == 2 and capped["mask"][3, 4] and capped["mask"][3, 90]


@pytest.mark.parametrize("calibrated", [False, True])
def test_sink_decode_equals_plain_attention_on_lossless_inputs(calibrated):
    """With the first token kept in the input precision, decode over lossless nuq inputs equals
    plain fp64 attention over the raw K/V, the first token included at position 0 (with and
    without calibrated key statistics: calibrating on such inputs recovers their grid)."""
    rng = np.random.default_rng(23)
    B, H, nb = 1, 2, 2
    cb = np.array([-1, -0.75, -0.5, -0.25, 0.25, 0.5, 0.75, 1.0], np.float32)
    ch = (2.0 ** (np.arange(128) % 3 - 2))[None, :]
    K = np.empty((B, H, nb * 128, 128), np.float32)
    V = np.empty_like(K)
    for h in range(H):
        qk = rng.integers(0, 8, (nb * 128, 128))
        qk[1::128], qk[2::128] = 0, 7                # every block's extremes off the sink row
        K[0, h] = cb[qk] * ch + 0.25 * ch
        qv = rng.integers(0, 8, (nb * 128, 128))
        qv[:, 0], qv[:, 1] = 0, 7
        V[0, h] = cb[qv] * 0.5 - 0.125
        K[0, h, 0] = rng.standard_normal(128) * 3    # the sink token: off every grid
        V[0, h, 0] = rng.standard_normal(128) * 3
    calib = None
    if calibrated:
        parts = [O.calibrate_keys(K[0, h], 0.0) for h in range(H)]
        calib = tuple(np.stack([p[i] for p in parts]) for i in range(3))
    cache = O.OracleCache("nuq", 3, B, H, H, pre_rope=True, outlier_frac=0.0, codebook=cb, key_calib=calib,
                          sink=True)
    cache.append(K, V)
    qv_ = rng.standard_normal((B, H, 128))
    tk, tv = rng.standard_normal((B, H, 3, 128)), rng.standard_normal((B, H, 3, 128))
    got = cache.decode(qv_, tk, tv)
    for h in range(H):
        Kf = O.rope(np.concatenate([K[0, h], tk[0, h]]).astype(np.float64), np.arange(nb * 128 + 3))
        Vf = np.concatenate([V[0, h], tv[0, h]]).astype(np.float64)
        ref = O.attention(qv_[0, h][None], Kf, Vf)[0]
        assert np.allclose(got[0, h], ref, rtol=1e-12, atol=1e-12)
