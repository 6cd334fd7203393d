"""CPU oracle for low-bit KV-cache quantization and decode attention over the packed cache.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` use it. It shares no code with the CUDA library and imports nothing
from it.

What it restates (the sources are three web pages; cited by page and section):

* [KVQ]  "KVQuant: Towards 10 Million Context Length LLM Inference with KV Cache
         Quantization" - reading notes (zhongzhuzhou.org, 2026-06-03).
* [KVN]  "KVarN: Variance-Normalized KV-Cache Quantization Mitigates Error
         Accumulation in Reasoning Tasks" - paper summary (paper.rainbus.top).
* [TQ]   TurboQuant KV-cache reproduction blog (pwwt.cn).

Precision. Every quantizer step that decides an integer code or a stored fp16
value is written as a sequence of IEEE fp32 operations in a fixed order
(numpy float32 ufuncs: one correctly rounded operation each, no fused
multiply-add), so the codes and the stored bytes are reproducible bit for bit.
The Hadamard transform and the Sinkhorn-style variance normalisation run in
fp64 (their codes are checked with a +-1 exemption at rounding boundaries).
Dequantisation, RoPE and attention run in fp64.

Readings taken where the pages are silent or disagree (each names the page
passage it settles):

* rounding is round-half-to-even; fp16 conversion is round-to-nearest-even.
* uniform RTN stores the zero point in units of the scale, x_dq = (q + z) * s
  ([KVN] preliminaries, KIVI form); [KVQ] §1.2 writes x_dq = q*s + z', the same
  with z' = z*s.
* keys: per-channel statistics over the 128 tokens of a block; values:
  per-token statistics over the 128 channels ([KVQ] §3.1, §3.6; [KVN] prelim).
* nuq keys/values are normalised to [-1, 1] by (x - zp)/s with zp = (max+min)/2,
  s = (max-min)/2 over the non-outlier entries ([KVQ] Algorithm 2 input,
  Algorithm 1 step 4, worked example step 2); the codebook is the 8 N(0,1)
  quantiles scaled to span [-1, 1]; outliers are the ceil(frac*16384)
  largest-|x| entries of a 128x128 tile (a per-tile fixed count stands in for
  the offline per-channel 99% threshold, which needs calibration data).
* int4 absmax blocks are one token's 128 channels, symmetric, two's complement
  nibbles ([TQ] §2.1 and §4.2 code); the variants take 8 bits ([TQ] §5.1's
  sensitive layers) and/or blocks of 64 channels ([TQ] §2.1), two per token.
* KVarN: x <- H x / sqrt(128) per token (Sylvester order); VarN alternates
  column then row population-std normalisation for 8 iterations with the
  scales accumulated in the log domain; for keys the channel scales merge into
  the per-channel RTN scale and s1 is the per-token scale, for values the token
  scales merge into the per-token RTN scale and s1 is the per-channel scale
  ([KVN] method steps 1-5).
"""
from __future__ import annotations

import math
from statistics import NormalDist

import numpy as np

T = 128            # tokens per block
D = 128            # head dim
TILE = T * D       # elements per tile

KIND_K, KIND_V = 0, 1


# =========================================================================== sizes

def kv_cache_bytes(n_layers: int, n_heads: int, head_dim: int, elem_bytes: int,
                   batch: int, seq_len: int) -> int:
    """Dense KV-cache size 2*n*h*d*e*b*l bytes: the factor 2 is K and V
    ([KVQ] §1.1 formula; [TQ] §1.1 formula and table)."""
    return 2 * n_layers * n_heads * head_dim * elem_bytes * batch * seq_len


# =========================================================================== helpers

def _f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32)


def _half(x) -> np.ndarray:
    """Round to fp16, nearest-even (from fp32 or fp64 directly)."""
    return np.asarray(x).astype(np.float16)


def _f32_of_half(h) -> np.ndarray:
    return np.asarray(h, dtype=np.float16).astype(np.float32)


# =========================================================================== packing

def codes_per_word(bits: int) -> int:
    """floor(32/b) codes per 32-bit word ([KVQ] §9.3: ten 3-bit codes per word)."""
    return 32 // bits


def words_per_row(bits: int) -> int:
    return -(-D // codes_per_word(bits))


def pack_rows(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack each row of 128 b-bit codes into 32-bit words.

    Code i of a row goes to bits [b*(i%n)+b-1 : b*(i%n)] of word i//n, n = floor(32/b);
    the bits above b*n in a word stay zero ([KVQ] §9.3 memory layout: codes 0..9 of a
    3-bit row at bits [2:0], [5:3], ..., [29:27], bits [31:30] unused).
    """
    codes = np.asarray(codes)
    n = codes_per_word(bits)
    W = words_per_row(bits)
    out = np.zeros(codes.shape[:-1] + (W,), dtype=np.uint64)
    mask = (1 << bits) - 1
    for i in range(D):
        out[..., i // n] |= (codes[..., i].astype(np.uint64) & mask) << np.uint64(bits * (i % n))
    return out.astype(np.uint32)


def unpack_rows(words: np.ndarray, bits: int) -> np.ndarray:
    """Inverse of pack_rows: uint32 [..., W] -> uint8 codes [..., 128]."""
    words = np.asarray(words, dtype=np.uint32)
    n = codes_per_word(bits)
    out = np.empty(words.shape[:-1] + (D,), dtype=np.uint8)
    mask = np.uint32((1 << bits) - 1)
    for i in range(D):
        out[..., i] = (words[..., i // n] >> np.uint32(bits * (i % n))) & mask
    return out


# Two packed layouts of a tile.
#
# LAYOUT_ROWS (the default): one row per token, for keys and values alike, each row its 128 codes
# in floor(32/b)-code words as `pack_rows` above ([KVQ] §9.3 bit layout; a 3-bit row is 13 words
# = 52 bytes).
#
# LAYOUT_MMA (the tensor-core decode's format): 2- and 4-bit value tiles hold one row per channel
# (its codes for the 128 tokens); 3-bit tiles take [KVQ] §9.3's other figure, 128 x 3 bits = 48
# bytes per vector, which ten codes per word cannot reach: 128 x 128 codes in 1536 words, every
# code's two low bits and its high bit in separate bit planes. The plane order follows the decode's
# matrix fragments: the tile is cut into 8 segments of 16 tokens, each segment into 32 groups of
# 64 codes (6 words each), and within a group the codes sit in 8 four-bit slots of 8 "nibble
# words" u (the low bits of nibble word u in word u//2 at bit 4k + 2(u%2), its high bit in word
# 4 + u//4 at bit 4k + (2, 3, 0, 1)[u%4], k = 0..7 the slot).
LAYOUT_ROWS, LAYOUT_MMA = 0, 1
TILE3_WORDS = 1536


def tile3_slot(kind: int, t, c):
    """Where code (token t, channel c) of a 3-bit tile lives: (low-bits word, its shift,
    high-bit word, its shift). Keys: group 4*(t%8) + (c//2)%4 of segment t//16, nibble word
    c//16, slot 4*((c//8)%2) + 2*((t%16)//8) + c%2. Values: group 4*(c%8) + t%4 of segment
    t//16, nibble word c//16, slot 4*((t%16)//4 % 2) + 2*((c//8)%2) + (t%16)//8."""
    t = np.asarray(t, np.int64)
    c = np.asarray(c, np.int64)
    s, tl = t >> 4, t & 15
    if kind == KIND_K:
        g, r = tl & 7, tl >> 3
        tq, kg, j = (c >> 1) & 3, c >> 3, c & 1
        u, k = kg >> 1, 4 * (kg & 1) + 2 * r + j
    else:
        tq, v = tl & 3, tl >> 2
        g, r, mt = c & 7, (c >> 3) & 1, c >> 4
        u, k = mt, 4 * (v & 1) + 2 * r + (v >> 1)
    base = s * 192 + (4 * g + tq) * 6
    hi_pos = np.array([2, 3, 0, 1])[u & 3]
    return base + (u >> 1), 4 * k + 2 * (u & 1), base + 4 + (u >> 2), 4 * k + hi_pos


def pack_tile3(codes: np.ndarray, kind: int) -> np.ndarray:
    """3-bit codes [128 tokens][128 channels] -> uint32[1536] in the tile3 plane layout."""
    codes = np.asarray(codes, np.uint64)
    t, c = np.meshgrid(np.arange(T), np.arange(D), indexing="ij")
    lw, ls, hw, hs = tile3_slot(kind, t.ravel(), c.ravel())
    q = codes.ravel()
    out = np.zeros(TILE3_WORDS, np.uint64)
    np.bitwise_or.at(out, lw, (q & np.uint64(3)) << ls.astype(np.uint64))
    np.bitwise_or.at(out, hw, ((q >> np.uint64(2)) & np.uint64(1)) << hs.astype(np.uint64))
    return out.astype(np.uint32)


def unpack_tile3(words: np.ndarray, kind: int) -> np.ndarray:
    """Inverse of pack_tile3: uint32[1536] -> uint8 codes [128 tokens][128 channels]."""
    w = np.asarray(words, np.uint64)
    t, c = np.meshgrid(np.arange(T), np.arange(D), indexing="ij")
    lw, ls, hw, hs = tile3_slot(kind, t.ravel(), c.ravel())
    lo = (w[lw] >> ls.astype(np.uint64)) & np.uint64(3)
    hi = (w[hw] >> hs.astype(np.uint64)) & np.uint64(1)
    return (lo | (hi << np.uint64(2))).astype(np.uint8).reshape(T, D)


def pack_tile(codes: np.ndarray, bits: int, kind: int, layout: int = LAYOUT_ROWS) -> np.ndarray:
    """Code words of one tile (codes [token][channel]) in `layout` (see above)."""
    if layout == LAYOUT_ROWS:
        return pack_rows(codes, bits)
    if bits == 3:
        return pack_tile3(codes, kind)
    return pack_rows(codes if kind == KIND_K else np.asarray(codes).T, bits)


def unpack_tile(words: np.ndarray, bits: int, kind: int, layout: int = LAYOUT_ROWS) -> np.ndarray:
    """Inverse of pack_tile: codes [token][channel]."""
    if layout == LAYOUT_ROWS:
        return unpack_rows(words, bits)
    if bits == 3:
        return unpack_tile3(words, kind)
    codes = unpack_rows(words, bits)
    return codes if kind == KIND_K else codes.T


# =========================================================================== uniform RTN

def rtn_meta(mx, mn, bits: int):
    """Scale and zero point of b-bit asymmetric RTN over one group.

    s = (max - min)/(2^b - 1) ([KVQ] §3.1 per-token and per-channel scale formulas),
    computed as one fp32 subtraction then one fp32 division, rounded to fp16; a zero
    scale becomes 1. The zero point is stored in units of s, z = min/s, so that
    x_dq = (q + z)*s ([KVN] preliminaries, KIVI representation).
    """
    s32 = (_f32(mx) - _f32(mn)) / np.float32(2 ** bits - 1)
    s16 = _half(s32)
    s16 = np.where(s16 == 0, np.float16(1.0), s16)
    with np.errstate(over="ignore"):
        z16 = _half(_f32(mn) / _f32_of_half(s16))
    return s16, z16


def rtn_encode(x, s16, z16, bits: int) -> np.ndarray:
    """q = clamp(rne(x/s - z), 0, 2^b-1): fp32 division, then fp32 subtraction, then
    round-half-even ([KVQ] §1.2, Q(x) = round((x - z)/s) in the (q+z)*s form)."""
    with np.errstate(invalid="ignore", over="ignore"):
        t = _f32(x) / _f32_of_half(s16) - _f32_of_half(z16)
        return np.clip(np.rint(t), 0, 2 ** bits - 1).astype(np.uint8)


def rtn_quantize(x: np.ndarray, bits: int, axis: int):
    """RTN of one 128x128 tile x[token][channel] (float32 values).

    axis=0: one (s, z) per channel over the 128 tokens (keys, per-channel);
    axis=1: one (s, z) per token over the 128 channels (values, per-token).
    Returns (codes uint8 [128][128], s16 [128], z16 [128]).
    """
    x = _f32(x)
    s16, z16 = rtn_meta(x.max(axis=axis), x.min(axis=axis), bits)
    if axis == 0:
        codes = rtn_encode(x, s16[None, :], z16[None, :], bits)
    else:
        codes = rtn_encode(x, s16[:, None], z16[:, None], bits)
    return codes, s16, z16


def rtn_dequant(codes, s16, z16, axis: int) -> np.ndarray:
    """x_dq = (q + z) * s in fp64 ([KVN] preliminaries)."""
    q = np.asarray(codes, np.float64)
    s = np.asarray(s16, np.float64)
    z = np.asarray(z16, np.float64)
    if axis == 0:
        return (q + z[None, :]) * s[None, :]
    return (q + z[:, None]) * s[:, None]


# =========================================================================== int4 / int8 absmax

def absmax_quantize(x: np.ndarray, bits: int = 4, group: int = 128):
    """Symmetric absmax integer blocks of `group` contiguous channels of one token: 128 (one
    scale per token's head vector, the reading of [TQ] §4.1 "a scale every 128 elements") or 64
    (two per token, [TQ] §2.1's smaller block), b = 4 bits or 8 (the "sensitive layer" precision
    of [TQ] §5.1).

    scale = absmax/(2^(b-1) - 1) (fp32 division), stored fp16 (saturating at the fp16 maximum);
    q = clamp(rne(x/scale), -2^(b-1), 2^(b-1) - 1) with fp32 division; a zero scale gives q = 0
    ([TQ] §2.1 block quantization and §4.2 quantize_kv_block, there with b = 4).
    Returns (q int16 [128][128], s16 [128/group][128]: s16[g][t] scales channels g*group ..
    g*group + group - 1 of token t).
    """
    assert bits in (4, 8) and group in (64, 128)
    x = _f32(x)
    qmax = 2 ** (bits - 1) - 1
    ng = D // group
    xg = x.reshape(T, ng, group)
    a = np.abs(xg).max(axis=2)                                       # [t][g]
    s16 = _half(np.minimum(a / np.float32(qmax), np.float32(65504.0)))
    sf = _f32_of_half(s16)
    with np.errstate(invalid="ignore", divide="ignore"):
        t = xg / sf[:, :, None]
        q = np.clip(np.rint(t), -qmax - 1, qmax)
    q[sf == 0] = 0
    return q.reshape(T, D).astype(np.int16), np.ascontiguousarray(s16.T)


def int4_quantize(x: np.ndarray):
    """absmax_quantize with b = 4 and one scale per token: (q int8 [128][128], s16 [128])."""
    q, s16 = absmax_quantize(x, 4, 128)
    return q.astype(np.int8), s16[0]


def absmax_codes(q: np.ndarray, bits: int = 4) -> np.ndarray:
    """Two's complement b-bit code q & (2^b - 1) ([TQ] §4.2, `q.to(int8) & 0xF` for b = 4)."""
    return (np.asarray(q, np.int16) & ((1 << bits) - 1)).astype(np.uint8)


def absmax_from_codes(codes: np.ndarray, bits: int = 4) -> np.ndarray:
    n = np.asarray(codes, np.int16)
    return np.where(n >= 2 ** (bits - 1), n - 2 ** bits, n).astype(np.int16)


def int4_nibbles(q: np.ndarray) -> np.ndarray:
    return absmax_codes(q, 4)


def int4_from_nibbles(nib: np.ndarray) -> np.ndarray:
    return absmax_from_codes(nib, 4).astype(np.int8)


def absmax_dequant(q, s16) -> np.ndarray:
    """x_dq = q * scale of the element's group (zero point 0), fp64. s16: [128] (one group per
    token) or [n_groups][128]."""
    s = np.asarray(s16, np.float64)
    if s.ndim == 1:
        s = s[None, :]
    group = D // s.shape[0]
    return np.asarray(q, np.float64) * np.repeat(s.T, group, axis=1)


def int4_dequant(q, s16) -> np.ndarray:
    """x_dq = q * scale (zero point 0), fp64."""
    return absmax_dequant(q, s16)


# =========================================================================== nuq (KVQuant)

def nuq_codebook(bits: int = 3) -> np.ndarray:
    """2^b-entry codebook: the N(0,1) quantiles at (j+1/2)/2^b, divided by the largest so
    that the table spans [-1, 1] like the worked example's C[15] ([KVQ] appendix step 3).
    Computed in fp64, stored fp32."""
    n = 2 ** bits
    inv = NormalDist().inv_cdf
    top = inv((n - 0.5) / n)
    return np.array([inv((j + 0.5) / n) / top for j in range(n)], np.float64).astype(np.float32)


FIT_SCALE = 2.0 ** 32   # fixed-point resolution of the weighted sums of fit_codebook


def fit_codebook(a: np.ndarray, w: np.ndarray, bits: int, max_iter: int = 50):
    """Sensitivity-weighted nuq codebook ([KVQ] §3.3, Algorithm 2): Lloyd iterations on the
    normalised samples a (clamped to [-1, 1]) with weights w (Fisher information, clamped to
    [0, 1]). Start from k = 2^b centres spaced evenly over [-1, 1] (reading: c_j = -1 + 2j/(k-1)).
    Each iteration assigns every sample to its nearest centre (|a - c_j| in fp32, the lowest j
    on ties), stops if no assignment changed, else moves each centre to the weighted mean of its
    members (a centre without members stays). The weighted sums are exact: w*a and w (products
    exact in fp64) are scaled by 2^32, rounded half-even to 64-bit integers and added as
    integers; each centre is the fp64 quotient of the two sums rounded to fp32.
    Returns (codebook fp32 [k], iterations run)."""
    a = np.clip(np.asarray(a, np.float32), np.float32(-1.0), np.float32(1.0))
    w = np.clip(np.asarray(w, np.float32), np.float32(0.0), np.float32(1.0))
    k = 2 ** bits
    c = np.array([-1.0 + 2.0 * j / (k - 1) for j in range(k)], np.float64).astype(np.float32)
    P = np.rint(w.astype(np.float64) * a.astype(np.float64) * FIT_SCALE).astype(np.int64)
    W = np.rint(w.astype(np.float64) * FIT_SCALE).astype(np.int64)
    prev = None
    it = 0
    for it in range(1, max_iter + 1):
        d = np.abs(a[:, None] - c[None, :])             # fp32 subtraction, then |.|
        assign = np.argmin(d, axis=1)                    # first index on ties
        if prev is not None and np.array_equal(assign, prev):
            break
        for j in range(k):
            m = assign == j
            if m.any():
                sw = int(W[m].sum())
                if sw > 0:
                    c[j] = np.float32(np.float64(int(P[m].sum())) / np.float64(sw))
        prev = assign
    return c, it


def n_outliers(frac: float) -> int:
    """Outliers per 128x128 tile: ceil(frac * 16384), frac taken as an fp32 value."""
    return int(math.ceil(float(np.float32(frac)) * TILE))


def threshold_split(k: np.ndarray, tau: np.ndarray):
    """The pages' per-channel threshold form of the dense-and-sparse split: entries with
    |k[c]| > tau[c] move to the sparse part and are zeroed in the dense part
    ([KVQ] §3.4 formula, worked example step 1). Returns (dense, sparse)."""
    k = np.asarray(k, np.float64)
    m = np.abs(k) > np.asarray(tau, np.float64)
    return np.where(m, 0.0, k), np.where(m, k, 0.0)


def outlier_mask(x: np.ndarray, n_out: int) -> np.ndarray:
    """The n_out largest-|x| entries of a tile ([KVQ] §3.4 dense-and-sparse split,
    about 1% of entries kept in fp16). Order: fp16 magnitude descending, then the
    lower flat index t*128 + c first."""
    mag = (np.asarray(x, np.float32).astype(np.float16).view(np.uint16) & 0x7FFF).ravel()
    idx = np.arange(mag.size)
    order = np.lexsort((idx, -mag.astype(np.int64)))
    mask = np.zeros(mag.size, dtype=bool)
    mask[order[:n_out]] = True
    return mask.reshape(np.shape(x))


def csr_of(x: np.ndarray, mask: np.ndarray):
    """CSR with rows = tokens (new tokens append as new rows, [KVQ] §3.4 storage):
    row_ptr uint16[129], col uint8[nnz] (channel), val fp16 bits uint16[nnz]."""
    counts = mask.sum(axis=1)
    row_ptr = np.zeros(T + 1, np.int64)
    row_ptr[1:] = np.cumsum(counts)
    tt, cc = np.nonzero(mask)            # row-major order: sorted by (t, c)
    val = np.asarray(x, np.float32)[tt, cc].astype(np.float16).view(np.uint16)
    return row_ptr.astype(np.uint16), cc.astype(np.uint8), val


def csc_of(x: np.ndarray, mask: np.ndarray):
    """CSC with columns = channels, the value storage of [KVQ] §3.4 ("by column"):
    col_ptr uint16[129], row uint8[nnz] (token), val fp16 bits uint16[nnz], entries sorted by
    (channel, token)."""
    counts = mask.sum(axis=0)
    col_ptr = np.zeros(D + 1, np.int64)
    col_ptr[1:] = np.cumsum(counts)
    cc, tt = np.nonzero(np.asarray(mask).T)  # column-major order: sorted by (c, t)
    val = np.asarray(x, np.float32)[tt, cc].astype(np.float16).view(np.uint16)
    return col_ptr.astype(np.uint16), tt.astype(np.uint8), val


def to_csc(rec: dict, x: np.ndarray) -> dict:
    """The same quantised tile with its outliers stored by column (the outlier set, codes and
    metadata unchanged): keys col_ptr, row, val replace row_ptr, col, val."""
    out = {k: v for k, v in rec.items() if k not in ("row_ptr", "col", "val")}
    out["col_ptr"], out["row"], out["val"] = csc_of(x, rec["mask"])
    return out


def nuq_meta(x: np.ndarray, mask: np.ndarray, axis: int):
    """Centre zp and half-range s of the non-outlier entries of each group
    ([KVQ] Algorithm 1 offline step 4: normalise to [-1,1] excluding outliers):
    zp = (max+min)/2, s = (max-min)/2 in fp32, stored fp16. An empty group gets
    zp = s = 0."""
    x = _f32(x)
    inf = np.float32(np.inf)
    mx = np.where(mask, -inf, x).max(axis=axis)
    mn = np.where(mask, inf, x).min(axis=axis)
    empty = np.isinf(mx)
    with np.errstate(invalid="ignore"):
        zp32 = (mx + mn) / np.float32(2.0)
        h32 = (mx - mn) / np.float32(2.0)
    zp16 = _half(np.where(empty, np.float32(0), zp32))
    s16 = _half(np.where(empty, np.float32(0), h32))
    return s16, zp16


def nuq_normalise(x, s16, zp16) -> np.ndarray:
    """t = clamp((x - zp)/s, -1, 1) with an fp32 subtraction then an fp32 division
    ([KVQ] Algorithm 1 step 2; worked example: 1.45 clamps to 1.0). A zero scale gives t = 0."""
    sf = _f32_of_half(s16)
    with np.errstate(invalid="ignore", divide="ignore"):
        t = (_f32(x) - _f32_of_half(zp16)) / sf
        t = np.clip(t, np.float32(-1.0), np.float32(1.0))
    return np.where(sf == 0, np.float32(0.0), t).astype(np.float32)


def nuq_encode(t: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """q = argmin_j |t - C_j| with fp32 |t - C_j|; the lowest index wins ties
    ([KVQ] §1.2 NUQ definition, Algorithm 1 step 3)."""
    d = np.abs(_f32(t)[..., None] - _f32(codebook))
    return np.argmin(d, axis=-1).astype(np.uint8)


def nuq_quantize(x: np.ndarray, codebook: np.ndarray, axis: int, n_out: int):
    """Dense-and-sparse nuq of one tile (Algorithm 1 inference steps 1-4).

    1. the n_out largest-|x| entries go to CSR in fp16 and are zeroed in the dense part;
    2. each group (axis 0: per channel, keys; axis 1: per token, values) is normalised
       with the centre/half-range of its non-outlier entries;
    3. each dense entry (zeros at outlier positions included) takes the nearest codebook
       index.
    Returns dict(codes, s16, zp16, mask, row_ptr, col, val).
    """
    x = _f32(x)
    mask = outlier_mask(x, n_out)
    dense = np.where(mask, np.float32(0.0), x)
    s16, zp16 = nuq_meta(x, mask, axis)
    if axis == 0:
        t = nuq_normalise(dense, s16[None, :], zp16[None, :])
    else:
        t = nuq_normalise(dense, s16[:, None], zp16[:, None])
    codes = nuq_encode(t, codebook)
    row_ptr, col, val = csr_of(x, mask)
    return dict(codes=codes, s16=s16, zp16=zp16, mask=mask, row_ptr=row_ptr, col=col, val=val)


def calibrate_keys(K: np.ndarray, outlier_frac: float):
    """Offline per-channel key statistics of one head ([KVQ] Algorithm 1 offline steps 3-4 and
    §3.5): K [N][128] calibration keys (values representable in the input dtype), token 0 (the
    attention sink) excluded. Per channel c over the M = N - 1 remaining tokens:
      tau_c = the ceil((1 - f) M)-th smallest |K[t, c]|   (f = 0: no threshold, tau = inf),
      zp_c, s_c = centre and half-range of the entries with |K[t, c]| <= tau_c (fp32, stored fp16).
    Entries above tau_c are the channel's outliers. Returns (tau fp32[128], s16, zp16)."""
    x = _f32(K)[1:]
    M = x.shape[0]
    a = np.sort(np.abs(x), axis=0)
    f = float(np.float32(outlier_frac))
    if f > 0.0:
        r = max(1, int(math.ceil((1.0 - f) * M)))
        tau = a[r - 1].astype(np.float32)
    else:
        tau = np.full(D, np.inf, np.float32)
    mask = np.abs(x) > tau[None, :]
    s16, zp16 = nuq_meta(x, mask, 0)
    return tau, s16, zp16


def nuq_quantize_calibrated(x: np.ndarray, codebook: np.ndarray, tau, s16, zp16, n_out: int):
    """Key tile quantised with calibrated statistics ([KVQ] Algorithm 1 inference steps 1-4):
    1. entries with |x[t, c]| > tau_c are outliers, at most n_out of them per tile (the largest,
       in the order of `outlier_mask`); they go to CSR in fp16 and are zeroed in the dense part;
    2. the dense part is normalised with the calibrated zp_c, s_c;
    3. each dense entry takes the nearest codebook index.
    Returns dict(codes, s16, zp16, mask, row_ptr, col, val)."""
    x = _f32(x)
    over = np.abs(x) > np.asarray(tau, np.float32)[None, :]
    mask = outlier_mask(x, n_out) & over
    dense = np.where(mask, np.float32(0.0), x)
    s16 = np.asarray(s16, np.float16)
    zp16 = np.asarray(zp16, np.float16)
    codes = nuq_encode(nuq_normalise(dense, s16[None, :], zp16[None, :]), codebook)
    row_ptr, col, val = csr_of(x, mask)
    return dict(codes=codes, s16=s16.copy(), zp16=zp16.copy(), mask=mask, row_ptr=row_ptr, col=col, val=val)


def nuq_dequant(codes, s16, zp16, codebook, axis: int, row_ptr=None, col=None, val=None, col_ptr=None, row=None):
    """x_dq = C[q]*s + zp, then the fp16 outliers are added back
    ([KVQ] Algorithm 1 dequantisation: K_hat[mask] += outlier_vals), from CSR (row_ptr, col,
    val) or from CSC (col_ptr, row, val)."""
    c = np.asarray(codebook, np.float64)[np.asarray(codes, np.intp)]
    s = np.asarray(s16, np.float64)
    zp = np.asarray(zp16, np.float64)
    x = c * s[None, :] + zp[None, :] if axis == 0 else c * s[:, None] + zp[:, None]
    if row_ptr is not None:
        vals = np.asarray(val, np.uint16).view(np.float16).astype(np.float64)
        for t in range(T):
            for j in range(int(row_ptr[t]), int(row_ptr[t + 1])):
                x[t, int(col[j])] += vals[j]
    if col_ptr is not None:
        vals = np.asarray(val, np.uint16).view(np.float16).astype(np.float64)
        for c in range(D):
            for j in range(int(col_ptr[c]), int(col_ptr[c + 1])):
                x[int(row[j]), c] += vals[j]
    return x


# =========================================================================== RoPE

def rope_angles(positions, theta: float = 10000.0, d: int = D) -> np.ndarray:
    """n * theta_i with theta_i = theta^(-2i/d), i = 0..d/2-1 ([KVQ] §1.3), fp64."""
    i = np.arange(d // 2, dtype=np.float64)
    th = np.float64(theta) ** (-2.0 * i / d)
    return np.asarray(positions, np.float64)[:, None] * th[None, :]


def rope(x: np.ndarray, positions, theta: float = 10000.0) -> np.ndarray:
    """Rotate each channel pair (2i, 2i+1) of row n by angle n*theta_i:
    [x0', x1'] = [[cos, -sin], [sin, cos]] [x0, x1] ([KVQ] §1.3 rotation matrix)."""
    x = np.asarray(x, np.float64)
    ang = rope_angles(positions, theta, x.shape[-1])
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = c * x0 - s * x1
    out[..., 1::2] = s * x0 + c * x1
    return out


# =========================================================================== KVarN

def hadamard(n: int = D) -> np.ndarray:
    """Sylvester Hadamard matrix: H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]]."""
    H = np.ones((1, 1))
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def fwht(x: np.ndarray) -> np.ndarray:
    """x <- H x / sqrt(128) on the channel dimension of every token row ([KVN] method
    step 1, Hadamard rotation on channels). H is symmetric, so the row form is x H."""
    return np.asarray(x, np.float64) @ hadamard(x.shape[-1]) / math.sqrt(x.shape[-1])


def varn(X: np.ndarray, iters: int = 8):
    """Sinkhorn-style two-axis variance normalisation ([KVN] method step 2): repeat
    {divide every column by its population std, then every row by its std}, keeping the
    accumulated log-std per column (lc) and per row (lr). Returns (Y, r, c) with
    X = diag(r) Y diag(c), r = exp(lr), c = exp(lc). fp64."""
    Y = np.array(X, dtype=np.float64)
    lr = np.zeros(Y.shape[0])
    lc = np.zeros(Y.shape[1])
    for _ in range(iters):
        sc = Y.std(axis=0)
        ok = sc > 0
        Y[:, ok] /= sc[ok]
        lc[ok] += np.log(sc[ok])
        sr = Y.std(axis=1)
        ok = sr > 0
        Y[ok, :] /= sr[ok, None]
        lr[ok] += np.log(sr[ok])
    return Y, np.exp(lr), np.exp(lc)


def varn_quantize(x: np.ndarray, bits: int, kind: int, iters: int = 8, use_hadamard: bool = True):
    """KVarN encode of one tile ([KVN] method steps 1-4).

    X = FWHT(x); (Y, r, c) = VarN(X). Keys (per-channel RTN): Z = Y diag(c), s1 = r
    (one extra scale per token). Values (per-token RTN): Z = diag(r) Y, s1 = c (one
    per channel). Z is rounded to fp32 and RTN-quantised as in rtn_quantize.
    Returns dict(codes, s16, z16, s1 (fp16), r, c (fp64), Z (fp64)).
    """
    X = fwht(x) if use_hadamard else np.asarray(x, np.float64)
    Y, r, c = varn(X, iters)
    if kind == KIND_K:
        Z, s1, axis = Y * c[None, :], r, 0
    else:
        Z, s1, axis = Y * r[:, None], c, 1
    codes, s16, z16 = rtn_quantize(Z.astype(np.float32), bits, axis)
    return dict(codes=codes, s16=s16, z16=z16, s1=_half(s1), r=r, c=c, Z=Z, axis=axis)


def varn_dequant(codes, s16, z16, s1, kind: int) -> np.ndarray:
    """x_dq = (q + z) * s_RTN * s1 in the Hadamard domain ([KVN] method step 5)."""
    base = rtn_dequant(codes, s16, z16, 0 if kind == KIND_K else 1)
    s1 = np.asarray(s1, np.float64)
    return base * s1[:, None] if kind == KIND_K else base * s1[None, :]


def norm_direction_errors(K: np.ndarray, Kdq: np.ndarray):
    """Per-row split of the squared error into a norm part E_M = (|K| - |K_dq|)^2 and a
    direction part E_D = 2|K||K_dq|(1 - cos theta) ([KVN] key innovation, Figure 1a)."""
    K = np.asarray(K, np.float64)
    Kdq = np.asarray(Kdq, np.float64)
    nk = np.linalg.norm(K, axis=-1)
    nd = np.linalg.norm(Kdq, axis=-1)
    dot = (K * Kdq).sum(axis=-1)
    with np.errstate(invalid="ignore", divide="ignore"):
        cos = np.where(nk * nd > 0, dot / (nk * nd), 1.0)
    return (nk - nd) ** 2, 2.0 * nk * nd * (1.0 - cos)


def token_error_stats(X: np.ndarray, Xdq: np.ndarray) -> np.ndarray:
    """Per row (one token's 128 channels) of an input X and its reconstruction Xdq, fp64:
    (|x|, |x_dq| - |x|, E_T = |x - x_dq|^2, E_D) with E_D the direction part of [KVN]'s split
    |x - x_dq|^2 = (|x| - |x_dq|)^2 + 2|x||x_dq|(1 - cos theta) (key innovation, Figure 1a); the
    norm part is E_M = (|x_dq| - |x|)^2, the square of the second column, and the second column
    itself is the token-norm deviation of Figure 1b. Rows with a zero norm on either side have
    no direction, so E_D = 0 there."""
    X = np.asarray(X, np.float64)
    Xdq = np.asarray(Xdq, np.float64)
    nx = np.sqrt((X * X).sum(axis=-1))
    nq = np.sqrt((Xdq * Xdq).sum(axis=-1))
    et = ((X - Xdq) ** 2).sum(axis=-1)
    both = (nx > 0) & (nq > 0)
    cos = np.where(both, (X * Xdq).sum(axis=-1) / np.where(both, nx * nq, 1.0), 1.0)
    ed = np.where(both, 2.0 * nx * nq * (1.0 - cos), 0.0)
    return np.stack([nx, nq - nx, et, ed], axis=-1)


def topk_error_share(stats: np.ndarray, fracs) -> np.ndarray:
    """For each fraction f: the k = ceil(f * n) rows with the largest E_T (stats column 2; equal
    errors: the lower row first) and, over them, (k, sum E_T, sum E_M, sum E_D) with E_M the
    square of column 1 ([KVN] Figure 1a plots sum E_M / sum E_T against the top-k% of errors).
    The sums run in fp64 over the rows' values as given."""
    stats = np.asarray(stats).reshape(-1, 4)
    n = stats.shape[0]
    et = stats[:, 2].astype(np.float64)
    em = stats[:, 1].astype(np.float64) ** 2
    ed = stats[:, 3].astype(np.float64)
    order = np.lexsort((np.arange(n), -et))  # E_T descending, then row ascending
    out = np.zeros((len(fracs), 4))
    for i, f in enumerate(fracs):
        k = min(n, int(math.ceil(float(f) * n)))
        sel = order[:k]
        out[i] = (k, et[sel].sum(), em[sel].sum(), ed[sel].sum())
    return out


# =========================================================================== attention

def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """softmax(q K^T / sqrt(d)) V for a set of queries q [G][d] over keys/values [n][d],
    fp64 with a max shift ([KVQ] Algorithm 1: attn_score = dot(Q, K_rot)/sqrt(d_h))."""
    q = np.asarray(q, np.float64)
    s = q @ np.asarray(K, np.float64).T / math.sqrt(q.shape[-1])
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    return (p @ np.asarray(V, np.float64)) / p.sum(axis=-1, keepdims=True)


# =========================================================================== cache model

class OracleCache:
    """A packed cache kept as per-tile records plus the decode that reads it.

    One record per (batch b, KV head h, block, kind): the packed code words (pack_tile in the
    cache's layout), the fp16 metadata and, for nuq, the CSR outliers. decode() unpacks and dequantises every
    record in fp64 (RoPE at absolute positions for pre-RoPE keys; the Hadamard domain
    for KVarN, with the query transformed the same way and the output transformed back),
    appends the fp residual tail and evaluates softmax attention. Query head j reads KV
    head j // (H_q / H_kv).

    nuq only: key_calib = (tau [H][128], s16 [H][128], zp16 [H][128]) from calibrate_keys makes
    key tiles use the calibrated statistics (nuq_quantize_calibrated); sink = True keeps the first
    token of every sequence in the input precision ([KVQ] §3.5): its K and V rows of block 0 are
    zero in the quantised tiles, and decode attends the kept rows at position 0 instead of the
    quantised token 0.

    nuq only: v_csc = True stores the value tiles' outliers by column (to_csc).
    """

    def __init__(self, method: str, bits: int, batch: int, n_kv_heads: int, n_q_heads: int,
                 pre_rope: bool = False, rope_theta: float = 10000.0, outlier_frac: float = 0.01,
                 varn_iters: int = 8, use_hadamard: bool = True, codebook=None, layout: int = LAYOUT_ROWS,
                 key_calib=None, sink: bool = False, scale_group: int = 128, v_csc: bool = False):
        assert method in ("rtn", "nuq", "varn", "int4")
        assert scale_group == 128 or method == "int4"
        self.scale_group = scale_group
        assert layout in (LAYOUT_ROWS, LAYOUT_MMA)
        self.method, self.bits, self.layout = method, bits, layout
        self.batch, self.n_kv_heads, self.n_q_heads = batch, n_kv_heads, n_q_heads
        self.pre_rope, self.rope_theta = pre_rope, rope_theta
        self.outlier_frac, self.varn_iters, self.use_hadamard = outlier_frac, varn_iters, use_hadamard
        if method == "nuq":
            cb = nuq_codebook(bits) if codebook is None else np.asarray(codebook, np.float32)
            self.codebook = np.broadcast_to(cb, (n_kv_heads, 2 ** bits)) if cb.ndim == 1 else cb
            self.n_out = n_outliers(outlier_frac)
        assert (key_calib is None and not sink) or method == "nuq"
        self.key_calib, self.sink = key_calib, bool(sink)
        assert not v_csc or method == "nuq"
        self.v_csc = bool(v_csc)
        self.sink_kv = {}  # (b, h) -> (k row, v row) of the first token
        self.recs = {}
        self.n_blocks = 0

    @classmethod
    def for_workload(cls, w, **kw):
        return cls(w.method, w.bits, kw.pop("batch", w.batch), w.n_kv_heads, w.n_q_heads,
                   pre_rope=w.pre_rope, rope_theta=w.rope_theta, outlier_frac=w.outlier_frac,
                   varn_iters=w.varn_iters, scale_group=getattr(w, "scale_group", 128), **kw)

    # ------------------------------------------------------------------ encode
    def quantize_tile(self, x: np.ndarray, kind: int, h: int = 0) -> dict:
        m, b = self.method, self.bits
        if m == "rtn":
            codes, s16, z16 = rtn_quantize(x, b, 0 if kind == KIND_K else 1)
            rec = dict(codes=codes, s16=s16, z16=z16)
        elif m == "int4":
            q, s16 = absmax_quantize(x, b, self.scale_group)
            rec = dict(codes=absmax_codes(q, b), s16=s16[0] if s16.shape[0] == 1 else s16)
        elif m == "nuq" and kind == KIND_K and self.key_calib is not None:
            tau, s16, zp16 = (np.asarray(a)[h] for a in self.key_calib)
            rec = nuq_quantize_calibrated(x, self.codebook[h], tau, s16, zp16, self.n_out)
        elif m == "nuq":
            rec = nuq_quantize(x, self.codebook[h], 0 if kind == KIND_K else 1, self.n_out)
            if kind == KIND_V and self.v_csc:
                rec = to_csc(rec, x)
        else:
            rec = varn_quantize(x, b, kind, self.varn_iters, self.use_hadamard)
        rec["words"] = pack_tile(rec["codes"], b, kind, self.layout)
        return rec

    def append(self, K: np.ndarray, V: np.ndarray, only_heads=None):
        """K, V: float32 [B][H_kv][n*128][128]. only_heads restricts the work to a list of
        (b, h) pairs (the others are left out of the model)."""
        n = K.shape[2] // T
        for blk in range(n):
            for b in range(self.batch):
                for h in range(self.n_kv_heads):
                    if only_heads is not None and (b, h) not in only_heads:
                        continue
                    first = self.sink and self.n_blocks + blk == 0
                    if first:
                        self.sink_kv[(b, h)] = (np.array(K[b, h, 0], np.float64), np.array(V[b, h, 0], np.float64))
                    for kind, X in ((KIND_K, K), (KIND_V, V)):
                        x = np.array(X[b, h, blk * T:(blk + 1) * T], np.float32)
                        if first:
                            x[0] = 0.0
                        self.recs[(b, h, self.n_blocks + blk, kind)] = self.quantize_tile(x, kind, h)
        self.n_blocks += n

    # ------------------------------------------------------------------ decode
    def dequant_tile(self, rec: dict, kind: int, h: int, blk: int, domain: str) -> np.ndarray:
        """domain 'stored': the quantised representation (pre-RoPE keys un-rotated, KVarN
        in the Hadamard domain); 'input': back in the input domain (inverse Hadamard for
        KVarN); 'attn': what attention reads (RoPE applied to pre-RoPE keys)."""
        codes = unpack_tile(rec["words"], self.bits, kind, self.layout)
        m = self.method
        if m == "rtn":
            x = rtn_dequant(codes, rec["s16"], rec["z16"], 0 if kind == KIND_K else 1)
        elif m == "int4":
            x = absmax_dequant(absmax_from_codes(codes, self.bits), rec["s16"])
        elif m == "nuq":
            x = nuq_dequant(codes, rec["s16"], rec["zp16"], self.codebook[h], 0 if kind == KIND_K else 1,
                            rec.get("row_ptr"), rec.get("col"), rec["val"], rec.get("col_ptr"), rec.get("row"))
        else:
            x = varn_dequant(codes, rec["s16"], rec["z16"], rec["s1"], kind)
            if domain == "input" and self.use_hadamard:
                x = fwht(x)
        if domain == "attn" and kind == KIND_K and self.pre_rope:
            x = rope(x, np.arange(blk * T, (blk + 1) * T), self.rope_theta)
        return x

    def dequant(self, b: int, h: int, kind: int, domain: str = "stored", first: int = 0, n=None):
        n = self.n_blocks - first if n is None else n
        return np.concatenate([self.dequant_tile(self.recs[(b, h, blk, kind)], kind, h, blk, domain)
                               for blk in range(first, first + n)], axis=0) if n > 0 \
            else np.zeros((0, D))

    def decode(self, q: np.ndarray, tail_k=None, tail_v=None, only_heads=None) -> np.ndarray:
        """q [B][H_q][128] (post-RoPE for pre-RoPE caches); tail_k/tail_v [B][H_kv][n_tail][128]
        fp residual tokens at positions n_blocks*128 + j (pre-RoPE keys are rotated there).
        Returns fp64 [B][H_q][128] (rows of heads outside only_heads are NaN)."""
        G = self.n_q_heads // self.n_kv_heads
        out = np.full((self.batch, self.n_q_heads, D), np.nan)
        n_tail = 0 if tail_k is None else tail_k.shape[2]
        pos0 = self.n_blocks * T
        for b in range(self.batch):
            for h in range(self.n_kv_heads):
                if only_heads is not None and (b, h) not in only_heads:
                    continue
                qg = np.asarray(q[b, h * G:(h + 1) * G], np.float64)
                Kc = self.dequant(b, h, KIND_K, "attn")
                Vc = self.dequant(b, h, KIND_V, "attn")
                is_varn = self.method == "varn" and self.use_hadamard
                qc = fwht(qg) if is_varn else qg
                s = qc @ Kc.T / math.sqrt(D)
                if self.sink and Kc.shape[0]:  # the kept first token replaces quantised token 0
                    ks, vs = self.sink_kv[(b, h)]
                    s[:, 0] = qg @ ks / math.sqrt(D)  # position 0: RoPE is the identity
                    Vc = Vc.copy()
                    Vc[0] = vs
                if n_tail:
                    kt = np.asarray(tail_k[b, h], np.float64)
                    if self.pre_rope:
                        kt = rope(kt, np.arange(pos0, pos0 + n_tail), self.rope_theta)
                    s = np.concatenate([s, qg @ kt.T / math.sqrt(D)], axis=1)
                mx = s.max(axis=1, keepdims=True)
                p = np.exp(s - mx)
                oc = p[:, :Kc.shape[0]] @ Vc
                if is_varn:
                    oc = fwht(oc)
                if n_tail:
                    oc = oc + p[:, Kc.shape[0]:] @ np.asarray(tail_v[b, h], np.float64)
                out[b, h * G:(h + 1) * G] = oc / p.sum(axis=1, keepdims=True)
        return out
