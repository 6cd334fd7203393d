"""Helpers shared by the tests: build a device cache for a workload, upload seeded inputs,
read the device records back through the layout, compare them with the oracle's records."""
from __future__ import annotations

import numpy as np

import oracle as O
import workloads as WL

T, D = 128, 128


def torch_mod():
    import torch
    return torch


def cfg_for(w: WL.Workload, max_blocks=None, batch=None, layout="rows", v_csc=False):
    import bit_kv_cache_block_gb300 as K
    return K.make_config(w.method, w.bits, batch or w.batch, w.n_kv_heads, w.n_q_heads,
                         max_blocks or w.n_blocks, in_dtype=w.dtype, pre_rope=w.pre_rope,
                         rope_theta=w.rope_theta, outlier_frac=w.outlier_frac, varn_iters=w.varn_iters,
                         hadamard=True, layout=layout, scale_group=w.scale_group, v_csc=v_csc)


def oracle_layout(layout: str) -> int:
    return O.LAYOUT_MMA if layout == "mma" else O.LAYOUT_ROWS


def codebook_for(w: WL.Workload):
    if w.method != "nuq":
        return None
    return np.broadcast_to(O.nuq_codebook(w.bits), (w.n_kv_heads, 2 ** w.bits)).copy()


def to_device(x: np.ndarray, dtype: str, device="cuda"):
    """float32 values (exactly representable in dtype) -> device tensor of that dtype."""
    torch = torch_mod()
    bits = WL.to_storage(np.ascontiguousarray(x), dtype)
    t = torch.from_numpy(bits.view(np.int16).copy()).to(device)
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def new_cache(w: WL.Workload, max_blocks=None, batch=None, layout="rows", v_csc=False):
    import bit_kv_cache_block_gb300 as K
    torch = torch_mod()
    cb = codebook_for(w)
    return K.KVCache(cfg_for(w, max_blocks, batch, layout, v_csc), None if cb is None else torch.from_numpy(cb))


def sparse_parts(otile: dict):
    """(pointer array, index array, values) of an oracle nuq tile, CSR or CSC: the three arrays in
    the order the record's outlier region stores them."""
    if "col_ptr" in otile:
        return otile["col_ptr"], otile["row"], otile["val"]
    return otile["row_ptr"], otile["col"], otile["val"]


def records_np(cache) -> np.ndarray:
    return cache.record_view().cpu().numpy()


def tile_fields(rec: np.ndarray, lay, kind: int, method: str, bits: int, layout: str = "rows") -> dict:
    """Decode one record's K (kind 0) or V (kind 1) regions into arrays (code words shaped as the
    oracle's pack_tile returns them: flat planes for 3-bit "mma" tiles, else [128 rows][W])."""
    W = lay.words_per_row
    co, cb = int(lay.codes_off[kind]), int(lay.codes_bytes[kind])
    mo, mb = int(lay.meta_off[kind]), int(lay.meta_bytes[kind])
    words = rec[co:co + cb].view(np.uint32).copy()
    out = dict(words=words if (bits == 3 and layout == "mma") else words.reshape(T, W))
    meta = rec[mo:mo + mb].view(np.uint16).reshape(-1, T)
    out["s16"] = meta[0].view(np.float16).copy()
    if method == "int4" and meta.shape[0] == 2:  # one scale per 64 channels: [2][128]
        out["s16"] = meta.view(np.float16).copy()
    if method in ("rtn", "varn"):
        out["z16"] = meta[1].view(np.float16).copy()
    if method == "varn":
        out["s1"] = meta[2].view(np.float16).copy()
    if method == "nuq":
        out["zp16"] = meta[1].view(np.float16).copy()
        n = int(lay.n_outliers)
        if n:
            so = int(lay.csr_off[kind])
            csr = rec[so:so + int(lay.csr_bytes[kind])]
            out["val"] = csr[:2 * n].view(np.uint16).copy()
            out["row_ptr"] = csr[2 * n:2 * n + 2 * (T + 1)].view(np.uint16).copy()
            out["col"] = csr[2 * n + 2 * (T + 1):3 * n + 2 * (T + 1)].copy()
            out["csr_pad"] = csr[3 * n + 2 * (T + 1):].copy()
    return out


def serialize_tile(rec: np.ndarray, lay, kind: int, otile: dict, method: str) -> None:
    """Write an oracle tile record into the byte layout (for feeding oracle planes to the GPU)."""
    co, mo = int(lay.codes_off[kind]), int(lay.meta_off[kind])
    words = np.ascontiguousarray(otile["words"], np.uint32)
    rec[co:co + words.nbytes] = words.view(np.uint8).ravel()
    vecs = [otile["s16"]]
    if method in ("rtn", "varn"):
        vecs.append(otile["z16"])
    if method == "varn":
        vecs.append(otile["s1"])
    if method == "nuq":
        vecs.append(otile["zp16"])
    meta = np.stack([np.asarray(v, np.float16) for v in vecs]).view(np.uint8).ravel()
    rec[mo:mo + meta.size] = meta
    n = int(lay.n_outliers)
    if method == "nuq" and n:
        so = int(lay.csr_off[kind])
        rec[so:so + 2 * n] = np.asarray(otile["val"], np.uint16).view(np.uint8)
        ptr, idx, _ = sparse_parts(otile)
        rec[so + 2 * n:so + 2 * n + 2 * (T + 1)] = np.asarray(ptr, np.uint16).view(np.uint8)
        rec[so + 2 * n + 2 * (T + 1):so + 3 * n + 2 * (T + 1)] = np.asarray(idx, np.uint8)


def f16_bits(x) -> np.ndarray:
    return np.asarray(x, np.float16).view(np.uint16)


def near_f16_midpoint(v: np.ndarray, rel: float = 1e-5) -> np.ndarray:
    """True where a positive/negative value lies within rel of a rounding midpoint of fp16."""
    v = np.asarray(v, np.float64)
    h = v.astype(np.float16)
    hf = h.astype(np.float64)
    up = np.nextafter(h, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(h, np.float16(-np.inf)).astype(np.float64)
    other = np.where(hf <= v, up, dn)
    mid = (hf + other) / 2
    return np.abs(v - mid) <= rel * np.maximum(np.abs(v), 1e-30)


def ulp_apart(a16: np.ndarray, b16: np.ndarray) -> np.ndarray:
    """|ordinal(a) - ordinal(b)| for fp16 arrays (works across zero)."""
    def ordn(x):
        u = np.asarray(x, np.float16).view(np.uint16).astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7fff), u)
    return np.abs(ordn(a16) - ordn(b16))


def varn_check_tile(got: dict, exp: dict, kind: int, dbg_rc, layout: str, bits: int = 2) -> dict:
    """KVarN record of one tile against the oracle's, under the exemptions the fp32 kernel may take
    against the fp64 oracle (KVarN summary, method steps 2-5; the window is 1e-5 relative
    throughout):

    - VarN scales r, c (dbg_rc, or None to skip) within 1e-5 relative of the oracle's;
    - s1 and the RTN scale s equal to the oracle's fp16 values, or one fp16 ulp apart only where
      the oracle's unrounded value lies within 1e-5 relative of an fp16 rounding midpoint;
    - in groups whose s equals the oracle's: the zero point z equal to the oracle's, or one ulp
      apart only next to a midpoint of the oracle's unrounded min/s; the codes equal to the
      oracle's, or +-1 only where the oracle's x/s - z lies within 1e-5 (relative to the larger of
      |x/s - z| and 1) of a rounding boundary n + 1/2;
    - groups whose s took the one-ulp exemption form their own class: their z is derived from that
      s, so z and the codes are judged the same way but against the oracle's Z under the kernel's
      s (the values the oracle would store with that scale).

    Returns counts: s1/s/z cells one ulp apart, codes +-1, and the groups and codes of the
    derived class."""
    if dbg_rc is not None:
        r_o, c_o = exp["r"], exp["c"]
        assert np.all(np.abs(dbg_rc[0] - r_o) <= 1e-5 * np.abs(r_o)), "VarN token scales r"
        assert np.all(np.abs(dbg_rc[1] - c_o) <= 1e-5 * np.abs(c_o)), "VarN channel scales c"
    cnt = dict(s1_ulp=0, s_ulp=0, z_ulp=0, codes_pm1=0, derived_groups=0, derived_codes_pm1=0)
    s1_true = exp["r"] if kind == 0 else exp["c"]
    d = ulp_apart(got["s1"], exp["s1"])
    assert np.all((d == 0) | ((d == 1) & near_f16_midpoint(s1_true))), "s1"
    cnt["s1_ulp"] = int((d == 1).sum())
    axis = 0 if kind == 0 else 1
    Z32 = exp["Z"].astype(np.float32)
    mx = Z32.max(axis=axis).astype(np.float32)
    mn = Z32.min(axis=axis).astype(np.float32)
    s32 = (mx - mn) / np.float32(2 ** bits - 1)
    ds = ulp_apart(got["s16"], exp["s16"])
    assert np.all((ds == 0) | ((ds == 1) & near_f16_midpoint(s32))), "RTN scale"
    cnt["s_ulp"] = int((ds == 1).sum())
    same = ds == 0
    # zero point: against the oracle's where s agrees; derived from the kernel's s where it does not
    s_ref = np.where(same, exp["s16"], got["s16"]).astype(np.float16)
    z_ref = np.where(same, exp["z16"], (mn / s_ref.astype(np.float32)).astype(np.float16)).astype(np.float16)
    zt = mn.astype(np.float64) / s_ref.astype(np.float64)
    dz = ulp_apart(got["z16"], z_ref)
    assert np.all((dz == 0) | ((dz == 1) & near_f16_midpoint(zt))), "RTN zero point"
    cnt["z_ulp"] = int(((dz == 1) & same).sum())
    # codes: the oracle's Z under the reference metadata (the oracle's own where s agrees)
    s = s_ref.astype(np.float32)
    z = z_ref.astype(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        tt = Z32 / s[None, :] - z[None, :] if axis == 0 else Z32 / s[:, None] - z[:, None]
    e = np.clip(np.rint(tt), 0, 2 ** bits - 1)
    codes = O.unpack_tile(got["words"], bits, kind, oracle_layout(layout)).astype(np.int64)
    diff = np.abs(codes - e)
    t64 = tt.astype(np.float64)
    near = np.abs(t64 - np.floor(t64) - 0.5) <= 1e-5 * np.maximum(1.0, np.abs(t64))
    assert np.all((diff == 0) | ((diff == 1) & near)), f"codes: {int(((diff > 0) & ~near).sum())} off"
    derived = np.broadcast_to(~same[None, :] if axis == 0 else ~same[:, None], diff.shape)
    cnt["codes_pm1"] = int(((diff == 1) & ~derived).sum())
    cnt["derived_groups"] = int((~same).sum())
    cnt["derived_codes_pm1"] = int(((diff == 1) & derived).sum())
    return cnt
