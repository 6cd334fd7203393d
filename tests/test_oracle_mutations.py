"""Planted mistakes: each test swaps one oracle function for a plausibly wrong version
(on the CPU, inside the oracle only) and checks that at least one pin then fails."""
import numpy as np
import pytest

import oracle as O
import oracle.kvq_oracle as K
import tests.test_oracle_pins as P


def _fails(fn, *args, **kw):
    try:
        fn(*args, **kw)
    except (AssertionError, IndexError, ValueError):
        return True
    return False


def test_rope_sign_flip_is_caught(monkeypatch, golden_dir):
    orig = K.rope
    monkeypatch.setattr(K, "rope", lambda x, pos, theta=10000.0: orig(x, -np.asarray(pos), theta))
    monkeypatch.setattr(O, "rope", K.rope)
    assert _fails(P.test_rope_norm_identity_and_relative_position, golden_dir)


def test_rope_rotate_half_layout_is_caught(monkeypatch, golden_dir):
    def rotate_half(x, positions, theta=10000.0):
        x = np.asarray(x, np.float64)
        ang = K.rope_angles(positions, theta, x.shape[-1])
        c, s = np.cos(ang), np.sin(ang)
        x0, x1 = x[..., :64], x[..., 64:]
        return np.concatenate([c * x0 - s * x1, s * x0 + c * x1], axis=-1)
    monkeypatch.setattr(K, "rope", rotate_half)
    monkeypatch.setattr(O, "rope", rotate_half)
    assert _fails(P.test_rope_norm_identity_and_relative_position, golden_dir)


def test_rtn_axis_swap_in_cache_is_caught(monkeypatch):
    orig = K.rtn_quantize
    monkeypatch.setattr(K, "rtn_quantize", lambda x, bits, axis: orig(x, bits, 1 - axis))
    assert _fails(P.test_cache_decode_equals_plain_attention_on_lossless_inputs, "rtn", 1, False)


def test_rtn_floor_instead_of_rint_is_caught(monkeypatch):
    def enc(x, s16, z16, bits):
        t = np.float32(x) / s16.astype(np.float32) - z16.astype(np.float32)
        return np.clip(np.floor(t), 0, 2 ** bits - 1).astype(np.uint8)
    monkeypatch.setattr(K, "rtn_encode", enc)
    assert _fails(P.test_rtn_error_bound, 2, 0)


def test_missing_sqrt_d_is_caught(monkeypatch):
    def att(q, Kx, V):
        s = np.asarray(q, np.float64) @ np.asarray(Kx, np.float64).T
        p = np.exp(s - s.max(axis=-1, keepdims=True))
        return (p @ V) / p.sum(axis=-1, keepdims=True)
    monkeypatch.setattr(K, "attention", att)
    monkeypatch.setattr(O, "attention", att)
    assert _fails(P.test_attention_brute_force, 127)


def test_argmin_last_index_tie_is_caught(monkeypatch):
    def enc(t, cb):
        d = np.abs(np.float32(t)[..., None] - np.float32(cb))
        return (len(cb) - 1 - np.argmin(d[..., ::-1], axis=-1)).astype(np.uint8)
    monkeypatch.setattr(K, "nuq_encode", enc)
    monkeypatch.setattr(O, "nuq_encode", enc)
    assert _fails(P.test_nuq_argmin_equals_brute_force)


def test_pack_msb_first_is_caught(monkeypatch, golden_dir):
    def pack(codes, bits):
        n = 32 // bits
        W = -(-128 // n)
        out = np.zeros(np.shape(codes)[:-1] + (W,), np.uint64)
        for i in range(128):
            out[..., i // n] |= np.asarray(codes)[..., i].astype(np.uint64) << np.uint64(bits * (n - 1 - i % n))
        return out.astype(np.uint32)
    monkeypatch.setattr(K, "pack_rows", pack)
    monkeypatch.setattr(O, "pack_rows", pack)
    assert _fails(P.test_3bit_layout_printed_words, golden_dir)


def test_tile3_swapped_high_bit_planes_are_caught(monkeypatch):
    orig = K.tile3_slot

    def slot(kind, t, c):
        lw, ls, hw, hs = orig(kind, t, c)
        u = np.asarray(c, np.int64) >> 4  # the nibble word, for keys and values alike
        # high bits of nibble words 2 and 3 exchanged: still a valid permutation
        return lw, ls, hw, np.where((u & 3) >= 2, hs ^ 1, hs)
    monkeypatch.setattr(K, "tile3_slot", slot)
    monkeypatch.setattr(O, "tile3_slot", slot)
    assert _fails(P.test_tile3_slots_follow_the_documented_rule)


def test_tile3_value_token_order_is_caught(monkeypatch):
    orig = K.tile3_slot

    def slot(kind, t, c):
        if kind == K.KIND_V:  # tokens t and t^8 of each segment exchanged
            t = np.asarray(t, np.int64) ^ 8
        return orig(kind, t, c)
    monkeypatch.setattr(K, "tile3_slot", slot)
    monkeypatch.setattr(O, "tile3_slot", slot)
    assert _fails(P.test_tile3_groups_hold_one_lanes_fragment_codes, 1) or \
        _fails(P.test_tile3_slots_follow_the_documented_rule)


def test_varn_column_only_is_caught(monkeypatch):
    def varn_cols(X, iters=8):
        Y = np.array(X, np.float64)
        lc = np.zeros(Y.shape[1])
        for _ in range(iters):
            sc = Y.std(axis=0)
            Y /= sc
            lc += np.log(sc)
        return Y, np.ones(Y.shape[0]), np.exp(lc)
    monkeypatch.setattr(K, "varn", varn_cols)
    monkeypatch.setattr(O, "varn", varn_cols)
    assert _fails(P.test_varn_recomposition_and_stds)


def test_hadamard_unnormalised_is_caught(monkeypatch):
    monkeypatch.setattr(K, "fwht", lambda x: np.asarray(x, np.float64) @ K.hadamard(x.shape[-1]))
    monkeypatch.setattr(O, "fwht", K.fwht)
    assert _fails(P.test_hadamard_sylvester_and_orthogonality)


def test_int4_asymmetric_clamp_is_caught(monkeypatch):
    orig = K.int4_quantize
    def q8(x):
        q, s = orig(x)
        return np.where(q == -7, -8, q).astype(np.int8), s
    monkeypatch.setattr(K, "int4_quantize", q8)
    monkeypatch.setattr(O, "int4_quantize", q8)
    assert _fails(P.test_int4_codes_range_and_bound)


def test_outlier_tie_break_reversed_is_caught(monkeypatch):
    def mask_rev(x, n_out):
        mag = (np.asarray(x, np.float32).astype(np.float16).view(np.uint16) & 0x7FFF).ravel()
        idx = np.arange(mag.size)
        order = np.lexsort((-idx, -mag.astype(np.int64)))
        m = np.zeros(mag.size, bool)
        m[order[:n_out]] = True
        return m.reshape(np.shape(x))
    monkeypatch.setattr(K, "outlier_mask", mask_rev)
    monkeypatch.setattr(O, "outlier_mask", mask_rev)
    assert _fails(P.test_outlier_selection_planted_and_ties)


def test_gqa_mapping_interleaved_is_caught(monkeypatch):
    orig = K.OracleCache.decode
    def dec(self, q, tail_k=None, tail_v=None, only_heads=None):
        G = self.n_q_heads // self.n_kv_heads
        qq = np.asarray(q).copy()
        if G > 1:       # read KV head j % H_kv instead of j // G
            idx = np.array([(j % self.n_kv_heads) * G + (j // self.n_kv_heads) for j in range(self.n_q_heads)])
            qq = qq[:, idx]
            out = orig(self, qq, tail_k, tail_v, only_heads)
            res = np.empty_like(out)
            res[:, idx] = out
            return res
        return orig(self, q, tail_k, tail_v, only_heads)
    monkeypatch.setattr(K.OracleCache, "decode", dec)
    assert _fails(P.test_cache_decode_equals_plain_attention_on_lossless_inputs, "rtn", 4, False)


def test_calibration_including_the_first_token_is_caught(monkeypatch):
    orig = K.calibrate_keys
    monkeypatch.setattr(K, "calibrate_keys", lambda Kc, f: orig(np.concatenate([Kc[:1], Kc]), f))
    monkeypatch.setattr(O, "calibrate_keys", K.calibrate_keys)
    assert _fails(P.test_calibrate_keys_brute_force)


def test_calibrated_threshold_off_by_one_is_caught(monkeypatch):
    def calib(Kc, f):  # the next order statistic up: one outlier fewer per channel
        x = np.asarray(Kc, np.float32)[1:]
        a = np.sort(np.abs(x), axis=0)
        r = min(x.shape[0], int(np.ceil((1.0 - float(np.float32(f))) * x.shape[0])) + 1)
        tau = a[r - 1].astype(np.float32) if f > 0 else np.full(128, np.inf, np.float32)
        s16, zp16 = K.nuq_meta(x, np.abs(x) > tau[None, :], 0)
        return tau, s16, zp16
    monkeypatch.setattr(K, "calibrate_keys", calib)
    monkeypatch.setattr(O, "calibrate_keys", calib)
    assert _fails(P.test_calibrate_keys_brute_force)


def test_sink_row_left_in_the_tiles_is_caught(monkeypatch):
    orig = K.OracleCache.append
    def append(self, Kx, Vx, only_heads=None):  # keeps the first token but never zeroes it
        sink, self.sink = self.sink, False
        first = self.n_blocks == 0
        orig(self, Kx, Vx, only_heads)
        self.sink = sink
        if sink and first:
            for b in range(self.batch):
                for h in range(self.n_kv_heads):
                    self.sink_kv[(b, h)] = (np.array(Kx[b, h, 0], np.float64), np.array(Vx[b, h, 0], np.float64))
    monkeypatch.setattr(K.OracleCache, "append", append)
    assert _fails(P.test_sink_decode_equals_plain_attention_on_lossless_inputs, False)


def test_direction_error_without_factor_two_is_caught(monkeypatch):
    orig = K.token_error_stats

    def half_ed(X, Xdq):
        s = orig(X, Xdq)
        s[..., 3] *= 0.5
        return s
    monkeypatch.setattr(K, "token_error_stats", half_ed)
    monkeypatch.setattr(O, "token_error_stats", half_ed)
    assert _fails(P.test_token_error_stats_closed_forms)


def test_norm_deviation_sign_flip_is_caught(monkeypatch):
    orig = K.token_error_stats

    def flipped(X, Xdq):
        s = orig(X, Xdq)
        s[..., 1] *= -1.0
        return s
    monkeypatch.setattr(K, "token_error_stats", flipped)
    monkeypatch.setattr(O, "token_error_stats", flipped)
    assert _fails(P.test_token_error_stats_closed_forms)


def test_topk_ties_to_the_higher_row_are_caught(monkeypatch):
    def later_first(stats, fracs):
        stats = np.asarray(stats).reshape(-1, 4)
        n = stats.shape[0]
        order = np.lexsort((-np.arange(n), -stats[:, 2].astype(np.float64)))
        out = np.zeros((len(fracs), 4))
        for i, f in enumerate(fracs):
            sel = order[:min(n, int(np.ceil(float(f) * n)))]
            out[i] = (len(sel), stats[sel, 2].sum(), (stats[sel, 1] ** 2).sum(), stats[sel, 3].sum())
        return out
    monkeypatch.setattr(K, "topk_error_share", later_first)
    monkeypatch.setattr(O, "topk_error_share", later_first)
    assert _fails(P.test_topk_error_share_brute_force)


def test_int8_divisor_128_is_caught(monkeypatch):
    orig = K.absmax_quantize

    def wrong(x, bits=4, group=128):
        if bits != 8:
            return orig(x, bits, group)
        x = np.asarray(x, np.float32)
        ng = 128 // group
        xg = x.reshape(128, ng, group)
        s16 = np.minimum(np.abs(xg).max(axis=2) / np.float32(128.0), np.float32(65504.0)).astype(np.float16)
        sf = s16.astype(np.float32)
        with np.errstate(invalid="ignore", divide="ignore"):
            q = np.clip(np.rint(xg / sf[:, :, None]), -128, 127)
        q[sf == 0] = 0
        return q.reshape(128, 128).astype(np.int16), np.ascontiguousarray(s16.T)
    monkeypatch.setattr(K, "absmax_quantize", wrong)
    monkeypatch.setattr(O, "absmax_quantize", wrong)
    assert _fails(P.test_absmax_variants_codes_range_and_bound, 8, 128)


def test_group64_scales_of_the_wrong_half_are_caught(monkeypatch):
    orig = K.absmax_dequant

    def swapped(q, s16):
        s = np.asarray(s16)
        return orig(q, s[::-1] if s.ndim == 2 and s.shape[0] == 2 else s)
    monkeypatch.setattr(K, "absmax_dequant", swapped)
    assert _fails(P.test_cache_decode_equals_plain_attention_on_lossless_inputs, "int4g64", 1, False)


def test_unweighted_codebook_update_is_caught(monkeypatch):
    orig = K.fit_codebook
    monkeypatch.setattr(K, "fit_codebook", lambda a, w, bits, max_iter=50: orig(a, np.ones_like(np.asarray(w)), bits,
                                                                               max_iter))
    monkeypatch.setattr(O, "fit_codebook", K.fit_codebook)
    assert _fails(P.test_fit_codebook_weighted_means_of_separated_groups)


def test_codebook_ties_to_the_higher_centre_are_caught(monkeypatch):
    orig = K.fit_codebook

    def flipped(a, w, bits, max_iter=50):
        c, it = orig(-np.asarray(a, np.float32), w, bits, max_iter)  # mirrored data: ties go the other way
        return -c[::-1], it
    monkeypatch.setattr(K, "fit_codebook", flipped)
    monkeypatch.setattr(O, "fit_codebook", flipped)
    assert _fails(P.test_fit_codebook_converged_state_and_ties)



def test_csc_in_row_order_is_caught(monkeypatch):
    def row_order(x, mask):  # entries left in (token, channel) order under column pointers
        col_ptr = np.zeros(O.D + 1, np.int64)
        col_ptr[1:] = np.cumsum(np.asarray(mask).sum(axis=0))
        tt, cc = np.nonzero(mask)
        return col_ptr.astype(np.uint16), tt.astype(np.uint8), np.asarray(x, np.float32)[tt, cc].astype(np.float16).view(np.uint16)
    monkeypatch.setattr(K, "csc_of", row_order)
    monkeypatch.setattr(O, "csc_of", row_order)
    assert _fails(P.test_csc_of_brute_force_and_same_entries_as_csr)
