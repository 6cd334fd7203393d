"""bit_kv_cache_block_gb300: low-bit KV-cache quantization in 128-token blocks and decode
attention over the packed cache, as hand-written CUDA kernels for sm_103a behind a C ABI
(include/kvq.h, libkvq.so).

This module is the thin Python binding: the functions carry the C names and only marshal
arguments (torch tensors -> device pointers, the current torch stream -> cudaStream_t).
Every step of the path runs in the library's kernels; there is no Python or CPU fallback.
PyTorch only provides device memory and streams.
"""
from __future__ import annotations

import ctypes as C

from . import _lib
from ._lib import (KVQ_BF16, KVQ_F16, KVQ_INT4, KVQ_LAYOUT_MMA, KVQ_LAYOUT_ROWS, KVQ_NUQ, KVQ_OK, KVQ_RTN, KVQ_VARN,
                   KVQError, LAYOUTS, METHODS,
                   kvq_cache, kvq_config, kvq_layout_t)

__all__ = ["make_config", "kvq_layout", "kvq_dense_kv_bytes", "kvq_cache_init", "kvq_append_block",
           "kvq_truncate", "kvq_reset", "kvq_decode_splits", "kvq_decode_workspace_bytes", "kvq_decode_bytes",
           "kvq_decode_attn", "kvq_decode_attn_ex", "kvq_decode_attn_static", "kvq_dequant", "kvq_error_stats", "kvq_error_topk",
           "kvq_error_topk_workspace_bytes", "error_topk", "fit_codebook", "kvq_status_str", "KVCache", "KVQError", "kvq_config",
           "kvq_layout_t", "kvq_cache", "lib_path"]


def lib_path() -> str:
    return _lib.LIB_PATH


def make_config(method: str, bits: int, batch: int, n_kv_heads: int, n_q_heads: int, max_blocks: int,
                in_dtype: str = "f16", pre_rope: bool = False, rope_theta: float = 10000.0,
                outlier_frac: float = 0.01, varn_iters: int = 8, hadamard: bool = True,
                layout: str = "rows", n_pages: int = 0, key_calib: bool = False, sink: bool = False,
                scale_group: int = 128, v_csc: bool = False) -> kvq_config:
    c = kvq_config()
    c.method = METHODS[method] if isinstance(method, str) else int(method)
    c.bits, c.batch, c.n_kv_heads, c.n_q_heads = bits, batch, n_kv_heads, n_q_heads
    c.head_dim, c.block, c.max_blocks = 128, 128, max_blocks
    c.in_dtype = KVQ_BF16 if in_dtype == "bf16" else KVQ_F16
    c.pre_rope = int(bool(pre_rope))
    c.rope_theta = float(rope_theta)
    c.outlier_frac = float(outlier_frac)
    c.varn_iters = int(varn_iters)
    c.hadamard = int(bool(hadamard))
    c.layout = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    c.n_pages = int(n_pages)
    c.key_calib = int(bool(key_calib))
    c.sink = int(bool(sink))
    c.scale_group = int(scale_group)
    c.v_csc = int(bool(v_csc))
    return c


def _stream(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if hasattr(stream, "cuda_stream"):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return C.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return C.c_void_p(t.data_ptr())


def kvq_status_str(s: int) -> str:
    return _lib.status_str(s)


def kvq_dense_kv_bytes(n_layers, n_heads, head_dim, elem_bytes, batch, seq_len) -> int:
    return int(_lib.lib().kvq_dense_kv_bytes(n_layers, n_heads, head_dim, elem_bytes, batch, seq_len))


def kvq_layout(cfg: kvq_config) -> kvq_layout_t:
    out = kvq_layout_t()
    _lib.check(_lib.lib().kvq_layout(C.byref(cfg), C.byref(out)), "kvq_layout")
    return out


def kvq_cache_init(cfg: kvq_config, base, codebook, status, stream=None) -> kvq_cache:
    """base: uint8 device tensor of >= layout.total_bytes; codebook: fp32 [H_kv][2^bits] (NUQ) or
    None; status: int32 device tensor of 1 element."""
    cache = kvq_cache()
    _lib.check(_lib.lib().kvq_cache_init(C.byref(cache), C.byref(cfg), _ptr(base), base.numel() * base.element_size(),
                                         _ptr(codebook), _ptr(status), _stream(stream)), "kvq_cache_init")
    return cache


def kvq_append_block(cache: kvq_cache, k, v, dbg_varn_scales=None, stream=None) -> None:
    """k, v: device [B][H_kv][n*128][128] in the cache's input dtype."""
    n = k.shape[2] // 128
    if tuple(k.shape) != tuple(v.shape) or k.shape[2] % 128 != 0:
        raise ValueError("k and v must have the same shape [B][H_kv][n*128][128]")
    _lib.check(_lib.lib().kvq_append_block(C.byref(cache), _ptr(k), _ptr(v), n, _ptr(dbg_varn_scales),
                                           _stream(stream)), "kvq_append_block")


def kvq_truncate(cache: kvq_cache, n_blocks: int) -> None:
    _lib.check(_lib.lib().kvq_truncate(C.byref(cache), int(n_blocks)), "kvq_truncate")


def kvq_reset(cache: kvq_cache) -> None:
    _lib.check(_lib.lib().kvq_reset(C.byref(cache)), "kvq_reset")


def kvq_debug_stall_decode(enable: bool) -> None:
    """Test switch: later nuq tensor-core decodes run with no copies and ~1 ms wait bounds, so they
    record KVQ_ERR_TIMEOUT and write NaN (see include/kvq.h)."""
    _lib.check(_lib.lib().kvq_debug_stall_decode(1 if enable else 0), "kvq_debug_stall_decode")


def kvq_decode_splits(cfg: kvq_config, n_blocks: int) -> int:
    return int(_lib.lib().kvq_decode_splits(C.byref(cfg), int(n_blocks)))


def kvq_decode_workspace_bytes(cfg: kvq_config, n_blocks: int) -> int:
    out = C.c_size_t()
    _lib.check(_lib.lib().kvq_decode_workspace_bytes(C.byref(cfg), int(n_blocks), C.byref(out)),
               "kvq_decode_workspace_bytes")
    return int(out.value)


def kvq_decode_bytes(cfg: kvq_config, n_blocks: int) -> int:
    return int(_lib.lib().kvq_decode_bytes(C.byref(cfg), int(n_blocks)))


def kvq_decode_attn(cache: kvq_cache, q, tail_k, tail_v, n_tail: int, out, workspace, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.check(_lib.lib().kvq_decode_attn(C.byref(cache), _ptr(q), _ptr(tail_k), _ptr(tail_v), int(n_tail),
                                          _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)),
               "kvq_decode_attn")


def kvq_decode_attn_ex(cache: kvq_cache, q, tail_k, tail_v, n_tail: int, bh_stride: int, token_stride: int, out,
                       workspace, stream=None) -> None:
    """kvq_decode_attn over tail buffers laid out by (b, h) and token strides, in elements."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.check(_lib.lib().kvq_decode_attn_ex(C.byref(cache), _ptr(q), _ptr(tail_k), _ptr(tail_v), int(n_tail),
                                             int(bh_stride), int(token_stride), _ptr(out), _ptr(workspace),
                                             ws_bytes, _stream(stream)), "kvq_decode_attn_ex")


def kvq_decode_attn_static(cache: kvq_cache, q, tail_k, tail_v, n_tail: int, out, stream=None) -> None:
    """kvq_decode_attn with the library's own fixed scratch instead of a caller workspace, for
    callers that cannot allocate device memory. Calls that may overlap on the GPU share that
    scratch and race; the first call on a device looks up its address (no allocation)."""
    _lib.check(_lib.lib().kvq_decode_attn_static(C.byref(cache), _ptr(q), _ptr(tail_k), _ptr(tail_v),
                                                 int(n_tail), _ptr(out), _stream(stream)),
               "kvq_decode_attn_static")


def kvq_dequant(cache: kvq_cache, first_block: int, n_blocks: int, domain: int, out_k, out_v, stream=None) -> None:
    _lib.check(_lib.lib().kvq_dequant(C.byref(cache), int(first_block), int(n_blocks), int(domain), _ptr(out_k),
                                      _ptr(out_v), _stream(stream)), "kvq_dequant")


def kvq_calibrate_keys(cache: kvq_cache, k_calib, stream=None) -> None:
    """k_calib: device [H_kv][n_tokens][128] in the cache's input dtype (calibration keys)."""
    if k_calib.dim() != 3 or k_calib.shape[2] != 128:
        raise ValueError("calibration keys must be [H_kv][n_tokens][128]")
    _lib.check(_lib.lib().kvq_calibrate_keys(C.byref(cache), _ptr(k_calib), int(k_calib.shape[1]),
                                             _stream(stream)), "kvq_calibrate_keys")


def kvq_error_stats(cache: kvq_cache, first_block: int, n_blocks: int, k, v, stats_k, stats_v, stream=None) -> None:
    """Per-token (|x|, |x_dq| - |x|, E_T, E_D) of cached blocks against their inputs; either
    (k, stats_k) or (v, stats_v) may be None."""
    _lib.check(_lib.lib().kvq_error_stats(C.byref(cache), _ptr(k), _ptr(v), int(first_block), int(n_blocks),
                                          _ptr(stats_k), _ptr(stats_v), _stream(stream)), "kvq_error_stats")


def kvq_error_topk_workspace_bytes() -> int:
    return int(_lib.lib().kvq_error_topk_workspace_bytes())


def kvq_error_topk(stats, fracs, out, workspace, stream=None) -> None:
    """stats: device fp32 [..., 4] rows from kvq_error_stats; fracs: host sequence of fractions;
    out: device fp64 [len(fracs)][4] = (k, sum E_T, sum E_M, sum E_D) over the k largest E_T."""
    if stats.shape[-1] != 4:
        raise ValueError("stats rows must have 4 columns")
    fr = (C.c_double * len(fracs))(*[float(f) for f in fracs])
    ws_bytes = workspace.numel() * workspace.element_size()
    _lib.check(_lib.lib().kvq_error_topk(_ptr(stats), int(stats.numel() // 4), fr, len(fracs), _ptr(out),
                                         _ptr(workspace), ws_bytes, _stream(stream)), "kvq_error_topk")


def error_topk(stats, fracs, stream=None):
    """kvq_error_topk with its own output and workspace: returns fp64 [len(fracs)][4] on the
    stats' device."""
    import torch
    out = torch.empty(len(fracs), 4, dtype=torch.float64, device=stats.device)
    ws = torch.empty(kvq_error_topk_workspace_bytes(), dtype=torch.uint8, device=stats.device)
    kvq_error_topk(stats, fracs, out, ws, stream)
    return out


def fit_codebook(a, w, bits: int, max_iter: int = 50, stream=None):
    """Sensitivity-weighted nuq codebook per KV head ([KVQ] Algorithm 2): a, w device fp32
    [n_heads][n] (normalised samples, Fisher weights); returns fp32 [n_heads][2^bits]."""
    import torch
    if a.dim() != 2 or tuple(w.shape) != tuple(a.shape) or a.dtype != torch.float32 or w.dtype != torch.float32:
        raise ValueError("a and w must be fp32 [n_heads][n] of one shape")
    H, n = int(a.shape[0]), int(a.shape[1])
    out = torch.empty(H, 2 ** int(bits), dtype=torch.float32, device=a.device)
    wsb = int(_lib.lib().kvq_fit_codebook_workspace_bytes(H, n))
    ws = torch.empty(max(16, wsb), dtype=torch.uint8, device=a.device)
    _lib.check(_lib.lib().kvq_fit_codebook(_ptr(a), _ptr(w), H, n, int(bits), int(max_iter), _ptr(out), _ptr(ws),
                                           ws.numel(), _stream(stream)), "kvq_fit_codebook")
    return out


class KVCache:
    """Convenience owner of the device buffers of one cache (allocated by PyTorch) plus the
    decode workspace; every call goes through the C ABI above."""

    def __init__(self, cfg: kvq_config, codebook=None, device="cuda", stream=None, block_table=None):
        """block_table: paged caches (cfg.n_pages > 0) only, int32 [B][max_blocks] of page ids;
        default: sequence b's block blk on page b * max_blocks + blk (needs n_pages >= B * max_blocks)."""
        import torch
        self.cfg = cfg
        self.layout = kvq_layout(cfg)
        self.device = torch.device(device)
        self.base = torch.empty(int(self.layout.total_bytes), dtype=torch.uint8, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.codebook = None if codebook is None else codebook.to(self.device, torch.float32).contiguous()
        self.cache = kvq_cache_init(cfg, self.base, self.codebook, self.status, stream)
        self.block_table = None
        if cfg.n_pages > 0:
            if block_table is None:
                block_table = torch.arange(cfg.batch * cfg.max_blocks, dtype=torch.int32).view(cfg.batch, cfg.max_blocks)
            self.set_block_table(block_table)
        self.workspace = torch.empty(max(16, kvq_decode_workspace_bytes(cfg, cfg.max_blocks)),
                                     dtype=torch.uint8, device=self.device)

    @property
    def n_blocks(self) -> int:
        return int(self.cache.n_blocks)

    def append(self, k, v, dbg_varn_scales=None, stream=None):
        kvq_append_block(self.cache, k, v, dbg_varn_scales, stream)

    def truncate(self, n_blocks: int):
        kvq_truncate(self.cache, n_blocks)

    def decode(self, q, tail_k=None, tail_v=None, out=None, stream=None, n_tail=None):
        """n_tail: tokens of the tail buffers to attend when they are allocated with a larger
        capacity ([B][H_kv][capacity][128]); default: all of them."""
        import torch
        if out is None:
            out = torch.empty(q.shape[0], q.shape[1], 128, dtype=torch.float32, device=self.device)
        stride = 0 if tail_k is None else int(tail_k.shape[2])
        n_tail = stride if n_tail is None else int(n_tail)
        need = kvq_decode_workspace_bytes(self.cfg, self.n_blocks)
        if self.workspace.numel() < need:
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        kvq_decode_attn_ex(self.cache, q, tail_k if n_tail else None, tail_v if n_tail else None, n_tail,
                           max(stride, n_tail) * 128, 128, out, self.workspace, stream)
        return out

    def dequant(self, first_block: int, n_blocks: int, domain: int = 0, stream=None):
        import torch
        shape = (self.cfg.batch, self.cfg.n_kv_heads, n_blocks * 128, 128)
        ok = torch.empty(shape, dtype=torch.float32, device=self.device)
        ov = torch.empty(shape, dtype=torch.float32, device=self.device)
        kvq_dequant(self.cache, first_block, n_blocks, domain, ok, ov, stream)
        return ok, ov

    def error_stats(self, k, v, first_block: int = 0, stream=None):
        """Per-token error statistics of blocks first_block .. first_block + n - 1 against the
        inputs k, v [B][H_kv][n*128][128] they were appended from (either may be None): fp32
        [B][H_kv][n*128][4] per kind = (|x|, |x_dq| - |x|, E_T, E_D)."""
        import torch
        src = k if k is not None else v
        n_blocks = int(src.shape[2]) // 128
        for x in (k, v):
            if x is not None and (tuple(x.shape) != (self.cfg.batch, self.cfg.n_kv_heads, n_blocks * 128, 128)
                                  or x.element_size() != 2):
                raise ValueError("inputs must be [B][H_kv][n*128][128] in the cache's 16-bit input dtype")
        shape = (self.cfg.batch, self.cfg.n_kv_heads, n_blocks * 128, 4)
        sk = None if k is None else torch.empty(shape, dtype=torch.float32, device=self.device)
        sv = None if v is None else torch.empty(shape, dtype=torch.float32, device=self.device)
        kvq_error_stats(self.cache, first_block, n_blocks, k, v, sk, sv, stream)
        return sk, sv

    def calibrate_keys(self, k_calib, stream=None):
        """Offline key statistics from calibration keys [H_kv][n_tokens][128] (key_calib caches)."""
        kvq_calibrate_keys(self.cache, k_calib, stream)

    def set_block_table(self, table):
        """Binds a page table (int32 [B][max_blocks]); it is read by every later call."""
        import torch
        t = table.to(self.device, torch.int32).contiguous()
        if tuple(t.shape) != (self.cfg.batch, self.cfg.max_blocks):
            raise ValueError("block table must be [batch][max_blocks]")
        self.block_table = t
        self.cache.block_table = t.data_ptr()

    def device_status(self) -> int:
        return int(self.status.item())

    def record_view(self):
        """The records as a uint8 tensor (for checking): [B][H_kv][max_blocks][record_bytes], or
        for paged caches the pool [n_pages][H_kv][record_bytes]."""
        c = self.cfg
        rb = int(self.layout.record_bytes)
        if c.n_pages > 0:
            return self.base[:c.n_pages * c.n_kv_heads * rb].view(c.n_pages, c.n_kv_heads, rb)
        n = c.batch * c.n_kv_heads * c.max_blocks * rb
        return self.base[:n].view(c.batch, c.n_kv_heads, c.max_blocks, rb)
