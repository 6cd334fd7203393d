"""kvq_decode_attn_static: the decode entry point that takes no workspace and allocates
nothing, for callers that cannot provide device scratch memory (an engine whose device memory
is all owned by another allocator, a loop where a cudaMalloc would synchronise the device).
Its partials live in a fixed array inside the library. This file is collected last on purpose.

Checked through the C ABI: on two calls in a row its output equals the output of
kvq_decode_attn (caller workspace) bit for bit (decode is deterministic: the same kernels run
with the same split, only the partials' address differs) and lies within max-abs 2e-3 of the
oracle's fp64 attention, and a decode needing more than the fixed scratch is refused with
KVQ_ERR_CAPACITY before anything is launched."""
import ctypes as C

import numpy as np
import pytest

import oracle as O
import workloads as WL
from tests import kvq_testutil as U

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def K():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_block_gb300 as K
    return K


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


@pytest.mark.parametrize("layout", ["rows", "mma"])
def test_static_scratch_matches_workspace_decode_twice(K, layout):
    import torch
    L = K._lib
    lib = L.lib()
    # nuq3 with pre-RoPE keys and CSR outliers, several sequence splits per head
    w = WL.WORKLOADS[2].scaled(batch=1, n_kv_heads=4, n_q_heads=4, ctx=12 * 128)
    cache = U.new_cache(w, layout=layout)
    Kx, Vx = WL.blocks(w, 0, w.n_blocks)
    cache.append(U.to_device(Kx, w.dtype), U.to_device(Vx, w.dtype))
    assert K.kvq_decode_workspace_bytes(cache.cfg, cache.n_blocks) <= L.KVQ_STATIC_WORKSPACE_BYTES
    oc = O.OracleCache.for_workload(w, codebook=U.codebook_for(w)[0], layout=U.oracle_layout(layout))
    oc.append(Kx, Vx)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for step, n_tail in ((0, 5), (1, 77)):
        q = U.to_device(WL.query(w, step), w.dtype)
        tk, tv = WL.tail(w, n_tail, step)
        tk, tv = U.to_device(tk, w.dtype), U.to_device(tv, w.dtype)
        ref = torch.empty(w.batch, w.n_q_heads, 128, dtype=torch.float32, device="cuda")
        ws = cache.workspace
        st = lib.kvq_decode_attn(C.byref(cache.cache), _p(q), _p(tk), _p(tv), n_tail, _p(ref), _p(ws),
                                 ws.numel(), stream)
        assert st == L.KVQ_OK
        got = torch.full_like(ref, float("nan"))
        st = lib.kvq_decode_attn_static(C.byref(cache.cache), _p(q), _p(tk), _p(tv), n_tail, _p(got), stream)
        assert st == L.KVQ_OK, K.kvq_status_str(st)
        torch.cuda.synchronize()
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(g))
        assert np.array_equal(g, r), f"max abs difference {np.max(np.abs(g - r)):.3e}"
        exp = oc.decode(WL.query(w, step), *WL.tail(w, n_tail, step))
        assert np.max(np.abs(g.astype(np.float64) - exp)) <= TOL
    assert cache.device_status() == 0


def test_static_scratch_refuses_oversized_decode(K):
    import torch
    L = K._lib
    lib = L.lib()
    # 128 sequences x 128 query heads: the split partials need more than the fixed scratch
    cfg = K.make_config("rtn", 2, 128, 8, 128, 1)
    need = K.kvq_decode_workspace_bytes(cfg, 1)
    assert need > L.KVQ_STATIC_WORKSPACE_BYTES
    cache = K.KVCache(cfg)
    cache.cache.n_blocks = 1          # nothing is launched: the size check comes first
    q = torch.zeros(128, 128, 128, dtype=torch.float16, device="cuda")
    out = torch.zeros(128, 128, 128, dtype=torch.float32, device="cuda")
    st = lib.kvq_decode_attn_static(C.byref(cache.cache), _p(q), None, None, 0, _p(out),
                                    C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == L.KVQ_ERR_CAPACITY
    torch.cuda.synchronize()
    assert not out.any()
