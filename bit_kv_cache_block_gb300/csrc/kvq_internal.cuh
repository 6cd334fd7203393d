// Internal definitions shared by the translation units of libkvq (not installed).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "../../include/kvq.h"

namespace kvq {

constexpr int T = 128;      // tokens per block
constexpr int D = 128;      // head dim
constexpr int TILE = T * D; // elements per tile

__host__ __device__ constexpr int codes_per_word(int bits) { return 32 / bits; }
// Words per 128-code row; 3-bit tiles in the plane layout (KVQ_LAYOUT_MMA) count as 12.
__host__ __device__ constexpr int words_per_row(int bits, int layout) {
  return (bits == 3 && layout == KVQ_LAYOUT_MMA) ? 12 : (D + codes_per_word(bits) - 1) / codes_per_word(bits);
}

// 3-bit tiles ([KVQ] §9.3: 48 bytes per 128 codes) keep each code's two low bits and its high
// bit in separate planes, in the order the tensor-core decode's fragments read them. The tile
// is 8 segments of 16 tokens; a segment is 32 groups of 6 words (one lane's codes); in a group,
// slot k (0..7) of nibble word u (0..7) has its low bits in word u/2 at bit 4k + 2(u%2) and its
// high bit in word 4 + u/4 at bit 4k + ((u%4) ^ 2).
constexpr int TILE3_WORDS = 1536;

// Token t and channel c of slot k of nibble word u in group grp of segment s.
__host__ __device__ inline void tile3_code_at(int kind, int s, int grp, int u, int k, int& t, int& c) {
  const int g = grp >> 2, tq = grp & 3;
  if (kind == 0) {  // keys: group = (token t%8, channel pair class (c/2)%4)
    t = 16 * s + g + 8 * ((k >> 1) & 1);
    c = 8 * (2 * u + (k >> 2)) + 2 * tq + (k & 1);
  } else {          // values: group = (channel c%8, token class t%4)
    const int v = 2 * (k & 1) + (k >> 2);
    t = 16 * s + tq + 4 * v;
    c = 16 * u + g + 8 * ((k >> 1) & 1);
  }
}

// Word indices and bit shifts of code (t, c): low bits at (lw, ls), high bit at (hw, hs).
__host__ __device__ inline void tile3_slot(int kind, int t, int c, int& lw, int& ls, int& hw, int& hs) {
  const int s = t >> 4, tl = t & 15;
  int grp, u, k;
  if (kind == 0) {
    grp = 4 * (tl & 7) + ((c >> 1) & 3);
    u = c >> 4;
    k = 4 * ((c >> 3) & 1) + 2 * (tl >> 3) + (c & 1);
  } else {
    const int v = tl >> 2;
    grp = 4 * (c & 7) + (tl & 3);
    u = c >> 4;
    k = 4 * (v & 1) + 2 * ((c >> 3) & 1) + (v >> 1);
  }
  const int base = s * 192 + grp * 6;
  lw = base + (u >> 1);
  ls = 4 * k + 2 * (u & 1);
  hw = base + 4 + (u >> 2);
  hs = 4 * k + ((u & 3) ^ 2);
}

__device__ __forceinline__ uint32_t tile3_code(const uint32_t* w, int kind, int t, int c) {
  int lw, ls, hw, hs;
  tile3_slot(kind, t, c, lw, ls, hw, hs);
  return ((w[lw] >> ls) & 3u) | (((w[hw] >> hs) & 1u) << 2);
}
__host__ __device__ constexpr uint64_t round16(uint64_t x) { return (x + 15) & ~uint64_t(15); }

// Number of fp16 vectors of 128 in a tile's metadata region.
__host__ __device__ inline int meta_vectors(int method, int scale_group) {
  switch (method) {
    case KVQ_RTN: return 2;    // s, z
    case KVQ_NUQ: return 2;    // s, zp
    case KVQ_VARN: return 3;   // s, z, s1
    default: return scale_group == 64 ? 2 : 1;  // INT4: s per token (or per half-token)
  }
}

// Outliers per tile: ceil(frac * 16384) with frac taken as the stored fp32 value.
inline int n_outliers_for(float frac) {
  if (!(frac > 0.0f)) return 0;
  double n = (double)frac * (double)TILE;
  long long c = (long long)n;
  if ((double)c < n) ++c;
  if (c > TILE) c = TILE;
  return (int)c;
}

inline uint64_t csr_bytes_for(int n_out) {
  if (n_out == 0) return 0;
  return round16((uint64_t)n_out * 2 + (uint64_t)(T + 1) * 2 + (uint64_t)n_out);
}

// Parameters every kernel needs, passed by value.
struct Geo {
  int method, bits, B, H, Hq, G, max_blocks, in_bf16, pre_rope, n_out, W;
  int layout;   // kvq_code_layout
  int planes3;  // 3-bit tiles in bit planes (KVQ_LAYOUT_MMA)
  int vrows_ch; // value tiles hold one row per channel (KVQ_LAYOUT_MMA, 2 and 4 bits)
  uint64_t rec_bytes;
  uint32_t codes_off[2], meta_off[2], csr_off[2];
  uint64_t rope_off;
  int n_pages;          // > 0: paged cache (records addressed through `table`)
  const int32_t* table; // paged caches: device block table [B][max_blocks] (else NULL)
  int key_calib;        // NUQ keys use the calibration table at calib_off
  int sink;             // NUQ: the first token of each sequence is kept at sink_off
  uint64_t calib_off, sink_off;
  int g64;              // INT4: one scale per 64 channels (meta vectors: channels 0..63, 64..127)
  int v_csc;            // NUQ: value outliers by column (col_ptr over channels, token per entry)
  // Bound of every stage wait, in SM clocks (about 1 s by default), and a test switch under which
  // the decode's producer issues no copies, so that its waits run out (kvq_debug_stall_decode).
  long long wait_cycles;
  int dbg_stall;
};

inline Geo make_geo(const kvq_config& c, const kvq_layout_t& l) {
  Geo g;
  g.method = c.method; g.bits = c.bits; g.B = c.batch; g.H = c.n_kv_heads; g.Hq = c.n_q_heads;
  g.G = c.n_q_heads / c.n_kv_heads; g.max_blocks = c.max_blocks; g.in_bf16 = c.in_dtype == KVQ_BF16;
  g.pre_rope = c.pre_rope; g.n_out = l.n_outliers; g.W = l.words_per_row; g.rec_bytes = l.record_bytes;
  g.layout = c.layout;
  g.planes3 = c.layout == KVQ_LAYOUT_MMA && c.bits == 3;
  g.vrows_ch = c.layout == KVQ_LAYOUT_MMA && c.bits != 3;
  for (int k = 0; k < 2; ++k) {
    g.codes_off[k] = (uint32_t)l.codes_off[k];
    g.meta_off[k] = (uint32_t)l.meta_off[k];
    g.csr_off[k] = (uint32_t)l.csr_off[k];
  }
  g.rope_off = l.rope_off;
  g.n_pages = c.n_pages;
  g.table = nullptr;
  g.key_calib = c.key_calib;
  g.sink = c.sink;
  g.calib_off = l.calib_off;
  g.sink_off = l.sink_off;
  g.g64 = c.method == KVQ_INT4 && c.scale_group == 64;
  g.v_csc = c.method == KVQ_NUQ && c.v_csc;
  g.wait_cycles = 2000000000LL;
  g.dbg_stall = 0;
  return g;
}

// Programmatic dependent launch: a kernel lets the next launch in its stream (when that launch
// allows programmatic serialization) be scheduled once every CTA of this grid has executed
// launch_dependents or exited; the dependent's grid_dependency_wait returns when this grid has
// completed and its memory is visible. Both are no-ops for ordinary launches.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Raises a kernel's dynamic shared-memory limit on the current device once (the setting is
// cached per device and kernel), so repeated launches make no extra runtime calls.
inline cudaError_t ensure_smem_attr(const void* fn, size_t smem) {
  static std::mutex mu;
  struct Entry { int dev; const void* fn; size_t smem; };
  static Entry tab[128];
  static int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (tab[i].dev == dev && tab[i].fn == fn && tab[i].smem >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && n < 128) tab[n++] = Entry{dev, fn, smem};
  return e;
}

// ----------------------------------------------------------------- device helpers

__device__ __forceinline__ float load_in(const uint16_t* p, int bf16) {
  uint16_t u = *p;
  return bf16 ? __bfloat162float(__ushort_as_bfloat16(u)) : __half2float(__ushort_as_half(u));
}

__device__ __forceinline__ float in_bits_to_f32(uint16_t u, int bf16) {
  return bf16 ? __bfloat162float(__ushort_as_bfloat16(u)) : __half2float(__ushort_as_half(u));
}

__device__ __forceinline__ float h2f(uint16_t u) { return __half2float(__ushort_as_half(u)); }
__device__ __forceinline__ uint16_t f2h_rn(float x) { return __half_as_ushort(__float2half_rn(x)); }

// First device-side error wins.
__device__ __forceinline__ void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrives on an mbarrier (release semantics at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier (bytes: multiple of 16,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Non-blocking probe of an mbarrier phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of an mbarrier for at most ~`max_cycles` SM clocks. Returns false
// (and records KVQ_ERR_TIMEOUT) when the wait gives up.
// try_wait that may suspend the thread until the phase completes or about 1 ms passes, so a
// waiting warp issues a few instructions per wait instead of spinning on the issue slots of
// the warps it waits for.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Byte offset from the cache base of the record of (b, h, block): contiguous records, or for
// paged caches page table[b][block] of the pool, whose pages hold the records of all H heads.
// A table entry outside [0, n_pages) is reported as KVQ_ERR_PAGE and page 0 used instead, so a
// bad table never addresses memory outside the pool.
__device__ __forceinline__ uint64_t record_offset(const Geo& g, int b, int h, int blk, int* status) {
  if (g.n_pages <= 0) return (((uint64_t)b * g.H + h) * g.max_blocks + blk) * g.rec_bytes;
  int page = __ldg(g.table + (size_t)b * g.max_blocks + blk);
  if (page < 0 || page >= g.n_pages) {
    report(status, KVQ_ERR_PAGE);
    page = 0;
  }
  return ((uint64_t)page * g.H + h) * g.rec_bytes;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status,
                                                  long long max_cycles = 2000000000LL) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (clock64() - t0 > max_cycles) {
      report(status, KVQ_ERR_TIMEOUT);
      return false;
    }
  }
}

// Waits like mbar_wait_bounded, for warps that run ahead of the ones they feed (producers and
// helpers): polls with the non-blocking probe and sleeps ~SLEEP_NS between probes, so that a
// waiting warp neither takes issue slots nor keeps the barrier unit busy for the warps doing the
// work. A probe that fails records KVQ_ERR_TIMEOUT after ~max_cycles SM clocks.
template <int SLEEP_NS = 64>
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, int* status,
                                                  long long max_cycles = 2000000000LL) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(SLEEP_NS);
    if (mbar_test_wait(bar, parity)) return true;
    if (clock64() - t0 > max_cycles) {
      report(status, KVQ_ERR_TIMEOUT);
      return false;
    }
  }
}

}  // namespace kvq
