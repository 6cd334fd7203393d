// Host side of the C ABI: argument checks, layout arithmetic and kernel launches.
#include <atomic>
#include <cmath>
#include <cstring>

#include "kvq_internal.cuh"

cudaError_t kvq_launch_append(const kvq::Geo& g, const uint16_t* k, const uint16_t* v, int n_new, int blk0,
                              uint8_t* base, const float* codebook, float* dbg, int* status, int varn_iters,
                              int hadamard, cudaStream_t st);
cudaError_t kvq_launch_decode(const kvq::Geo& g, const uint8_t* base, const float* codebook, const uint16_t* q,
                              const uint16_t* tail_k, const uint16_t* tail_v, int n_tail, long long tail_bh,
                              long long tail_tok, int n_blocks,
                              int n_split, float* ws, float* out, int* status, int hadamard, cudaStream_t st);
size_t kvq_decode_ws_floats(const kvq::Geo& g, int n_blocks, int v1_splits);
size_t kvq_decode_kernel_smem(const kvq::Geo& g);
cudaError_t kvq_launch_dequant(const kvq::Geo& g, const uint8_t* base, const float* codebook, int first, int n,
                               int domain, int hadamard, float* out_k, float* out_v, int* status, cudaStream_t st);
cudaError_t kvq_launch_rope_init(float2* tab, int max_blocks, double theta, cudaStream_t st);
cudaError_t kvq_launch_calibrate(const kvq::Geo& g, uint8_t* base, const uint16_t* k, int n_tokens, int rank,
                                 cudaStream_t st);
cudaError_t kvq_static_workspace(float** ptr, size_t* n_floats);
cudaError_t kvq_launch_error_stats(const kvq::Geo& g, const uint8_t* base, const float* codebook, int first, int n,
                                   int hadamard, const uint16_t* in_k, const uint16_t* in_v, float* st_k, float* st_v,
                                   int* status, cudaStream_t st);
size_t kvq_topk_ws_bytes();
size_t kvq_fit_ws_bytes(int n_heads, long long n);
cudaError_t kvq_launch_fit(const float* a, const float* w, int n_heads, long long n, int bits, int max_iter, float* c,
                           void* ws, cudaStream_t st);
cudaError_t kvq_launch_topk(const float* stats, unsigned long long n, const unsigned long long* k, int nf, double* out,
                            void* ws, cudaStream_t st);

namespace {

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

kvq_status check_config(const kvq_config* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->method < KVQ_RTN || c->method > KVQ_INT4) return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != KVQ_HEAD_DIM || c->block != KVQ_BLOCK) return KVQ_ERR_UNSUPPORTED;
  if (c->batch < 1 || c->n_kv_heads < 1 || c->n_q_heads < 1 || c->max_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (c->batch > 32767 || c->n_kv_heads > 65535 || c->n_q_heads > 65535 || c->max_blocks > (1 << 24))
    return KVQ_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (c->n_q_heads / c->n_kv_heads > KVQ_MAX_GROUP) return KVQ_ERR_UNSUPPORTED;
  if (c->in_dtype != KVQ_F16 && c->in_dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARG;
  if ((c->bits < 2 || c->bits > 4) && !(c->method == KVQ_INT4 && c->bits == 8)) return KVQ_ERR_UNSUPPORTED;
  if (c->layout != KVQ_LAYOUT_ROWS && c->layout != KVQ_LAYOUT_MMA) return KVQ_ERR_INVALID_ARG;
  if (c->n_pages < 0 || c->n_pages > (1 << 28)) return KVQ_ERR_INVALID_ARG;
  if ((c->key_calib != 0 && c->key_calib != 1) || (c->sink != 0 && c->sink != 1)) return KVQ_ERR_INVALID_ARG;
  if ((c->key_calib || c->sink) && c->method != KVQ_NUQ) return KVQ_ERR_UNSUPPORTED;
  if (c->method == KVQ_INT4 && c->bits != 4 && c->bits != 8) return KVQ_ERR_UNSUPPORTED;
  if (c->scale_group != 0 && c->scale_group != 128 && c->scale_group != 64) return KVQ_ERR_INVALID_ARG;
  if (c->scale_group == 64 && c->method != KVQ_INT4) return KVQ_ERR_UNSUPPORTED;
  if (c->v_csc != 0 && c->v_csc != 1) return KVQ_ERR_INVALID_ARG;
  if (c->v_csc && c->method != KVQ_NUQ) return KVQ_ERR_UNSUPPORTED;
  if (c->pre_rope != 0 && c->pre_rope != 1) return KVQ_ERR_INVALID_ARG;
  if (c->pre_rope && c->method != KVQ_NUQ) return KVQ_ERR_UNSUPPORTED;
  if (c->pre_rope && !(c->rope_theta > 1.0)) return KVQ_ERR_INVALID_ARG;
  if (c->method == KVQ_NUQ && !(c->outlier_frac >= 0.0f && c->outlier_frac <= 1.0f)) return KVQ_ERR_INVALID_ARG;
  if (c->method == KVQ_VARN) {
    if (c->varn_iters < 0 || c->varn_iters > 64) return KVQ_ERR_INVALID_ARG;
    if (c->hadamard != 0 && c->hadamard != 1) return KVQ_ERR_INVALID_ARG;
  }
  return KVQ_OK;
}

// Runs `fn` with the cache's device current, then restores the caller's device.
template <class F>
kvq_status on_device(int dev, F fn) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cur != dev && cudaSetDevice(dev) != cudaSuccess) return KVQ_ERR_CUDA;
  cudaError_t e = fn();
  if (cur != dev) cudaSetDevice(cur);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int hadamard_of(const kvq_config& c) { return c.method == KVQ_VARN ? c.hadamard : 0; }

// Test switch of kvq_debug_stall_decode (process-wide; read when a decode is launched).
std::atomic<int> g_dbg_stall{0};

// A decode's kernel parameters under the test switch: no copies, waits bounded at ~1 ms.
void apply_debug(kvq::Geo& g) {
  if (g_dbg_stall.load(std::memory_order_relaxed)) {
    g.dbg_stall = 1;
    g.wait_cycles = 2000000LL;
  }
}

// Kernel parameters of a cache; paged caches need their block table (non-null, 4-byte aligned).
kvq_status geo_of(const kvq_cache* cache, kvq::Geo& g) {
  g = kvq::make_geo(cache->cfg, cache->lay);
  if (cache->cfg.n_pages > 0) {
    if (!cache->block_table) return KVQ_ERR_INVALID_ARG;
    if (!aligned(cache->block_table, 4)) return KVQ_ERR_ALIGNMENT;
    g.table = cache->block_table;
  }
  return KVQ_OK;
}

}  // namespace

extern "C" {

const char* kvq_status_str(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CAPACITY: return "capacity exceeded";
    case KVQ_ERR_ALIGNMENT: return "misaligned pointer";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_TIMEOUT: return "device wait timed out";
    case KVQ_ERR_PAGE: return "block table entry out of range";
  }
  return "unknown status";
}

uint64_t kvq_dense_kv_bytes(int64_t n_layers, int64_t n_heads, int64_t head_dim, int64_t elem_bytes,
                            int64_t batch, int64_t seq_len) {
  return 2ull * (uint64_t)n_layers * (uint64_t)n_heads * (uint64_t)head_dim * (uint64_t)elem_bytes *
         (uint64_t)batch * (uint64_t)seq_len;
}

kvq_status kvq_layout(const kvq_config* c, kvq_layout_t* out) {
  kvq_status s = check_config(c);
  if (s != KVQ_OK) return s;
  if (!out) return KVQ_ERR_INVALID_ARG;
  kvq_layout_t l;
  std::memset(&l, 0, sizeof(l));
  l.words_per_row = kvq::words_per_row(c->bits, c->layout);
  l.n_outliers = c->method == KVQ_NUQ ? kvq::n_outliers_for(c->outlier_frac) : 0;
  const uint64_t codes = (uint64_t)kvq::T * l.words_per_row * 4;
  const uint64_t meta = (uint64_t)kvq::meta_vectors(c->method, c->scale_group) * kvq::T * 2;
  const uint64_t csr = kvq::csr_bytes_for(l.n_outliers);
  uint64_t off = 0;
  for (int k = 0; k < 2; ++k) {
    l.codes_off[k] = off; l.codes_bytes[k] = codes; off += codes;
    l.meta_off[k] = off; l.meta_bytes[k] = meta; off += meta;
    l.csr_off[k] = off; l.csr_bytes[k] = csr; off += csr;
  }
  l.record_bytes = off;
  l.records_bytes = c->n_pages > 0 ? (uint64_t)c->n_pages * c->n_kv_heads * l.record_bytes
                                   : (uint64_t)c->batch * c->n_kv_heads * (uint64_t)c->max_blocks * l.record_bytes;
  l.rope_off = (l.records_bytes + 127) & ~uint64_t(127);
  l.rope_bytes = c->pre_rope ? (uint64_t)((c->max_blocks + 1) + kvq::T) * 64 * 8 : 0;
  uint64_t end = c->pre_rope ? l.rope_off + l.rope_bytes : l.records_bytes;
  if (c->key_calib) {
    l.calib_off = (end + 127) & ~uint64_t(127);
    l.calib_bytes = (uint64_t)c->n_kv_heads * kvq::D * (4 + 2 + 2);
    end = l.calib_off + l.calib_bytes;
  }
  if (c->sink) {
    l.sink_off = (end + 127) & ~uint64_t(127);
    l.sink_bytes = (uint64_t)c->batch * c->n_kv_heads * 2 * kvq::D * 2;
    end = l.sink_off + l.sink_bytes;
  }
  l.total_bytes = end;
  l.format_version = KVQ_FORMAT_VERSION;
  // every cache must be decodable by the CUDA-core decode (large outlier fractions make its
  // three-record ring outgrow the 227 KB of shared memory one CTA may use)
  if (kvq_decode_kernel_smem(kvq::make_geo(*c, l)) > (size_t)227 * 1024) return KVQ_ERR_UNSUPPORTED;
  *out = l;
  return KVQ_OK;
}

kvq_status kvq_cache_init(kvq_cache* cache, const kvq_config* cfg, void* dev_base, size_t bytes,
                          const float* dev_codebook, int32_t* dev_status, cudaStream_t stream) {
  if (!cache || !cfg || !dev_base || !dev_status) return KVQ_ERR_INVALID_ARG;
  kvq_layout_t l;
  kvq_status s = kvq_layout(cfg, &l);
  if (s != KVQ_OK) return s;
  if (bytes < l.total_bytes) return KVQ_ERR_CAPACITY;
  if (!aligned(dev_base, 128) || !aligned(dev_status, 4)) return KVQ_ERR_ALIGNMENT;
  if (cfg->method == KVQ_NUQ) {
    if (!dev_codebook) return KVQ_ERR_INVALID_ARG;
    if (!aligned(dev_codebook, 16)) return KVQ_ERR_ALIGNMENT;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  kvq_cache c;
  std::memset(&c, 0, sizeof(c));
  c.cfg = *cfg;
  c.lay = l;
  c.base = dev_base;
  c.codebook = cfg->method == KVQ_NUQ ? dev_codebook : nullptr;
  c.dev_status = dev_status;
  c.n_blocks = 0;
  c.device = dev;
  s = on_device(dev, [&]() -> cudaError_t {
    cudaError_t e = cudaMemsetAsync(dev_status, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    if (cfg->pre_rope)
      e = kvq_launch_rope_init(reinterpret_cast<float2*>(static_cast<uint8_t*>(dev_base) + l.rope_off),
                               cfg->max_blocks, cfg->rope_theta, stream);
    return e;
  });
  if (s != KVQ_OK) return s;
  *cache = c;
  return KVQ_OK;
}

kvq_status kvq_append_block(kvq_cache* cache, const void* k, const void* v, int32_t n_blocks,
                            float* dbg_varn_scales, cudaStream_t stream) {
  if (!cache || !cache->base || !k || !v) return KVQ_ERR_INVALID_ARG;
  if (n_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (check_config(&cache->cfg) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16)) return KVQ_ERR_ALIGNMENT;
  if (dbg_varn_scales && !aligned(dbg_varn_scales, 16)) return KVQ_ERR_ALIGNMENT;
  if (n_blocks > 65535) return KVQ_ERR_INVALID_ARG;
  if ((int64_t)cache->n_blocks + n_blocks > cache->cfg.max_blocks) return KVQ_ERR_CAPACITY;
  if (cache->cfg.key_calib && !cache->calibrated) return KVQ_ERR_INVALID_ARG;
  kvq::Geo g;
  if (kvq_status gs = geo_of(cache, g); gs != KVQ_OK) return gs;
  float* dbg = cache->cfg.method == KVQ_VARN ? dbg_varn_scales : nullptr;
  kvq_status s = on_device(cache->device, [&]() {
    return kvq_launch_append(g, static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), n_blocks,
                             cache->n_blocks, static_cast<uint8_t*>(cache->base), cache->codebook, dbg,
                             cache->dev_status, cache->cfg.varn_iters, hadamard_of(cache->cfg), stream);
  });
  if (s == KVQ_OK) cache->n_blocks += n_blocks;
  return s;
}

kvq_status kvq_calibrate_keys(kvq_cache* cache, const void* k_calib, int32_t n_tokens, cudaStream_t stream) {
  if (!cache || !cache->base || !k_calib) return KVQ_ERR_INVALID_ARG;
  if (check_config(&cache->cfg) != KVQ_OK || !cache->cfg.key_calib) return KVQ_ERR_INVALID_ARG;
  if (n_tokens < 2 || n_tokens > (1 << 24)) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k_calib, 16)) return KVQ_ERR_ALIGNMENT;
  // rank of tau among the |k| of tokens 1 .. n_tokens-1, ascending (1-based); 0: no threshold
  const double f = (double)cache->cfg.outlier_frac, m = (double)(n_tokens - 1);
  int rank = 0;
  if (f > 0.0) {
    rank = (int)std::ceil((1.0 - f) * m);
    if (rank < 1) rank = 1;
  }
  const kvq::Geo g = kvq::make_geo(cache->cfg, cache->lay);
  kvq_status s = on_device(cache->device, [&]() {
    return kvq_launch_calibrate(g, static_cast<uint8_t*>(cache->base), static_cast<const uint16_t*>(k_calib),
                                n_tokens, rank, stream);
  });
  if (s == KVQ_OK) cache->calibrated = 1;
  return s;
}

kvq_status kvq_truncate(kvq_cache* cache, int32_t n_blocks) {
  if (!cache) return KVQ_ERR_INVALID_ARG;
  if (n_blocks < 0 || n_blocks > cache->n_blocks) return KVQ_ERR_INVALID_ARG;
  cache->n_blocks = n_blocks;
  return KVQ_OK;
}

kvq_status kvq_debug_stall_decode(int32_t enable) {
  if (enable != 0 && enable != 1) return KVQ_ERR_INVALID_ARG;
  g_dbg_stall.store(enable, std::memory_order_relaxed);
  return KVQ_OK;
}

kvq_status kvq_reset(kvq_cache* cache) { return kvq_truncate(cache, 0); }

int32_t kvq_decode_splits(const kvq_config* cfg, int32_t n_blocks) {
  if (!cfg || n_blocks <= 0) return 0;
  const int64_t heads = (int64_t)cfg->batch * cfg->n_kv_heads;
  const int64_t target = 1216;  // CTAs to aim for: 8 per SM of a 152-SM part
  int64_t s = (target + heads - 1) / heads;
  if (s > n_blocks) s = n_blocks;
  if (s > 1024) s = 1024;
  if (s < 1) s = 1;
  return (int32_t)s;
}

kvq_status kvq_decode_workspace_bytes(const kvq_config* cfg, int32_t n_blocks, size_t* out) {
  kvq_layout_t l;
  kvq_status s = kvq_layout(cfg, &l);
  if (s != KVQ_OK) return s;
  if (!out || n_blocks < 0) return KVQ_ERR_INVALID_ARG;
  const kvq::Geo g = kvq::make_geo(*cfg, l);
  *out = kvq_decode_ws_floats(g, n_blocks, kvq_decode_splits(cfg, n_blocks)) * sizeof(float);
  return KVQ_OK;
}

uint64_t kvq_decode_bytes(const kvq_config* cfg, int32_t n_blocks) {
  kvq_layout_t l;
  if (kvq_layout(cfg, &l) != KVQ_OK || n_blocks < 0) return 0;
  uint64_t per_tile_pair = 0;
  for (int k = 0; k < 2; ++k) {
    per_tile_pair += l.codes_bytes[k] + l.meta_bytes[k];
    if (l.n_outliers) per_tile_pair += 3ull * l.n_outliers + 2ull * (kvq::T + 1);
  }
  return per_tile_pair * (uint64_t)n_blocks * cfg->batch * cfg->n_kv_heads;
}

kvq_status kvq_decode_attn(const kvq_cache* cache, const void* q, const void* tail_k, const void* tail_v,
                           int32_t n_tail, float* out, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  return kvq_decode_attn_ex(cache, q, tail_k, tail_v, n_tail, (int64_t)n_tail * KVQ_HEAD_DIM, KVQ_HEAD_DIM, out,
                            workspace, workspace_bytes, stream);
}

kvq_status kvq_decode_attn_ex(const kvq_cache* cache, const void* q, const void* tail_k, const void* tail_v,
                              int32_t n_tail, int64_t tail_bh_stride, int64_t tail_token_stride, float* out,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!cache || !cache->base || !q || !out) return KVQ_ERR_INVALID_ARG;
  if (check_config(&cache->cfg) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  if (n_tail < 0 || n_tail >= KVQ_BLOCK) return KVQ_ERR_INVALID_ARG;
  if (n_tail > 0) {  // strides in elements, multiples of 8 (16-byte rows), within 2^40
    if (tail_bh_stride < 0 || tail_token_stride < KVQ_HEAD_DIM) return KVQ_ERR_INVALID_ARG;
    if (tail_bh_stride > ((int64_t)1 << 40) || tail_token_stride > ((int64_t)1 << 40)) return KVQ_ERR_INVALID_ARG;
    if ((tail_bh_stride & 7) || (tail_token_stride & 7)) return KVQ_ERR_ALIGNMENT;
  }
  if (n_tail > 0 && (!tail_k || !tail_v)) return KVQ_ERR_INVALID_ARG;
  const int nb = cache->n_blocks;
  if (nb + n_tail == 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16)) return KVQ_ERR_ALIGNMENT;
  if (n_tail > 0 && (!aligned(tail_k, 16) || !aligned(tail_v, 16))) return KVQ_ERR_ALIGNMENT;
  kvq::Geo g;
  if (kvq_status gs = geo_of(cache, g); gs != KVQ_OK) return gs;
  const int S = kvq_decode_splits(&cache->cfg, nb);
  const size_t need = kvq_decode_ws_floats(g, nb, S) * sizeof(float);
  if (nb > 0) {
    if (!workspace) return KVQ_ERR_INVALID_ARG;
    if (workspace_bytes < need) return KVQ_ERR_CAPACITY;
    if (!aligned(workspace, 16)) return KVQ_ERR_ALIGNMENT;
  }
  return on_device(cache->device, [&]() {
    apply_debug(g);
    return kvq_launch_decode(g, static_cast<const uint8_t*>(cache->base), cache->codebook,
                             static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(tail_k),
                             static_cast<const uint16_t*>(tail_v), n_tail, tail_bh_stride, tail_token_stride, nb, S,
                             static_cast<float*>(workspace),
                             out, cache->dev_status, hadamard_of(cache->cfg), stream);
  });
}

kvq_status kvq_decode_attn_static(const kvq_cache* cache, const void* q, const void* tail_k, const void* tail_v,
                                  int32_t n_tail, float* out, cudaStream_t stream) {
  if (!cache || !cache->base || !q || !out) return KVQ_ERR_INVALID_ARG;
  if (check_config(&cache->cfg) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  if (n_tail < 0 || n_tail >= KVQ_BLOCK) return KVQ_ERR_INVALID_ARG;
  if (n_tail > 0 && (!tail_k || !tail_v)) return KVQ_ERR_INVALID_ARG;
  const int nb = cache->n_blocks;
  if (nb + n_tail == 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16)) return KVQ_ERR_ALIGNMENT;
  if (n_tail > 0 && (!aligned(tail_k, 16) || !aligned(tail_v, 16))) return KVQ_ERR_ALIGNMENT;
  kvq::Geo g;
  if (kvq_status gs = geo_of(cache, g); gs != KVQ_OK) return gs;
  const int S = kvq_decode_splits(&cache->cfg, nb);
  const size_t need = kvq_decode_ws_floats(g, nb, S) * sizeof(float);
  if (need > KVQ_STATIC_WORKSPACE_BYTES) return KVQ_ERR_CAPACITY;
  kvq_status cap = KVQ_OK;
  kvq_status s = on_device(cache->device, [&]() -> cudaError_t {
    float* ws = nullptr;
    size_t n_floats = 0;
    cudaError_t e = kvq_static_workspace(&ws, &n_floats);
    if (e != cudaSuccess) return e;
    if (need > n_floats * sizeof(float)) {
      cap = KVQ_ERR_CAPACITY;
      return cudaSuccess;
    }
    apply_debug(g);
    return kvq_launch_decode(g, static_cast<const uint8_t*>(cache->base), cache->codebook,
                             static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(tail_k),
                             static_cast<const uint16_t*>(tail_v), n_tail, (long long)n_tail * kvq::D, kvq::D, nb, S,
                             ws, out, cache->dev_status,
                             hadamard_of(cache->cfg), stream);
  });
  return s != KVQ_OK ? s : cap;
}

kvq_status kvq_dequant(const kvq_cache* cache, int32_t first_block, int32_t n_blocks, int32_t domain, float* out_k,
                       float* out_v, cudaStream_t stream) {
  if (!cache || !cache->base) return KVQ_ERR_INVALID_ARG;
  if (check_config(&cache->cfg) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  if (first_block < 0 || n_blocks < 1 || (int64_t)first_block + n_blocks > cache->n_blocks)
    return KVQ_ERR_INVALID_ARG;
  if (n_blocks > 65535) return KVQ_ERR_INVALID_ARG;
  if (domain != 0 && domain != 1) return KVQ_ERR_INVALID_ARG;
  if (!out_k && !out_v) return KVQ_ERR_INVALID_ARG;
  if ((out_k && !aligned(out_k, 16)) || (out_v && !aligned(out_v, 16))) return KVQ_ERR_ALIGNMENT;
  kvq::Geo g;
  if (kvq_status gs = geo_of(cache, g); gs != KVQ_OK) return gs;
  return on_device(cache->device, [&]() {
    return kvq_launch_dequant(g, static_cast<const uint8_t*>(cache->base), cache->codebook, first_block, n_blocks,
                              domain, hadamard_of(cache->cfg), out_k, out_v, cache->dev_status, stream);
  });
}

kvq_status kvq_error_stats(const kvq_cache* cache, const void* k, const void* v, int32_t first_block,
                           int32_t n_blocks, float* stats_k, float* stats_v, cudaStream_t stream) {
  if (!cache || !cache->base) return KVQ_ERR_INVALID_ARG;
  if (check_config(&cache->cfg) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  if (first_block < 0 || n_blocks < 1 || (int64_t)first_block + n_blocks > cache->n_blocks)
    return KVQ_ERR_INVALID_ARG;
  if (n_blocks > 65535) return KVQ_ERR_INVALID_ARG;
  if (!k != !stats_k || !v != !stats_v || (!k && !v)) return KVQ_ERR_INVALID_ARG;
  for (const void* p : {k, v, (const void*)stats_k, (const void*)stats_v})
    if (p && !aligned(p, 16)) return KVQ_ERR_ALIGNMENT;
  kvq::Geo g;
  if (kvq_status gs = geo_of(cache, g); gs != KVQ_OK) return gs;
  return on_device(cache->device, [&]() {
    return kvq_launch_error_stats(g, static_cast<const uint8_t*>(cache->base), cache->codebook, first_block, n_blocks,
                                  hadamard_of(cache->cfg), static_cast<const uint16_t*>(k),
                                  static_cast<const uint16_t*>(v), stats_k, stats_v, cache->dev_status, stream);
  });
}

size_t kvq_error_topk_workspace_bytes(void) { return kvq_topk_ws_bytes(); }

size_t kvq_fit_codebook_workspace_bytes(int32_t n_heads, int64_t n) {
  if (n_heads < 1 || n < 1 || n > ((int64_t)1 << 30)) return 0;
  return kvq_fit_ws_bytes(n_heads, n);
}

kvq_status kvq_fit_codebook(const float* a, const float* w, int32_t n_heads, int64_t n, int32_t bits,
                            int32_t max_iter, float* codebook, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  if (!a || !w || !codebook || !workspace) return KVQ_ERR_INVALID_ARG;
  if (n_heads < 1 || n_heads > 65535 || n < 1 || n > ((int64_t)1 << 30)) return KVQ_ERR_INVALID_ARG;
  if (bits < 1 || bits > 4 || max_iter < 1 || max_iter > 10000) return KVQ_ERR_INVALID_ARG;
  if (workspace_bytes < kvq_fit_ws_bytes(n_heads, n)) return KVQ_ERR_CAPACITY;
  if (!aligned(a, 4) || !aligned(w, 4) || !aligned(codebook, 4) || !aligned(workspace, 16)) return KVQ_ERR_ALIGNMENT;
  return kvq_launch_fit(a, w, n_heads, n, bits, max_iter, codebook, workspace, stream) == cudaSuccess ? KVQ_OK
                                                                                                   : KVQ_ERR_CUDA;
}

kvq_status kvq_error_topk(const float* stats, int64_t n_rows, const double* fracs, int32_t n_fracs, double* out,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!stats || !fracs || !out || !workspace) return KVQ_ERR_INVALID_ARG;
  if (n_rows < 1 || n_rows > (int64_t)0xffffffffLL) return KVQ_ERR_INVALID_ARG;
  if (n_fracs < 1 || n_fracs > KVQ_TOPK_MAX_FRACS) return KVQ_ERR_INVALID_ARG;
  if (workspace_bytes < kvq_topk_ws_bytes()) return KVQ_ERR_CAPACITY;
  if (!aligned(stats, 16) || !aligned(out, 8) || !aligned(workspace, 16)) return KVQ_ERR_ALIGNMENT;
  unsigned long long kk[KVQ_TOPK_MAX_FRACS];
  for (int f = 0; f < n_fracs; ++f) {
    const double fr = fracs[f];
    if (!(fr > 0.0 && fr <= 1.0)) return KVQ_ERR_INVALID_ARG;
    double kd = std::ceil(fr * (double)n_rows);
    if (kd > (double)n_rows) kd = (double)n_rows;
    kk[f] = (unsigned long long)kd;
  }
  return kvq_launch_topk(stats, (unsigned long long)n_rows, kk, n_fracs, out, workspace, stream) == cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

}  // extern "C"
