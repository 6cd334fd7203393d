// Append: quantize new 128-token blocks of K and V into packed cache records.
//
// One CTA of 256 threads per tile (b, h, block, K|V). The tile is staged once from HBM into
// shared memory as fp32 (128 x 129, padded rows), then:
//   RTN  : per-group min/max -> fp16 s, z -> q = clamp(rne(x/s - z)) -> pack
//          ([KVN] preliminaries, KIVI representation (K_q + z) * s; [KVQ] §1.2, §3.1)
//   VARN : FWHT-128 on each token row, Sinkhorn-style variance normalisation (columns, then
//          rows, repeated), merge of the scales, RTN, second scale s1 ([KVN] method steps 1-4)
//   INT4 : per-token (or per-64-channel) absmax/(2^(b-1)-1) -> fp16 scale -> q = clamp(rne(x/s)) -> b-bit two's complement (b = 4, 8)
//          ([TQ] §2.1, §4.2 quantize_kv_block)
//   NUQ  : exact top-n |x| selection (radix select on the fp16 magnitude, ties to the lower
//          flat index) -> CSR (value tiles of v_csc caches: CSC); centre/half-range of the
//          non-outliers -> nearest codebook entry ([KVQ] §3.3-3.4, §3.8 Algorithm 1 steps 1-4)
// Every step that decides a code or a stored fp16 value uses single IEEE fp32 operations
// (explicit _rn intrinsics, no contraction) in a fixed order, so the records are bit-exact
// with a plain restatement of the definitions.
#include "kvq_internal.cuh"

namespace kvq {

constexpr int AP_THREADS = 256;
constexpr int XS = 129;  // padded row stride of the fp32 tile in shared memory

struct AppendArgs {
  Geo g;
  const uint16_t* k;
  const uint16_t* v;
  int n_new;
  int blk0;
  uint8_t* base;
  const float* codebook;
  float* dbg;
  int* status;
  int varn_iters;
  int hadamard;
};

struct AppendSmem {
  float x[T * XS];
  uint8_t codes[T * D];
  float gs[T], gz[T], gs1[T];     // per-group scale / zero (fp32 copies of the fp16 values)
  float racc[T], cacc[T];         // VarN token / channel scales
  uint32_t mask[TILE / 32];       // NUQ outlier bitmap, flat index t*128 + c
  int hist[256];
  int scan[16];
  int sel[4];
  float cb[16];
};

__device__ __forceinline__ int block_excl_scan(int v, int* sh, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < AP_THREADS / 32 ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < AP_THREADS / 32) sh[lane] = s;
  }
  __syncthreads();
  int excl = x - v + (wid > 0 ? sh[wid - 1] : 0);
  if (total) *total = sh[AP_THREADS / 32 - 1];
  __syncthreads();
  return excl;
}

// Element j (0..63) of half `half` of group `gi`: axis 0 = per channel (group = channel,
// elements over tokens), axis 1 = per token.
__device__ __forceinline__ int gidx(int axis, int gi, int half, int j) {
  int e = half * 64 + j;
  return axis == 0 ? e * XS + gi : gi * XS + e;
}

// RTN of the tile in sm->x along `axis`: fills gs/gz and the fp16 meta (s at m16[0..127],
// z at m16[128..255]) and sm->codes.
__device__ void rtn_tile(AppendSmem* sm, int axis, int bits, uint16_t* m16) {
  const int tid = threadIdx.x, gi = tid >> 1, half = tid & 1;
  float mx = -INFINITY, mn = INFINITY;
  for (int j = 0; j < 64; ++j) {
    float v = sm->x[gidx(axis, gi, half, j)];
    mx = fmaxf(mx, v);
    mn = fminf(mn, v);
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
  if (half == 0) {
    float s32 = __fdiv_rn(__fsub_rn(mx, mn), (float)((1 << bits) - 1));
    uint16_t s16 = f2h_rn(s32);
    if ((s16 & 0x7fff) == 0) s16 = 0x3c00;  // a zero scale becomes 1
    float sf = h2f(s16);
    uint16_t z16 = f2h_rn(__fdiv_rn(mn, sf));
    sm->gs[gi] = sf;
    sm->gz[gi] = h2f(z16);
    m16[gi] = s16;
    m16[T + gi] = z16;
  }
  __syncthreads();
  const float qmax = (float)((1 << bits) - 1);
  for (int e = tid; e < TILE; e += AP_THREADS) {
    int t = e >> 7, c = e & 127;
    int gg = axis == 0 ? c : t;
    float q = rintf(__fsub_rn(__fdiv_rn(sm->x[t * XS + c], sm->gs[gg]), sm->gz[gg]));
    q = fminf(fmaxf(q, 0.0f), qmax);
    sm->codes[e] = (uint8_t)q;
  }
  __syncthreads();
}

// Warp-wide selection over PER * 32 histogram bins (lane l holds bins PER*l .. PER*l + PER-1):
// the highest bin b such that base + (count in bins above b) < target <= base + (count in bins b
// and above); bin 0 when no bin qualifies. The lane holding b returns true with cum = base +
// count above b. Same result as scanning the bins one by one from the top.
template <int PER>
__device__ __forceinline__ bool select_bin(const int* hist, int base, int target, int lane, int& cum, int& bin) {
  int hv[PER], sl = 0;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    hv[k] = hist[PER * lane + k];
    sl += hv[k];
  }
  int incl = sl;  // bins of this lane and of the lanes above it
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  const int above = base + incl - sl;
  const bool here = (above < target && base + incl >= target) || (lane == 0 && base + incl < target);
  if (!here) return false;
  cum = above;
  int b = PER - 1;
#pragma unroll
  for (int k = PER - 1; k > 0; --k) {
    if (b == k) {
      if (cum + hv[k] >= target) break;
      cum += hv[k];
      b = k - 1;
    }
  }
  bin = PER * lane + b;
  return true;
}

// Pack sm->codes (token-major, [t][c]) into words. Rows: code i of a row at bits
// [b*(i%n)+b-1 : b*(i%n)] of word i/n, n = floor(32/b); one row per token, or (transpose) one row
// per channel (its codes for the 128 tokens). planes: the 3-bit plane layout of tile3_slot (one
// thread per output word; kind 0 keys, 1 values).
__device__ void pack_tile(const AppendSmem* sm, int bits, bool transpose, bool planes, int kind, uint32_t* dst) {
  if (planes) {  // thread = one 6-word group (segment s, group grp): each of its 64 codes read once
    for (int gi = threadIdx.x; gi < TILE3_WORDS / 6; gi += AP_THREADS) {
      const int s = gi >> 5, grp = gi & 31;
      uint32_t w[6] = {0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          int t, c;
          tile3_code_at(kind, s, grp, u, k, t, c);
          const uint32_t q = sm->codes[t * D + c];
          w[u >> 1] |= (q & 3u) << (4 * k + 2 * (u & 1));              // low bits
          w[4 + (u >> 2)] |= ((q >> 2) & 1u) << (4 * k + ((u & 3) ^ 2));  // high bit
        }
#pragma unroll
      for (int o = 0; o < 6; ++o) dst[gi * 6 + o] = w[o];
    }
    return;
  }
  const int n = 32 / bits, W = (D + n - 1) / n;
  for (int it = threadIdx.x; it < T * W; it += AP_THREADS) {
    int r = it / W, w = it - r * W;
    uint32_t word = 0;
    for (int j = 0; j < n; ++j) {
      int i = w * n + j;
      if (i < D) {
        uint32_t code = transpose ? sm->codes[i * D + r] : sm->codes[r * D + i];
        word |= (code & ((1u << bits) - 1)) << (bits * j);
      }
    }
    dst[it] = word;
  }
}

// In-place FWHT of every row (Sylvester order), then scaling by 1/sqrt(128).
__device__ void fwht_rows(AppendSmem* sm) {
  const int tid = threadIdx.x;
  for (int hh = 1; hh < D; hh <<= 1) {
    for (int it = tid; it < T * (D / 2); it += AP_THREADS) {
      int t = it >> 6, j = it & 63;
      int i0 = (j / hh) * (2 * hh) + (j % hh);
      float a = sm->x[t * XS + i0], b = sm->x[t * XS + i0 + hh];
      sm->x[t * XS + i0] = __fadd_rn(a, b);
      sm->x[t * XS + i0 + hh] = __fsub_rn(a, b);
    }
    __syncthreads();
  }
  const float inv = 0.08838834764831845f;  // 1/sqrt(128)
  for (int e = tid; e < TILE; e += AP_THREADS) {
    int t = e >> 7, c = e & 127;
    sm->x[t * XS + c] = __fmul_rn(sm->x[t * XS + c], inv);
  }
  __syncthreads();
}

// Population std of each group along `axis`, divide the group by it, multiply the
// accumulated scale. Two threads per group, four partial sums each.
__device__ void varn_axis(AppendSmem* sm, int axis, float* acc) {
  const int tid = threadIdx.x, gi = tid >> 1, half = tid & 1;
  float p[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < 64; ++j) p[j & 3] += sm->x[gidx(axis, gi, half, j)];
  float s = (p[0] + p[1]) + (p[2] + p[3]);
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  const float mean = s * (1.0f / 128.0f);
  float r[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < 64; ++j) {
    float d = sm->x[gidx(axis, gi, half, j)] - mean;
    r[j & 3] = fmaf(d, d, r[j & 3]);
  }
  float ss = (r[0] + r[1]) + (r[2] + r[3]);
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  const float sigma = sqrtf(ss * (1.0f / 128.0f));
  if (sigma > 0.0f) {
    for (int j = 0; j < 64; ++j) {
      int id = gidx(axis, gi, half, j);
      sm->x[id] = sm->x[id] / sigma;
    }
    if (half == 0) acc[gi] *= sigma;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(AP_THREADS) append_kernel(AppendArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  AppendSmem* sm = reinterpret_cast<AppendSmem*>(smem_raw);
  const Geo& g = a.g;
  const int tid = threadIdx.x;
  const int blk_src = blockIdx.x, h = blockIdx.y, b = blockIdx.z >> 1, kind = blockIdx.z & 1;
  const int blk = a.blk0 + blk_src;
  if (blk >= g.max_blocks) {  // host checks capacity; keep the kernel safe regardless
    if (tid == 0) report(a.status, KVQ_ERR_CAPACITY);
    return;
  }

  // ---- stage the tile (one read of HBM), fp32
  const uint16_t* src = (kind ? a.v : a.k) +
                        (((uint64_t)b * g.H + h) * (uint64_t)a.n_new * T + (uint64_t)blk_src * T) * D;
  const bool sink_row = g.sink && blk == 0;  // token 0 of the sequence: kept, zero in the tile
  for (int i = tid; i < TILE / 8; i += AP_THREADS) {
    uint4 u = reinterpret_cast<const uint4*>(src)[i];
    int e = i * 8, t = e >> 7, c = e & 127;
    if (sink_row && t == 0) {
      reinterpret_cast<uint4*>(a.base + g.sink_off + (((uint64_t)b * g.H + h) * 2 + kind) * D * 2)[i] = u;
      u = make_uint4(0u, 0u, 0u, 0u);
    }
    const uint16_t* hv = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
    for (int j = 0; j < 8; ++j) sm->x[t * XS + c + j] = in_bits_to_f32(hv[j], g.in_bf16);
  }
  if (tid < T) {
    sm->racc[tid] = 1.0f;
    sm->cacc[tid] = 1.0f;
  }
  __syncthreads();

  uint8_t* rec = a.base + record_offset(g, b, h, blk, a.status);
  uint32_t* codes_dst = reinterpret_cast<uint32_t*>(rec + g.codes_off[kind]);
  uint16_t* m16 = reinterpret_cast<uint16_t*>(rec + g.meta_off[kind]);
  const int axis = kind == 0 ? 0 : 1;  // keys per channel, values per token

  if (g.method == KVQ_RTN) {
    rtn_tile(sm, axis, g.bits, m16);
  } else if (g.method == KVQ_VARN) {
    if (a.hadamard) fwht_rows(sm);
    for (int it = 0; it < a.varn_iters; ++it) {
      varn_axis(sm, 0, sm->cacc);   // columns (channels) first
      varn_axis(sm, 1, sm->racc);   // then rows (tokens)
    }
    // keys: Z = Y diag(c), s1 = r; values: Z = diag(r) Y, s1 = c
    for (int e = tid; e < TILE; e += AP_THREADS) {
      int t = e >> 7, c = e & 127;
      float sc = kind == 0 ? sm->cacc[c] : sm->racc[t];
      sm->x[t * XS + c] = __fmul_rn(sm->x[t * XS + c], sc);
    }
    __syncthreads();
    if (tid < T) {
      float s1 = kind == 0 ? sm->racc[tid] : sm->cacc[tid];
      m16[2 * T + tid] = f2h_rn(s1);
      if (a.dbg) {
        float* d = a.dbg + ((((uint64_t)b * g.H + h) * a.n_new + blk_src) * 2 + kind) * 2 * T;
        d[tid] = sm->racc[tid];
        d[T + tid] = sm->cacc[tid];
      }
    }
    rtn_tile(sm, axis, g.bits, m16);
  } else if (g.method == KVQ_INT4) {
    // scale = absmax / qmax per token (or per half-token), q = clamp(rne(x / scale), -qmax-1, qmax)
    const float qmax = g.bits == 8 ? 127.0f : 7.0f;
    const uint32_t cmask = (1u << g.bits) - 1u;
    const int gi = tid >> 1, half = tid & 1;
    float am = 0.0f;
    for (int j = 0; j < 64; ++j) am = fmaxf(am, fabsf(sm->x[gi * XS + half * 64 + j]));
    if (!g.g64) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    if (g.g64 || half == 0) {
      float s32 = fminf(__fdiv_rn(am, qmax), 65504.0f);
      uint16_t s16 = f2h_rn(s32);
      (half ? sm->gz : sm->gs)[gi] = h2f(s16);  // g64: channels 64..127 in gz
      m16[half * T + gi] = s16;
    }
    __syncthreads();
    for (int e = tid; e < TILE; e += AP_THREADS) {
      int t = e >> 7, c = e & 127;
      float sf = (g.g64 && c >= 64) ? sm->gz[t] : sm->gs[t];
      int q = 0;
      if (sf != 0.0f) {
        float qf = rintf(__fdiv_rn(sm->x[t * XS + c], sf));
        q = (int)fminf(fmaxf(qf, -qmax - 1.0f), qmax);
      }
      sm->codes[e] = (uint8_t)((uint32_t)q & cmask);
    }
    __syncthreads();
  } else {  // KVQ_NUQ
    const int ncb = 1 << g.bits;
    if (tid < ncb) sm->cb[tid] = a.codebook[h * ncb + tid];
    for (int i = tid; i < TILE / 32; i += AP_THREADS) sm->mask[i] = 0u;
    uint8_t* csr = rec + g.csr_off[kind];
    const int n_out = g.n_out;
    // calibrated keys: per-channel threshold and statistics from the calibration table
    const bool calib = g.key_calib && kind == 0;
    const float* tau_tab = reinterpret_cast<const float*>(a.base + g.calib_off) + h * D;
    const uint16_t* s_tab = reinterpret_cast<const uint16_t*>(a.base + g.calib_off + (uint64_t)g.H * D * 4) + h * D;
    const uint16_t* zp_tab = s_tab + (uint64_t)g.H * D;
    __syncthreads();
    if (n_out > 0) {
      // pass 1: histogram of the high 8 bits of the 15-bit fp16 magnitude
      sm->hist[tid] = 0;
      __syncthreads();
      const int e0 = tid * 64;  // this thread's chunk of flat indices (half a row)
      const int t0 = e0 >> 7, c0 = e0 & 127;
      uint32_t mpk[32];         // the chunk's fp16 magnitudes, two per register
#pragma unroll
      for (int j = 0; j < 64; j += 2)
        mpk[j >> 1] = (uint32_t)(f2h_rn(sm->x[t0 * XS + c0 + j]) & 0x7fff) |
                      ((uint32_t)(f2h_rn(sm->x[t0 * XS + c0 + j + 1]) & 0x7fff) << 16);
      auto mag_of = [&](int j) -> int { return (int)((mpk[j >> 1] >> (16 * (j & 1))) & 0x7fffu); };
#pragma unroll
      for (int j = 0; j < 64; ++j) atomicAdd(&sm->hist[mag_of(j) >> 7], 1);
      __syncthreads();
      if (tid < 32) {  // the bin holding the n_out-th largest: suffix sums over 8 bins per lane
        int cum, bin;
        if (select_bin<8>(sm->hist, 0, n_out, tid, cum, bin)) {
          sm->sel[0] = bin;
          sm->sel[1] = cum;  // count strictly above this bin
        }
      }
      __syncthreads();
      const int bin1 = sm->sel[0];
      sm->hist[tid] = 0;
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int mag = mag_of(j);
        if ((mag >> 7) == bin1) atomicAdd(&sm->hist[mag & 0x7f], 1);
      }
      __syncthreads();
      if (tid < 32) {  // the same inside that bin: 128 bins of the low 7 bits, 4 per lane
        int cum, lo;
        if (select_bin<4>(sm->hist, sm->sel[1], n_out, tid, cum, lo)) {
          sm->sel[2] = (bin1 << 7) | lo;  // threshold magnitude
          sm->sel[3] = n_out - cum;       // how many entries equal to the threshold are taken
        }
      }
      __syncthreads();
      const int thr = sm->sel[2], need_eq = sm->sel[3];
      int n_eq = 0;
#pragma unroll
      for (int j = 0; j < 64; ++j) n_eq += mag_of(j) == thr;
      int eq_rank = block_excl_scan(n_eq, sm->scan, nullptr);
      uint64_t selbits = 0;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int mag = mag_of(j);
        bool s = mag > thr;
        if (mag == thr) {
          s = eq_rank < need_eq;
          ++eq_rank;
        }
        if (s) selbits |= 1ull << j;
      }
      if (calib) {  // of the tile's largest entries, only those over the channel's threshold
        for (int j = 0; j < 64; ++j)
          if (!(fabsf(sm->x[t0 * XS + c0 + j]) > tau_tab[c0 + j])) selbits &= ~(1ull << j);
      }
      const int n_sel = __popcll(selbits);
      int n_total = 0;
      int pos = block_excl_scan(n_sel, sm->scan, &n_total);
      uint16_t* val = reinterpret_cast<uint16_t*>(csr);
      uint16_t* ptr = reinterpret_cast<uint16_t*>(csr + 2 * n_out);  // row_ptr (CSR) or col_ptr (CSC)
      uint8_t* idx = csr + 2 * n_out + 2 * (T + 1);                   // channel (CSR) or token (CSC)
      for (int i = n_total + tid; i < n_out; i += AP_THREADS) {  // unused capacity (calibrated keys)
        val[i] = 0;
        idx[i] = 0;
      }
      sm->mask[e0 >> 5] = (uint32_t)selbits;
      sm->mask[(e0 >> 5) + 1] = (uint32_t)(selbits >> 32);
      if (!(g.v_csc && kind == 1)) {  // CSR: thread (t0, half) writes its row segment in channel order
        if ((tid & 1) == 0) ptr[t0] = (uint16_t)pos;
        if (tid == 0) ptr[T] = (uint16_t)n_total;
        for (int j = 0; j < 64; ++j) {
          if (selbits >> j & 1) {
            if (pos < n_out) {
              val[pos] = f2h_rn(sm->x[t0 * XS + c0 + j]);
              idx[pos] = (uint8_t)(c0 + j);
            } else {
              report(a.status, KVQ_ERR_INVALID_ARG);
            }
            ++pos;
          }
        }
      } else {  // CSC values: thread c writes column c in token order
        __syncthreads();  // every mask word written
        int cnt = 0;
        if (tid < D)
          for (int t = 0; t < T; ++t) cnt += (int)(sm->mask[(t * D + tid) >> 5] >> (tid & 31) & 1u);
        int cpos = block_excl_scan(cnt, sm->scan, nullptr);
        if (tid < D) {
          ptr[tid] = (uint16_t)cpos;
          if (tid == 0) ptr[D] = (uint16_t)n_total;
          for (int t = 0; t < T; ++t) {
            if (sm->mask[(t * D + tid) >> 5] >> (tid & 31) & 1u) {
              if (cpos < n_out) {
                val[cpos] = f2h_rn(sm->x[t * XS + tid]);
                idx[cpos] = (uint8_t)t;
              } else {
                report(a.status, KVQ_ERR_INVALID_ARG);
              }
              ++cpos;
            }
          }
        }
      }
      // zero the padding of the outlier region so that records are deterministic
      const int used = 3 * n_out + 2 * (T + 1);
      const int total = (int)round16((uint64_t)used);
      for (int i = used + tid; i < total; i += AP_THREADS) csr[i] = 0;
      __syncthreads();
    }
    // centre / half-range of the non-outlier entries of each group
    {
      const int gi = tid >> 1, half = tid & 1;
      float mx = -INFINITY, mn = INFINITY;
      for (int j = 0; j < 64; ++j) {
        int e = axis == 0 ? (half * 64 + j) * D + gi : gi * D + half * 64 + j;
        if (sm->mask[e >> 5] >> (e & 31) & 1) continue;
        float v = sm->x[gidx(axis, gi, half, j)];
        mx = fmaxf(mx, v);
        mn = fminf(mn, v);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
      if (half == 0) {
        uint16_t s16 = 0, zp16 = 0;
        if (calib) {
          s16 = s_tab[gi];
          zp16 = zp_tab[gi];
        } else if (mx != -INFINITY) {
          zp16 = f2h_rn(__fdiv_rn(__fadd_rn(mx, mn), 2.0f));
          s16 = f2h_rn(__fdiv_rn(__fsub_rn(mx, mn), 2.0f));
        }
        sm->gs[gi] = h2f(s16);
        sm->gz[gi] = h2f(zp16);
        m16[gi] = s16;
        m16[T + gi] = zp16;
      }
    }
    __syncthreads();
    for (int e = tid; e < TILE; e += AP_THREADS) {
      int t = e >> 7, c = e & 127;
      int gg = axis == 0 ? c : t;
      bool outl = sm->mask[e >> 5] >> (e & 31) & 1;
      float xd = outl ? 0.0f : sm->x[t * XS + c];
      float sf = sm->gs[gg];
      float tv = 0.0f;
      if (sf != 0.0f) tv = fminf(fmaxf(__fdiv_rn(__fsub_rn(xd, sm->gz[gg]), sf), -1.0f), 1.0f);
      int best = 0;
      float bd = fabsf(__fsub_rn(tv, sm->cb[0]));
      for (int j = 1; j < ncb; ++j) {
        float d = fabsf(__fsub_rn(tv, sm->cb[j]));
        if (d < bd) {
          bd = d;
          best = j;
        }
      }
      sm->codes[e] = (uint8_t)best;
    }
    __syncthreads();
  }
  pack_tile(sm, g.bits, kind == 1 && g.vrows_ch, g.planes3 != 0, kind, codes_dst);
}

size_t append_smem_bytes() { return sizeof(AppendSmem); }

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(AppendSmem);
  cudaError_t e = ensure_smem_attr((const void*)append_kernel, (size_t)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_new, a.g.H, a.g.B * 2);
  append_kernel<<<grid, AP_THREADS, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq

// C++ entry used by the API translation unit.
cudaError_t kvq_launch_append(const kvq::Geo& g, const uint16_t* k, const uint16_t* v, int n_new, int blk0,
                              uint8_t* base, const float* codebook, float* dbg, int* status, int varn_iters,
                              int hadamard, cudaStream_t st) {
  kvq::AppendArgs a;
  a.g = g; a.k = k; a.v = v; a.n_new = n_new; a.blk0 = blk0; a.base = base; a.codebook = codebook;
  a.dbg = dbg; a.status = status; a.varn_iters = varn_iters; a.hadamard = hadamard;
  return kvq::launch_append(a, st);
}
