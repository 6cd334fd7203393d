// Dequantisation of cached blocks to fp32 (checking only) and the RoPE angle tables.
#include "kvq_internal.cuh"

namespace kvq {

constexpr int DQ_THREADS = 128;

struct DequantArgs {
  Geo g;
  const uint8_t* base;
  const float* codebook;
  int first, n;
  int domain;
  int hadamard;
  float* out_k;
  float* out_v;
  int* status;
};

// Row t of one tile record dequantised to fp32 into row[0..127]: token t for key tiles and
// value tiles alike (the value planes of the tensor-core format hold channels per row and are
// indexed accordingly), CSR outliers added for nuq, and for KVarN with the Hadamard transform
// the inverse transform applied when to_input is set.
__device__ void dequant_row(const Geo& g, const uint8_t* rec, const float* codebook, int h, int kind, int t,
                            bool to_input, float* row) {
  const uint32_t* codes = reinterpret_cast<const uint32_t*>(rec + g.codes_off[kind]);
  const uint16_t* m = reinterpret_cast<const uint16_t*>(rec + g.meta_off[kind]);
  const int bits = g.bits, W = g.W, nw = 32 / bits;
  const uint32_t cmask = (1u << bits) - 1u;
  for (int c = 0; c < D; ++c) {
    // rows of tokens (value tiles: rows of channels when vrows_ch), or the 3-bit planes
    const uint32_t q = g.planes3 ? tile3_code(codes, kind, t, c)
                       : (kind == 0 || !g.vrows_ch) ? (codes[t * W + c / nw] >> (bits * (c % nw))) & cmask
                                                    : (codes[c * W + t / nw] >> (bits * (t % nw))) & cmask;
    float v;
    if (g.method == KVQ_RTN || g.method == KVQ_VARN) {
      const int gi = kind == 0 ? c : t;
      v = ((float)q + h2f(m[T + gi])) * h2f(m[gi]);
      if (g.method == KVQ_VARN) v *= h2f(m[2 * T + (kind == 0 ? t : c)]);
    } else if (g.method == KVQ_INT4) {  // b-bit two's complement times the scale of (t, c's group)
      v = (float)((int)(q << (32 - bits)) >> (32 - bits)) * h2f(m[(g.g64 && c >= 64 ? T : 0) + t]);
    } else {
      const int gi = kind == 0 ? c : t;
      v = codebook[h * (1 << bits) + q] * h2f(m[gi]) + h2f(m[T + gi]);
    }
    row[c] = v;
  }
  if (g.method == KVQ_NUQ && g.n_out > 0) {
    const uint8_t* csr = rec + g.csr_off[kind];
    const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
    const uint16_t* rp = reinterpret_cast<const uint16_t*>(csr + 2 * g.n_out);
    const uint8_t* col = csr + 2 * g.n_out + 2 * (T + 1);
    const int j1 = min((int)rp[t + 1], g.n_out);
    for (int j = min((int)rp[t], g.n_out); j < j1; ++j) row[col[j] & (D - 1)] += h2f(val[j]);
  }
  if (g.method == KVQ_VARN && to_input) {
    for (int hh = 1; hh < D; hh <<= 1)
      for (int j = 0; j < D / 2; ++j) {
        int i0 = (j / hh) * (2 * hh) + (j % hh);
        float x0 = row[i0], x1 = row[i0 + hh];
        row[i0] = x0 + x1;
        row[i0 + hh] = x0 - x1;
      }
    for (int c = 0; c < D; ++c) row[c] *= 0.08838834764831845f;
  }
}

// grid (n, H, B*2), thread = token row of the tile; rows staged in shared memory (stride 129)
// so that the inverse Hadamard transform and the stores run on whole rows.
__global__ void __launch_bounds__(DQ_THREADS) dequant_kernel(DequantArgs a) {
  extern __shared__ float xs[];
  const Geo& g = a.g;
  const int t = threadIdx.x;
  const int bi = blockIdx.x, h = blockIdx.y, b = blockIdx.z >> 1, kind = blockIdx.z & 1;
  float* out = kind ? a.out_v : a.out_k;
  if (!out) return;
  const int blk = a.first + bi;
  const uint8_t* rec = a.base + record_offset(g, b, h, blk, a.status);
  dequant_row(g, rec, a.codebook, h, kind, t, a.hadamard && a.domain == 1, xs + t * 129);
  __syncthreads();
  float* dst = out + (((uint64_t)b * g.H + h) * (uint64_t)a.n * T + (uint64_t)bi * T) * D;
  for (int e = t; e < TILE; e += DQ_THREADS) dst[e] = xs[(e >> 7) * 129 + (e & 127)];
}

// Per-token error statistics ([KVN] key innovation: |x - x_dq|^2 = E_M + E_D). grid (n, H, B*2),
// ES_THREADS threads, one instantiation per (method, bits). The tile's part of the record (codes,
// metadata, CSR) is copied into shared memory; value tiles stored as channel rows get a row
// stride of W + 1 words (odd), so the 32 channels a warp reads at once sit in 32 banks. Then warp
// w takes token rows w, w + 8, ...: lane l holds channels l + 32j (j = 0..3), dequantises them
// (per-channel scales kept in registers), applies the row's CSR entries and, for KVarN, the
// inverse Hadamard transform (distances 1 .. 16 across lanes, 32 and 64 inside the lane), and
// the sums close with xor shuffles.
constexpr int ES_THREADS = 256;

struct ErrArgs {
  Geo g;
  const uint8_t* base;
  const float* codebook;
  int first, n;
  int hadamard;
  const uint16_t* in_k;
  const uint16_t* in_v;
  float* st_k;
  float* st_v;
  int* status;
};

template <int BITS>
struct EsGeom {
  static constexpr int NWC = 32 / BITS;             // codes per word
  static constexpr int W = (D + NWC - 1) / NWC;     // words per row
  static constexpr uint32_t MASK = (1u << BITS) - 1u;
};

// Shared-memory bytes of the staged code region (channel rows padded to W + 1 words).
template <int BITS>
__host__ __device__ inline uint32_t es_codes_bytes(bool padded, uint32_t plain_bytes) {
  return padded ? (uint32_t)round16((uint64_t)T * (EsGeom<BITS>::W + 1) * 4) : plain_bytes;
}

template <int METHOD, int BITS>
__global__ void __launch_bounds__(ES_THREADS) error_stats_kernel(ErrArgs a) {
  using E = EsGeom<BITS>;
  extern __shared__ __align__(16) uint8_t es_smem[];
  const Geo& g = a.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bi = blockIdx.x, h = blockIdx.y, b = blockIdx.z >> 1, kind = blockIdx.z & 1;
  const uint16_t* in = kind ? a.in_v : a.in_k;
  float* st = kind ? a.st_v : a.st_k;
  if (!in || !st) return;
  const int blk = a.first + bi;
  const uint8_t* rec = a.base + record_offset(g, b, h, blk, a.status);
  const bool planes = BITS == 3 && g.planes3;
  const bool chrows = kind == 1 && g.vrows_ch && !planes;  // value codes as channel rows
  const uint32_t off = g.codes_off[kind], moff = g.meta_off[kind];
  const uint32_t end = kind ? (uint32_t)g.rec_bytes : g.codes_off[1];
  const uint32_t cbytes = es_codes_bytes<BITS>(chrows, moff - off);
  {
    if (chrows) {  // row r (channel) at word r * (W + 1)
      const uint32_t* src = reinterpret_cast<const uint32_t*>(rec + off);
      uint32_t* dst = reinterpret_cast<uint32_t*>(es_smem);
      for (int i = tid; i < T * E::W; i += ES_THREADS) dst[(i / E::W) * (E::W + 1) + i % E::W] = src[i];
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(rec + off);
      uint4* dst = reinterpret_cast<uint4*>(es_smem);
      for (uint32_t i = tid; i < (moff - off) / 16; i += ES_THREADS) dst[i] = src[i];
    }
    const uint4* src = reinterpret_cast<const uint4*>(rec + moff);  // metadata and CSR
    uint4* dst = reinterpret_cast<uint4*>(es_smem + cbytes);
    for (uint32_t i = tid; i < (end - moff) / 16; i += ES_THREADS) dst[i] = src[i];
  }
  const uint32_t* codes = reinterpret_cast<const uint32_t*>(es_smem);
  const uint16_t* m = reinterpret_cast<const uint16_t*>(es_smem + cbytes);
  __shared__ float cb[16];  // nuq codebook of this head
  if (METHOD == KVQ_NUQ && tid < (1 << BITS)) cb[tid] = a.codebook[h * (1 << BITS) + tid];
  __syncthreads();
  // per-channel metadata of the lane's channels l + 32j (keys: s, z or zp; values: s1)
  float cs[4], cz[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = lane + 32 * j;
    cs[j] = 1.0f;
    cz[j] = 0.0f;
    if (kind == 0 && METHOD != KVQ_INT4) {
      cs[j] = h2f(m[c]);
      cz[j] = h2f(m[T + c]);
    } else if (kind == 1 && METHOD == KVQ_VARN) {
      cs[j] = h2f(m[2 * T + c]);  // s1 per channel
    }
  }
  const bool to_input = METHOD == KVQ_VARN && a.hadamard;
  const uint64_t tok0 = ((uint64_t)b * g.H + h) * (uint64_t)a.n * T + (uint64_t)bi * T;
  for (int t = warp; t < T; t += ES_THREADS / 32) {
    const uint16_t* xr = in + (tok0 + t) * D + lane;
    float x[4], q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = in_bits_to_f32(xr[32 * j], g.in_bf16);
    if (g.sink && blk == 0 && t == 0) {  // the kept first token: what decode attends
      const uint16_t* kept =
          reinterpret_cast<const uint16_t*>(a.base + g.sink_off) + (((uint64_t)b * g.H + h) * 2 + kind) * D + lane;
#pragma unroll
      for (int j = 0; j < 4; ++j) q[j] = in_bits_to_f32(kept[32 * j], g.in_bf16);
    } else {
      // per-token metadata of this row (values: s, z or zp; keys: KVarN s1; absmax: s per block)
      const float ts0 = (kind == 1 || METHOD == KVQ_INT4) ? h2f(m[t]) : 1.0f;
      const float ts1 = (METHOD == KVQ_INT4 && g.g64) ? h2f(m[T + t]) : ts0;  // channels 64..127
      const float tz = (kind == 1 && METHOD != KVQ_INT4) ? h2f(m[T + t]) : 0.0f;
      const float tk1 = (kind == 0 && METHOD == KVQ_VARN) ? h2f(m[2 * T + t]) : 1.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = lane + 32 * j;
        uint32_t code;
        if (planes) code = tile3_code(codes, kind, t, c);
        else if (chrows) code = (codes[c * (E::W + 1) + t / E::NWC] >> (BITS * (t % E::NWC))) & E::MASK;
        else code = (codes[t * E::W + c / E::NWC] >> (BITS * (c % E::NWC))) & E::MASK;
        const float ts = j < 2 ? ts0 : ts1;
        float v;
        if (METHOD == KVQ_RTN || METHOD == KVQ_VARN) {
          v = kind == 0 ? ((float)code + cz[j]) * cs[j] : ((float)code + tz) * ts;
          if (METHOD == KVQ_VARN) v *= kind == 0 ? tk1 : cs[j];
        } else if (METHOD == KVQ_INT4) {
          constexpr int SH = 32 - BITS;
          v = (float)((int)(code << SH) >> SH) * ts;
        } else {
          v = kind == 0 ? cb[code] * cs[j] + cz[j] : cb[code] * ts + tz;
        }
        q[j] = v;
      }
      if (METHOD == KVQ_NUQ && g.n_out > 0) {  // this row's outliers (few): the owning lane adds
        const uint8_t* csr = es_smem + cbytes + (g.csr_off[kind] - moff);
        const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
        const uint16_t* rp = reinterpret_cast<const uint16_t*>(csr + 2 * g.n_out);
        const uint8_t* col = csr + 2 * g.n_out + 2 * (T + 1);
        const int e1 = min((int)rp[t + 1], g.n_out);
        for (int e = min((int)rp[t], g.n_out); e < e1; ++e) {
          const int c = col[e] & (D - 1);
          if ((c & 31) == lane) {
            const float vv = h2f(val[e]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if ((c >> 5) == j) q[j] += vv;
          }
        }
      }
      if (to_input) {  // inverse Hadamard (H / sqrt(128) is its own inverse), Sylvester order
#pragma unroll
        for (int hl = 1; hl < 32; hl <<= 1) {  // channel distance hl: across lanes
          const bool upper = lane & hl;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float o = __shfl_xor_sync(0xffffffffu, q[j], hl);
            q[j] = upper ? o - q[j] : q[j] + o;
          }
        }
        const float y0 = q[0] + q[1], y1 = q[0] - q[1], y2 = q[2] + q[3], y3 = q[2] - q[3];  // distance 32
        q[0] = (y0 + y2) * 0.08838834764831845f;  // distance 64
        q[2] = (y0 - y2) * 0.08838834764831845f;
        q[1] = (y1 + y3) * 0.08838834764831845f;
        q[3] = (y1 - y3) * 0.08838834764831845f;
      }
    }
    float sxx = 0.0f, sqq = 0.0f, sdd = 0.0f, spm = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float dd = x[j] - q[j];
      sxx = fmaf(x[j], x[j], sxx);
      sqq = fmaf(q[j], q[j], sqq);
      sdd = fmaf(dd, dd, sdd);
      spm = fmaf(q[j] - x[j], q[j] + x[j], spm);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sxx += __shfl_xor_sync(0xffffffffu, sxx, o);
      sqq += __shfl_xor_sync(0xffffffffu, sqq, o);
      sdd += __shfl_xor_sync(0xffffffffu, sdd, o);
      spm += __shfl_xor_sync(0xffffffffu, spm, o);
    }
    const float nx = sqrtf(sxx), nq = sqrtf(sqq);
    const float dn = nx + nq > 0.0f ? spm / (nx + nq) : 0.0f;
    float ed = 0.0f;
    if (nx > 0.0f && nq > 0.0f) {  // warp-uniform
      const float ix = 1.0f / nx, iq = 1.0f / nq;
      float su = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float u = __fsub_rn(__fmul_rn(x[j], ix), __fmul_rn(q[j], iq));  // 0 when x_dq = x
        su = fmaf(u, u, su);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) su += __shfl_xor_sync(0xffffffffu, su, o);
      ed = nx * nq * su;
    }
    if (lane == 0) reinterpret_cast<float4*>(st)[tok0 + t] = make_float4(nx, dn, sdd, ed);
  }
}

// RoPE tables: (cos, sin) of blk*128*theta_i for blk = 0..max_blocks, then of t*theta_i for
// t = 0..127; theta_i = rope_theta^(-2i/128), angles and sin/cos in fp64, stored fp32.
__global__ void rope_table_kernel(float2* tab, int max_blocks, double theta) {
  const int n_blk = (max_blocks + 1) * 64;
  const int total = n_blk + T * 64;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
    const int i = e & 63;
    const double th = pow(theta, -2.0 * (double)i / (double)D);
    const double pos = e < n_blk ? (double)(e >> 6) * (double)T : (double)((e - n_blk) >> 6);
    double s, c;
    sincos(pos * th, &s, &c);
    tab[e] = make_float2((float)c, (float)s);
  }
}

}  // namespace kvq

cudaError_t kvq_launch_dequant(const kvq::Geo& g, const uint8_t* base, const float* codebook, int first, int n,
                               int domain, int hadamard, float* out_k, float* out_v, int* status, cudaStream_t st) {
  kvq::DequantArgs a;
  a.g = g; a.base = base; a.codebook = codebook; a.first = first; a.n = n; a.domain = domain;
  a.hadamard = hadamard; a.out_k = out_k; a.out_v = out_v; a.status = status;
  const int smem = kvq::T * 129 * (int)sizeof(float);
  cudaError_t e = kvq::ensure_smem_attr((const void*)kvq::dequant_kernel, (size_t)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n, g.H, g.B * 2);
  kvq::dequant_kernel<<<grid, kvq::DQ_THREADS, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t kvq_launch_error_stats(const kvq::Geo& g, const uint8_t* base, const float* codebook, int first, int n,
                                   int hadamard, const uint16_t* in_k, const uint16_t* in_v, float* st_k, float* st_v,
                                   int* status, cudaStream_t st) {
  kvq::ErrArgs a;
  a.g = g; a.base = base; a.codebook = codebook; a.first = first; a.n = n; a.hadamard = hadamard;
  a.in_k = in_k; a.in_v = in_v; a.st_k = st_k; a.st_v = st_v; a.status = status;
  // largest staged region: a kind's record part, plus the padding of value channel rows
  const uint32_t kb = g.codes_off[1] - g.codes_off[0], vb = (uint32_t)g.rec_bytes - g.codes_off[1];
  const int smem = (int)(kb > vb ? kb : vb) + (int)kvq::round16((uint64_t)kvq::T * 4) + 16;
  using Fn = void (*)(kvq::ErrArgs);
  Fn fn = nullptr;
  const int m = g.method, b = g.bits;
#define KVQ_ES(M, B) if (m == M && b == B) fn = kvq::error_stats_kernel<M, B>;
  KVQ_ES(KVQ_RTN, 2) KVQ_ES(KVQ_RTN, 3) KVQ_ES(KVQ_RTN, 4)
  KVQ_ES(KVQ_NUQ, 2) KVQ_ES(KVQ_NUQ, 3) KVQ_ES(KVQ_NUQ, 4)
  KVQ_ES(KVQ_VARN, 2) KVQ_ES(KVQ_VARN, 3) KVQ_ES(KVQ_VARN, 4)
  KVQ_ES(KVQ_INT4, 4) KVQ_ES(KVQ_INT4, 8)
#undef KVQ_ES
  if (!fn) return cudaErrorInvalidValue;
  cudaError_t e = kvq::ensure_smem_attr((const void*)fn, (size_t)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n, g.H, g.B * 2);
  fn<<<grid, kvq::ES_THREADS, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t kvq_launch_rope_init(float2* tab, int max_blocks, double theta, cudaStream_t st) {
  const int total = (max_blocks + 1 + kvq::T) * 64;
  int blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  kvq::rope_table_kernel<<<blocks, 256, 0, st>>>(tab, max_blocks, theta);
  return cudaGetLastError();
}
