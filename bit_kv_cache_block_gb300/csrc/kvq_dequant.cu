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
// indexed accordingly), outliers added for nuq (CSR, or CSC value tiles), and for KVarN with
// the Hadamard transform the inverse transform applied when to_input is set.
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
    if (g.v_csc && kind == 1) {  // by column: rp is the column pointer, col the token of each entry
      for (int c = 0; c < D; ++c) {
        const int j1 = min((int)rp[c + 1], g.n_out);
        for (int j = min((int)rp[c], g.n_out); j < j1; ++j)
          if (col[j] == t) row[c] += h2f(val[j]);
      }
    } else {
      const int j1 = min((int)rp[t + 1], g.n_out);
      for (int j = min((int)rp[t], g.n_out); j < j1; ++j) row[col[j] & (D - 1)] += h2f(val[j]);
    }
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
// ES_THREADS threads, one instantiation per (method, bits). Two bulk copies bring the tile's
// 32 KB of input rows and its part of the record (codes, metadata, CSR) into shared memory; the
// codes are unpacked once into a token-major byte tile (value channel rows are transposed on the
// way). Then 8 lanes take one
// token row: lane j holds channels 16j .. 16j+15, reads their codes with one 16-byte load and
// the input with two, dequantises (per-channel scales in registers), adds the row's CSR entries,
// applies the inverse Hadamard transform for KVarN (distances 1..8 inside the lane, 16..64
// across the 8 lanes), and the sums close over the 8 lanes; a warp finishes 4 rows at a time.
constexpr int ES_THREADS = 256;
constexpr int ES_BROW = D + 16;  // bytes per token row of the unpacked code tile

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

template <int METHOD, int BITS>
__global__ void __launch_bounds__(ES_THREADS, 2) error_stats_kernel(ErrArgs a) {
  constexpr int NWC = 32 / BITS, W = (D + NWC - 1) / NWC;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  extern __shared__ __align__(16) uint8_t es_smem[];
  const Geo& g = a.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bi = blockIdx.x, h = blockIdx.y, b = blockIdx.z >> 1, kind = blockIdx.z & 1;
  const uint16_t* in = kind ? a.in_v : a.in_k;
  float* st = kind ? a.st_v : a.st_k;
  if (!in || !st) return;
  const int blk = a.first + bi;
  const uint8_t* rec = a.base + record_offset(g, b, h, blk, a.status);
  const uint32_t off = g.codes_off[kind], end = kind ? (uint32_t)g.rec_bytes : g.codes_off[1];
  const uint64_t tok0 = ((uint64_t)b * g.H + h) * (uint64_t)a.n * T + (uint64_t)bi * T;
  uint16_t* xs = reinterpret_cast<uint16_t*>(es_smem);        // [128 tokens][128] input rows
  uint8_t* ctile = es_smem + TILE * 2;                        // [128 tokens][ES_BROW] codes
  uint8_t* part = ctile + T * ES_BROW;                        // the record's part of this kind
  __shared__ uint64_t landed;
  __shared__ float cb[16];  // nuq codebook of this head
  if (tid == 0) {
    mbar_init(&landed, 1);
    fence_mbar_init();
  }
  if (METHOD == KVQ_NUQ && tid < (1 << BITS)) cb[tid] = a.codebook[h * (1 << BITS) + tid];
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&landed, (uint32_t)(TILE * 2) + (end - off));
    bulk_g2s(xs, in + tok0 * D, (uint32_t)(TILE * 2), &landed);
    bulk_g2s(part, rec + off, end - off, &landed);
  }
  const bool got = mbar_wait_bounded(&landed, 0u, a.status);
  if (__syncthreads_or(!got)) return;  // every thread leaves together
  const uint32_t* codes = reinterpret_cast<const uint32_t*>(part);
  const uint16_t* m = reinterpret_cast<const uint16_t*>(part + (g.meta_off[kind] - off));
  if (BITS == 3 && g.planes3) {  // bit planes: element by element
    for (int e = tid; e < TILE; e += ES_THREADS) {
      const int t = e >> 7, c = e & 127;
      ctile[t * ES_BROW + c] = (uint8_t)tile3_code(codes, kind, t, c);
    }
  } else {
    const bool chrows = kind == 1 && g.vrows_ch;  // value codes stored as channel rows
    for (int i = tid; i < T * W; i += ES_THREADS) {
      const int r = i / W, w = i - r * W;
      const uint32_t word = codes[i];
#pragma unroll
      for (int j = 0; j < NWC; ++j) {
        const int pos = w * NWC + j;
        if (pos < D) {
          const uint8_t q = (uint8_t)((word >> (BITS * j)) & MASK);
          if (chrows) ctile[pos * ES_BROW + r] = q;  // row r = channel, pos = token
          else ctile[r * ES_BROW + pos] = q;
        }
      }
    }
  }
  __syncthreads();
  const int sub = lane >> 3, j8 = lane & 7, c0 = 16 * j8;  // row within the warp's 4, channel group
  // per-channel metadata of the lane's 16 channels (keys: s, z or zp; values: s1)
  float cs[16], cz[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    cs[i] = 1.0f;
    cz[i] = 0.0f;
    if (kind == 0 && METHOD != KVQ_INT4) {
      cs[i] = h2f(m[c0 + i]);
      cz[i] = h2f(m[T + c0 + i]);
    } else if (kind == 1 && METHOD == KVQ_VARN) {
      cs[i] = h2f(m[2 * T + c0 + i]);  // s1 per channel
    }
  }
  const bool to_input = METHOD == KVQ_VARN && a.hadamard;
  for (int t = 4 * warp + sub; t < T; t += 4 * (ES_THREADS / 32)) {
    float x[16], q[16];
    {
      const uint4* xp = reinterpret_cast<const uint4*>(xs + t * D + c0);
      const uint4 x0 = xp[0], x1 = xp[1];
      const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = in_bits_to_f32((uint16_t)(xw[i] & 0xffffu), g.in_bf16);
        x[2 * i + 1] = in_bits_to_f32((uint16_t)(xw[i] >> 16), g.in_bf16);
      }
    }
    if (g.sink && blk == 0 && t == 0) {  // the kept first token: what decode attends
      const uint16_t* kept =
          reinterpret_cast<const uint16_t*>(a.base + g.sink_off) + (((uint64_t)b * g.H + h) * 2 + kind) * D + c0;
#pragma unroll
      for (int i = 0; i < 16; ++i) q[i] = in_bits_to_f32(kept[i], g.in_bf16);
    } else {
      const uint4 cw = *reinterpret_cast<const uint4*>(ctile + t * ES_BROW + c0);
      const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
      // per-token metadata of this row (values: s, z or zp; keys: KVarN s1; absmax: s per block)
      const float ts = (kind == 1 || METHOD == KVQ_INT4) ? h2f(m[(METHOD == KVQ_INT4 && g.g64 && c0 >= 64 ? T : 0) + t])
                                                         : 1.0f;
      const float tz = (kind == 1 && METHOD != KVQ_INT4) ? h2f(m[T + t]) : 0.0f;
      const float tk1 = (kind == 0 && METHOD == KVQ_VARN) ? h2f(m[2 * T + t]) : 1.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t code = (cws[i >> 2] >> (8 * (i & 3))) & 0xffu;
        float v;
        if (METHOD == KVQ_RTN || METHOD == KVQ_VARN) {
          v = kind == 0 ? ((float)code + cz[i]) * cs[i] : ((float)code + tz) * ts;
          if (METHOD == KVQ_VARN) v *= kind == 0 ? tk1 : cs[i];
        } else if (METHOD == KVQ_INT4) {
          constexpr int SH = 32 - BITS;
          v = (float)((int)(code << SH) >> SH) * ts;
        } else {
          v = kind == 0 ? cb[code] * cs[i] + cz[i] : cb[code] * ts + tz;
        }
        q[i] = v;
      }
      if (METHOD == KVQ_NUQ && g.n_out > 0) {  // this row's outliers (few): the owning lane adds
        const uint8_t* csr = part + (g.csr_off[kind] - off);
        const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
        const uint16_t* rp = reinterpret_cast<const uint16_t*>(csr + 2 * g.n_out);
        const uint8_t* col = csr + 2 * g.n_out + 2 * (T + 1);
        if (g.v_csc && kind == 1) {  // by column: the lane scans its 16 columns for token t
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 16 * j8 + i;
            const int e1 = min((int)rp[c + 1], g.n_out);
            for (int e = min((int)rp[c], g.n_out); e < e1; ++e)
              if (col[e] == t) q[i] += h2f(val[e]);
          }
        } else {
          const int e1 = min((int)rp[t + 1], g.n_out);
          for (int e = min((int)rp[t], g.n_out); e < e1; ++e) {
            const int c = col[e] & (D - 1);
            const float vv = (c >> 4) == j8 ? h2f(val[e]) : 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) q[i] += (c & 15) == i ? vv : 0.0f;  // no indexed register
          }
        }
      }
      if (to_input) {  // inverse Hadamard (H / sqrt(128) is its own inverse), Sylvester order
#pragma unroll
        for (int d = 1; d < 16; d <<= 1)  // distances 1..8: inside the lane
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (!(i & d)) {
              const float u0 = q[i], u1 = q[i + d];
              q[i] = u0 + u1;
              q[i + d] = u0 - u1;
            }
#pragma unroll
        for (int dl = 1; dl < 8; dl <<= 1) {  // distances 16, 32, 64: across the row's 8 lanes
          const bool upper = j8 & dl;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, q[i], dl);
            q[i] = upper ? o - q[i] : q[i] + o;
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] *= 0.08838834764831845f;
      }
    }
    float sxx = 0.0f, sqq = 0.0f, sdd = 0.0f, spm = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float dd = x[i] - q[i];
      sxx = fmaf(x[i], x[i], sxx);
      sqq = fmaf(q[i], q[i], sqq);
      sdd = fmaf(dd, dd, sdd);
      spm = fmaf(q[i] - x[i], q[i] + x[i], spm);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      sxx += __shfl_xor_sync(0xffffffffu, sxx, o);
      sqq += __shfl_xor_sync(0xffffffffu, sqq, o);
      sdd += __shfl_xor_sync(0xffffffffu, sdd, o);
      spm += __shfl_xor_sync(0xffffffffu, spm, o);
    }
    const float nx = sqrtf(sxx), nq = sqrtf(sqq);
    const float dn = nx + nq > 0.0f ? spm / (nx + nq) : 0.0f;
    float su = 0.0f;
    const bool both = nx > 0.0f && nq > 0.0f;  // uniform over the row's 8 lanes
    const float ix = both ? 1.0f / nx : 0.0f, iq = both ? 1.0f / nq : 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float u = __fsub_rn(__fmul_rn(x[i], ix), __fmul_rn(q[i], iq));  // 0 when x_dq = x
      su = fmaf(u, u, su);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) su += __shfl_xor_sync(0xffffffffu, su, o);
    const float ed = both ? nx * nq * su : 0.0f;
    if (j8 == 0) reinterpret_cast<float4*>(st)[tok0 + t] = make_float4(nx, dn, sdd, ed);
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
  // the unpacked code tile, then the larger of the two kinds' record parts
  const uint32_t kb = g.codes_off[1] - g.codes_off[0], vb = (uint32_t)g.rec_bytes - g.codes_off[1];
  const int smem = kvq::TILE * 2 + kvq::T * kvq::ES_BROW + (int)(kb > vb ? kb : vb);
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
