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

// Per-token error statistics ([KVN] key innovation: |x - x_dq|^2 = E_M + E_D). grid (n, H, B*2):
// the tile is dequantised row by row into shared memory as above (input domain), then each warp
// takes rows w, w + 4, ...: lane l reads channels l + 32j of the input row (coalesced) and of the
// staged row (conflict-free), and the sums close with xor shuffles.
__global__ void __launch_bounds__(DQ_THREADS) error_stats_kernel(ErrArgs a) {
  extern __shared__ float xs[];
  const Geo& g = a.g;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int bi = blockIdx.x, h = blockIdx.y, b = blockIdx.z >> 1, kind = blockIdx.z & 1;
  const uint16_t* in = kind ? a.in_v : a.in_k;
  float* st = kind ? a.st_v : a.st_k;
  if (!in || !st) return;
  const int blk = a.first + bi;
  const uint8_t* rec = a.base + record_offset(g, b, h, blk, a.status);
  float* row = xs + t * 129;
  if (g.sink && blk == 0 && t == 0) {  // the kept first token: what decode attends
    const uint16_t* kept = reinterpret_cast<const uint16_t*>(a.base + g.sink_off) + (((uint64_t)b * g.H + h) * 2 + kind) * D;
    for (int c = 0; c < D; ++c) row[c] = in_bits_to_f32(kept[c], g.in_bf16);
  } else {
    dequant_row(g, rec, a.codebook, h, kind, t, a.hadamard != 0, row);
  }
  __syncthreads();
  const uint64_t tok0 = ((uint64_t)b * g.H + h) * (uint64_t)a.n * T + (uint64_t)bi * T;
  for (int r = warp; r < T; r += DQ_THREADS / 32) {
    const uint16_t* xr = in + (tok0 + r) * D;
    const float* qr = xs + r * 129;
    float x[4], q[4];
    float sxx = 0.0f, sqq = 0.0f, sdd = 0.0f, spm = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[j] = in_bits_to_f32(xr[lane + 32 * j], g.in_bf16);
      q[j] = qr[lane + 32 * j];
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
    if (lane == 0) reinterpret_cast<float4*>(st)[tok0 + r] = make_float4(nx, dn, sdd, ed);
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
  const int smem = kvq::T * 129 * (int)sizeof(float);
  cudaError_t e = kvq::ensure_smem_attr((const void*)kvq::error_stats_kernel, (size_t)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n, g.H, g.B * 2);
  kvq::error_stats_kernel<<<grid, kvq::DQ_THREADS, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t kvq_launch_rope_init(float2* tab, int max_blocks, double theta, cudaStream_t st) {
  const int total = (max_blocks + 1 + kvq::T) * 64;
  int blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  kvq::rope_table_kernel<<<blocks, 256, 0, st>>>(tab, max_blocks, theta);
  return cudaGetLastError();
}
