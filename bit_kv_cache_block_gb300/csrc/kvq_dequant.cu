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
  const uint32_t* codes = reinterpret_cast<const uint32_t*>(rec + g.codes_off[kind]);
  const uint16_t* m = reinterpret_cast<const uint16_t*>(rec + g.meta_off[kind]);
  const int bits = g.bits, W = g.W, nw = 32 / bits;
  const uint32_t cmask = (1u << bits) - 1u;
  float* row = xs + t * 129;
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
    } else if (g.method == KVQ_INT4) {
      v = (float)((int)(q << 28) >> 28) * h2f(m[t]);
    } else {
      const int gi = kind == 0 ? c : t;
      v = a.codebook[h * (1 << bits) + q] * h2f(m[gi]) + h2f(m[T + gi]);
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
  if (g.method == KVQ_VARN && a.hadamard && a.domain == 1) {
    for (int hh = 1; hh < D; hh <<= 1)
      for (int j = 0; j < D / 2; ++j) {
        int i0 = (j / hh) * (2 * hh) + (j % hh);
        float x0 = row[i0], x1 = row[i0 + hh];
        row[i0] = x0 + x1;
        row[i0 + hh] = x0 - x1;
      }
    for (int c = 0; c < D; ++c) row[c] *= 0.08838834764831845f;
  }
  __syncthreads();
  float* dst = out + (((uint64_t)b * g.H + h) * (uint64_t)a.n * T + (uint64_t)bi * T) * D;
  for (int e = t; e < TILE; e += DQ_THREADS) dst[e] = xs[(e >> 7) * 129 + (e & 127)];
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

cudaError_t kvq_launch_rope_init(float2* tab, int max_blocks, double theta, cudaStream_t st) {
  const int total = (max_blocks + 1 + kvq::T) * 64;
  int blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  kvq::rope_table_kernel<<<blocks, 256, 0, st>>>(tab, max_blocks, theta);
  return cudaGetLastError();
}
