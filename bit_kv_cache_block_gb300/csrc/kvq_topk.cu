// Shares of the largest token errors ([KVN] Figure 1a: E_M / E_T over the top-k% of errors).
//
// For each requested fraction the k largest E_T are found by a radix select over 64-bit keys
// (E_T bits << 32 | (2^32 - 1 - row)): the keys are distinct, so the k-th largest key is one
// exact threshold and equal errors go to the lower row. Eight passes of 8 bits each run a
// histogram kernel over the rows whose key starts with the prefix chosen so far (one histogram
// per fraction) and a one-CTA kernel that picks the next digit. A last pass sums E_T, E_M and
// E_D over the keys at or above each threshold in fp64: every thread walks a fixed set of rows,
// the CTA reduces in a fixed tree, one thread per fraction adds the CTA partials in order, so
// the result does not depend on scheduling. No host synchronisation anywhere.
#include "kvq_internal.cuh"

namespace kvq {
namespace topk {

constexpr int NF = KVQ_TOPK_MAX_FRACS;
constexpr int THREADS = 256;
constexpr int SUM_CTAS = 296;  // 2 per SM

struct State {
  unsigned int hist[NF][256];
  unsigned long long prefix[NF];  // digits chosen so far (high bits of the threshold key)
  unsigned long long rest[NF];    // rank of the threshold among keys with that prefix (1-based)
  double part[SUM_CTAS][NF][3];   // per-CTA sums of E_T, E_M, E_D
};

struct Args {
  const float4* stats;
  unsigned long long n;
  int nf;
  unsigned long long k[NF];
  State* ws;
  double* out;
};

__device__ __forceinline__ unsigned long long key_of(const float4* stats, unsigned long long r) {
  unsigned int u = __float_as_uint(__ldg(&stats[r].z));
  if (u & 0x80000000u) u = 0u;  // -0 (and any negative) ranks as 0
  return ((unsigned long long)u << 32) | (0xffffffffull - r);
}

__global__ void init_kernel(Args a) {
  State* s = a.ws;
  for (int i = threadIdx.x; i < NF * 256; i += blockDim.x) (&s->hist[0][0])[i] = 0u;
  if (threadIdx.x < NF) {
    s->prefix[threadIdx.x] = 0ull;
    s->rest[threadIdx.x] = threadIdx.x < a.nf ? a.k[threadIdx.x] : 0ull;
  }
}

// Histogram of digit `pass` (bits 63-8*pass .. 56-8*pass) over keys matching each prefix.
__global__ void __launch_bounds__(THREADS) hist_kernel(Args a, int pass) {
  __shared__ unsigned int h[NF][256];
  __shared__ unsigned long long pre[NF];
  for (int i = threadIdx.x; i < NF * 256; i += THREADS) (&h[0][0])[i] = 0u;
  if (threadIdx.x < NF) pre[threadIdx.x] = a.ws->prefix[threadIdx.x];
  __syncthreads();
  const int shift = 56 - 8 * pass;
  for (unsigned long long r = blockIdx.x * (unsigned long long)THREADS + threadIdx.x; r < a.n;
       r += (unsigned long long)gridDim.x * THREADS) {
    const unsigned long long key = key_of(a.stats, r);
    const unsigned int digit = (unsigned int)(key >> shift) & 0xffu;
    for (int f = 0; f < a.nf; ++f)
      if (pass == 0 || ((key ^ pre[f]) >> (shift + 8)) == 0ull) atomicAdd(&h[f][digit], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a.nf * 256; i += THREADS) {
    const unsigned int c = (&h[0][0])[i];
    if (c) atomicAdd(&(&a.ws->hist[0][0])[i], c);
  }
}

// One CTA: for each fraction, the digit whose bin holds the rest-th largest key; then clear.
__global__ void pick_kernel(Args a, int pass) {
  State* s = a.ws;
  const int shift = 56 - 8 * pass;
  if (threadIdx.x < a.nf) {
    const int f = threadIdx.x;
    unsigned long long rest = s->rest[f], above = 0ull;
    int d = 255;
    for (; d > 0; --d) {
      const unsigned long long c = s->hist[f][d];
      if (above + c >= rest) break;
      above += c;
    }
    s->rest[f] = rest - above;
    s->prefix[f] |= (unsigned long long)d << shift;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < NF * 256; i += blockDim.x) (&s->hist[0][0])[i] = 0u;
}

// Sums over keys >= threshold, per CTA in a fixed order.
__global__ void __launch_bounds__(THREADS) sum_kernel(Args a) {
  __shared__ double red[THREADS / 32][NF][3];
  __shared__ unsigned long long thr[NF];
  if (threadIdx.x < NF) thr[threadIdx.x] = a.ws->prefix[threadIdx.x];
  __syncthreads();
  double acc[NF][3];
#pragma unroll
  for (int f = 0; f < NF; ++f) acc[f][0] = acc[f][1] = acc[f][2] = 0.0;
  for (unsigned long long r = blockIdx.x * (unsigned long long)THREADS + threadIdx.x; r < a.n;
       r += (unsigned long long)gridDim.x * THREADS) {
    const unsigned long long key = key_of(a.stats, r);
    const float4 v = __ldg(&a.stats[r]);
    const double et = v.z, em = (double)v.y * (double)v.y, ed = v.w;
#pragma unroll
    for (int f = 0; f < NF; ++f)
      if (f < a.nf && key >= thr[f]) {
        acc[f][0] += et;
        acc[f][1] += em;
        acc[f][2] += ed;
      }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int f = 0; f < NF; ++f)
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      double v = acc[f][j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[warp][f][j] = v;
    }
  __syncthreads();
  if (threadIdx.x < NF * 3) {
    const int f = threadIdx.x / 3, j = threadIdx.x % 3;
    double v = 0.0;
    for (int w = 0; w < THREADS / 32; ++w) v += red[w][f][j];
    a.ws->part[blockIdx.x][f][j] = v;
  }
}

__global__ void final_kernel(Args a) {
  const int f = threadIdx.x;
  if (f >= a.nf) return;
  double s[3] = {0.0, 0.0, 0.0};
  for (int c = 0; c < SUM_CTAS; ++c)
    for (int j = 0; j < 3; ++j) s[j] += a.ws->part[c][f][j];
  a.out[4 * f + 0] = (double)a.k[f];
  a.out[4 * f + 1] = s[0];
  a.out[4 * f + 2] = s[1];
  a.out[4 * f + 3] = s[2];
}

}  // namespace topk
}  // namespace kvq

size_t kvq_topk_ws_bytes() { return sizeof(kvq::topk::State); }

cudaError_t kvq_launch_topk(const float* stats, unsigned long long n, const unsigned long long* k, int nf, double* out,
                            void* ws, cudaStream_t st) {
  using namespace kvq::topk;
  Args a;
  a.stats = reinterpret_cast<const float4*>(stats);
  a.n = n;
  a.nf = nf;
  for (int f = 0; f < NF; ++f) a.k[f] = f < nf ? k[f] : 0ull;
  a.ws = static_cast<State*>(ws);
  a.out = out;
  unsigned long long want = (n + THREADS - 1) / THREADS;
  const int hist_ctas = (int)(want < 4 * 152ull ? (want ? want : 1) : 4 * 152ull);
  init_kernel<<<1, 256, 0, st>>>(a);
  for (int pass = 0; pass < 8; ++pass) {
    hist_kernel<<<hist_ctas, THREADS, 0, st>>>(a, pass);
    pick_kernel<<<1, 256, 0, st>>>(a, pass);
  }
  sum_kernel<<<SUM_CTAS, THREADS, 0, st>>>(a);
  final_kernel<<<1, 32, 0, st>>>(a);
  return cudaGetLastError();
}
