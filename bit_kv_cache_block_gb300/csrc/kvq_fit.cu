// Sensitivity-weighted nuq codebook fitting ([KVQ] §3.3, Algorithm 2): Lloyd iterations per KV
// head on normalised calibration samples with Fisher weights.
//
// Per iteration, an assign kernel (grid: sample chunks x heads) gives every sample its nearest
// centre (|a - c_j| in fp32, the lowest j on ties), counts the samples whose centre changed, and
// adds w*a and w, each scaled by 2^32 and rounded half-even to a 64-bit integer, into the centre's
// sums (integer atomics: exact, so the result does not depend on their order); an update kernel
// (one CTA per head) then stops the head when nothing changed, else moves each centre with
// members of nonzero weight to the fp64 quotient of its sums rounded to fp32. The host issues
// max_iter iterations without synchronising; a stopped head is skipped by the later ones.
#include "kvq_internal.cuh"

namespace kvq {
namespace fit {

constexpr int THREADS = 256;
constexpr int KMAX = 16;
constexpr double SCALE = 4294967296.0;  // 2^32

struct Ws {  // per head
  unsigned long long sum[KMAX][2];  // sum of round(w*a*2^32) (two's complement), sum of round(w*2^32)
  int changes;
  int done;
  int pad[2];
};

struct Args {
  const float* a;
  const float* w;
  long long n;
  int k;
  float* c;         // [H][k]
  Ws* ws;           // [H]
  uint8_t* prev;    // [H][n] assignment of the previous iteration (255: none)
  int it;
};

__global__ void init_kernel(Args g, int n_heads) {
  const long long total = (long long)n_heads * g.n;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x)
    g.prev[i] = 255;
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e < n_heads * KMAX; e += blockDim.x) {
      const int h = e / KMAX, j = e % KMAX;
      if (j < g.k) g.c[h * g.k + j] = (float)(-1.0 + 2.0 * (double)j / (double)(g.k - 1));
      g.ws[h].sum[j][0] = 0ull;
      g.ws[h].sum[j][1] = 0ull;
      if (j == 0) {
        g.ws[h].changes = 0;
        g.ws[h].done = 0;
      }
    }
}

__global__ void __launch_bounds__(THREADS) assign_kernel(Args g) {
  __shared__ float c[KMAX];
  __shared__ unsigned long long s[KMAX][2];
  __shared__ int changed;
  const int h = blockIdx.y;
  Ws& ws = g.ws[h];
  if (ws.done) return;  // uniform over the CTA
  if (threadIdx.x < KMAX) {
    c[threadIdx.x] = threadIdx.x < g.k ? g.c[h * g.k + threadIdx.x] : 0.0f;
    s[threadIdx.x][0] = 0ull;
    s[threadIdx.x][1] = 0ull;
  }
  if (threadIdx.x == 0) changed = 0;
  __syncthreads();
  const float* a = g.a + (uint64_t)h * g.n;
  const float* w = g.w + (uint64_t)h * g.n;
  uint8_t* prev = g.prev + (uint64_t)h * g.n;
  int my_changes = 0;
  for (long long i = blockIdx.x * (long long)THREADS + threadIdx.x; i < g.n; i += (long long)gridDim.x * THREADS) {
    const float x = fminf(fmaxf(a[i], -1.0f), 1.0f);
    const float wt = fminf(fmaxf(w[i], 0.0f), 1.0f);
    int best = 0;
    float bd = fabsf(__fsub_rn(x, c[0]));
    for (int j = 1; j < g.k; ++j) {
      const float d = fabsf(__fsub_rn(x, c[j]));
      if (d < bd) {
        bd = d;
        best = j;
      }
    }
    if (prev[i] != (uint8_t)best) {
      ++my_changes;
      prev[i] = (uint8_t)best;
    }
    const long long P = __double2ll_rn(__dmul_rn(__dmul_rn((double)wt, (double)x), SCALE));  // exact product
    const long long W = __double2ll_rn(__dmul_rn((double)wt, SCALE));
    if (W != 0) {
      atomicAdd(&s[best][0], (unsigned long long)P);
      atomicAdd(&s[best][1], (unsigned long long)W);
    }
  }
  if (my_changes) atomicAdd(&changed, my_changes);
  __syncthreads();
  if (threadIdx.x < g.k) {
    if (s[threadIdx.x][1] != 0ull) {
      atomicAdd(&ws.sum[threadIdx.x][0], s[threadIdx.x][0]);
      atomicAdd(&ws.sum[threadIdx.x][1], s[threadIdx.x][1]);
    }
  }
  if (threadIdx.x == 0 && changed) atomicAdd(&ws.changes, changed);
}

__global__ void update_kernel(Args g) {
  const int h = blockIdx.x, j = threadIdx.x;
  Ws& ws = g.ws[h];
  if (ws.done) return;
  const bool stop = g.it > 0 && ws.changes == 0;  // every assignment as in the last iteration
  __syncthreads();
  if (j < g.k) {
    const long long sp = (long long)ws.sum[j][0], sw = (long long)ws.sum[j][1];
    if (!stop && sw > 0) g.c[h * g.k + j] = (float)__ddiv_rn((double)sp, (double)sw);
    ws.sum[j][0] = 0ull;
    ws.sum[j][1] = 0ull;
  }
  __syncthreads();
  if (j == 0) {
    ws.changes = 0;
    if (stop) ws.done = 1;
  }
}

}  // namespace fit
}  // namespace kvq

size_t kvq_fit_ws_bytes(int n_heads, long long n) {
  return (size_t)n_heads * sizeof(kvq::fit::Ws) + (size_t)kvq::round16((uint64_t)n_heads * (uint64_t)n);
}

cudaError_t kvq_launch_fit(const float* a, const float* w, int n_heads, long long n, int bits, int max_iter, float* c,
                           void* ws, cudaStream_t st) {
  using namespace kvq::fit;
  Args g;
  g.a = a; g.w = w; g.n = n; g.k = 1 << bits; g.c = c;
  g.ws = static_cast<Ws*>(ws);
  g.prev = static_cast<uint8_t*>(ws) + (size_t)n_heads * sizeof(Ws);
  g.it = 0;
  long long blocks = ((long long)n_heads * n + 255) / 256;
  init_kernel<<<(int)(blocks < 1024 ? (blocks > 0 ? blocks : 1) : 1024), 256, 0, st>>>(g, n_heads);
  long long chunks = (n + THREADS * 8 - 1) / (THREADS * 8);
  const long long cap = 1216 / n_heads > 0 ? 1216 / n_heads : 1;
  if (chunks > cap) chunks = cap;
  if (chunks < 1) chunks = 1;
  const dim3 grid((unsigned)chunks, (unsigned)n_heads);
  for (int it = 0; it < max_iter; ++it) {
    g.it = it;
    assign_kernel<<<grid, THREADS, 0, st>>>(g);
    update_kernel<<<n_heads, 32, 0, st>>>(g);
  }
  return cudaGetLastError();
}
