// Sensitivity-weighted nuq codebook fitting ([KVQ] §3.3, Algorithm 2): Lloyd iterations per KV
// head on normalised calibration samples with Fisher weights.
//
// Per iteration, an assign kernel (grid: sample chunks x heads) gives every sample its nearest
// centre (|a - c_j| in fp32, the lowest j on ties) and adds w*a and w, each scaled by 2^32 and
// rounded half-even to a 64-bit integer, into that centre's sums. The sums are integers, so the
// result does not depend on the order of the additions. Each thread owns one (sum w*a, sum w)
// slot per centre in shared memory (no contention, no atomics in the sample loop); the CTA folds
// its slots and adds them to the head's sums with one global atomic per centre and sum.
//
// An update kernel (one warp per head) then moves each centre whose members weigh more than zero
// to the fp64 quotient of its sums rounded to fp32. A head stops when an update leaves every
// centre's bits unchanged. That gives the codebook of the rule "stop when no assignment changed"
// for every iteration cap: equal assignments give equal centres (same members, same sums; a
// centre without weight keeps its value), and equal centres give equal assignments on the next
// pass; so the two rules stop at most one pass apart with the same centres. No per-sample state
// is kept between passes, and a pass reads 8 bytes per sample.
//
// The pass is bound by the integer/logic pipe, so the per-sample work is kept small: the
// fixed-point products are taken in integer arithmetic (the two 24-bit significands make a 48-bit
// integer, shifted into place with round-half-even; fp64 runs at a small fraction of the integer
// rate on this part), and the nearest centre comes from a descent over precomputed decision
// thresholds whenever the centres allow it (see well_separated).
#include "kvq_internal.cuh"

namespace kvq {
namespace fit {

constexpr int THREADS = 256;
constexpr int KMAX = 16;

struct Ws {  // per head
  unsigned long long sum[KMAX][2];  // sum of round(w*a*2^32) (two's complement), sum of round(w*2^32)
  int done;
  int pad[3];
};

struct Args {
  const float* a;
  const float* w;
  long long n;
  int k;
  float* c;  // [H][k]
  Ws* ws;    // [H]
};

// rint(w * a * 2^32), exactly, for w in [0, 1] and a in [-1, 1] (fp32, finite): the significands
// multiply into a signed 48-bit integer m, and w*a*2^32 = m * 2^-s with s >= 14. Half-even
// rounding of m / 2^s in two's complement: floor((m + 2^(s-1) - 1 + parity(floor(m / 2^s))) / 2^s).
// A zero or subnormal operand makes s >= 141 (clamped to 63), where the result is 0 as it should be.
__device__ __forceinline__ long long fixed_product(float w, float a) {
  const uint32_t bw = __float_as_uint(w), ba = __float_as_uint(a);
  const int s = min(268 - (int)((bw >> 23) & 0xFFu) - (int)((ba >> 23) & 0xFFu), 63);
  const int ma = (int)((ba & 0x7FFFFFu) | 0x800000u);
  const long long m = (long long)((bw & 0x7FFFFFu) | 0x800000u) * (long long)((int)ba < 0 ? -ma : ma);
  return (m + ((1ll << (s - 1)) - 1ll + ((m >> s) & 1ll))) >> s;
}

// Nearest centre of x: |x - c_j| in fp32, the lowest j on ties.
template <int K>
__device__ __forceinline__ int nearest(float x, const float (&c)[K]) {
  int best = 0;
  float bd = fabsf(__fsub_rn(x, c[0]));
#pragma unroll
  for (int j = 1; j < K; ++j) {
    const float d = fabsf(__fsub_rn(x, c[j]));
    if (d < bd) {
      bd = d;
      best = j;
    }
  }
  return best;
}

// Order-preserving map of fp32 values to int32 (and back).
__device__ __forceinline__ int order_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float from_order_key(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7FFFFFFF); }

// When adjacent centres are sorted and more than 2^-21 apart, the fp32 differences x - c_j keep
// their order for every x in [-1, 1] (each is off by at most 2^-24), so the nearest centre is a
// non-decreasing function of x: nearest(x) = #{j >= 1 : x >= t_j}, with t_j the smallest fp32 value
// whose nearest centre is j or above. t_j is found by bisection over the ordered fp32 values of
// [-1, 1], and the K - 1 thresholds are kept in Eytzinger order (node i, children 2i and 2i + 1)
// for a branch-free descent.
template <int K>
__device__ bool well_separated(const float (&c)[K]) {
  bool ok = true;
#pragma unroll
  for (int j = 0; j + 1 < K; ++j) ok &= __fsub_rn(c[j + 1], c[j]) > 4.76837158203125e-7f;  // 2^-21
  return ok;
}

template <int K>
__device__ float threshold(int j, const float (&c)[K]) {
  int lo = order_key(-1.0f), hi = order_key(1.0f);  // nearest(-1) = 0 < j <= K - 1 = nearest(1)
  while (hi - lo > 1) {
    const int mid = (int)(((long long)lo + (long long)hi) >> 1);
    if (nearest<K>(from_order_key(mid), c) >= j)
      hi = mid;
    else
      lo = mid;
  }
  return from_order_key(hi);
}

template <int K, bool SORTED>
__device__ __forceinline__ void add_sample(float x, float wt, const float (&c)[K], const float* eyt, float root,
                                           ulonglong2* slot) {
  x = fminf(fmaxf(x, -1.0f), 1.0f);
  wt = __saturatef(wt);
  int best;
  if (SORTED) {
    int i = 2 + (x >= root ? 1 : 0);
#pragma unroll
    for (int l = 1; (1 << l) < K; ++l) i = 2 * i + (x >= eyt[i] ? 1 : 0);
    best = i - K;
  } else {
    best = nearest<K>(x, c);
  }
  const unsigned long long P = (unsigned long long)fixed_product(wt, x);
  const unsigned long long W = __float2ull_rn(__fmul_rn(wt, 4294967296.0f));  // w * 2^32 is exact in fp32
  ulonglong2& s = slot[best * THREADS];
  ulonglong2 v = s;
  v.x += P;
  v.y += W;
  s = v;
}

__global__ void init_kernel(Args g, int n_heads) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n_heads * KMAX; e += gridDim.x * blockDim.x) {
    const int h = e / KMAX, j = e % KMAX;
    if (j < g.k) g.c[h * g.k + j] = (float)(-1.0 + 2.0 * (double)j / (double)(g.k - 1));  // evenly spaced
    g.ws[h].sum[j][0] = 0ull;
    g.ws[h].sum[j][1] = 0ull;
    if (j == 0) g.ws[h].done = 0;
  }
}

template <int K, bool VEC, bool SORTED>
__device__ __forceinline__ void sample_loop(const Args& g, int h, int t, const float (&c)[K], const float* eyt,
                                            ulonglong2* my) {
  const float root = eyt[1];
  const float* a = g.a + (uint64_t)h * g.n;
  const float* w = g.w + (uint64_t)h * g.n;
  const long long stride = (long long)gridDim.x * THREADS;
  if (VEC) {  // n % 4 == 0 and 16-byte aligned rows
    const float4* a4 = reinterpret_cast<const float4*>(a);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const long long n4 = g.n >> 2;
    long long i = blockIdx.x * (long long)THREADS + t;
    for (; i + stride < n4; i += 2 * stride) {  // two float4 pairs in flight
      const float4 x0 = __ldg(a4 + i), w0 = __ldg(w4 + i), x1 = __ldg(a4 + i + stride), w1 = __ldg(w4 + i + stride);
      add_sample<K, SORTED>(x0.x, w0.x, c, eyt, root, my);
      add_sample<K, SORTED>(x0.y, w0.y, c, eyt, root, my);
      add_sample<K, SORTED>(x0.z, w0.z, c, eyt, root, my);
      add_sample<K, SORTED>(x0.w, w0.w, c, eyt, root, my);
      add_sample<K, SORTED>(x1.x, w1.x, c, eyt, root, my);
      add_sample<K, SORTED>(x1.y, w1.y, c, eyt, root, my);
      add_sample<K, SORTED>(x1.z, w1.z, c, eyt, root, my);
      add_sample<K, SORTED>(x1.w, w1.w, c, eyt, root, my);
    }
    if (i < n4) {
      const float4 x0 = __ldg(a4 + i), w0 = __ldg(w4 + i);
      add_sample<K, SORTED>(x0.x, w0.x, c, eyt, root, my);
      add_sample<K, SORTED>(x0.y, w0.y, c, eyt, root, my);
      add_sample<K, SORTED>(x0.z, w0.z, c, eyt, root, my);
      add_sample<K, SORTED>(x0.w, w0.w, c, eyt, root, my);
    }
  } else {
    for (long long i = blockIdx.x * (long long)THREADS + t; i < g.n; i += stride)
      add_sample<K, SORTED>(__ldg(a + i), __ldg(w + i), c, eyt, root, my);
  }
}

// grid (chunks, heads), THREADS threads, K * THREADS * 16 bytes of dynamic shared memory
template <int K, bool VEC>
__global__ void __launch_bounds__(THREADS) assign_kernel(Args g) {
  extern __shared__ ulonglong2 slots[];  // [K][THREADS]
  __shared__ float eyt[KMAX];            // thresholds, Eytzinger order (nodes 1 .. K-1)
  const int h = blockIdx.y, t = threadIdx.x;
  Ws& ws = g.ws[h];
  if (*(volatile int*)&ws.done) return;  // uniform over the CTA
  float c[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    c[j] = g.c[h * K + j];
    slots[j * THREADS + t] = make_ulonglong2(0ull, 0ull);
  }
  const bool sorted = well_separated<K>(c);  // the same in every thread
  if (t < KMAX) eyt[t] = 0.0f;
  if (sorted && t >= 1 && t < K) {
    // node t at depth d holds the threshold of in-order rank (2 (t - 2^d) + 1) 2^(log2 K - d - 1)
    const int d = 31 - __clz(t), lk = 31 - __clz(K);
    eyt[t] = threshold<K>((2 * (t - (1 << d)) + 1) << (lk - d - 1), c);
  }
  __syncthreads();
  ulonglong2* my = slots + t;
  if (sorted)
    sample_loop<K, VEC, true>(g, h, t, c, eyt, my);
  else
    sample_loop<K, VEC, false>(g, h, t, c, eyt, my);
  __syncthreads();
  // fold: warp q sums centres q, q + 8, ...; lane l reads slots l, l + 32, ...
  const int warp = t >> 5, lane = t & 31;
  for (int j = warp; j < K; j += THREADS / 32) {
    unsigned long long sp = 0ull, sw = 0ull;
#pragma unroll
    for (int r = lane; r < THREADS; r += 32) {
      const ulonglong2 v = slots[j * THREADS + r];
      sp += v.x;
      sw += v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sp += __shfl_xor_sync(0xffffffffu, sp, o);
      sw += __shfl_xor_sync(0xffffffffu, sw, o);
    }
    if (lane == 0 && sw != 0ull) {
      atomicAdd(&ws.sum[j][0], sp);
      atomicAdd(&ws.sum[j][1], sw);
    }
  }
}

// grid n_heads, 32 threads
__global__ void update_kernel(Args g) {
  const int h = blockIdx.x, j = threadIdx.x;
  Ws& ws = g.ws[h];
  if (ws.done) return;
  bool moved = false;
  if (j < g.k) {
    const long long sp = (long long)ws.sum[j][0], sw = (long long)ws.sum[j][1];
    const float old = g.c[h * g.k + j];
    const float nc = sw > 0 ? (float)__ddiv_rn((double)sp, (double)sw) : old;
    moved = __float_as_uint(nc) != __float_as_uint(old);
    g.c[h * g.k + j] = nc;
    ws.sum[j][0] = 0ull;
    ws.sum[j][1] = 0ull;
  }
  if (!__any_sync(0xffffffffu, moved) && j == 0) ws.done = 1;
}

template <int K>
cudaError_t launch_iterations(const Args& g, int n_heads, int max_iter, cudaStream_t st) {
  const bool vec = (g.n & 3) == 0 && ((uintptr_t)g.a & 15) == 0 && ((uintptr_t)g.w & 15) == 0;
  const int smem = K * THREADS * (int)sizeof(ulonglong2);
  const void* fn = vec ? (const void*)assign_kernel<K, true> : (const void*)assign_kernel<K, false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, THREADS, smem)) != cudaSuccess) return e;
  // enough CTAs to fill the GPU once over all heads, each with at least 32 samples per thread
  long long chunks = (g.n + THREADS * 32 - 1) / (THREADS * 32);
  const long long cap = (long long)sms * (per_sm > 0 ? per_sm : 1) / n_heads;
  if (chunks > cap) chunks = cap;
  if (chunks < 1) chunks = 1;
  const dim3 grid((unsigned)chunks, (unsigned)n_heads);
  for (int it = 0; it < max_iter; ++it) {
    if (vec)
      assign_kernel<K, true><<<grid, THREADS, smem, st>>>(g);
    else
      assign_kernel<K, false><<<grid, THREADS, smem, st>>>(g);
    update_kernel<<<n_heads, 32, 0, st>>>(g);
  }
  return cudaGetLastError();
}

}  // namespace fit
}  // namespace kvq

size_t kvq_fit_ws_bytes(int n_heads, long long) { return (size_t)n_heads * sizeof(kvq::fit::Ws); }

cudaError_t kvq_launch_fit(const float* a, const float* w, int n_heads, long long n, int bits, int max_iter, float* c,
                           void* ws, cudaStream_t st) {
  using namespace kvq::fit;
  Args g;
  g.a = a; g.w = w; g.n = n; g.k = 1 << bits; g.c = c;
  g.ws = static_cast<Ws*>(ws);
  init_kernel<<<(n_heads * KMAX + 255) / 256, 256, 0, st>>>(g, n_heads);
  switch (bits) {
    case 1: return launch_iterations<2>(g, n_heads, max_iter, st);
    case 2: return launch_iterations<4>(g, n_heads, max_iter, st);
    case 3: return launch_iterations<8>(g, n_heads, max_iter, st);
    default: return launch_iterations<16>(g, n_heads, max_iter, st);
  }
}
