// Offline key calibration for KVQuant-style caches ([KVQ] §3.6, Algorithm 1 offline steps 3-4;
// the first token excluded as §3.5 asks): per (KV head, channel), the outlier threshold tau and
// the centre / half-range of the entries at or below it.
//
// One CTA per (channel, head). The magnitude of an fp16 or bf16 value is its low 15 bits read
// as an integer (monotone in |x| for finite values), so tau, the rank-th smallest |k| over tokens
// 1 .. n-1, comes from a two-pass radix select: a 256-bin histogram of the high 8 bits, then a
// 128-bin histogram of the low 7 bits inside the bin that holds the rank. A third pass takes the
// minimum and maximum of the entries whose magnitude does not exceed tau.
#include "kvq_internal.cuh"

namespace kvq {

constexpr int CAL_THREADS = 256;

__global__ void __launch_bounds__(CAL_THREADS) calibrate_kernel(Geo g, uint8_t* base, const uint16_t* k,
                                                                int n_tokens, int rank) {
  __shared__ int hist[256];
  __shared__ int sel[2];
  __shared__ float red[2][CAL_THREADS / 32];
  const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const uint16_t* col = k + (uint64_t)h * n_tokens * D + c;  // token t at col[t * D]
  float* tau_tab = reinterpret_cast<float*>(base + g.calib_off);
  uint16_t* s_tab = reinterpret_cast<uint16_t*>(base + g.calib_off + (uint64_t)g.H * D * 4);
  uint16_t* zp_tab = s_tab + (uint64_t)g.H * D;

  int tau_key = 0x7fff;  // rank 0: no threshold (every finite magnitude is kept)
  if (rank > 0) {
    hist[tid] = 0;
    __syncthreads();
    for (int t = 1 + tid; t < n_tokens; t += CAL_THREADS) atomicAdd(&hist[(col[(uint64_t)t * D] & 0x7fff) >> 7], 1);
    __syncthreads();
    if (tid == 0) {
      int cum = 0, bin = 0;
      for (; bin < 255; ++bin) {
        if (cum + hist[bin] >= rank) break;
        cum += hist[bin];
      }
      sel[0] = bin;
      sel[1] = cum;  // entries in lower bins
    }
    __syncthreads();
    const int bin = sel[0];
    hist[tid] = 0;
    __syncthreads();
    for (int t = 1 + tid; t < n_tokens; t += CAL_THREADS) {
      const int m = col[(uint64_t)t * D] & 0x7fff;
      if ((m >> 7) == bin) atomicAdd(&hist[m & 127], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int cum = sel[1], lo = 0;
      for (; lo < 127; ++lo) {
        if (cum + hist[lo] >= rank) break;
        cum += hist[lo];
      }
      sel[0] = (bin << 7) | lo;
    }
    __syncthreads();
    tau_key = sel[0];
  }

  // centre / half-range of the entries with |k| <= tau
  float mx = -INFINITY, mn = INFINITY;
  for (int t = 1 + tid; t < n_tokens; t += CAL_THREADS) {
    const uint16_t u = col[(uint64_t)t * D];
    if ((u & 0x7fff) > tau_key) continue;
    const float v = in_bits_to_f32(u, g.in_bf16);
    mx = fmaxf(mx, v);
    mn = fminf(mn, v);
  }
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if ((tid & 31) == 0) {
    red[0][tid >> 5] = mx;
    red[1][tid >> 5] = mn;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < CAL_THREADS / 32; ++w) {
      mx = fmaxf(mx, red[0][w]);
      mn = fminf(mn, red[1][w]);
    }
    uint16_t s16 = 0, zp16 = 0;
    if (mx != -INFINITY) {
      zp16 = f2h_rn(__fdiv_rn(__fadd_rn(mx, mn), 2.0f));
      s16 = f2h_rn(__fdiv_rn(__fsub_rn(mx, mn), 2.0f));
    }
    tau_tab[h * D + c] = rank > 0 ? in_bits_to_f32((uint16_t)tau_key, g.in_bf16) : INFINITY;
    s_tab[h * D + c] = s16;
    zp_tab[h * D + c] = zp16;
  }
}

}  // namespace kvq

cudaError_t kvq_launch_calibrate(const kvq::Geo& g, uint8_t* base, const uint16_t* k, int n_tokens, int rank,
                                 cudaStream_t st) {
  dim3 grid(kvq::D, g.H);
  kvq::calibrate_kernel<<<grid, kvq::CAL_THREADS, 0, st>>>(g, base, k, n_tokens, rank);
  return cudaGetLastError();
}
