// Decode attention over the packed cache: split-K flash-decode plus a combine kernel.
//
// decode_kernel: grid (n_split, H_kv, B), 128 threads. A CTA owns a contiguous range of
// blocks of one (b, h) and all G = H_q/H_kv query heads that share it. Whole block records
// (K tile + V tile: codes, fp16 metadata, CSR) stream from HBM into a 3-stage shared-memory
// ring by 1-D bulk copies (cp.async.bulk, completion on an mbarrier; every wait is bounded).
// Per block:
//   K phase (thread = token): unpack, dequantise in registers ((q+z)*s, C[q]*s+zp, q*s, times
//     s1), add the CSR outliers, rotate pre-RoPE keys at their absolute position, dot with the
//     G queries ([KVQ] §3.7 key matvec steps 1-6, Algorithm 1 dequantisation).
//   online softmax over the block's 128 scores (running max and sum per head, base 2).
//   V phase (thread = channel): unpack, dequantise, weighted sum with the probabilities, plus
//     the channel's value outliers (CSR, or CSC for v_csc caches) ([KVQ] §3.7 value matvec;
//     [KVN] step 5 with s1; [TQ] §5.2: dequantise inside attention).
// No dequantised value is written to memory. Each CTA writes (m, l, o[128]) per query head.
//
// combine_kernel: grid (H_q, B), 128 threads: merges the splits, applies the inverse FWHT for
// KVarN caches, attends the fp tail (< 128 tokens, RoPE'd at its positions for pre-RoPE
// caches) and writes out = o / l.
#include "kvq_internal.cuh"

namespace kvq {

constexpr int DC_THREADS = 128;
constexpr int NSTAGE = 3;
constexpr float LOG2E_RSQRT_D = 1.4426950408889634f * 0.08838834764831845f;  // log2(e)/sqrt(128)

struct DecodeArgs {
  Geo g;
  const uint8_t* base;
  const float* codebook;
  const uint16_t* q;
  int n_blocks;
  int n_split;
  float* ws_m;
  float* ws_l;
  float* ws_o;
  int* status;
  int hadamard;
};

struct CombineArgs {
  Geo g;
  const uint8_t* base;
  const uint16_t* q;
  const uint16_t* tail_k;
  const uint16_t* tail_v;
  int n_tail;
  long long tail_bh;    // elements between the tail rows of consecutive (b, h)
  long long tail_tok;   // elements between consecutive tokens of a tail row
  int n_blocks;
  int n_split;          // partial rows per (b, query head) in the workspace
  int tail_ws;          // 1: the decode kernel attended the fp tail into the last of those rows
  long long ranges;     // > 0: partials come from the range-split tensor-core decode
  int per_range;        // partial rows per range and (b, query head)
  long long total;      // B * H * n_blocks
  const float* ws_m;
  const float* ws_l;
  const float* ws_o;
  float* out;
  int hadamard;
  const int* status;    // the cache's status word: a decode that timed out left its partials unwritten
};

// 1/sqrt(128)-scaled FWHT of `n` rows of 128 fp32 values in shared memory (row stride 128).
__device__ void smem_fwht(float* x, int n) {
  for (int hh = 1; hh < D; hh <<= 1) {
    for (int it = threadIdx.x; it < n * (D / 2); it += blockDim.x) {
      int r = it >> 6, j = it & 63;
      int i0 = (j / hh) * (2 * hh) + (j % hh);
      float a = x[r * D + i0], b = x[r * D + i0 + hh];
      x[r * D + i0] = a + b;
      x[r * D + i0 + hh] = a - b;
    }
    __syncthreads();
  }
  for (int it = threadIdx.x; it < n * D; it += blockDim.x) x[it] *= 0.08838834764831845f;
  __syncthreads();
}

template <int GMAX>
struct DecSmem {
  float qraw[GMAX][D];    // query (Hadamard domain for KVarN)
  float qs[GMAX][D];      // query used by the K phase (rotated by the block's base angle if pre-RoPE)
  float pv[GMAX][T];      // probabilities times the per-token value scale
  float osp[GMAX][D];     // NUQ value outliers weighted by p
  float red[2][GMAX][DC_THREADS / 32];
  float cb[16];
  uint64_t bar[NSTAGE];
};

template <int METHOD, int GMAX>
__global__ void __launch_bounds__(DC_THREADS) decode_kernel(DecodeArgs a) {
  launch_dependents();  // the combine kernel may be scheduled once every CTA of this grid runs
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const Geo& g = a.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = g.G;
  const int rec = (int)g.rec_bytes;
  uint8_t* stages = smem_raw;
  DecSmem<GMAX>* sm = reinterpret_cast<DecSmem<GMAX>*>(smem_raw + NSTAGE * rec);

  const int nb = a.n_blocks;
  const int blk_begin = (int)((long long)nb * split / a.n_split);
  const int blk_end = (int)((long long)nb * (split + 1) / a.n_split);
  const int n_my = blk_end - blk_begin;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&sm->bar[s], 1);
    fence_mbar_init();
    fence_proxy_async();
    for (int s = 0; s < NSTAGE && s < n_my; ++s) {
      mbar_arrive_expect_tx(&sm->bar[s], (uint32_t)rec);
      bulk_g2s(stages + s * rec, a.base + record_offset(g, b, h, blk_begin + s, a.status), (uint32_t)rec, &sm->bar[s]);
    }
  }
  // queries of this KV head's group
  for (int i = tid; i < G * D; i += DC_THREADS) {
    int gg = i >> 7, c = i & 127;
    sm->qraw[gg][c] = load_in(a.q + ((uint64_t)b * g.Hq + h * G + gg) * D + c, g.in_bf16);
  }
  if (METHOD == KVQ_NUQ && tid < (1 << g.bits)) sm->cb[tid] = a.codebook[h * (1 << g.bits) + tid];
  __syncthreads();
  if (METHOD == KVQ_VARN && a.hadamard) smem_fwht(&sm->qraw[0][0], G);
  if (!g.pre_rope) {
    for (int i = tid; i < G * D; i += DC_THREADS) sm->qs[i >> 7][i & 127] = sm->qraw[i >> 7][i & 127];
  }
  __syncthreads();

  const int bits = g.bits, W = g.W, nw = 32 / bits;
  const uint32_t cmask = (1u << bits) - 1u;
  const float2* rope_blk = reinterpret_cast<const float2*>(a.base + g.rope_off);
  const float2* rope_off = rope_blk + (size_t)(g.max_blocks + 1) * 64;

  float m_run[GMAX], l_run[GMAX], o[GMAX];
#pragma unroll
  for (int k = 0; k < GMAX; ++k) {
    m_run[k] = -INFINITY;
    l_run[k] = 0.0f;
    o[k] = 0.0f;
  }

  bool ok = true;
  int failed_at = n_my;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % NSTAGE;
    const int blk = blk_begin + i;
    const bool got = mbar_wait_bounded(&sm->bar[s], (uint32_t)((i / NSTAGE) & 1), a.status);
    if (__syncthreads_or(!got)) {  // every thread leaves together
      ok = false;
      failed_at = i;
      break;
    }
    const uint8_t* st = stages + s * rec;
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(st + g.codes_off[0]);
    const uint16_t* km = reinterpret_cast<const uint16_t*>(st + g.meta_off[0]);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + g.codes_off[1]);
    const uint16_t* vm = reinterpret_cast<const uint16_t*>(st + g.meta_off[1]);

    if (g.pre_rope) {  // q0 = R(n0)^T q, n0 = blk*128
      for (int it = tid; it < G * 64; it += DC_THREADS) {
        int gg = it >> 6, p = it & 63;
        float2 cs = rope_blk[(size_t)blk * 64 + p];
        float x0 = sm->qraw[gg][2 * p], x1 = sm->qraw[gg][2 * p + 1];
        sm->qs[gg][2 * p] = cs.x * x0 + cs.y * x1;
        sm->qs[gg][2 * p + 1] = -cs.y * x0 + cs.x * x1;
      }
    }
    if (METHOD == KVQ_NUQ) {
#pragma unroll
      for (int k = 0; k < GMAX; ++k)
        if (k < G) sm->osp[k][tid] = 0.0f;
    }
    __syncthreads();

    // ---------------- K phase: thread = token t
    const int t = tid;
    float acc[GMAX];
#pragma unroll
    for (int k = 0; k < GMAX; ++k) acc[k] = 0.0f;
    for (int c = 0; c < D; c += 2) {
      {
        uint32_t c0, c1;
        if (g.planes3) {
          c0 = tile3_code(kc, 0, t, c);
          c1 = tile3_code(kc, 0, t, c + 1);
        } else {  // n = floor(32/bits) (16, 10, 8, 4) is even: a channel pair never straddles two words
          const int w = c / nw, j = c - w * nw;
          const uint32_t word = kc[t * W + w];
          c0 = (word >> (bits * j)) & cmask;
          c1 = (word >> (bits * (j + 1))) & cmask;
        }
        float k0, k1;
        if (METHOD == KVQ_RTN || METHOD == KVQ_VARN) {
          k0 = ((float)c0 + h2f(km[T + c])) * h2f(km[c]);
          k1 = ((float)c1 + h2f(km[T + c + 1])) * h2f(km[c + 1]);
        } else if (METHOD == KVQ_INT4) {  // b-bit two's complement; per-half scales applied here
          k0 = (float)((int)(c0 << (32 - bits)) >> (32 - bits));
          k1 = (float)((int)(c1 << (32 - bits)) >> (32 - bits));
          if (g.g64) {
            const float sc = h2f(km[(c >> 6) * T + t]);
            k0 *= sc;
            k1 *= sc;
          }
        } else {
          k0 = sm->cb[c0] * h2f(km[c]) + h2f(km[T + c]);
          k1 = sm->cb[c1] * h2f(km[c + 1]) + h2f(km[T + c + 1]);
        }
        if (g.pre_rope) {
          float2 cs = rope_off[t * 64 + (c >> 1)];
          float r0 = cs.x * k0 - cs.y * k1, r1 = cs.y * k0 + cs.x * k1;
          k0 = r0;
          k1 = r1;
        }
#pragma unroll
        for (int k = 0; k < GMAX; ++k)
          if (k < G) acc[k] += sm->qs[k][c] * k0 + sm->qs[k][c + 1] * k1;
      }
    }
    if (METHOD == KVQ_NUQ && g.n_out > 0) {
      const uint8_t* csr = st + g.csr_off[0];
      const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
      const uint16_t* rp = reinterpret_cast<const uint16_t*>(csr + 2 * g.n_out);
      const uint8_t* col = csr + 2 * g.n_out + 2 * (T + 1);
      const int j1 = min((int)rp[t + 1], g.n_out);
      for (int j = min((int)rp[t], g.n_out); j < j1; ++j) {
        const int c = col[j] & (D - 1);
        const float v = h2f(val[j]);
        if (g.pre_rope) {
          float2 cs = rope_off[t * 64 + (c >> 1)];
#pragma unroll
          for (int k = 0; k < GMAX; ++k) {
            if (k < G) {
              float a0 = sm->qs[k][c & ~1], a1 = sm->qs[k][c | 1];
              float qq = (c & 1) ? (-cs.y * a0 + cs.x * a1) : (cs.x * a0 + cs.y * a1);
              acc[k] += v * qq;
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < GMAX; ++k)
            if (k < G) acc[k] += v * sm->qs[k][c];
        }
      }
    }
    float tscale = LOG2E_RSQRT_D;
    if (METHOD == KVQ_INT4 && !g.g64) tscale *= h2f(km[t]);
    if (METHOD == KVQ_VARN) tscale *= h2f(km[2 * T + t]);

    // ---------------- online softmax (base 2)
    float s2[GMAX];
#pragma unroll
    for (int k = 0; k < GMAX; ++k) {
      s2[k] = acc[k] * tscale;
      if (METHOD == KVQ_NUQ && g.sink && blk == 0 && t == 0) s2[k] = -INFINITY;  // the kept first token
      float mx = s2[k];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane == 0 && k < G) sm->red[0][k][warp] = mx;
    }
    __syncthreads();
    float alpha[GMAX];
#pragma unroll
    for (int k = 0; k < GMAX; ++k) {
      if (k < G) {
        float mb = fmaxf(fmaxf(sm->red[0][k][0], sm->red[0][k][1]), fmaxf(sm->red[0][k][2], sm->red[0][k][3]));
        float mn = fmaxf(m_run[k], mb);
        alpha[k] = exp2f(m_run[k] - mn);
        m_run[k] = mn;
        float p = exp2f(s2[k] - mn);
        float ps = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        if (lane == 0) sm->red[1][k][warp] = ps;
        float vs = 1.0f;
        if (METHOD != KVQ_NUQ && !(METHOD == KVQ_INT4 && g.g64)) vs = h2f(vm[t]);  // per-token value scale folded into p
        sm->pv[k][t] = p * vs;
      } else {
        alpha[k] = 1.0f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < GMAX; ++k)
      if (k < G)
        l_run[k] = l_run[k] * alpha[k] +
                   ((sm->red[1][k][0] + sm->red[1][k][1]) + (sm->red[1][k][2] + sm->red[1][k][3]));

    if (METHOD == KVQ_NUQ && g.n_out > 0) {  // value outliers, weighted by p
      const uint8_t* csr = st + g.csr_off[1];
      const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
      const uint16_t* rp = reinterpret_cast<const uint16_t*>(csr + 2 * g.n_out);
      const uint8_t* col = csr + 2 * g.n_out + 2 * (T + 1);
      // thread c adds the entries of channel c in token order (the sum does not depend on timing,
      // and it is the same for CSR and CSC tiles)
      const int c = tid;
      float acc[GMAX];
#pragma unroll
      for (int k = 0; k < GMAX; ++k) acc[k] = 0.0f;
      if (g.v_csc) {  // column c is one run of entries; rp is the column pointer, col the token
        const int j1 = min((int)rp[c + 1], g.n_out);
        for (int j = min((int)rp[c], g.n_out); j < j1; ++j) {
          const int tj = col[j] & (T - 1);
          const float v = h2f(val[j]);
#pragma unroll
          for (int k = 0; k < GMAX; ++k)
            if (k < G) acc[k] = fmaf(sm->pv[k][tj], v, acc[k]);
        }
      } else {
        uint8_t* vtag = reinterpret_cast<uint8_t*>(sm + 1);  // the token of each entry
        {
          const int j1 = min((int)rp[t + 1], g.n_out);
          for (int j = min((int)rp[t], g.n_out); j < j1; ++j) vtag[j] = (uint8_t)t;
        }
        __syncthreads();
        const int n_v = min((int)rp[T], g.n_out);
        for (int j = 0; j < n_v; ++j) {
          if ((col[j] & (D - 1)) != c) continue;
          const int tj = vtag[j];
          const float v = h2f(val[j]);
#pragma unroll
          for (int k = 0; k < GMAX; ++k)
            if (k < G) acc[k] = fmaf(sm->pv[k][tj], v, acc[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < GMAX; ++k)
        if (k < G) sm->osp[k][c] += acc[k];
      __syncthreads();
    }

    // ---------------- V phase: thread = channel c (value rows are channels)
    {
      const int c = tid;
      float bs[GMAX];
#pragma unroll
      for (int k = 0; k < GMAX; ++k) bs[k] = 0.0f;
      for (int tt = 0; tt < T; ++tt) {
        const uint32_t code = g.planes3 ? tile3_code(vc, 1, tt, c)
                              : g.vrows_ch ? (vc[c * W + tt / nw] >> (bits * (tt % nw))) & cmask
                                           : (vc[tt * W + c / nw] >> (bits * (c % nw))) & cmask;
        float val;
        if (METHOD == KVQ_RTN || METHOD == KVQ_VARN) {
          val = (float)code + h2f(vm[T + tt]);
        } else if (METHOD == KVQ_INT4) {
          val = (float)((int)(code << (32 - bits)) >> (32 - bits));
          if (g.g64) val *= h2f(vm[(c >> 6) * T + tt]);
        } else {
          val = sm->cb[code] * h2f(vm[tt]) + h2f(vm[T + tt]);
        }
#pragma unroll
        for (int k = 0; k < GMAX; ++k)
          if (k < G) bs[k] += sm->pv[k][tt] * val;
      }
      float s1c = 1.0f;
      if (METHOD == KVQ_VARN) s1c = h2f(vm[2 * T + c]);
#pragma unroll
      for (int k = 0; k < GMAX; ++k) {
        if (k < G) {
          float add = bs[k];
          if (METHOD == KVQ_NUQ) add += sm->osp[k][c];
          o[k] = o[k] * alpha[k] + add * s1c;
        }
      }
    }
    __syncthreads();  // every thread is done with stage s
    if (tid == 0 && i + NSTAGE < n_my) {
      fence_proxy_async();
      mbar_arrive_expect_tx(&sm->bar[s], (uint32_t)rec);
      bulk_g2s(stages + s * rec, a.base + record_offset(g, b, h, blk + NSTAGE, a.status), (uint32_t)rec, &sm->bar[s]);
    }
  }

  if (!ok) {
    // a wait gave up: wait (bounded) for the copies still in flight before the CTA exits
    if (tid == 0) {
      for (int j = failed_at; j < n_my && j < failed_at + NSTAGE; ++j)
        mbar_wait_bounded(&sm->bar[j % NSTAGE], (uint32_t)((j / NSTAGE) & 1), nullptr, 200000000LL);
    }
    __syncthreads();
    return;
  }
#pragma unroll
  for (int k = 0; k < GMAX; ++k) {
    if (k < G) {
      const uint64_t row = ((uint64_t)b * g.Hq + h * G + k) * a.n_split + split;
      a.ws_o[row * D + tid] = o[k];
      if (tid == 0) {
        a.ws_m[row] = m_run[k];
        a.ws_l[row] = l_run[k];
      }
    }
  }
}

constexpr int CB_THREADS = 512, CB_GROUPS = CB_THREADS / D;  // 4 thread groups of 128 channels
// Words per staged tail-key row: 64 channel pairs padded to 68, so that the 32 lanes reading
// pair 4j + q of tokens t (lane = 4t + q) hit 32 distinct banks (68t + q = 4t + q mod 32).
constexpr int TK_STRIDE = 68;

// Block-wide reductions over CB_THREADS threads (red: CB_THREADS/32 floats of scratch).
__device__ __forceinline__ float cb_max(float v, float* red) {
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < CB_THREADS / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}
__device__ __forceinline__ float cb_sum(float v, float* red) {
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.0f;
  for (int w = 0; w < CB_THREADS / 32; ++w) r += red[w];
  return r;
}

// grid (H_q, B), CB_THREADS threads: thread (grp, c) = (tid / 128, tid % 128).
__global__ void __launch_bounds__(CB_THREADS) combine_kernel(CombineArgs a) {
  __shared__ float red[CB_THREADS / 32];
  __shared__ float part[CB_GROUPS][D];
  __shared__ float ob[D];
  __shared__ float qv[D];
  __shared__ float sc[T];
  __shared__ uint32_t tkw[(T - 1) * TK_STRIDE];  // tail keys, one word per channel pair (input dtype bits)
  const Geo& g = a.g;
  const int tid = threadIdx.x, c = tid & (D - 1), grp = tid >> 7;
  const int hq = blockIdx.x, b = blockIdx.y, h = hq / g.G;

  // ---- first what reads only the call's inputs: the kept first token and the fp tail, as one
  // softmax state (Mt, Lt, Ot). Launched as a programmatic dependent of the decode kernel, this
  // part overlaps the decode's last blocks; the partials are read after the grid dependency.
  float Mt = -INFINITY, Lt = 0.0f, Ot = 0.0f;
  // the kept first token of the sequence (attention sink, [KVQ] §3.5) at position 0, where RoPE
  // is the identity: quantised token 0 was left out of the partials
  if (g.sink && a.n_blocks > 0) {
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(a.base + g.sink_off) + ((uint64_t)b * g.H + h) * 2 * D;
    const float qk = grp == 0 ? load_in(a.q + ((uint64_t)b * g.Hq + hq) * D + c, g.in_bf16) *
                                    in_bits_to_f32(ks[c], g.in_bf16)
                              : 0.0f;
    Mt = cb_sum(qk, red) * LOG2E_RSQRT_D;
    Lt = 1.0f;
    Ot = in_bits_to_f32(ks[D + c], g.in_bf16);
  }
  if (a.n_tail > 0 && !a.tail_ws) {  // the fp residual tail (< 128 tokens)
    const int nt = a.n_tail;
    const uint16_t* tk = a.tail_k + ((uint64_t)b * g.H + h) * a.tail_bh;
    const uint16_t* tv = a.tail_v + ((uint64_t)b * g.H + h) * a.tail_bh;
    for (int e = tid; e < nt * (D / 2); e += CB_THREADS)  // channel pairs
      tkw[(e >> 6) * TK_STRIDE + (e & 63)] = *reinterpret_cast<const uint32_t*>(tk + (e >> 6) * a.tail_tok + 2 * (e & 63));
    const float2* rope_blk = reinterpret_cast<const float2*>(a.base + g.rope_off);
    const float2* rope_loc = rope_blk + (size_t)(g.max_blocks + 1) * 64;
    if (grp == 0) {
      const float qc = load_in(a.q + ((uint64_t)b * g.Hq + hq) * D + c, g.in_bf16);
      qv[c] = qc;
    }
    __syncthreads();
    float qr = 0.0f;
    if (grp == 0 && g.pre_rope) {  // q0 = R(n0)^T q with n0 = n_blocks*128
      const int p = c >> 1;
      const float2 cs = rope_blk[(size_t)a.n_blocks * 64 + p];
      const float x0 = qv[2 * p], x1 = qv[2 * p + 1];
      qr = (c & 1) ? (-cs.y * x0 + cs.x * x1) : (cs.x * x0 + cs.y * x1);
    }
    __syncthreads();
    if (grp == 0 && g.pre_rope) qv[c] = qr;
    __syncthreads();
    // scores: token t = tid / 4, channel pairs 4j + tid%4 (j = 0..15)
    {
      const int t = tid >> 2, q4 = tid & 3;
      float acc = 0.0f;
      if (t < nt) {
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
          const int p = 4 * j + q4;
          const uint32_t kw = tkw[t * TK_STRIDE + p];
          float k0 = in_bits_to_f32((uint16_t)(kw & 0xffffu), g.in_bf16), k1 = in_bits_to_f32((uint16_t)(kw >> 16), g.in_bf16);
          if (g.pre_rope) {
            const float2 cs = rope_loc[t * 64 + p];
            const float r0 = cs.x * k0 - cs.y * k1, r1 = cs.y * k0 + cs.x * k1;
            k0 = r0;
            k1 = r1;
          }
          acc = fmaf(qv[2 * p], k0, fmaf(qv[2 * p + 1], k1, acc));
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (t < nt && q4 == 0) sc[t] = acc * LOG2E_RSQRT_D;
    }
    __syncthreads();
    const float mt = cb_max(tid < nt ? sc[tid] : -INFINITY, red);
    const float Mn = fmaxf(Mt, mt);
    const float f = exp2f(Mt - Mn);  // 0 when there is no sink term
    Lt *= f;
    Ot *= f;
    float pl = 0.0f;
    if (tid < nt) {
      pl = exp2f(sc[tid] - Mn);
      sc[tid] = pl;
    }
    Lt += cb_sum(pl, red);  // (also orders the sc[] stores)
    // values: group grp sums tokens grp, grp+4, ..., four of them per iteration with their
    // loads side by side
    float ov[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int j = grp;
    for (; j + 3 * CB_GROUPS < nt; j += 4 * CB_GROUPS) {
      float vv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) vv[k] = load_in(tv + (uint64_t)(j + k * CB_GROUPS) * a.tail_tok + c, g.in_bf16);
#pragma unroll
      for (int k = 0; k < 4; ++k) ov[k] = fmaf(sc[j + k * CB_GROUPS], vv[k], ov[k]);
    }
    for (; j < nt; j += CB_GROUPS) ov[0] = fmaf(sc[j], load_in(tv + (uint64_t)j * a.tail_tok + c, g.in_bf16), ov[0]);
    __syncthreads();
    part[grp][c] = (ov[0] + ov[1]) + (ov[2] + ov[3]);
    __syncthreads();
    Ot += (part[0][c] + part[1][c]) + (part[2][c] + part[3][c]);
    Mt = Mn;
  }

  grid_dependency_wait();  // the decode kernel's partials are complete and visible
  // A decode kernel whose bounded wait ran out returned without writing its partial rows, so the
  // workspace holds an earlier call's values: the output is marked NaN rather than merged.
  // (one thread reads the word, so that the whole CTA takes the same branch)
  __shared__ int timed_out;
  if (tid == 0)
    timed_out = a.n_blocks > 0 && a.status && *reinterpret_cast<const volatile int*>(a.status) == KVQ_ERR_TIMEOUT;
  __syncthreads();
  if (timed_out) {
    if (grp == 0) a.out[((uint64_t)b * g.Hq + hq) * D + c] = __int_as_float(0x7fc00000);
    return;
  }
  if (a.n_blocks <= 0) {
    if (grp == 0) a.out[((uint64_t)b * g.Hq + hq) * D + c] = Ot / Lt;
    return;
  }
  const uint64_t row0 = ((uint64_t)b * g.Hq + hq) * a.n_split;
  const int range_rows = a.n_split - (a.ranges > 0 && a.tail_ws ? 1 : 0);
  int n_part = a.n_split;
  if (a.ranges > 0) {  // the ranges that hold blocks of this (b, h)
    const long long u = (long long)b * g.H + h;
    const long long r0 = ((u * a.n_blocks + 1) * a.ranges - 1) / a.total;
    const long long r1 = (((u + 1) * a.n_blocks) * a.ranges - 1) / a.total;
    n_part = (int)(r1 - r0 + 1) * a.per_range;
    if (n_part > range_rows) n_part = range_rows;
  }
  if (a.tail_ws) {  // the tail's softmax state, attended by the decode kernel, joins the sink's
    const uint64_t tr = row0 + (uint64_t)(a.n_split - 1);
    const float m2 = a.ws_m[tr], l2 = a.ws_l[tr], o2 = a.ws_o[tr * D + c];
    const float Mn = fmaxf(Mt, m2);
    const float f1 = exp2f(Mt - Mn), f2 = exp2f(m2 - Mn);
    Lt = Lt * f1 + l2 * f2;
    Ot = Ot * f1 + o2 * f2;
    Mt = Mn;
  }

  // ---- merge the partials in one pass: group grp takes partials grp, grp+4, ..., eight of them
  // per chunk with their loads side by side (they sit in L2), against its own running maximum;
  // then the four groups meet in shared memory (fixed order: the result does not depend on timing)
  __shared__ float gm[CB_GROUPS], gl[CB_GROUPS];
  __syncthreads();  // part[] is reused below
  float mg = -INFINITY, Lg = 0.0f, Og = 0.0f;
  for (int s0 = grp; s0 < n_part; s0 += 8 * CB_GROUPS) {
    float mv[8], lv[8], ovv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int s = s0 + k * CB_GROUPS;
      const uint64_t r = row0 + (s < n_part ? s : s0);
      mv[k] = s < n_part ? a.ws_m[r] : -INFINITY;
      lv[k] = a.ws_l[r];
      ovv[k] = a.ws_o[r * D + c];
    }
    float mc = mg;
#pragma unroll
    for (int k = 0; k < 8; ++k) mc = fmaxf(mc, mv[k]);
    if (mc > mg) {  // group-uniform
      const float f = exp2f(mg - mc);
      Lg *= f;
      Og *= f;
      mg = mc;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float f = mv[k] == -INFINITY ? 0.0f : exp2f(mv[k] - mg);
      Lg = fmaf(lv[k], f, Lg);
      Og = fmaf(ovv[k], f, Og);
    }
  }
  part[grp][c] = Og;
  if (c == 0) {
    gm[grp] = mg;
    gl[grp] = Lg;
  }
  __syncthreads();
  float M = gm[0];
#pragma unroll
  for (int k = 1; k < CB_GROUPS; ++k) M = fmaxf(M, gm[k]);
  float L = 0.0f, O = 0.0f;
#pragma unroll
  for (int k = 0; k < CB_GROUPS; ++k) {
    const float f = gm[k] == -INFINITY ? 0.0f : exp2f(gm[k] - M);
    L = fmaf(gl[k], f, L);
    O = fmaf(part[k][c], f, O);
  }
  if (g.method == KVQ_VARN && a.hadamard && n_part > 0) {
    __syncthreads();
    if (grp == 0) ob[c] = O;
    __syncthreads();
    smem_fwht(ob, 1);
    O = ob[c];
  }
  // ---- the cached part and the sink/tail state together
  const float Mf = fmaxf(M, Mt);
  const float fc = exp2f(M - Mf), ft = exp2f(Mt - Mf);
  L = L * fc + Lt * ft;
  O = O * fc + Ot * ft;
  if (grp == 0) a.out[((uint64_t)b * g.Hq + hq) * D + c] = O / L;
}

template <int GMAX>
size_t decode_smem_bytes(const Geo& g) {
  return (size_t)NSTAGE * g.rec_bytes + sizeof(DecSmem<GMAX>) + round16((uint64_t)g.n_out);
}

template <int METHOD, int GMAX>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
  size_t smem = decode_smem_bytes<GMAX>(a.g);
  cudaError_t e = ensure_smem_attr((const void*)decode_kernel<METHOD, GMAX>, (size_t)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_split, a.g.H, a.g.B);
  decode_kernel<METHOD, GMAX><<<grid, DC_THREADS, smem, st>>>(a);
  return cudaGetLastError();
}

template <int METHOD>
cudaError_t launch_decode_m(const DecodeArgs& a, cudaStream_t st) {
  const int G = a.g.G;
  if (G <= 1) return launch_decode_t<METHOD, 1>(a, st);
  if (G <= 2) return launch_decode_t<METHOD, 2>(a, st);
  if (G <= 4) return launch_decode_t<METHOD, 4>(a, st);
  if (G <= 8) return launch_decode_t<METHOD, 8>(a, st);
  return launch_decode_t<METHOD, 16>(a, st);
}

}  // namespace kvq

// Dynamic shared memory of the CUDA-core decode for this geometry: it serves every cache, so a
// configuration whose records do not fit it three times over (with its other buffers) in one
// SM's shared memory cannot be decoded.
size_t kvq_decode_kernel_smem(const kvq::Geo& g) {
  using namespace kvq;
  const int G = g.G;
  if (G <= 1) return decode_smem_bytes<1>(g);
  if (G <= 2) return decode_smem_bytes<2>(g);
  if (G <= 4) return decode_smem_bytes<4>(g);
  if (G <= 8) return decode_smem_bytes<8>(g);
  return decode_smem_bytes<16>(g);
}

long long kvq_mma_ranges(const kvq::Geo& g);
long long kvq_nuq_ranges(const kvq::Geo& g);
int kvq_nuq_parts_per_range();
cudaError_t kvq_launch_decode_nuq(const kvq::Geo& g, const uint8_t* base, const float* codebook, const uint16_t* q,
                                  int n_blocks, long long ranges, long long slots, long long rows_ph, float* ws_m,
                                  float* ws_l, float* ws_o, int* status, const uint16_t* tail_k,
                                  const uint16_t* tail_v, int n_tail, long long tail_bh, long long tail_tok,
                                  cudaStream_t st);
long long kvq_mma_slots(const kvq::Geo& g, int n_blocks, long long ranges);
cudaError_t kvq_launch_decode_mma(const kvq::Geo& g, const uint8_t* base, const uint16_t* q, int n_blocks,
                                  long long ranges, long long slots, float* ws_m, float* ws_l, float* ws_o,
                                  int* status, int hadamard, cudaStream_t st);
int32_t kvq_decode_splits(const kvq_config* cfg, int32_t n_blocks);

namespace {
// Which decode runs for this geometry on the current device, and how many partial rows per
// (b, query head) it writes.
struct DecodePlan {
  long long ranges;  // > 0: tensor-core decode over this many ranges (warps, or CTAs for nuq)
  long long rows;    // partial rows per (b, query head)
  bool nuq;          // the 3-bit nuq pre-RoPE decode
  long long slots;   // range slots per (b, query head) (rows = slots * per_range [+ 1])
  int per_range;     // partial rows one range writes per (b, query head)
  bool tail_row;     // the last row of each (b, query head) holds the tail (the nuq decode's idle warps)
};

DecodePlan plan_decode(const kvq::Geo& g, int n_blocks, int v1_splits) {
  DecodePlan p{0, v1_splits, false, v1_splits, 1, false};
  if (n_blocks <= 0) return DecodePlan{0, 0, false, 0, 1, false};
  long long ranges = kvq_nuq_ranges(g);
  p.nuq = ranges > 0;
  if (!p.nuq) ranges = kvq_mma_ranges(g);
  const long long total = (long long)g.B * g.H * n_blocks;
  if (ranges > total) ranges = total;  // every range holds at least one block
  if (ranges > 0 && total < (1LL << 62) / ranges) {
    p.ranges = ranges;
    p.slots = kvq_mma_slots(g, n_blocks, ranges);
    p.per_range = p.nuq ? kvq_nuq_parts_per_range() : 1;
    p.tail_row = p.nuq;
    p.rows = p.slots * p.per_range + (p.tail_row ? 1 : 0);
  }
  return p;
}
}  // namespace

cudaError_t kvq_launch_decode(const kvq::Geo& g, const uint8_t* base, const float* codebook, const uint16_t* q,
                              const uint16_t* tail_k, const uint16_t* tail_v, int n_tail, long long tail_bh,
                              long long tail_tok, int n_blocks,
                              int n_split, float* ws, float* out, int* status, int hadamard, cudaStream_t st) {
  using namespace kvq;
  const DecodePlan plan = plan_decode(g, n_blocks, n_split);
  const uint64_t rows = (uint64_t)g.B * g.Hq * plan.rows;
  float* ws_m = ws;
  float* ws_l = ws + rows;
  float* ws_o = ws + 2 * rows + ((4 - (2 * rows) % 4) % 4);  // keep o 16-byte aligned
  if (n_blocks > 0) {
    cudaError_t e;
    if (plan.ranges > 0 && plan.nuq) {
      e = kvq_launch_decode_nuq(g, base, codebook, q, n_blocks, plan.ranges, plan.slots, plan.rows, ws_m, ws_l, ws_o,
                                status, tail_k, tail_v, n_tail, tail_bh, tail_tok, st);
    } else if (plan.ranges > 0) {
      e = kvq_launch_decode_mma(g, base, q, n_blocks, plan.ranges, plan.slots, ws_m, ws_l, ws_o, status, hadamard,
                                st);
    } else {
      DecodeArgs a;
      a.g = g; a.base = base; a.codebook = codebook; a.q = q; a.n_blocks = n_blocks; a.n_split = n_split;
      a.ws_m = ws_m; a.ws_l = ws_l; a.ws_o = ws_o; a.status = status; a.hadamard = hadamard;
      switch (g.method) {
        case KVQ_RTN: e = launch_decode_m<KVQ_RTN>(a, st); break;
        case KVQ_NUQ: e = launch_decode_m<KVQ_NUQ>(a, st); break;
        case KVQ_VARN: e = launch_decode_m<KVQ_VARN>(a, st); break;
        default: e = launch_decode_m<KVQ_INT4>(a, st); break;
      }
    }
    if (e != cudaSuccess) return e;
  }
  CombineArgs c;
  c.g = g; c.base = base; c.q = q; c.tail_k = tail_k; c.tail_v = tail_v; c.n_tail = n_tail;
  c.tail_bh = tail_bh;
  c.tail_tok = tail_tok;
  c.n_blocks = n_blocks; c.n_split = (int)plan.rows; c.ranges = plan.ranges; c.per_range = plan.per_range;
  c.tail_ws = (plan.tail_row && n_tail > 0) ? 1 : 0;
  c.total = (long long)g.B * g.H * n_blocks;
  c.ws_m = ws_m; c.ws_l = ws_l; c.ws_o = ws_o; c.out = out; c.hadamard = hadamard; c.status = status;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(g.Hq, g.B);
  lc.blockDim = dim3(CB_THREADS);
  lc.dynamicSmemBytes = 0;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // after a decode kernel (which releases its dependents once all its CTAs run), the combine may
  // start early and attend the tail meanwhile; with no cached blocks it is an ordinary launch
  lc.attrs = attr;
  lc.numAttrs = n_blocks > 0 ? 1 : 0;
  return cudaLaunchKernelEx(&lc, combine_kernel, c);
}

// Workspace floats the decode of n_blocks blocks needs on the current device (v1_splits: the
// split count of the CUDA-core decode).
size_t kvq_decode_ws_floats(const kvq::Geo& g, int n_blocks, int v1_splits) {
  const DecodePlan plan = plan_decode(g, n_blocks, v1_splits);
  const uint64_t rows = (uint64_t)g.B * g.Hq * plan.rows;
  return 2 * rows + 4 + rows * kvq::D;
}

// ------------------------------------------------------------------ library-owned decode scratch
//
// kvq_decode_attn_static runs the same decode as kvq_decode_attn but keeps the split partials in
// this file-scope device array instead of a caller buffer. The array exists once per GPU that
// loads the library and lives until the process exits. Host code must not pass its name to a
// kernel (on the host it is only a stand-in); kvq_static_workspace() looks up its device
// address with cudaGetSymbolAddress, once per device, with that device current.
#include <mutex>

namespace {
constexpr size_t kStaticWsFloats = (size_t)KVQ_STATIC_WORKSPACE_BYTES / sizeof(float);
static __device__ __align__(256) float g_decode_scratch[kStaticWsFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {};
}  // namespace

// Device address of the scratch array on the current device (looked up on first use).
cudaError_t kvq_static_workspace(float** ptr, size_t* n_floats) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *ptr = g_scratch_ptr[dev];
  *n_floats = kStaticWsFloats;
  return cudaSuccess;
}
