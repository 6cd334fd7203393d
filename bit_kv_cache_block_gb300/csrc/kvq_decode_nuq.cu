// Decode attention over 3-bit nuq caches whose keys are stored before RoPE, on the tensor cores
// (one query head per KV head).
//
// Work split. The (b, h, block) sequence of the whole batch is cut into one contiguous range
// per CTA (persistent: one wave). A CTA of 8 warps streams whole block records (K tile, V tile,
// fp16 metadata, CSR outliers) through a ring of shared-memory stages with 1-D bulk copies
// (cp.async.bulk, mbarrier completion, bounded waits). Warp w owns tokens 16w..16w+15 of every
// block and keeps its own flash-decode state (running max, sum, output); at the end of each
// (b, h) segment the 8 states merge into one partial (m, l, o[128]) for the combine kernel.
//
// Keys ([KVQ] §3.2 pre-RoPE quantisation, Algorithm 1 dequantisation, worked example step 5):
// the key at absolute position n = n0 + t (n0 = 128 * block) is k_n = R(n) (s*C[q] + zp + o),
// so q . k_n = (R(t)^T q_b) . (s*C[q] + zp + o) with q_b = R(n0)^T q. Per channel pair i
// (angle t*theta_i) this is cos * X_i + sin * Y_i with
//     X_i = q_b0 k0 + q_b1 k1,    Y_i = q_b1 k0 - q_b0 k1.
// X and Y of 16 tokens x 4 pairs come out of one mma.sync m16n8k16: A = the codebook values
// C[q] of 16 tokens x 8 channels (looked up from the packed codes with byte permutes on an fp16
// table held in registers; the 8 channels repeated in k = 8..15), B = the block's q_b * s as an
// fp16 high part (k < 8) and low part (k >= 8) in the X and Y columns of each pair, C = the
// zero-point terms. The cos/sin of a lane's own (token, pair) cells are fixed over blocks and
// stay in registers; the fp16 outliers of the CSR add their rotated contribution per entry.
// Values ([KVQ] §3.7 value matvec): O[channel] = sum_t p_t s_t C[q] + sum_t p_t zp_t + outliers,
// one m16n8k16 per 16 channels x the warp's 16 tokens; B = p*s in high/low fp16 columns.
// Softmax in base 2 with the running max per warp (rescaling only when the max grows).
#include "kvq_internal.cuh"

namespace kvq {
namespace nuqdec {

constexpr int NW = 8;  // warps per CTA (16 tokens of each block per warp)
constexpr int NT = NW * 32;
constexpr float LOG2E_RSQRT_D = 1.4426950408889634f * 0.08838834764831845f;

#ifndef KVQ_NUQ_NB
#define KVQ_NUQ_NB 4
#endif
constexpr int NB = KVQ_NUQ_NB;  // record stages in the ring

struct Args {
  Geo g;
  const uint8_t* base;
  const float* codebook;  // [H][8] fp32
  const uint16_t* q;
  int nb;                 // cached blocks per (b, h)
  long long total;        // B * H * nb
  int n_ranges;           // CTAs in the grid
  int n_slots;            // partial slots per (b, query head)
  float* ws_m;
  float* ws_l;
  float* ws_o;
  int* status;
};

// Per-block operands shared by the 8 warps (double-buffered by block parity).
struct Prep {
  uint32_t bk[9][36];  // score B fragments of column g (16 k-groups x (high, low)), padded rows;
                       // row 8 stays zero (read by the lanes whose B entries are zero)
  float cz[4][36];     // zero-point terms (X, Y) of pair 4*kgroup + tq, per tq, padded rows
  float qb[D];         // q rotated back by the block's start angle
};

struct Smem {
  float2 rope_loc[T * 64];  // (cos, sin) of t * theta_i, t = 0..127 (for the key outliers)
  Prep prep[2];
  float q[D];               // query of the current (b, h), times log2(e)/sqrt(128)
  float outv[NW][D];        // value outliers weighted by p, per warp
  float red_o[NW][D];       // per-warp outputs at a segment end
  float red_ml[NW][2];
  uint64_t bar[NB];
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// Nibble word u of a lane's 6-word code group: 8 codes in 4-bit slots (bit 3 of each slot clear),
// ready to serve as byte-permute selectors (low 16 bits: slots 0..3, high 16 bits: slots 4..7).
__device__ __forceinline__ uint32_t nibble_word(const uint32_t (&w)[6], const int U) {  // U: unrolled
  const uint32_t L = w[U >> 1], H = w[4 + (U >> 2)];
  const uint32_t lo = (U & 1) ? (L >> 2) : L;
  const uint32_t hi = (U & 3) == 0 ? H : (U & 3) == 1 ? (H >> 1) : (U & 3) == 2 ? (H << 2) : (H << 1);
  return (lo & 0x33333333u) | (hi & 0x44444444u);
}

// Codebook values of the 4 codes selected by sel[15:0] as two fp16 pairs: (slot 0, slot 1) and
// (slot 2, slot 3). tl/th: low and high bytes of the 8 fp16 entries.
__device__ __forceinline__ void lookup4(uint32_t sel, uint32_t tl0, uint32_t tl1, uint32_t th0, uint32_t th1,
                                        uint32_t& p01, uint32_t& p23) {
  const uint32_t lo = __byte_perm(tl0, tl1, sel), hi = __byte_perm(th0, th1, sel);
  p01 = __byte_perm(lo, hi, 0x5140);
  p23 = __byte_perm(lo, hi, 0x7362);
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__host__ __device__ inline long long range_of(long long x, long long total, long long N) {
  return ((x + 1) * N - 1) / total;
}

template <int NBS>
__global__ void __launch_bounds__(NT, 1) decode_nuq_kernel(Args a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const Geo& g = a.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const uint32_t rec = (uint32_t)g.rec_bytes;
  uint8_t* ring = smem_raw;
  Smem* sm = reinterpret_cast<Smem*>(smem_raw + (size_t)NBS * rec);

  const long long R = blockIdx.x;
  if (R >= a.n_ranges) return;
  const long long x0 = R * a.total / a.n_ranges, x1 = (R + 1) * a.total / a.n_ranges;
  const int n = (int)(x1 - x0);
  if (n <= 0) return;

  const float2* rope_blk = reinterpret_cast<const float2*>(a.base + g.rope_off);
  const float2* rope_loc = rope_blk + (size_t)(g.max_blocks + 1) * 64;

  long long u = x0 / a.nb;
  int blk = (int)(x0 - u * a.nb);
  // producer state (thread 0): next record to copy
  int pnext = 0, pbuf = 0, pblk = blk;
  const uint8_t* psrc = a.base + ((uint64_t)u * g.max_blocks + (uint64_t)blk) * g.rec_bytes;
  auto issue_next = [&]() {
    if (pnext >= n) return;
    mbar_arrive_expect_tx(&sm->bar[pbuf], rec);
    bulk_g2s(ring + (size_t)pbuf * rec, psrc, rec, &sm->bar[pbuf]);
    ++pnext;
    if (++pbuf == NBS) pbuf = 0;
    if (++pblk == a.nb) {
      pblk = 0;
      psrc += (uint64_t)(g.max_blocks - a.nb + 1) * g.rec_bytes;
    } else {
      psrc += g.rec_bytes;
    }
  };
  if (tid == 0) {
    for (int s = 0; s < NBS; ++s) mbar_init(&sm->bar[s], 1);
    fence_mbar_init();
    fence_proxy_async();
    for (int s = 0; s < NBS; ++s) issue_next();
  }

  // the in-block angle table, staged once per CTA
  {
    const float4* src = reinterpret_cast<const float4*>(rope_loc);
    float4* dst = reinterpret_cast<float4*>(sm->rope_loc);
    for (int e = tid; e < T * 32; e += NT) dst[e] = __ldg(src + e);
  }
  // cos/sin of the lane's (token, pair) cells: tokens 16w + gq + 8r, pairs 4kg + tq
  float wc[2][16], ws[2][16];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int kg = 0; kg < 16; ++kg) {
      const float2 cs = __ldg(rope_loc + (16 * warp + gq + 8 * r) * 64 + 4 * kg + tq);
      wc[r][kg] = cs.x;
      ws[r][kg] = cs.y;
    }
  // the block-start angle of the prep's channel pair, loaded one block ahead
  const int prep_pair = tid >> 2;
  float2 cs_next = __ldg(rope_blk + (size_t)blk * 64 + prep_pair);
  const int brow = (gq >> 1) == tq ? gq : 8;             // lanes holding nonzero score B entries
  for (int e = tid; e < 2 * 36; e += NT) sm->prep[e / 36].bk[8][e % 36] = 0u;
  const int src_a = 4 * tq + (gq < 2 ? gq : 2);          // value B: (high, low, zero) source lanes
  const uint32_t xsel = tq == 0 ? 0xffffffffu : 0u;      // this lane sends p' high (tq 0) ...
  const uint32_t ysel = tq == 1 ? 0xffffffffu : 0u;      // ... or low (tq 1) or zero

  uint32_t tl0 = 0, tl1 = 0, th0 = 0, th1 = 0;
  float acc[8][4];
  float m_w = -INFINITY, l_w = 0.0f, z_w = 0.0f;
  long long cur_u = -1;
  bool ok = true;
  int failed_at = n;

  auto flush = [&](long long uu) {
    // per-warp totals over its 16 tokens (l, z replicated over tq: reduce over gq only)
    float lt = l_w, zt = z_w;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lt += __shfl_xor_sync(0xffffffffu, lt, o);
      zt += __shfl_xor_sync(0xffffffffu, zt, o);
    }
    __syncwarp();
    if (tq == 0) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int c0 = 16 * mt + gq, c1 = c0 + 8;
        sm->red_o[warp][c0] = acc[mt][0] + acc[mt][1] + zt + sm->outv[warp][c0];
        sm->red_o[warp][c1] = acc[mt][2] + acc[mt][3] + zt + sm->outv[warp][c1];
      }
    }
    if (lane == 0) {
      sm->red_ml[warp][0] = m_w;
      sm->red_ml[warp][1] = lt;
    }
    __syncthreads();
    const long long b = uu / g.H, h = uu - b * g.H;
    const long long slot = R - range_of(uu * a.nb, a.total, a.n_ranges);
    if (tid < D && slot >= 0 && slot < a.n_slots) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, sm->red_ml[w][0]);
      float L = 0.0f, O = 0.0f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = exp2f(sm->red_ml[w][0] - M);
        L = fmaf(sm->red_ml[w][1], f, L);
        O = fmaf(sm->red_o[w][tid], f, O);
      }
      const uint64_t row = ((uint64_t)(b * g.Hq + h)) * a.n_slots + slot;
      a.ws_o[row * D + tid] = O;
      if (tid == 0) {
        a.ws_m[row] = M;
        a.ws_l[row] = L;
      }
    }
    __syncthreads();
  };

  for (int i = 0; i < n; ++i) {
    if (u != cur_u) {
      if (cur_u >= 0) flush(cur_u);
      cur_u = u;
      const long long b = u / g.H, h = u - b * g.H;
      if (tid < D) sm->q[tid] = load_in(a.q + ((uint64_t)(b * g.Hq + h)) * D + tid, g.in_bf16) * LOG2E_RSQRT_D;
      {
        uint32_t hb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) hb[j] = f2h_rn(__ldg(a.codebook + h * 8 + j));
        tl0 = (hb[0] & 0xffu) | (hb[1] & 0xffu) << 8 | (hb[2] & 0xffu) << 16 | (hb[3] & 0xffu) << 24;
        tl1 = (hb[4] & 0xffu) | (hb[5] & 0xffu) << 8 | (hb[6] & 0xffu) << 16 | (hb[7] & 0xffu) << 24;
        th0 = (hb[0] >> 8) | (hb[1] >> 8) << 8 | (hb[2] >> 8) << 16 | (hb[3] >> 8) << 24;
        th1 = (hb[4] >> 8) | (hb[5] >> 8) << 8 | (hb[6] >> 8) << 16 | (hb[7] >> 8) << 24;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) sm->outv[warp][lane + 32 * k] = 0.0f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
      m_w = -INFINITY;
      l_w = 0.0f;
      z_w = 0.0f;
      __syncthreads();  // the query is visible to the block preparation
    }

    // ---- wait for the record; prepare the block's score operands (all 256 threads)
    const int slot_i = i % NBS;
    const bool got = mbar_wait_bounded(&sm->bar[slot_i], (uint32_t)((i / NBS) & 1), a.status);
    const uint8_t* st = ring + (size_t)slot_i * rec;
    Prep& pr = sm->prep[i & 1];
    if (got) {
      const uint16_t* km = reinterpret_cast<const uint16_t*>(st + g.meta_off[0]);
      const int pi = prep_pair, sub = tid & 3, kg = pi >> 2, tqp = pi & 3;
      const float2 cs = cs_next;
      const float q0 = sm->q[2 * pi], q1 = sm->q[2 * pi + 1];
      const float qb0 = cs.x * q0 + cs.y * q1, qb1 = -cs.y * q0 + cs.x * q1;
      if (sub < 2) {
        const float s0 = h2f(km[2 * pi]), s1 = h2f(km[2 * pi + 1]);
        const float v0 = sub == 0 ? qb0 * s0 : qb1 * s0;
        const float v1 = sub == 0 ? qb1 * s1 : -qb0 * s1;
        const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
        const float r0 = v0 - __half2float(h0), r1 = v1 - __half2float(h1);
        uint32_t* dst = &pr.bk[2 * tqp + sub][2 * kg];
        dst[0] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
        dst[1] = pack_h2(r0, r1);
      } else if (sub == 2) {
        const float z0 = h2f(km[T + 2 * pi]), z1 = h2f(km[T + 2 * pi + 1]);
        pr.cz[tqp][2 * kg] = qb0 * z0 + qb1 * z1;
        pr.cz[tqp][2 * kg + 1] = qb1 * z0 - qb0 * z1;
      } else {
        pr.qb[2 * pi] = qb0;
        pr.qb[2 * pi + 1] = qb1;
      }
    }
    if (__syncthreads_or(!got)) {  // every thread leaves together
      ok = false;
      failed_at = i;
      break;
    }
    if (tid == 0 && i > 0) {  // every thread is done with block i-1: refill its stage
      fence_proxy_async();
      issue_next();
    }
    if (i + 1 < n) cs_next = __ldg(rope_blk + (size_t)(blk + 1 == a.nb ? 0 : blk + 1) * 64 + prep_pair);

    // ---- scores of the warp's 16 tokens
    float s0 = 0.0f, s1 = 0.0f;
    {
      uint32_t cw[6];
      const uint2* kp = reinterpret_cast<const uint2*>(st + g.codes_off[0] + warp * 768 + lane * 24);
      const uint2 k0 = kp[0], k1 = kp[1], k2 = kp[2];
      cw[0] = k0.x; cw[1] = k0.y; cw[2] = k1.x; cw[3] = k1.y; cw[4] = k2.x; cw[5] = k2.y;
      uint32_t bf[32];
      {
        const uint4* bp = reinterpret_cast<const uint4*>(&pr.bk[brow][0]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 v = bp[j];
          bf[4 * j] = v.x; bf[4 * j + 1] = v.y; bf[4 * j + 2] = v.z; bf[4 * j + 3] = v.w;
        }
      }
      const float4* cp = reinterpret_cast<const float4*>(&pr.cz[tq][0]);
#pragma unroll
      for (int uu = 0; uu < 8; ++uu) {
        const uint32_t nw = nibble_word(cw, uu);
        const float4 z = cp[uu];  // (ZX, ZY) of k-groups 2uu and 2uu+1
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int kg = 2 * uu + hf;
          uint32_t a0, a1;
          lookup4(hf ? (nw >> 16) : nw, tl0, tl1, th0, th1, a0, a1);
          const float c4[4] = {hf ? z.z : z.x, hf ? z.w : z.y, hf ? z.z : z.x, hf ? z.w : z.y};
          float d[4];
          mma16816(d, a0, a1, a0, a1, bf[2 * kg], bf[2 * kg + 1], c4);
          s0 = fmaf(wc[0][kg], d[0], fmaf(ws[0][kg], d[1], s0));
          s1 = fmaf(wc[1][kg], d[2], fmaf(ws[1][kg], d[3], s1));
        }
      }
    }
    // key outliers of the warp's tokens: entries split over the 4 lanes of each token
    const int t0 = 16 * warp + gq, t1 = t0 + 8;
    if (g.n_out > 0) {
      const uint8_t* csr = st + g.csr_off[0];
      const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
      const uint16_t* rp = reinterpret_cast<const uint16_t*>(csr + 2 * g.n_out);
      const uint8_t* col = csr + 2 * g.n_out + 2 * (T + 1);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int t = r ? t1 : t0;
        const int j1 = min((int)rp[t + 1], g.n_out);
        float add = 0.0f;
        for (int j = min((int)rp[t], g.n_out) + tq; j < j1; j += 4) {
          const int c = col[j] & (D - 1);
          const float2 cs = sm->rope_loc[t * 64 + (c >> 1)];
          const float qa = pr.qb[c & ~1], qc = pr.qb[c | 1];
          const float qq = (c & 1) ? (-cs.y * qa + cs.x * qc) : (cs.x * qa + cs.y * qc);
          add = fmaf(h2f(val[j]), qq, add);
        }
        if (r) s1 += add; else s0 += add;
      }
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);

    // ---- online softmax over the warp's tokens (base 2)
    float mloc = fmaxf(s0, s1);
    mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 4));
    mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 8));
    mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16));
    if (mloc > m_w) {  // warp-uniform; rare after the first blocks
      const float al = exp2f(m_w - mloc);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        acc[mt][0] *= al; acc[mt][1] *= al; acc[mt][2] *= al; acc[mt][3] *= al;
      }
      l_w *= al;
      z_w *= al;
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 4; ++k) sm->outv[warp][lane + 32 * k] *= al;
      __syncwarp();
      m_w = mloc;
    }
    const float p0 = exp2f(s0 - m_w), p1 = exp2f(s1 - m_w);
    l_w += p0 + p1;

    // ---- value B fragments: p' = p * s_token, high and low fp16 columns
    const uint16_t* vm = reinterpret_cast<const uint16_t*>(st + g.meta_off[1]);
    uint32_t vb0, vb1;
    {
      const float pp0 = p0 * h2f(vm[t0]), pp1 = p1 * h2f(vm[t1]);
      z_w = fmaf(p0, h2f(vm[T + t0]), fmaf(p1, h2f(vm[T + t1]), z_w));
      const __half h0 = __float2half_rn(pp0), h1 = __float2half_rn(pp1);
      const uint32_t hi = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
      const uint32_t lo = pack_h2(pp0 - __half2float(h0), pp1 - __half2float(h1));
      const uint32_t x = (hi & xsel) | (lo & ysel);
      vb0 = __shfl_sync(0xffffffffu, x, src_a);
      vb1 = __shfl_sync(0xffffffffu, x, src_a + 16);
    }
    // value outliers of the warp's tokens, weighted by p
    if (g.n_out > 0) {
      const uint8_t* csr = st + g.csr_off[1];
      const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
      const uint16_t* rp = reinterpret_cast<const uint16_t*>(csr + 2 * g.n_out);
      const uint8_t* col = csr + 2 * g.n_out + 2 * (T + 1);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int t = r ? t1 : t0;
        const float p = r ? p1 : p0;
        const int j1 = min((int)rp[t + 1], g.n_out);
        for (int j = min((int)rp[t], g.n_out) + tq; j < j1; j += 4)
          atomicAdd(&sm->outv[warp][col[j] & (D - 1)], p * h2f(val[j]));
      }
    }

    // ---- outputs: 8 m-tiles of 16 channels x the warp's 16 tokens
    {
      uint32_t cw[6];
      const uint2* vp = reinterpret_cast<const uint2*>(st + g.codes_off[1] + warp * 768 + lane * 24);
      const uint2 v0 = vp[0], v1 = vp[1], v2 = vp[2];
      cw[0] = v0.x; cw[1] = v0.y; cw[2] = v1.x; cw[3] = v1.y; cw[4] = v2.x; cw[5] = v2.y;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint32_t nw = nibble_word(cw, mt);
        uint32_t a0, a1, a2, a3;
        lookup4(nw, tl0, tl1, th0, th1, a0, a1);
        lookup4(nw >> 16, tl0, tl1, th0, th1, a2, a3);
        mma16816(acc[mt], a0, a1, a2, a3, vb0, vb1, acc[mt]);
      }
    }
    if (++blk == a.nb) {
      blk = 0;
      ++u;
    }
  }

  if (!ok) {  // drain the copies still in flight (bounded) before the CTA exits
    if (tid == 0) {
      for (int j = failed_at; j < pnext; ++j)
        mbar_wait_bounded(&sm->bar[j % NBS], (uint32_t)((j / NBS) & 1), nullptr, 200000000LL);
    }
    __syncthreads();
    return;
  }
  if (cur_u >= 0) flush(cur_u);
}

size_t smem_bytes(const Geo& g) { return (size_t)NB * g.rec_bytes + sizeof(Smem); }

}  // namespace nuqdec
}  // namespace kvq

// ------------------------------------------------------------------ host entry points

namespace {
struct NuqOcc {
  int dev = -1;
  size_t smem = 0;
  int ctas = 0;
};
thread_local NuqOcc t_nuq_occ[4];
}  // namespace

bool kvq_nuq_supported(const kvq::Geo& g) {
  return g.method == KVQ_NUQ && g.bits == 3 && g.G == 1 && g.pre_rope == 1 &&
         kvq::nuqdec::smem_bytes(g) <= 227 * 1024;
}

// CTAs (ranges) the nuq decode uses on the current device, or 0 if the path does not apply.
// Without a usable device it assumes a 152-SM part with one CTA per SM.
long long kvq_nuq_ranges(const kvq::Geo& g) {
  using namespace kvq::nuqdec;
  if (!kvq_nuq_supported(g)) return 0;
  const size_t smem = smem_bytes(g);
  auto fn = decode_nuq_kernel<NB>;
  int dev = 0, sms = 152, ctas = 1;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
    NuqOcc* hit = nullptr;
    for (auto& c : t_nuq_occ)
      if (c.dev == dev && c.smem == smem) hit = &c;
    if (!hit) {
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      int occ = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, NT, smem) != cudaSuccess || occ < 1) occ = 1;
      for (auto& c : t_nuq_occ)
        if (c.dev < 0 || &c == &t_nuq_occ[3]) {
          c.dev = dev; c.smem = smem; c.ctas = occ;
          hit = &c;
          break;
        }
    }
    ctas = hit->ctas;
  } else {
    cudaGetLastError();
    sms = 152;
  }
  return (long long)sms * ctas;
}

cudaError_t kvq_launch_decode_nuq(const kvq::Geo& g, const uint8_t* base, const float* codebook, const uint16_t* q,
                                  int n_blocks, long long ranges, long long slots, float* ws_m, float* ws_l,
                                  float* ws_o, int* status, cudaStream_t st) {
  using namespace kvq::nuqdec;
  const size_t smem = smem_bytes(g);
  auto fn = decode_nuq_kernel<NB>;
  cudaError_t e = kvq::ensure_smem_attr((const void*)fn, smem);
  if (e != cudaSuccess) return e;
  Args a;
  a.g = g; a.base = base; a.codebook = codebook; a.q = q; a.nb = n_blocks;
  a.total = (long long)g.B * g.H * n_blocks; a.n_ranges = (int)ranges; a.n_slots = (int)slots;
  a.ws_m = ws_m; a.ws_l = ws_l; a.ws_o = ws_o; a.status = status;
  fn<<<(int)ranges, NT, smem, st>>>(a);
  return cudaGetLastError();
}
