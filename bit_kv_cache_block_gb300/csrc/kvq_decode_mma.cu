// Decode attention over the packed cache on the tensor cores (linear codes: RTN, KVarN, int4;
// 2- and 4-bit codes, and 8-bit absmax codes; up to 4 query heads per KV head).
//
// Work split. The (b, h, block) sequence of the whole batch is cut into one contiguous range
// per resident warp (persistent: one wave, equal ranges). A warp streams its blocks through
// its own ring of shared-memory stages with 1-D bulk copies (cp.async.bulk, mbarrier
// completion, bounded waits) and keeps a flash-decode state (running max, sum and output)
// per query head. When its range crosses from one (b, h) to the next, it writes a partial
// (m, l, o[128]) for the finished segment; the combine kernel merges the partials.
//
// Contractions. Both products run as mma.sync m16n8k16 (fp16 in, fp32 accumulate):
//   scores   S[token][col] = K_codes[token][channel] . Bq[channel][col]
//   outputs  O[channel][col] = V_codes[channel][token] . Bp[token][col]      (V tiles are
//            stored one row per channel, so both A operands are adjacent codes of a row)
// A operands are the packed codes themselves, masked in place into fp16 subnormals: a 2-bit
// code at bits [2p, 2p+1] of a 16-bit half becomes the exact value code * 4^p * 2^-24 (p <= 4;
// the upper positions are shifted down first), a 4-bit code code * 16^p * 2^-24; int4 codes
// are biased by 8 with one xor. One LOP3 yields two operands, about half an instruction per
// element. The power of two of each position is divided out of the matching B entry. 8-bit
// codes take one byte per half (code * 2^-24, biased by 128 with one xor), two operands per
// word.
// B columns are (query head, hi/lo): the per-channel key scales (RTN/KVarN, [KVN]
// preliminaries (K_q + z) * s) are folded into q, and the per-token value scales into the
// probabilities, each split into a high and a low fp16 half so the products keep about 22
// bits; a per-block power of two keeps them in range. Zero points enter as one scalar per
// head and block. The softmax (base 2, running max) runs on the score fragments in
// registers ([KVQ] §3.7 fused matvec kernels; [TQ] §5.2 dequantisation inside attention).
#include "kvq_internal.cuh"

#include <type_traits>

namespace kvq {
namespace mmadec {

constexpr int GQ = 4;  // query heads per KV head on this path: 8 MMA columns = 4 heads x (hi, lo)
constexpr float LOG2E_RSQRT_D = 1.4426950408889634f * 0.08838834764831845f;

struct Args {
  Geo g;
  const uint8_t* base;
  const uint16_t* q;
  int nb;                 // cached blocks per (b, h)
  long long total;        // B * H * nb
  int n_ranges;           // warps in the grid
  int n_slots;            // partial slots per (b, h, query head)
  float* ws_m;
  float* ws_l;
  float* ws_o;
  int* status;
  int hadamard;
};

// Staged B columns are FRAG_COL words apart (64 used; 2 * 68 = 8 mod 32): the writes of the 4
// column pairs by the lanes of one row group fall on distinct banks and the 16-byte fragment loads
// meet half as many conflicts. Query rows are padded for the reads of lanes that serve
// different heads.
constexpr int FRAG_COL = 68, QROW = D + 8;

struct WarpSmemQ {
  float q[GQ][QROW];          // queries of the current (b, h) (Hadamard domain for KVarN)
  uint32_t frag[8 * FRAG_COL];  // B columns staged for the score product, then the value product
  uint64_t bar[4];
};
// Absmax keys carry no per-channel scale, so q is read only while the fixed score operand of a
// (b, h) is built: q and the staging area share their memory.
struct WarpSmemU {
  union {
    float q[GQ][QROW];
    uint32_t frag[8 * FRAG_COL];
  };
  uint64_t bar[4];
};
template <int METHOD>
using WarpSmem = typename std::conditional<METHOD == KVQ_INT4, WarpSmemU, WarpSmemQ>::type;

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Signed codes enter offset-binary: one xor of the whole word flips the top bit of every code
// (int4: +8 per nibble; int8: +128 per byte), before the operands are masked out of it.
template <int BITS, bool BIAS8>
__device__ __forceinline__ uint32_t bias_word(uint32_t w) {
  return BIAS8 ? (w ^ (BITS == 8 ? 0x80808080u : 0x88888888u)) : w;
}
template <bool BIAS8>
__device__ __forceinline__ uint4 bias_words4(uint4 v) {
  return BIAS8 ? make_uint4(v.x ^ 0x88888888u, v.y ^ 0x88888888u, v.z ^ 0x88888888u, v.w ^ 0x88888888u) : v;
}

// Operand register `qr` of a packed word (signed codes already biased by bias_word): two codes
// (positions qr and qr + n/2 of the word) as fp16 subnormals. One mask each.
template <int BITS>
__device__ __forceinline__ uint32_t operand(uint32_t w, int qr) {
  if (BITS == 8) return (qr ? (w >> 8) : w) & 0x00ff00ffu;  // bytes 0, 2 (qr 0) or 1, 3 (qr 1)
  if (BITS == 2)
    return qr <= 4 ? (w & (0x00030003u << (2 * qr))) : ((w >> 10) & (0x00030003u << (2 * (qr - 5))));
  return (qr < 2 ? w : (w >> 8)) & ((qr & 1) ? 0x00f000f0u : 0x000f000fu);
}

// hi/lo fp16 split of x: hi = fp16(x), lo = fp16(x - hi).
__device__ __forceinline__ void split_hl(float x, __half& hi, __half& lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn(x - __half2float(hi));
}

// 2^e for the exponent that keeps max|v| * 2^e below 2^14 (0 for an all-zero block).
__device__ __forceinline__ int range_exp(float mx) {
  if (!(mx > 0.0f)) return 0;
  int e;
  frexpf(mx, &e);  // mx = m * 2^e, m in [0.5, 1)
  int s = 14 - e;
  return s > 100 ? 100 : (s < -100 ? -100 : s);
}

__device__ __forceinline__ float exp2i(int e) { return ldexpf(1.0f, e); }

__device__ __forceinline__ float warp_max_tq(float v) {  // over lanes with the same lane & 3
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}
__device__ __forceinline__ float warp_sum_tq(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  return v + __shfl_xor_sync(0xffffffffu, v, 16);
}
__device__ __forceinline__ float warp_max_all(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_all(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Range containing block x of the flattened (b, h, block) sequence: range r holds
// [floor(r*total/N), floor((r+1)*total/N)).
__host__ __device__ inline long long range_of(long long x, long long total, long long N) {
  return ((x + 1) * N - 1) / total;
}

// acc[mt] += (rows 16mt+gq and 16mt+gq+8 of a 128-row code tile) . B, for the 8 m-tiles of the
// tile; the k-step loop is outermost so that consecutive MMAs use independent accumulators.
// Only m-tiles MT0 .. MT1-1 are computed (the halves of a tile whose rows carry two scale sets).
template <int BITS, bool BIAS8, int MT0 = 0, int MT1 = 8>
__device__ __forceinline__ void tile_mma(float (&acc)[8][4], const uint32_t* codes, int gq, int tq,
                                         const uint32_t (&b)[16]) {
  if (BITS == 8) {  // rows of 32 words; lane tq feeds k-step ks from word 8*tq + ks of its rows
#pragma unroll
    for (int hm = 0; hm < 4; ++hm) {  // 2 m-tiles at a time
      if (2 * hm < MT0 || 2 * hm >= MT1) continue;
      uint4 w0[2][2], w1[2][2];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int mt = 2 * hm + m;
        const uint4* r0 = reinterpret_cast<const uint4*>(codes + (16 * mt + gq) * 32 + 8 * tq);
        const uint4* r1 = reinterpret_cast<const uint4*>(codes + (16 * mt + gq + 8) * 32 + 8 * tq);
        w0[m][0] = r0[0]; w0[m][1] = r0[1];
        w1[m][0] = r1[0]; w1[m][1] = r1[1];
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t x0 = bias_word<8, BIAS8>((&w0[m][ks >> 2].x)[ks & 3]);
          const uint32_t x1 = bias_word<8, BIAS8>((&w1[m][ks >> 2].x)[ks & 3]);
          mma16816(acc[2 * hm + m], operand<8>(x0, 0), operand<8>(x1, 0), operand<8>(x0, 1), operand<8>(x1, 1),
                   b[2 * ks], b[2 * ks + 1]);
        }
      }
    }
  } else if (BITS == 2) {
    uint2 w0[8], w1[8];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      if (mt < MT0 || mt >= MT1) continue;
      w0[mt] = *reinterpret_cast<const uint2*>(codes + (16 * mt + gq) * 8 + 2 * tq);
      w1[mt] = *reinterpret_cast<const uint2*>(codes + (16 * mt + gq + 8) * 8 + 2 * tq);
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int qr = 2 * (ks & 3);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        if (mt < MT0 || mt >= MT1) continue;
        const uint32_t x0 = ks < 4 ? w0[mt].x : w0[mt].y, x1 = ks < 4 ? w1[mt].x : w1[mt].y;
        mma16816(acc[mt], operand<2>(x0, qr), operand<2>(x1, qr), operand<2>(x0, qr + 1), operand<2>(x1, qr + 1),
                 b[2 * ks], b[2 * ks + 1]);
      }
    }
  } else {
#pragma unroll
    for (int hm = 0; hm < 2; ++hm) {  // 4 m-tiles at a time
      if (4 * hm + 3 < MT0 || 4 * hm >= MT1) continue;
      uint4 w0[4], w1[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int mt = 4 * hm + m;
        w0[m] = bias_words4<BIAS8>(*reinterpret_cast<const uint4*>(codes + (16 * mt + gq) * 16 + 4 * tq));
        w1[m] = bias_words4<BIAS8>(*reinterpret_cast<const uint4*>(codes + (16 * mt + gq + 8) * 16 + 4 * tq));
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int qr = 2 * (ks & 1);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t* p0 = &w0[m].x;
          const uint32_t* p1 = &w1[m].x;
          const uint32_t x0 = p0[ks >> 1], x1 = p1[ks >> 1];
          mma16816(acc[4 * hm + m], operand<4>(x0, qr), operand<4>(x1, qr), operand<4>(x0, qr + 1),
                   operand<4>(x1, qr + 1), b[2 * ks], b[2 * ks + 1]);
        }
      }
    }
  }
}

// The lane's code words of a 128-row tile of 2- or 4-bit codes (rows 16mt+gq and 16mt+gq+8 of every
// m-tile), held in registers so that the shared-memory buffer can be handed back before the
// products run.
template <int BITS>
struct TileWords {
  uint32_t w[8][BITS == 2 ? 4 : 8];
};

template <int BITS, bool BIAS8>
__device__ __forceinline__ void load_tile(TileWords<BITS>& t, const uint32_t* codes, int gq, int tq) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    if (BITS == 2) {
      const uint2 a = *reinterpret_cast<const uint2*>(codes + (16 * mt + gq) * 8 + 2 * tq);
      const uint2 b = *reinterpret_cast<const uint2*>(codes + (16 * mt + gq + 8) * 8 + 2 * tq);
      t.w[mt][0] = a.x; t.w[mt][1] = a.y; t.w[mt][2] = b.x; t.w[mt][3] = b.y;
    } else {
      const uint4 a = bias_words4<BIAS8>(*reinterpret_cast<const uint4*>(codes + (16 * mt + gq) * 16 + 4 * tq));
      const uint4 b = bias_words4<BIAS8>(*reinterpret_cast<const uint4*>(codes + (16 * mt + gq + 8) * 16 + 4 * tq));
      t.w[mt][0] = a.x; t.w[mt][1] = a.y; t.w[mt][2] = a.z; t.w[mt][3] = a.w;
      t.w[mt][4] = b.x; t.w[mt][5] = b.y; t.w[mt][6] = b.z; t.w[mt][7] = b.w;
    }
  }
}

// acc[mt] += the tile's m-tile mt . B for mt in [MT0, MT1), from the words in registers (biased by
// load_tile; the same operands as tile_mma reads from shared memory).
template <int BITS, int MT0 = 0, int MT1 = 8>
__device__ __forceinline__ void words_mma(float (&acc)[8][4], const TileWords<BITS>& t, const uint32_t (&b)[16]) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
    for (int mt = MT0; mt < MT1; ++mt) {
      const int qr = BITS == 2 ? 2 * (ks & 3) : 2 * (ks & 1);
      const int wi = BITS == 2 ? (ks >> 2) : (ks >> 1);
      const uint32_t x0 = t.w[mt][wi], x1 = t.w[mt][(BITS == 2 ? 2 : 4) + wi];
      mma16816(acc[mt], operand<BITS>(x0, qr), operand<BITS>(x1, qr), operand<BITS>(x0, qr + 1),
               operand<BITS>(x1, qr + 1), b[2 * ks], b[2 * ks + 1]);
    }
  }
}

// Half offset inside one staged B column of the code at row position x = 16*mt + gq + 8*hlf
// (the positions a lane owns), and the power of two that lane's operands carry (both follow from
// operand() and the fragment layout).
template <int BITS>
__device__ __forceinline__ int col_off(int mt, int gq, int hlf) {
  if (BITS == 8)  // code x = 16mt + gq + 8hlf: word x/4 (lane x/32, k-step (x/4)%8), byte x%4
    return 16 * mt + 8 * hlf + 4 * (gq >> 2) + 2 * (gq & 1) + ((gq >> 1) & 1);
  return BITS == 2 ? 16 * mt + 2 * gq + hlf : 16 * mt + 8 * hlf + 2 * (gq & 3) + (gq >> 2);
}
template <int BITS>
__device__ __forceinline__ float lane_inv_f(int gq) {
  if (BITS == 8) return 1.0f;  // every byte operand is code * 2^-24
  if (BITS == 2) {
    const int e = gq <= 4 ? 2 * gq : 2 * (gq - 5);
    return __int_as_float((127 - e) << 23);
  }
  return (gq & 1) ? 0.0625f : 1.0f;
}

// Reductions over the lanes that hold the same query head (8 row groups x the replicas).
template <int GT>
__device__ __forceinline__ float head_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  if (GT <= 2) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  if (GT == 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return v;
}
template <int GT>
__device__ __forceinline__ float head_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  if (GT <= 2) v += __shfl_xor_sync(0xffffffffu, v, 2);
  if (GT == 1) v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

// Stages the hi/lo halves of v (one value per position the lane owns) into columns 2h, 2h+1.
template <int BITS, int NMT>
__device__ __forceinline__ void stage_cols(uint32_t* frag, int h, int gq, int rho, int RP, const float (&v)[2 * NMT]) {
  __half* col_hi = reinterpret_cast<__half*>(frag) + (2 * h) * (2 * FRAG_COL);
  __half* col_lo = col_hi + 2 * FRAG_COL;
#pragma unroll
  for (int j = 0; j < NMT; ++j) {
    const int mt = rho + RP * j;
    __half h0, l0, h1, l1;
    split_hl(v[2 * j], h0, l0);
    split_hl(v[2 * j + 1], h1, l1);
    if (BITS == 2) {  // the two positions of an m-tile are adjacent halves
      const int o = col_off<2>(mt, gq, 0);
      *reinterpret_cast<__half2*>(col_hi + o) = __halves2half2(h0, h1);
      *reinterpret_cast<__half2*>(col_lo + o) = __halves2half2(l0, l1);
    } else {
      const int o0 = col_off<BITS>(mt, gq, 0), o1 = col_off<BITS>(mt, gq, 1);
      col_hi[o0] = h0; col_lo[o0] = l0;
      col_hi[o1] = h1; col_lo[o1] = l1;
    }
  }
}

// The lane's j-th own m-tile (mt = rho + RP*j) of an accumulator array, with static indices.
template <int RP>
__device__ __forceinline__ void pick_tile(const float (&acc)[8][4], int j, int rho, float (&c)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float v = acc[RP * j][k];
#pragma unroll
    for (int r = 1; r < RP; ++r) v = (rho == r) ? acc[r + RP * j][k] : v;
    c[k] = v;
  }
}

// Loads the lane's 16 B registers: lane (g', t') reads staged column g' mod 2G.
__device__ __forceinline__ void load_frag(const uint32_t* frag, int lane, int G, uint32_t (&b)[16]) {
  const int col = (lane >> 2) % (2 * G);
  const uint4* src = reinterpret_cast<const uint4*>(frag + col * FRAG_COL + (lane & 3) * 16);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 v = src[k];
    b[4 * k] = v.x; b[4 * k + 1] = v.y; b[4 * k + 2] = v.z; b[4 * k + 3] = v.w;
  }
}

// GT: query heads per KV head this instantiation serves (1, 2 or 4; G = 3 runs on GT = 4). Each
// head's B columns are replicated over the 4 column pairs (RP = 4/GT copies), so every lane holds
// real scores and finishes 16/RP of the block's tokens.
// NW warps per CTA; NB shared-memory buffers per warp, each holding one half-record (the K tile
// or the V tile of a block, with its metadata): the ring streams K(0), V(0), K(1), V(1), ...
// G64 (absmax only): every token has two scales, one per 64 channels. Scores run the key tile
// twice, against q restricted to each half, and the value product runs m-tiles 0-3 (channels
// 0..63) and 4-7 against probabilities scaled by the matching half's scales.
// 4-bit codes go to registers as soon as their buffer lands, and the buffer is handed back at once,
// so every buffer of the warp but the one being read stays in flight while it computes (8-bit
// tiles, and 4-bit tiles with two scale sets, are too large to hold; 2-bit tiles measured no
// faster this way and are read from shared memory).
template <int BITS, bool G64>
constexpr bool early_release() { return BITS == 4 && !G64; }
// CTAs per SM the register budget must allow (the shared-memory ring allows as many).
#ifndef KVQ_MMA2_G1_MINB
#define KVQ_MMA2_G1_MINB 1
#endif
template <int BITS, int GT, bool G64>
constexpr int min_ctas() {
  return early_release<BITS, G64>() ? 2 : (BITS == 2 && GT == 1) ? KVQ_MMA2_G1_MINB : 1;
}

template <int METHOD, int BITS, int GT, int NW, int NB, bool WHOLE, bool G64>
__global__ void __launch_bounds__(NW * 32, (min_ctas<BITS, GT, G64>())) decode_mma_kernel(Args a) {
  launch_dependents();  // the combine kernel may be scheduled once every CTA of this grid runs
  constexpr bool BIAS8 = METHOD == KVQ_INT4;          // signed codes enter biased by 8 (or 128)
  constexpr float BIASF = BITS == 8 ? 128.0f : 8.0f;
  constexpr int RP = 4 / GT;
  constexpr int NMT = 8 / RP;  // m-tiles (16 rows) a lane finishes
  constexpr bool EARLY = early_release<BITS, G64>();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const Geo& g = a.g;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const int G = g.G;
  const int hl = tq % GT, rho = tq / GT;  // the lane's head and replica
  const bool head_ok = hl < G;
  const float inv_f = lane_inv_f<BITS>(gq);
  const int halfk = (int)g.codes_off[1];               // K half: K codes, K meta (, K csr)
  const int halfv = (int)g.rec_bytes - halfk;          // V half
  const int hb = WHOLE ? (int)g.rec_bytes : (halfk > halfv ? halfk : halfv);  // bytes per buffer
  uint8_t* ring = smem_raw + (size_t)warp * NB * hb;
  WarpSmem<METHOD>* sw = reinterpret_cast<WarpSmem<METHOD>*>(smem_raw + (size_t)NW * NB * hb) + warp;

  const long long R = (long long)blockIdx.x * NW + warp;
  if (R >= a.n_ranges) return;  // the last CTA may carry warps beyond the range count
  const long long x0 = R * a.total / a.n_ranges, x1 = (R + 1) * a.total / a.n_ranges;
  const int n = (int)(x1 - x0);
  if (n <= 0) return;

  if (lane == 0) {
    for (int s = 0; s < NB; ++s) mbar_init(&sw->bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  // (unit, block) being processed; lane 0 also tracks the next half-record to prefetch
  long long u = x0 / a.nb;
  int blk = (int)(x0 - u * a.nb);
  const int n_units = WHOLE ? n : 2 * n;  // copies: whole records, or K and V halves
  int pnext = 0, pbuf = 0, pblk = blk;              // next copy to issue, its buffer, its block
  int pb = (int)(u / g.H), ph = (int)(u - (long long)pb * g.H);  // and its (b, h)
  const uint8_t* psrc = a.base + record_offset(g, pb, ph, pblk, a.status);
  auto issue_next = [&]() {  // lane 0 only
    if (pnext >= n_units) return;
    const bool is_v = !WHOLE && (pnext & 1);
    const uint32_t bytes = (uint32_t)(WHOLE ? (int)g.rec_bytes : (is_v ? halfv : halfk));
    mbar_arrive_expect_tx(&sw->bar[pbuf], bytes);
    bulk_g2s(ring + (size_t)pbuf * hb, psrc + (is_v ? halfk : 0), bytes, &sw->bar[pbuf]);
    ++pnext;
    if (++pbuf == NB) pbuf = 0;
    if (WHOLE || is_v) {  // next block: the next record, or the first record of the next (b, h)
      if (g.n_pages <= 0) {  // contiguous: the next record, or the first one of the next (b, h)
        if (++pblk == a.nb) {
          pblk = 0;
          psrc += (uint64_t)(g.max_blocks - a.nb + 1) * g.rec_bytes;
        } else {
          psrc += g.rec_bytes;
        }
      } else {                // paged: through the block table
        if (++pblk == a.nb) {
          pblk = 0;
          if (++ph == g.H) {
            ph = 0;
            ++pb;
          }
        }
        if (pnext < n_units) psrc = a.base + record_offset(g, pb, ph, pblk, a.status);
      }
    }
  };
  int cbuf = 0;          // buffer of the next half-record to consume
  uint32_t parity = 0;   // bit b: phase parity of buffer b's next completion
  auto wait_next = [&](const uint8_t*& buf) -> bool {
    const bool got = mbar_wait_bounded(&sw->bar[cbuf], (parity >> cbuf) & 1u, a.status);
    buf = ring + (size_t)cbuf * hb;
    parity ^= 1u << cbuf;
    if (++cbuf == NB) cbuf = 0;
    return got;
  };
  if (lane == 0) {
    fence_proxy_async();
    for (int s = 0; s < NB; ++s) issue_next();
  }

  float m_run = -INFINITY, l_run = 0.0f, zv = 0.0f, zv1 = 0.0f;
  float O[8][4];
  int g1_cur = 0;
  uint32_t bk[16], bv[16], bk1[16], bv1[16];  // bk1, bv1: second scale half (G64)
  float zk = 0.0f, sumq = 0.0f, sumq1 = 0.0f;
  int g0_fixed = 0;
  long long cur_u = -1;
  bool ok = true;
  int failed_at = n;

  auto flush = [&](long long uu) {
    const long long b = uu / g.H, h = uu - b * g.H;
    const long long slot = R - range_of(uu * a.nb, a.total, a.n_ranges);
    if (rho == 0 && head_ok && slot >= 0 && slot < a.n_slots) {
      const uint64_t row = ((uint64_t)(b * g.Hq + h * G + hl)) * a.n_slots + slot;
      const float sc = (METHOD == KVQ_VARN) ? 1.0f : exp2i(24 - g1_cur);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float add = (METHOD == KVQ_VARN) ? 0.0f : (G64 && mt >= 4) ? zv1 : zv;
        a.ws_o[row * D + 16 * mt + gq] = (O[mt][0] + O[mt][1]) * sc + add;
        a.ws_o[row * D + 16 * mt + gq + 8] = (O[mt][2] + O[mt][3]) * sc + add;
      }
      if (gq == 0) {
        a.ws_m[row] = m_run;
        a.ws_l[row] = l_run;
      }
    }
  };

  for (int i = 0; i < n; ++i) {
    if (u != cur_u) {
      if (cur_u >= 0) flush(cur_u);
      cur_u = u;
      const long long b = u / g.H, h = u - b * g.H;
      __syncwarp();
      for (int e = lane; e < GQ * D; e += 32) {
        const int hh = e >> 7, c = e & 127;
        sw->q[hh][c] = hh < G ? load_in(a.q + ((uint64_t)(b * g.Hq + h * G + hh)) * D + c, g.in_bf16) : 0.0f;
      }
      __syncwarp();
      if (METHOD == KVQ_VARN && a.hadamard) {  // q in the Hadamard domain
        for (int hh = 0; hh < G; ++hh) {
          float* v = sw->q[hh];
          for (int st = 1; st < D; st <<= 1) {
            for (int j = lane; j < D / 2; j += 32) {
              const int i0 = (j / st) * (2 * st) + (j % st);
              const float p0 = v[i0], p1 = v[i0 + st];
              v[i0] = p0 + p1;
              v[i0 + st] = p0 - p1;
            }
            __syncwarp();
          }
          for (int c = lane; c < D; c += 32) v[c] *= 0.08838834764831845f;
          __syncwarp();
        }
      }
      m_run = -INFINITY;
      l_run = 0.0f;
      zv = 0.0f;
      zv1 = 0.0f;
      g1_cur = 0;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) O[mt][0] = O[mt][1] = O[mt][2] = O[mt][3] = 0.0f;
      if (METHOD == KVQ_INT4) {  // absmax keys carry no per-channel scale: B is fixed per (b, h)
        float mx = 0.0f, sq = 0.0f, sq1 = 0.0f;
        float v[2 * NMT], v1[2 * NMT];
#pragma unroll
        for (int j = 0; j < NMT; ++j)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const float qv = head_ok ? sw->q[hl][16 * (rho + RP * j) + gq + 8 * hf] : 0.0f;
            const bool lo = !G64 || rho + RP * j < 4;  // channel < 64
            v[2 * j + hf] = lo ? qv : 0.0f;
            v1[2 * j + hf] = lo ? 0.0f : qv;
            if (lo) sq += qv;
            else sq1 += qv;
            mx = fmaxf(mx, fabsf(qv));
          }
        mx = warp_max_all(mx);
        sumq = head_sum<GT>(sq);
        if (G64) sumq1 = head_sum<GT>(sq1);
        g0_fixed = range_exp(mx);
        __syncwarp();  // every lane has read its q values: the staging area may be overwritten
        const float sc = exp2i(g0_fixed) * inv_f;
#pragma unroll
        for (int k = 0; k < 2 * NMT; ++k) {
          v[k] *= sc;
          v1[k] *= sc;
        }
        if (head_ok) stage_cols<BITS, NMT>(sw->frag, hl, gq, rho, RP, v);
        __syncwarp();
        load_frag(sw->frag, lane, G, bk);
        if (G64) {
          __syncwarp();
          if (head_ok) stage_cols<BITS, NMT>(sw->frag, hl, gq, rho, RP, v1);
          __syncwarp();
          load_frag(sw->frag, lane, G, bk1);
        }
      }
    }

    // ---- wait for this block's record or K half (bounded; all lanes leave together on failure)
    const uint8_t* kbuf;
    if (__any_sync(0xffffffffu, !wait_next(kbuf))) {
      ok = false;
      failed_at = WHOLE ? i : 2 * i;
      break;
    }
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(kbuf + g.codes_off[0]);
    const uint16_t* km = reinterpret_cast<const uint16_t*>(kbuf + g.meta_off[0]);

    // ---- per-token key metadata of the lane's tokens (int4: scales; KVarN: the token scale)
    float ktok[2 * NMT], ktok1[2 * NMT];
#pragma unroll
    for (int j = 0; j < NMT; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int tok = 16 * (rho + RP * j) + gq + 8 * hf;
        ktok[2 * j + hf] = METHOD == KVQ_INT4 ? h2f(km[tok]) : METHOD == KVQ_VARN ? h2f(km[2 * T + tok]) : 0.0f;
        ktok1[2 * j + hf] = G64 ? h2f(km[T + tok]) : 0.0f;
      }

    // ---- B fragments of the score product: q * s_channel (RTN, KVarN)
    int g0 = g0_fixed;
    if (METHOD != KVQ_INT4) {
      float v[2 * NMT];
      float mx = 0.0f, zp = 0.0f;
#pragma unroll
      for (int j = 0; j < NMT; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int c = 16 * (rho + RP * j) + gq + 8 * hf;
          const float qs = head_ok ? sw->q[hl][c] * h2f(km[c]) : 0.0f;
          v[2 * j + hf] = qs;
          mx = fmaxf(mx, fabsf(qs));
          zp = fmaf(qs, h2f(km[T + c]), zp);
        }
      mx = warp_max_all(mx);
      zk = head_sum<GT>(zp);
      g0 = range_exp(mx);
      const float sc = exp2i(g0) * inv_f;
#pragma unroll
      for (int k = 0; k < 2 * NMT; ++k) v[k] *= sc;
      __syncwarp();  // the staging buffer is free (last block's value fragments are loaded)
      if (head_ok) stage_cols<BITS, NMT>(sw->frag, hl, gq, rho, RP, v);
      __syncwarp();
      load_frag(sw->frag, lane, G, bk);
    }

    // ---- the V half's metadata and codes (value scale and zero point of the lane's tokens;
    // KVarN: s1 of the lane's channel rows), read as soon as the half is in shared memory
    const uint8_t* vbuf = kbuf + halfk;
    float vtok[2 * NMT], vtok1[2 * NMT], s1r[16];
    TileWords<EARLY ? BITS : 2> kw, vw;
    auto read_v = [&]() {
      const uint16_t* vm = reinterpret_cast<const uint16_t*>(vbuf + (g.meta_off[1] - g.codes_off[1]));
#pragma unroll
      for (int j = 0; j < NMT; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int tok = 16 * (rho + RP * j) + gq + 8 * hf;
          vtok[2 * j + hf] = h2f(vm[tok]);
          vtok1[2 * j + hf] = METHOD == KVQ_INT4 && !G64 ? 0.0f : h2f(vm[T + tok]);
        }
      if (METHOD == KVQ_VARN) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          s1r[2 * mt] = h2f(vm[2 * T + 16 * mt + gq]);
          s1r[2 * mt + 1] = h2f(vm[2 * T + 16 * mt + gq + 8]);
        }
      }
      if (EARLY) load_tile<EARLY ? BITS : 2, BIAS8>(vw, reinterpret_cast<const uint32_t*>(vbuf), gq, tq);
    };
    if (EARLY) {  // take the K half (or the whole record) into registers and hand the buffer back
      load_tile<EARLY ? BITS : 2, BIAS8>(kw, kc, gq, tq);
      if (WHOLE) read_v();
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async();
        issue_next();
      }
    }

    // ---- scores: S = K . Bq  (8 m-tiles of 16 tokens x 8 k-steps of 16 channels)
    float sc8[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) sc8[mt][0] = sc8[mt][1] = sc8[mt][2] = sc8[mt][3] = 0.0f;
    float sc8b[8][4];  // G64: the scores of channels 64..127
    if (G64) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) sc8b[mt][0] = sc8b[mt][1] = sc8b[mt][2] = sc8b[mt][3] = 0.0f;
    }
    if constexpr (EARLY) {
      words_mma<BITS>(sc8, kw, bk);
      if (G64) words_mma<BITS>(sc8b, kw, bk1);
    } else {
      tile_mma<BITS, BIAS8>(sc8, kc, gq, tq, bk);
      if (G64) tile_mma<BITS, BIAS8>(sc8b, kc, gq, tq, bk1);
    }

    // ---- finish the scores of the lane's tokens, online softmax (base 2)
    const float ksc = exp2i(24 - g0);
    float sv[2 * NMT];
    float mloc = -INFINITY;
#pragma unroll
    for (int j = 0; j < NMT; ++j) {
      float c4[4], d4[4];
      pick_tile<RP>(sc8, j, rho, c4);
      if (G64) pick_tile<RP>(sc8b, j, rho, d4);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float v = (c4[2 * hf] + c4[2 * hf + 1]) * ksc;
        if (METHOD == KVQ_INT4) {
          v = (v - BIASF * sumq) * ktok[2 * j + hf];
          if (G64) v += ((d4[2 * hf] + d4[2 * hf + 1]) * ksc - BIASF * sumq1) * ktok1[2 * j + hf];
        } else {
          v += zk;
        }
        if (METHOD == KVQ_VARN) v *= ktok[2 * j + hf];
        v *= LOG2E_RSQRT_D;
        sv[2 * j + hf] = v;
        mloc = fmaxf(mloc, v);
      }
    }
    if (!WHOLE) {  // the K half is consumed: refill its buffer (unless done above), then wait for the V half
      if (!EARLY) {
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async();
          issue_next();
        }
      }
      if (__any_sync(0xffffffffu, !wait_next(vbuf))) {
        ok = false;
        failed_at = 2 * i + 1;
        break;
      }
      read_v();
      if (EARLY) {
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async();
          issue_next();
        }
      }
    } else if (!EARLY) {
      read_v();
    }

    mloc = head_max<GT>(mloc);
    const float m_new = fmaxf(m_run, mloc);
    const float alpha = exp2f(m_run - m_new);
    float lsum = 0.0f, zsum_blk = 0.0f, zsum1 = 0.0f, pmax = 0.0f;
    float sv1[2 * NMT];  // G64: probabilities times the scales of channels 64..127
#pragma unroll
    for (int j = 0; j < NMT; ++j) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const float p = exp2f(sv[2 * j + hf] - m_new);
        lsum += p;
        const float pp = p * vtok[2 * j + hf];  // per-token value scale folded into p
        sv[2 * j + hf] = pp;
        if (METHOD == KVQ_INT4) zsum_blk -= BIASF * pp;
        else zsum_blk = fmaf(pp, vtok1[2 * j + hf], zsum_blk);
        pmax = fmaxf(pmax, pp);
        if (G64) {
          const float pp1 = p * vtok1[2 * j + hf];
          sv1[2 * j + hf] = pp1;
          zsum1 -= BIASF * pp1;
          pmax = fmaxf(pmax, pp1);
        }
      }
    }
    lsum = head_sum<GT>(lsum);
    zsum_blk = head_sum<GT>(zsum_blk);
    if (G64) zsum1 = head_sum<GT>(zsum1);
    l_run = l_run * alpha + lsum;
    m_run = m_new;
    const int g1 = range_exp(warp_max_all(head_ok ? pmax : 0.0f));

    // ---- B fragments of the value product: p' (hi, lo) per head
    {
      const float sc = exp2i(g1) * inv_f;
#pragma unroll
      for (int k = 0; k < 2 * NMT; ++k) sv[k] *= sc;
      __syncwarp();  // every lane has loaded its score fragments
      if (head_ok) stage_cols<BITS, NMT>(sw->frag, hl, gq, rho, RP, sv);
      __syncwarp();
      load_frag(sw->frag, lane, G, bv);
      if (G64) {
#pragma unroll
        for (int k = 0; k < 2 * NMT; ++k) sv1[k] *= sc;
        __syncwarp();
        if (head_ok) stage_cols<BITS, NMT>(sw->frag, hl, gq, rho, RP, sv1);
        __syncwarp();
        load_frag(sw->frag, lane, G, bv1);
      }
    }

    // ---- outputs: O = V . Bp  (8 m-tiles of 16 channels x 8 k-steps of 16 tokens)
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(vbuf);
    if (METHOD != KVQ_VARN) {
      const float rs = alpha * exp2i(g1 - g1_cur);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        O[mt][0] *= rs; O[mt][1] *= rs; O[mt][2] *= rs; O[mt][3] *= rs;
      }
      zv = zv * alpha + zsum_blk;
      g1_cur = g1;
      if constexpr (EARLY) {
        if (G64) {
          zv1 = zv1 * alpha + zsum1;
          words_mma<BITS, 0, 4>(O, vw, bv);
          words_mma<BITS, 4, 8>(O, vw, bv1);
        } else {
          words_mma<BITS>(O, vw, bv);
        }
      } else {
        if (G64) {
          zv1 = zv1 * alpha + zsum1;
          tile_mma<BITS, BIAS8, 0, 4>(O, vc, gq, tq, bv);
          tile_mma<BITS, BIAS8, 4, 8>(O, vc, gq, tq, bv1);
        } else {
          tile_mma<BITS, BIAS8>(O, vc, gq, tq, bv);
        }
      }
    } else {  // second scale s1 per channel: o_c += s1_c * (P.V_c + sum p' z)
      float acc[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
      if constexpr (EARLY) words_mma<BITS>(acc, vw, bv);
      else tile_mma<BITS, BIAS8>(acc, vc, gq, tq, bv);
      const float usc = exp2i(24 - g1);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float s1a = s1r[2 * mt], s1b = s1r[2 * mt + 1];
        O[mt][0] = O[mt][0] * alpha + (acc[mt][0] * usc + zsum_blk) * s1a;
        O[mt][1] = O[mt][1] * alpha + acc[mt][1] * usc * s1a;
        O[mt][2] = O[mt][2] * alpha + (acc[mt][2] * usc + zsum_blk) * s1b;
        O[mt][3] = O[mt][3] * alpha + acc[mt][3] * usc * s1b;
      }
    }

    if (!EARLY) {
      __syncwarp();  // every lane is done with the record / V half: refill its buffer
      if (lane == 0) {
        fence_proxy_async();
        issue_next();
      }
    }
    if (++blk == a.nb) { blk = 0; ++u; }
  }

  if (!ok) {  // drain the copies still in flight (bounded) before the warp exits
    if (lane == 0) {
      for (int j = failed_at; j < pnext; ++j)
        mbar_wait_bounded(&sw->bar[j % NB], (uint32_t)((j / NB) & 1), nullptr, 200000000LL);
    }
    __syncwarp();
    return;
  }
  if (cur_u >= 0) flush(cur_u);
}

struct Plan {
  void (*fn)(Args);
  int nw, ns;  // warps per CTA, buffers per warp
  bool whole;  // buffers hold whole records (else K and V halves)
  int ws;      // bytes of per-warp state after the rings
};

// Warps per CTA and half-record buffers per warp (compile-time tuning; the defaults are the
// measured best on GB300).
#ifndef KVQ_MMA2_NW
#define KVQ_MMA2_NW 4
#endif
#ifndef KVQ_MMA2_NB
#define KVQ_MMA2_NB 2
#endif
#ifndef KVQ_MMA2_G1_NW
#define KVQ_MMA2_G1_NW KVQ_MMA2_NW
#endif
#ifndef KVQ_MMA2_WHOLE
#define KVQ_MMA2_WHOLE 1
#endif
#ifndef KVQ_MMA2_WHOLE_G1
#define KVQ_MMA2_WHOLE_G1 0
#endif
#ifndef KVQ_MMA4_NW
#define KVQ_MMA4_NW 4  // 2 CTAs per SM: 2 warps per scheduler, registers for a whole tile of words
#endif
#ifndef KVQ_MMA4G64_NW
#define KVQ_MMA4G64_NW 5
#endif
#ifndef KVQ_MMA4_NB
#define KVQ_MMA4_NB 2
#endif
#ifndef KVQ_MMA4_INT4_NB
#define KVQ_MMA4_INT4_NB 2  // 3 fit beside the smaller warp state; measured the same (208 vs 211 us)
#endif
#ifndef KVQ_MMA4_WHOLE
#define KVQ_MMA4_WHOLE 0
#endif

#ifndef KVQ_MMA8_NW
#define KVQ_MMA8_NW 4
#endif
#ifndef KVQ_MMA8_NB
#define KVQ_MMA8_NB 2
#endif

template <int METHOD, int BITS, int GT, bool G64>
Plan plan_for() {
  constexpr int NW = BITS == 2 ? (GT == 1 ? KVQ_MMA2_G1_NW : KVQ_MMA2_NW)
                     : BITS == 4 ? (G64 ? KVQ_MMA4G64_NW : KVQ_MMA4_NW) : KVQ_MMA8_NW;
  constexpr int NB = BITS == 2 ? KVQ_MMA2_NB
                     : BITS == 4 ? ((METHOD == KVQ_INT4 && !G64) ? KVQ_MMA4_INT4_NB : KVQ_MMA4_NB)
                                 : KVQ_MMA8_NB;
  // one query head (GT 1, four replicas of its columns): a long stream of light records runs
  // best from K/V half buffers; several heads per record: whole records
  constexpr bool WH = BITS == 2 ? (GT == 1 ? KVQ_MMA2_WHOLE_G1 : KVQ_MMA2_WHOLE) : BITS == 4 ? KVQ_MMA4_WHOLE : false;
  constexpr int WS = METHOD == KVQ_INT4 ? (int)sizeof(WarpSmemU) : (int)sizeof(WarpSmemQ);
  return Plan{decode_mma_kernel<METHOD, BITS, GT, NW, NB, WH, G64>, NW, NB, WH, WS};
}

template <int METHOD, int BITS, bool G64 = false>
Plan plan_g(int G) {
  if (G == 1) return plan_for<METHOD, BITS, 1, G64>();
  if (G == 2) return plan_for<METHOD, BITS, 2, G64>();
  return plan_for<METHOD, BITS, 4, G64>();
}

bool supported(const Geo& g) {
  if (g.layout != KVQ_LAYOUT_MMA) return false;  // value tiles must hold one row per channel
  if (g.G > GQ) return false;
  if (g.bits != 2 && g.bits != 4 && !(g.bits == 8 && g.method == KVQ_INT4)) return false;
  return g.method == KVQ_RTN || g.method == KVQ_VARN || g.method == KVQ_INT4;
}

Plan get_plan(const Geo& g) {
  if (g.method == KVQ_RTN) return g.bits == 2 ? plan_g<KVQ_RTN, 2>(g.G) : plan_g<KVQ_RTN, 4>(g.G);
  if (g.method == KVQ_VARN) return g.bits == 2 ? plan_g<KVQ_VARN, 2>(g.G) : plan_g<KVQ_VARN, 4>(g.G);
  if (g.g64) return g.bits == 8 ? plan_g<KVQ_INT4, 8, true>(g.G) : plan_g<KVQ_INT4, 4, true>(g.G);
  return g.bits == 8 ? plan_g<KVQ_INT4, 8>(g.G) : plan_g<KVQ_INT4, 4>(g.G);
}

size_t smem_bytes(const Geo& g, const Plan& p) {
  const uint64_t hk = g.codes_off[1], hv = g.rec_bytes - hk;
  const uint64_t hb = p.whole ? g.rec_bytes : (hk > hv ? hk : hv);
  return (size_t)p.nw * p.ns * hb + (size_t)p.nw * p.ws;
}

}  // namespace mmadec
}  // namespace kvq

// ------------------------------------------------------------------ host entry points

namespace {
struct OccCache {
  int dev = -1;
  void* fn = nullptr;
  size_t smem = 0;
  int ctas = 0;
};
thread_local OccCache t_occ[8];
}  // namespace

// Ranges (warps) the tensor-core decode uses on the current device for this geometry, or 0 if
// the path does not apply. Without a usable device it assumes a 152-SM part with one CTA per SM.
long long kvq_mma_ranges(const kvq::Geo& g) {
  using namespace kvq::mmadec;
  if (!supported(g)) return 0;
  const Plan p = get_plan(g);
  const size_t smem = smem_bytes(g, p);
  if (smem > 227 * 1024) return 0;
  int dev = 0, sms = 152, ctas = 1;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
    OccCache* hit = nullptr;
    for (auto& c : t_occ)
      if (c.dev == dev && c.fn == (void*)p.fn && c.smem == smem) hit = &c;
    if (!hit) {
      // raise (never lower) the kernel's shared-memory limit through the shared bookkeeping
      if (kvq::ensure_smem_attr((const void*)p.fn, smem) != cudaSuccess) cudaGetLastError();
      int occ = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, p.fn, p.nw * 32, smem) != cudaSuccess || occ < 1)
        occ = 1;
      for (auto& c : t_occ)
        if (c.fn == nullptr || &c == &t_occ[7]) {
          c.dev = dev; c.fn = (void*)p.fn; c.smem = smem; c.ctas = occ;
          hit = &c;
          break;
        }
    }
    ctas = hit->ctas;
  } else {
    cudaGetLastError();
    sms = 152;
  }
  return (long long)sms * ctas * p.nw;
}

// Partial slots per (b, query head) for n_blocks blocks split into `ranges` ranges.
long long kvq_mma_slots(const kvq::Geo& g, int n_blocks, long long ranges) {
  const long long total = (long long)g.B * g.H * n_blocks;
  if (total <= 0 || ranges <= 0) return 0;
  long long p = (long long)(n_blocks - 1) * ranges / total + 2;
  return p < n_blocks ? p : n_blocks;
}

cudaError_t kvq_launch_decode_mma(const kvq::Geo& g, const uint8_t* base, const uint16_t* q, int n_blocks,
                                  long long ranges, long long slots, float* ws_m, float* ws_l, float* ws_o,
                                  int* status, int hadamard, cudaStream_t st) {
  using namespace kvq::mmadec;
  const Plan p = get_plan(g);
  const size_t smem = smem_bytes(g, p);
  cudaError_t e = kvq::ensure_smem_attr((const void*)p.fn, (size_t)smem);
  if (e != cudaSuccess) return e;
  Args a;
  a.g = g; a.base = base; a.q = q; a.nb = n_blocks; a.total = (long long)g.B * g.H * n_blocks;
  a.n_ranges = (int)ranges; a.n_slots = (int)slots; a.ws_m = ws_m; a.ws_l = ws_l; a.ws_o = ws_o;
  a.status = status; a.hadamard = hadamard;
  const int grid = (int)((ranges + p.nw - 1) / p.nw);
  p.fn<<<grid, p.nw * 32, smem, st>>>(a);
  return cudaGetLastError();
}
