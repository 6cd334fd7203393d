// Decode attention over 3-bit nuq caches whose keys are stored before RoPE, on the tensor cores
// (one query head per KV head).
//
// Work split. The (b, h, block) sequence of the whole batch is cut into one contiguous range
// per CTA (persistent: one wave). A CTA runs 4 warpgroups whose roles meet only on mbarriers
// (every wait bounded):
//   producer warp     : copies each block record (K tile, V tile, fp16 metadata, CSR outliers)
//                       and the block's RoPE start-angle row into an NB-stage ring with 1-D bulk
//                       copies, as soon as the consumers have released the stage;
//   4 aux warps       : two groups taking alternate blocks; they build each block's shared score
//                       operands, turn the key outliers into one additive score term per token
//                       and tag every outlier with its token;
//   8 consumer warps  : warp w owns tokens 16w..16w+15 of every block and keeps its own
//                       flash-decode state (running max, sum, output), written as its own
//                       partial (m, l, o[128]) at the end of each (b, h) segment; the combine
//                       kernel merges the partials.
// The consumer warpgroups run with 168 registers per thread, the others with 88 (setmaxnreg).
//
// Keys ([KVQ] §3.2 pre-RoPE quantisation, Algorithm 1 dequantisation, worked example step 5):
// the key at absolute position n = n0 + t (n0 = 128 * block) is k_n = R(n) (s*C[q] + zp + o),
// so q . k_n = (R(t)^T q_b) . (s*C[q] + zp + o) with q_b = R(n0)^T q. Per channel pair i
// (angle t*theta_i) this is cos * X_i + sin * Y_i with
//     X_i = q_b0 k0 + q_b1 k1,    Y_i = q_b1 k0 - q_b0 k1.
// X and Y of 16 tokens x 4 pairs come out of one mma.sync m16n8k8: A = the codebook values C[q]
// of 16 tokens x 8 channels (looked up from the packed codes with byte permutes on an fp16 table
// held in registers), B = the block's q_b * s in fp16 in the X and Y columns of each pair, C =
// the zero-point terms. The cos/sin of a lane's own (token, pair) cells are fixed over blocks
// and stay in registers; the fp16 outliers o of the CSR enter as per-token score terms.
// Values ([KVQ] §3.7 value matvec): O[channel] = sum_t p_t s_t C[q] + sum_t p_t zp_t + outliers,
// one m16n8k16 per 16 channels x the warp's 16 tokens; B = p*s in high/low fp16 columns.
// Softmax in base 2 with the running max per warp (rescaling only when the max grows).
#include "kvq_internal.cuh"

#include <type_traits>

namespace kvq {
namespace nuqdec {

constexpr int NW = 8;               // consumer warps (16 tokens of each block per warp)
constexpr int NAUX = 128;           // aux threads: two groups that take alternate blocks
constexpr int AUX_GROUP = 64;       // threads of one aux group: one per channel pair, two tokens each
constexpr int PRODUCER_WARP = NW + NAUX / 32;  // issues the bulk copies; the warpgroup's other 3 warps idle
constexpr int NTHREADS = 512;       // 4 warpgroups: consumers (2), aux, producer
// Register split (setmaxnreg): launched at 65536 / 512 = 128 per thread; the consumer warpgroups
// take 168 and the others give back down to 88 (2 x 128 x 168 + 2 x 128 x 88 = 65536).
constexpr int REGS_CONSUMER = 168, REGS_OTHER = 88;
static_assert(2 * 128 * REGS_CONSUMER + 2 * 128 * REGS_OTHER <= 65536, "register split over the launch total");
constexpr int ROPE_ROW = 64 * 8;    // bytes of one (cos, sin) row of 64 pairs
constexpr int MAX_OUTLIERS = 2048;  // per tile, on this path
constexpr float LOG2E_RSQRT_D = 1.4426950408889634f * 0.08838834764831845f;
// The running reference of a warp's softmax moves only when a score exceeds it by more than this
// (base-2 units): probabilities then stay below 2^8, so p * s of a token stays far inside fp16.
constexpr float RESCALE_SLACK = 8.0f;
// Value outliers are summed as 64-bit fixed point with OUTV_FRAC fraction bits: integer addition
// is exact, so the sums do not depend on the order of the shared-memory atomics. |p * v| < 2^24
// (p <= 2^RESCALE_SLACK, |v| <= 65504), so 2^19 entries per warp and (b, h) segment stay inside
// the range even at that bound; the rounding is 2^-21 per entry.
constexpr int OUTV_FRAC = 20;
constexpr float OUTV_ONE = (float)(1 << OUTV_FRAC), OUTV_UNIT = 1.0f / OUTV_ONE;

#ifndef KVQ_NUQ_NB
#define KVQ_NUQ_NB 8
#endif
constexpr int NB = KVQ_NUQ_NB;  // ring stages

struct Args {
  Geo g;
  const uint8_t* base;
  const float* codebook;  // [H][8] fp32
  const uint16_t* q;
  int nb;                 // cached blocks per (b, h)
  long long total;        // B * H * nb
  int n_ranges;           // CTAs in the grid
  int n_slots;            // range slots per (b, query head)
  float* ws_m;
  float* ws_l;
  float* ws_o;
  int* status;
};

// Per-stage operands the aux warps prepare for the consumer warps.
struct Ops {
  uint32_t bk[9][20];  // score B rows 0..7 (q_b * s) of column g, 16 k-groups, padded; row 8 stays zero
  uint32_t bz[9][20];  // score B rows 8, 9 of column g: zero-point term (high, low); row 8 stays zero
  float sk[T];         // key-outlier score term per token
};

struct Smem {
  float2 rope_loc[T * 64];  // (cos, sin) of t * theta_i, t = 0..127
  Ops op[NB];
  float qb[2][D];           // per aux group: q rotated back by the block's start angle
  long long outv[NW][D];    // value outliers weighted by p, per consumer warp, in units of 2^-OUTV_FRAC
  uint64_t rec_full[NB];    // record and RoPE row landed (bulk copies)
  uint64_t ops_full[NB];    // score operands and outlier terms ready (AUX_GROUP arrivals)
  uint64_t empty[NB];       // the consumer warps are done with the stage (NW arrivals)
  // followed by NB x 2 x round16(n_outliers) bytes, per stage: the token of each key outlier,
  // then the token of each value outlier; then 2 x round16(n_outliers) floats, per aux group:
  // the score term of each key outlier
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// Nibble word U of a lane's 6-word code group: 8 codes in 4-bit slots (bit 3 of each slot clear),
// ready to serve as byte-permute selectors (low 16 bits: slots 0..3, high 16 bits: slots 4..7).
__device__ __forceinline__ uint32_t nibble_word(const uint32_t (&w)[6], const int U) {  // U: unrolled
  const uint32_t L = w[U >> 1], H = w[4 + (U >> 2)];
  const uint32_t lo = (U & 1) ? (L >> 2) : L;
  const uint32_t hi = (U & 3) == 0 ? H : (U & 3) == 1 ? (H >> 1) : (U & 3) == 2 ? (H << 2) : (H << 1);
  return (lo & 0x33333333u) | (hi & 0x44444444u);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Codebook values of the 4 codes selected by sel[15:0] as two fp16 pairs: (slot 0, slot 1) and
// (slot 2, slot 3). tl/th: low and high bytes of the 8 fp16 entries.
__device__ __forceinline__ void lookup4(uint32_t sel, uint32_t tl0, uint32_t tl1, uint32_t th0, uint32_t th1,
                                        uint32_t& p01, uint32_t& p23) {
  const uint32_t lo = prmt(tl0, tl1, sel), hi = prmt(th0, th1, sel);
  p01 = prmt(lo, hi, 0x5140u);
  p23 = prmt(lo, hi, 0x7362u);
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__host__ __device__ inline long long range_of(long long x, long long total, long long N) {
  return ((x + 1) * N - 1) / total;
}

// Query pair pi of (b, h) = u, scaled by log2(e)/sqrt(128).
__device__ __forceinline__ float2 load_q_pair(const Args& a, long long u, int pi) {
  const long long b = u / a.g.H, h = u - b * a.g.H;
  const uint16_t* qp = a.q + ((uint64_t)(b * a.g.Hq + h)) * D;
  return make_float2(load_in(qp + 2 * pi, a.g.in_bf16) * LOG2E_RSQRT_D,
                     load_in(qp + 2 * pi + 1, a.g.in_bf16) * LOG2E_RSQRT_D);
}

// __syncthreads_or over the 64 threads of aux group grp (named barrier 1 + grp).
__device__ __forceinline__ bool bar_or_group(int grp, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(1 + grp)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void bar_group(int grp) { asm volatile("bar.sync %0, 64;" ::"r"(1 + grp) : "memory"); }

__device__ __forceinline__ uint32_t stage_bytes(const Geo& g) { return (uint32_t)g.rec_bytes + ROPE_ROW; }

// Per-stage outlier area (after the ring and Smem): the token tag of each key outlier
// [round16(n)], the run index of each value outlier [round16(n)] (token for CSR value tiles,
// channel for CSC ones), and for CSC value tiles the permutation grouping the value entries by
// consumer warp (uint16 [n], 16-byte padded) followed by the 9 group offsets (uint16, 32 bytes).
__host__ __device__ inline int csc_off_of(int n_out) {  // from the value tags to the offsets
  return (int)round16((uint64_t)n_out) + (int)round16(2 * (uint64_t)n_out);
}
__host__ __device__ inline int rows_stride_of(int n_out, bool csc) {
  return 2 * (int)round16((uint64_t)n_out) + (csc ? (int)round16(2 * (uint64_t)n_out) + 32 : 0);
}

template <uint32_t R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(R));
}

// Producer warp: copies block p of the range into stage p % NBS once the consumer warps have
// released the stage's previous block (NW arrivals on empty). A block's three copies (K half;
// V half with the CSR; the block's RoPE start-angle row) go out as one instruction from three
// lanes, and the lane triple rotates over blocks: a thread services its own bulk copies one
// after another, a few hundred cycles each whatever their size, so copies from distinct lanes
// overlap. Before leaving it waits (bounded) for the last copies it issued.
template <int NBS>
__device__ void producer(const Args& a, Smem* sm, uint8_t* ring, long long x0, int n, int lane) {
  const Geo& g = a.g;
  const uint32_t rec = (uint32_t)g.rec_bytes, khalf = g.codes_off[1], sb = stage_bytes(g);
  long long u = x0 / a.nb;
  int blk = (int)(x0 - u * a.nb);
  int pb = (int)(u / g.H), ph = (int)(u - (long long)pb * g.H);  // (b, h) of block p
  int issued = 0;
  for (int p = 0; p < n; ++p) {
    const int s = p % NBS;
    if (p >= NBS) {
      const bool got = mbar_wait_bounded(&sm->empty[s], (uint32_t)(((p / NBS) - 1) & 1), a.status);
      if (__any_sync(0xffffffffu, !got)) break;
    }
    const int set = 3 * (p & 7), part = lane - set;  // lanes set .. set+2 copy this block
    if (lane == set) mbar_arrive_expect_tx(&sm->rec_full[s], rec + ROPE_ROW);
    __syncwarp();
    if (part >= 0 && part < 3) {
      fence_proxy_async();
      const uint32_t off = part == 0 ? 0u : part == 1 ? khalf : rec;
      const uint32_t bytes = part == 0 ? khalf : part == 1 ? rec - khalf : (uint32_t)ROPE_ROW;
      const uint8_t* from =
          part == 2 ? a.base + g.rope_off + (size_t)blk * ROPE_ROW : a.base + record_offset(g, pb, ph, blk, a.status) + off;
      bulk_g2s(ring + (size_t)s * sb + off, from, bytes, &sm->rec_full[s]);
    }
    issued = p + 1;
    if (++blk == a.nb) {
      blk = 0;
      if (++ph == g.H) {
        ph = 0;
        ++pb;
      }
    }
  }
  for (int p = max(0, issued - NBS); p < issued; ++p)
    mbar_wait_bounded(&sm->rec_full[p % NBS], (uint32_t)((p / NBS) & 1), nullptr, 200000000LL);
}

// Aux warps: two groups of 64 threads, group grp preparing blocks grp, grp + 2, grp + 4, ... of
// the range (named barrier 1 + grp), so each group has two block periods per block. Per block,
// thread j of a group first handles channel pair j (score B operand, zero-point terms, q_b) and
// tokens j and j + 64 (the token tag of each of their key- and value-outlier entries); then it
// computes the score terms of the key-outlier entries e = j, j + 64, ...
//     v * (R(t)^T q_b)_c    (entry e = (t, c, v) of the CSR)
// and, after a group barrier, the sum sk[t] of each of its two tokens' terms in entry order.
// The consumers scatter p_t * v for the value outliers.
template <int NBS, bool CSC>
__device__ void aux_warps(const Args& a, Smem* sm, uint8_t* ring, uint8_t* rows, int rows_stride, long long x0,
                          int n, int ax) {
  const Geo& g = a.g;
  const uint32_t rec = (uint32_t)g.rec_bytes, sb = stage_bytes(g);
  const int n_out = g.n_out;
  const int grp = ax >> 6, j = ax & 63;
  const int tag_bytes = (int)round16((uint64_t)n_out);
  long long u = x0 / a.nb;
  int blk = (int)(x0 - u * a.nb);
  if (grp == 1 && ++blk == a.nb) {
    blk = 0;
    ++u;
  }
  long long cur_u = -1;
  float2 qv = make_float2(0.0f, 0.0f);
  float* qb = sm->qb[grp];
  float* kterm = reinterpret_cast<float*>(rows + (size_t)NBS * rows_stride) + grp * tag_bytes;  // per group
  // CSC value tiles: per group, entries per consumer warp [8] and the scatter cursors [8]
  int* gcnt = reinterpret_cast<int*>(reinterpret_cast<float*>(rows + (size_t)NBS * rows_stride) + 2 * tag_bytes) +
              grp * 16;
  const int tA = j, tB = j + 64;
  for (int p = grp; p < n; p += 2) {
    if (u != cur_u) {
      cur_u = u;
      qv = load_q_pair(a, u, j);
    }
    const int s = p % NBS;
    const bool got = mbar_wait_bounded(&sm->rec_full[s], (uint32_t)((p / NBS) & 1), a.status);
    if (bar_or_group(grp, !got)) break;  // the consumers time out on their own waits
    const uint8_t* st = ring + (size_t)s * sb;
    Ops& op = sm->op[s];
    {
      const float2 cs = reinterpret_cast<const float2*>(st + rec)[j];
      const float qb0 = cs.x * qv.x + cs.y * qv.y, qb1 = -cs.y * qv.x + cs.x * qv.y;
      const uint16_t* km = reinterpret_cast<const uint16_t*>(st + g.meta_off[0]);
      const int kg = j >> 2, tqp = j & 3;
      const float s0 = h2f(km[2 * j]), s1 = h2f(km[2 * j + 1]);
      const float z0 = h2f(km[T + 2 * j]), z1 = h2f(km[T + 2 * j + 1]);
      op.bk[2 * tqp][kg] = pack_h2(qb0 * s0, qb1 * s1);       // X column of pair j
      op.bk[2 * tqp + 1][kg] = pack_h2(qb1 * s0, -qb0 * s1);  // Y column
      const float zx = qb0 * z0 + qb1 * z1, zy = qb1 * z0 - qb0 * z1;
      const __half zxh = __float2half_rn(zx), zyh = __float2half_rn(zy);
      op.bz[2 * tqp][kg] = pack_h2(zx, zx - __half2float(zxh));      // X column: (high, low)
      op.bz[2 * tqp + 1][kg] = pack_h2(zy, zy - __half2float(zyh));  // Y column
      *reinterpret_cast<float2*>(&qb[2 * j]) = make_float2(qb0, qb1);
    }
    float skA = 0.0f, skB = 0.0f;
    if (n_out > 0) {
      uint8_t* ktag = rows + (size_t)s * rows_stride;
      uint8_t* vtag = ktag + tag_bytes;
      const uint8_t* csr = st + g.csr_off[0];
      const uint16_t* rp = reinterpret_cast<const uint16_t*>(csr + 2 * n_out);
      const uint16_t* rpv = reinterpret_cast<const uint16_t*>(st + g.csr_off[1] + 2 * n_out);
      const int ka0 = min((int)rp[tA], n_out), ka1 = min((int)rp[tA + 1], n_out);
      const int kb0 = min((int)rp[tB], n_out), kb1 = min((int)rp[tB + 1], n_out);
      {
        const int va0 = min((int)rpv[tA], n_out), va1 = min((int)rpv[tA + 1], n_out);
        const int vb0 = min((int)rpv[tB], n_out), vb1 = min((int)rpv[tB + 1], n_out);
        for (int e = ka0; e < ka1; ++e) ktag[e] = (uint8_t)tA;
        for (int e = kb0; e < kb1; ++e) ktag[e] = (uint8_t)tB;
        for (int e = va0; e < va1; ++e) vtag[e] = (uint8_t)tA;
        for (int e = vb0; e < vb1; ++e) vtag[e] = (uint8_t)tB;
        if (CSC && j < 16) gcnt[j] = 0;
      }
      bar_group(grp);  // q_b and the key tags visible
      if (CSC) {  // group the value entries by consumer warp (16 tokens each): count, offsets, scatter
        const uint8_t* vtok = st + g.csr_off[1] + 2 * n_out + 2 * (T + 1);  // token of each entry
        uint16_t* perm = reinterpret_cast<uint16_t*>(vtag + tag_bytes);
        uint16_t* off = reinterpret_cast<uint16_t*>(vtag + csc_off_of(n_out));
        const int n_v = min((int)rpv[T], n_out);
        for (int e = j; e < n_v; e += 64) atomicAdd(&gcnt[(vtok[e] >> 4) & 7], 1);
        bar_group(grp);
        if (j == 0) {
          int acc = 0;
          for (int w = 0; w < 8; ++w) {
            off[w] = (uint16_t)acc;
            gcnt[8 + w] = acc;
            acc += gcnt[w];
          }
          off[8] = (uint16_t)acc;
        }
        bar_group(grp);
        for (int e = j; e < n_v; e += 64) perm[atomicAdd(&gcnt[8 + ((vtok[e] >> 4) & 7)], 1)] = (uint16_t)e;
      }
      const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
      const uint8_t* col = csr + 2 * n_out + 2 * (T + 1);
      const int n_k = min((int)rp[T], n_out);
      auto key_term = [&](int e) {  // score term of key-outlier entry e < n_k
        const int c = col[e] & (D - 1), t = ktag[e] & (T - 1);
        const float2 cr = sm->rope_loc[t * 64 + (c >> 1)];
        const float qa = qb[c & ~1], qc = qb[c | 1];
        const float qq = (c & 1) ? (-cr.y * qa + cr.x * qc) : (cr.x * qa + cr.y * qc);
        return h2f(val[e]) * qq;
      };
      // every entry's term (up to 4 per thread side by side; 1% of a tile is 164 entries), then
      // each token's terms summed in entry order: the result does not depend on thread timing
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (j + AUX_GROUP * k < n_k) kterm[j + AUX_GROUP * k] = key_term(j + AUX_GROUP * k);
      for (int e = j + 4 * AUX_GROUP; e < n_k; e += AUX_GROUP) kterm[e] = key_term(e);
      bar_group(grp);
      for (int e = ka0; e < ka1; ++e) skA += kterm[e];
      for (int e = kb0; e < kb1; ++e) skB += kterm[e];
    }
    op.sk[tA] = skA;
    op.sk[tB] = skB;
    mbar_arrive(&sm->ops_full[s]);  // AUX_GROUP arrivals complete the phase
    blk += 2;
    while (blk >= a.nb) {
      blk -= a.nb;
      ++u;
    }
  }
}

// Scores of a consumer warp's 16 tokens in one block (after the reduction over the 4 lanes of a
// token and the key-outlier terms): s0 for token 16w + gq, s1 for token 16w + gq + 8.
__device__ __forceinline__ void block_scores(const uint8_t* st, const Ops& op, uint32_t codes_off, int warp, int lane,
                                             int brow, int zrow, uint32_t ones, int t0, int t1, uint32_t tl0,
                                             uint32_t tl1, uint32_t th0, uint32_t th1, const float2 (&w)[2][16],
                                             float& s0, float& s1) {
  uint32_t cw[6];
  const uint2* kp = reinterpret_cast<const uint2*>(st + codes_off + warp * 768 + lane * 24);
  const uint2 k0 = kp[0], k1 = kp[1], k2 = kp[2];
  cw[0] = k0.x; cw[1] = k0.y; cw[2] = k1.x; cw[3] = k1.y; cw[4] = k2.x; cw[5] = k2.y;
  const uint4* bp = reinterpret_cast<const uint4*>(&op.bk[brow][0]);
  const uint4* zp = reinterpret_cast<const uint4*>(&op.bz[zrow][0]);
  const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float2 acc[2][2] = {{{0.0f, 0.0f}, {0.0f, 0.0f}}, {{0.0f, 0.0f}, {0.0f, 0.0f}}};
#pragma unroll
  for (int uu = 0; uu < 8; ++uu) {
    const uint32_t nw = nibble_word(cw, uu);
    const uint4 bq = bp[uu >> 1], zq = zp[uu >> 1];  // k-groups 4(uu/2) .. 4(uu/2)+3
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int kg = 2 * uu + hf;
      uint32_t a0, a1;
      lookup4(hf ? (nw >> 16) : nw, tl0, tl1, th0, th1, a0, a1);
      const uint32_t bb = (kg & 3) == 0 ? bq.x : (kg & 3) == 1 ? bq.y : (kg & 3) == 2 ? bq.z : bq.w;
      const uint32_t bz = (kg & 3) == 0 ? zq.x : (kg & 3) == 1 ? zq.y : (kg & 3) == 2 ? zq.z : zq.w;
      float d[4];
      mma16816(d, a0, a1, ones, ones, bb, bz, zero4);  // X, Y of pair 4kg+tq incl. the zero-point term
      acc[0][hf] = __ffma2_rn(w[0][kg], make_float2(d[0], d[1]), acc[0][hf]);
      acc[1][hf] = __ffma2_rn(w[1][kg], make_float2(d[2], d[3]), acc[1][hf]);
    }
  }
  s0 = (acc[0][0].x + acc[0][1].x) + (acc[0][0].y + acc[0][1].y);
  s1 = (acc[1][0].x + acc[1][1].x) + (acc[1][0].y + acc[1][1].y);
  s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
  s0 += __shfl_xor_sync(0xffffffffu, s0, 2) + op.sk[t0];
  s1 += __shfl_xor_sync(0xffffffffu, s1, 2) + op.sk[t1];
}

// Value product of one block for a consumer warp: p' = p * s_token as high/low B columns, the
// zero-point sum and 8 m16n8k16 over the V codes.
__device__ __forceinline__ void block_values(const uint8_t* st, const Geo& g, int warp, int lane, int t0, int t1,
                                             int src_a, uint32_t xsel, uint32_t ysel, float p0, float p1,
                                             uint32_t tl0, uint32_t tl1, uint32_t th0, uint32_t th1, float& z_w,
                                             float (&acc)[8][4]) {
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

// Value outliers of a consumer warp's tokens in one block. rw: the stage's value-outlier area
// written by the aux warps: each entry's pointer-run index (the token for CSR tiles, the channel
// for CSC tiles), then for CSC tiles a permutation of the entries that groups them by consumer
// warp (16 tokens each) and the 9 group offsets. Entry k of the warp's span goes to lane
// (k - e0) mod 32, which takes p of its token from the token's owner lane and adds p * v to the
// warp's outv (integer atomics: the sum does not depend on the order). The first 32 entries run
// as one batch placed with the tensor-core work of the block; later ones loop.
template <bool CSC>
__device__ __forceinline__ void value_outlier_span(const uint8_t* st, const uint8_t* rw, const Geo& g, int warp,
                                                   int& e0, int& e1) {
  const int n_out = g.n_out;
  if (CSC) {
    const uint16_t* off = reinterpret_cast<const uint16_t*>(rw + csc_off_of(n_out));
    e0 = off[warp];
    e1 = off[warp + 1];
  } else {
    const uint16_t* rp = reinterpret_cast<const uint16_t*>(st + g.csr_off[1] + 2 * n_out);
    e0 = min((int)rp[16 * warp], n_out);
    e1 = min((int)rp[16 * warp + 16], n_out);
  }
}

// Value-outlier entry k of the lane (k >= e1: none): p_t * v added to the warp's outv[c] in
// fixed point (a shared-memory integer atomic; no branch, so it sits among the tensor-core work).
template <bool CSC>
__device__ __forceinline__ void value_outlier_entry(const uint8_t* st, const Geo& g, const uint8_t* rw, int k, int e1,
                                                    int t0, float p0, float p1, long long* outv) {
  const int n_out = g.n_out;
  const uint8_t* csr = st + g.csr_off[1];
  const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
  const uint8_t* idx = csr + 2 * n_out + 2 * (T + 1);  // CSR: channel; CSC: token
  const bool valid = k < e1;
  int e = k, t;
  if (CSC) {
    e = valid ? (int)reinterpret_cast<const uint16_t*>(rw + round16((uint64_t)n_out))[k] : 0;
    t = valid ? idx[e] : t0;
  } else {
    t = valid ? rw[e] : t0;
  }
  const int src = 4 * (t & 7);
  const float pa = __shfl_sync(0xffffffffu, p0, src), pb = __shfl_sync(0xffffffffu, p1, src);
  if (valid) {
    const float x = ((t & 8) ? pb : pa) * h2f(val[e]);
    atomicAdd(reinterpret_cast<unsigned long long*>(&outv[(CSC ? rw[e] : idx[e]) & (D - 1)]),
              (unsigned long long)llrintf(x * OUTV_ONE));
  }
}

// Consumer warp w: tokens 16w..16w+15 of every block of the CTA's range. Within a (b, h) segment
// the value product of block j and the scores of block j + 1 form one straight-line stretch, so
// their dependency chains overlap. Its flash-decode state goes to its own partial row at the end
// of each segment.
template <int NBS, bool CSC>
__device__ void consumer(const Args& a, Smem* sm, const uint8_t* ring, const uint8_t* rows, int rows_stride, long long R,
                         long long x0, int n, int warp, int lane) {
  const Geo& g = a.g;
  const uint32_t sb = stage_bytes(g);
  const int gq = lane >> 2, tq = lane & 3;
  // (cos, sin) of the lane's (token, pair) cells: tokens 16w + gq + 8r, pairs 4kg + tq
  float2 wcs[2][16];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int kg = 0; kg < 16; ++kg) wcs[r][kg] = sm->rope_loc[(16 * warp + gq + 8 * r) * 64 + 4 * kg + tq];
  const int brow = (gq >> 1) == tq ? gq : 8;             // lanes holding nonzero score B rows 0..7
  const int zrow = tq == 0 ? gq : 8;                     // lanes holding the zero-point rows 8, 9
  const uint32_t ones = tq == 0 ? 0x3c003c00u : 0u;      // A columns 8, 9 = 1.0 (fp16), others 0
  const int src_a = 4 * tq + (gq < 2 ? gq : 2);          // value B: (high, low, zero) source lanes
  const uint32_t xsel = tq == 0 ? 0xffffffffu : 0u;      // this lane sends p' high (tq 0) ...
  const uint32_t ysel = tq == 1 ? 0xffffffffu : 0u;      // ... or low (tq 1) or zero
  const int t0 = 16 * warp + gq, t1 = t0 + 8;
  long long* outv = sm->outv[warp];

  auto ready_now = [&](int i) -> bool {  // the stage of range block i is ready (no waiting)
    const int s = i % NBS;
    const uint32_t par = (uint32_t)((i / NBS) & 1);
    return mbar_test_wait(&sm->ops_full[s], par) & mbar_test_wait(&sm->rec_full[s], par);
  };
  auto wait_stage = [&](int i) -> bool {  // false when a wait gave up
    const int s = i % NBS;
    const uint32_t par = (uint32_t)((i / NBS) & 1);
    const bool got = mbar_wait_bounded(&sm->ops_full[s], par, a.status) &&
                     mbar_wait_bounded(&sm->rec_full[s], par, a.status);
    return !__any_sync(0xffffffffu, !got);
  };
  auto release = [&](int s) {  // this warp is done with stage s
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm->empty[s]);
  };

  long long u = x0 / a.nb;
  int blk = (int)(x0 - u * a.nb);
  float acc[8][4];
  int i = 0;
  while (i < n) {
    const int iend = (int)min((long long)n, (long long)i + (a.nb - blk));  // this (b, h) segment
    uint32_t tl0, tl1, th0, th1;
    {
      const long long h = u % g.H;
      uint32_t hb[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) hb[k] = f2h_rn(__ldg(a.codebook + h * 8 + k));
      tl0 = (hb[0] & 0xffu) | (hb[1] & 0xffu) << 8 | (hb[2] & 0xffu) << 16 | (hb[3] & 0xffu) << 24;
      tl1 = (hb[4] & 0xffu) | (hb[5] & 0xffu) << 8 | (hb[6] & 0xffu) << 16 | (hb[7] & 0xffu) << 24;
      th0 = (hb[0] >> 8) | (hb[1] >> 8) << 8 | (hb[2] >> 8) << 16 | (hb[3] >> 8) << 24;
      th1 = (hb[4] >> 8) | (hb[5] >> 8) << 8 | (hb[6] >> 8) << 16 | (hb[7] >> 8) << 24;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) outv[lane + 32 * k] = 0;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
    float m_w = -INFINITY, l_w = 0.0f, z_w = 0.0f;
    __syncwarp();
    if (!wait_stage(i)) return;
    float sv0, sv1;
    block_scores(ring + (size_t)(i % NBS) * sb, sm->op[i % NBS], g.codes_off[0], warp, lane, brow, zrow, ones, t0, t1,
                 tl0, tl1, th0, th1, wcs, sv0, sv1);
    for (int j = i; j < iend; ++j) {
      const int s = j % NBS;
      const uint8_t* st = ring + (size_t)s * sb;
      const bool more = j + 1 < iend;  // warp-uniform
      const bool ready = more ? ready_now(j + 1) : true;  // its latency overlaps the softmax
      if (g.sink && blk + (j - i) == 0 && warp == 0 && gq == 0) sv0 = -INFINITY;  // the kept first token
      // online softmax with block j's scores (base 2). m_w is the reference the warp's sums are
      // kept relative to; it moves up only when a score passes it by more than RESCALE_SLACK, so
      // p = 2^(s - m_w) stays below 2^RESCALE_SLACK and the usual block needs one vote instead of
      // a max reduction.
      if (__any_sync(0xffffffffu, fmaxf(sv0, sv1) > m_w + RESCALE_SLACK)) {  // rare after the first blocks
        float mloc = fmaxf(sv0, sv1);
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 4));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 8));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16));
        mloc = fmaxf(mloc, m_w);
        const float al = exp2f(m_w - mloc);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          acc[mt][0] *= al; acc[mt][1] *= al; acc[mt][2] *= al; acc[mt][3] *= al;
        }
        l_w *= al;
        z_w *= al;
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k) outv[lane + 32 * k] = llrintf((float)outv[lane + 32 * k] * al);
        __syncwarp();
        m_w = mloc;
      }
      const float p0 = exp2f(sv0 - m_w), p1 = exp2f(sv1 - m_w);
      l_w += p0 + p1;
      const uint8_t* rw = rows + (size_t)s * rows_stride + round16((uint64_t)g.n_out);
      int e0 = 0, e1 = 0;
      if (g.n_out > 0) value_outlier_span<CSC>(st, rw, g, warp, e0, e1);
      if (more) {
        if (!__all_sync(0xffffffffu, ready) && !wait_stage(j + 1)) return;
        const int s1 = (j + 1) % NBS;
        value_outlier_entry<CSC>(st, g, rw, e0 + lane, e1, t0, p0, p1, outv);
        block_values(st, g, warp, lane, t0, t1, src_a, xsel, ysel, p0, p1, tl0, tl1, th0, th1, z_w, acc);
        block_scores(ring + (size_t)s1 * sb, sm->op[s1], g.codes_off[0], warp, lane, brow, zrow, ones, t0, t1, tl0,
                     tl1, th0, th1, wcs, sv0, sv1);
      } else {
        value_outlier_entry<CSC>(st, g, rw, e0 + lane, e1, t0, p0, p1, outv);
        block_values(st, g, warp, lane, t0, t1, src_a, xsel, ysel, p0, p1, tl0, tl1, th0, th1, z_w, acc);
      }
      for (int e = e0 + 32 + lane; e - lane < e1; e += 32)  // more than 32 entries: uniform trip count
        value_outlier_entry<CSC>(st, g, rw, e, e1, t0, p0, p1, outv);
      release(s);
    }
    // the segment's partial row
    {
      float lt = l_w, zt = z_w;  // replicated over tq: reduce over gq only
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        lt += __shfl_xor_sync(0xffffffffu, lt, o);
        zt += __shfl_xor_sync(0xffffffffu, zt, o);
      }
      __syncwarp();
      const long long b = u / g.H, h = u - b * g.H;
      const long long slot = R - range_of(u * a.nb, a.total, a.n_ranges);
      if (slot >= 0 && slot < a.n_slots) {
        const uint64_t row = (((uint64_t)(b * g.Hq + h)) * a.n_slots + slot) * NW + warp;
        if (tq == 0) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int c0 = 16 * mt + gq, c1 = c0 + 8;
            a.ws_o[row * D + c0] = acc[mt][0] + acc[mt][1] + zt + (float)outv[c0] * OUTV_UNIT;
            a.ws_o[row * D + c1] = acc[mt][2] + acc[mt][3] + zt + (float)outv[c1] * OUTV_UNIT;
          }
        }
        if (lane == 0) {
          a.ws_m[row] = m_w;
          a.ws_l[row] = lt;
        }
      }
      __syncwarp();
    }
    i = iend;
    blk = 0;
    ++u;
  }
}

template <int NBS, bool CSC>
__global__ void __launch_bounds__(NTHREADS, 1) decode_nuq_kernel(Args a) {
  launch_dependents();  // the combine kernel may be scheduled once every CTA of this grid runs
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* ring = smem_raw;
  Smem* sm = reinterpret_cast<Smem*>(smem_raw + (size_t)NBS * stage_bytes(a.g));
  uint8_t* rows = reinterpret_cast<uint8_t*>(sm + 1);
  const int rows_stride = rows_stride_of(a.g.n_out, CSC);
  const long long R = blockIdx.x;
  if (R >= a.n_ranges) return;
  const long long x0 = R * a.total / a.n_ranges, x1 = (R + 1) * a.total / a.n_ranges;
  const int n = (int)(x1 - x0);
  if (n <= 0) return;
  {  // the in-block angle table, staged once per CTA
    const float4* src = reinterpret_cast<const float4*>(a.base + a.g.rope_off) + (size_t)(a.g.max_blocks + 1) * 32;
    float4* dst = reinterpret_cast<float4*>(sm->rope_loc);
    for (int e = tid; e < T * 32; e += NTHREADS) dst[e] = __ldg(src + e);
  }
  for (int e = tid; e < NBS * 20; e += NTHREADS) {
    sm->op[e / 20].bk[8][e % 20] = 0u;
    sm->op[e / 20].bz[8][e % 20] = 0u;
  }
  if (tid == 0) {
    for (int s = 0; s < NBS; ++s) {
      mbar_init(&sm->rec_full[s], 1);
      mbar_init(&sm->ops_full[s], AUX_GROUP);
      mbar_init(&sm->empty[s], NW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp < NW) {
    regs_inc<REGS_CONSUMER>();
    consumer<NBS, CSC>(a, sm, ring, rows, rows_stride, R, x0, n, warp, lane);
  } else {
    regs_dec<REGS_OTHER>();
    if (warp < PRODUCER_WARP) aux_warps<NBS, CSC>(a, sm, ring, rows, rows_stride, x0, n, tid - NW * 32);
    else if (warp == PRODUCER_WARP) producer<NBS>(a, sm, ring, x0, n, lane);
  }
}

size_t smem_bytes(const Geo& g) {
  return (size_t)NB * ((size_t)g.rec_bytes + ROPE_ROW) + sizeof(Smem) + (size_t)NB * rows_stride_of(g.n_out, g.v_csc) +
         2 * sizeof(float) * round16((uint64_t)g.n_out) + (g.v_csc ? 2 * 16 * sizeof(int) : 0);
}

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
  return g.method == KVQ_NUQ && g.bits == 3 && g.planes3 && g.G == 1 && g.pre_rope == 1 &&
         g.n_out <= kvq::nuqdec::MAX_OUTLIERS && kvq::nuqdec::smem_bytes(g) <= 227 * 1024;
}

// CTAs (ranges) the nuq decode uses on the current device, or 0 if the path does not apply.
// Without a usable device it assumes a 152-SM part with one CTA per SM.
long long kvq_nuq_ranges(const kvq::Geo& g) {
  using namespace kvq::nuqdec;
  if (!kvq_nuq_supported(g)) return 0;
  const size_t smem = smem_bytes(g);
  auto fn = g.v_csc ? decode_nuq_kernel<NB, true> : decode_nuq_kernel<NB, false>;
  int dev = 0, sms = 152, ctas = 1;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
    NuqOcc* hit = nullptr;
    for (auto& c : t_nuq_occ)
      if (c.dev == dev && c.smem == smem) hit = &c;
    if (!hit) {
      // raise (never lower) the kernel's shared-memory limit through the shared bookkeeping
      if (kvq::ensure_smem_attr((const void*)fn, smem) != cudaSuccess) cudaGetLastError();
      int occ = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, NTHREADS, smem) != cudaSuccess || occ < 1)
        occ = 1;
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

// Partial rows each range writes per (b, query head): one per consumer warp.
int kvq_nuq_parts_per_range() { return kvq::nuqdec::NW; }

// slots: range slots per (b, query head); the workspace holds slots * NW partial rows each.
cudaError_t kvq_launch_decode_nuq(const kvq::Geo& g, const uint8_t* base, const float* codebook, const uint16_t* q,
                                  int n_blocks, long long ranges, long long slots, float* ws_m, float* ws_l,
                                  float* ws_o, int* status, cudaStream_t st) {
  using namespace kvq::nuqdec;
  const size_t smem = smem_bytes(g);
  auto fn = g.v_csc ? decode_nuq_kernel<NB, true> : decode_nuq_kernel<NB, false>;
  cudaError_t e = kvq::ensure_smem_attr((const void*)fn, smem);
  if (e != cudaSuccess) return e;
  Args a;
  a.g = g; a.base = base; a.codebook = codebook; a.q = q; a.nb = n_blocks;
  a.total = (long long)g.B * g.H * n_blocks; a.n_ranges = (int)ranges; a.n_slots = (int)slots;
  a.ws_m = ws_m; a.ws_l = ws_l; a.ws_o = ws_o; a.status = status;
  fn<<<(int)ranges, NTHREADS, smem, st>>>(a);
  return cudaGetLastError();
}
