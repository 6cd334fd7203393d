// Decode attention over 3-bit nuq caches whose keys are stored before RoPE, on the tensor cores
// (one query head per KV head).
//
// Work split. The (b, h, block) sequence of the whole batch is cut into one contiguous range
// per CTA (persistent: one wave). A CTA runs 4 warpgroups whose roles meet only on mbarriers
// (every wait bounded):
//   producer warp     : copies each block record (K tile; V tile with the CSR outliers) into an
//                       NB-stage ring with two 1-D bulk copies, as soon as the consumers have
//                       released the stage;
//   4 aux warps       : two groups taking alternate blocks; per block they build the shared score
//                       operands, turn the key outliers into one additive score term per token
//                       and tag every outlier with its token;
//   8 consumer warps  : warp w owns tokens 16w..16w+15 of every block and keeps its own
//                       flash-decode state (running max, sum, output), written as its own
//                       partial (m, l, o[128]) at the end of each (b, h) segment; the combine
//                       kernel merges the partials. They publish each block's probabilities;
//   2 value-outlier warps: add the value outliers weighted by those probabilities into the
//                       consumers' outlier vectors, off the consumers' dependency chain;
//   1 tail warp       : attends the fp tail of the call (one warp per (b, head) over the grid).
// The consumer warpgroups run with 168 registers per thread, the others with 88 (setmaxnreg).
//
// Keys ([KVQ] §3.2 pre-RoPE quantisation, Algorithm 1 dequantisation, worked example step 5):
// the key at absolute position n = n0 + t (n0 = 128 * block) is k_n = R(n) (s*C[q] + zp + o),
// so q . k_n = (R(t)^T q_b) . (s*C[q] + zp + o) with q_b = R(n0)^T q. Per channel pair i
// (angle t*theta_i) this is cos * X_i + sin * Y_i with
//     X_i = q_b0 k0 + q_b1 k1,    Y_i = q_b1 k0 - q_b0 k1.
// X and Y of 16 tokens x 4 pairs come out of one mma.sync m16n8k16: A = the codebook values C[q]
// of 16 tokens x 8 channels (looked up from the packed codes with byte permutes on an fp16 table
// held in registers) and ones, B = the block's q_b * s in fp16 in the X and Y columns of each
// pair and the zero-point terms against the ones. The cos/sin of a lane's own (token, pair)
// cells are fixed over blocks and stay in registers; the fp16 outliers o of the CSR enter as
// per-token score terms.
// Values ([KVQ] §3.7 value matvec): O[channel] = sum_t p_t s_t C[q] + sum_t p_t zp_t + outliers,
// one m16n8k16 per 16 channels x the warp's 16 tokens with B = p*s in high/low fp16 columns; the
// value outliers add p_t * v per channel in token order (a fixed sequence of fp32 additions, the
// same for CSR and CSC value tiles), by the value-outlier warps.
// Softmax in base 2 with the running max per warp (rescaling only when the max grows).
#include "kvq_internal.cuh"

#include <type_traits>

namespace kvq {
namespace nuqdec {

constexpr int NW = 8;               // consumer warps (16 tokens of each block per warp)
constexpr int NAUX = 128;           // aux threads: two groups that take alternate blocks
constexpr int AUX_GROUP = 64;       // threads of one aux group: one per channel pair, two tokens each
constexpr int PRODUCER_WARP = NW + NAUX / 32;  // issues the bulk copies
constexpr int TAIL_WARP = PRODUCER_WARP + 1;     // attends the fp tail
constexpr int VOUT_WARP = TAIL_WARP + 1;         // first of the warps that add the value outliers
constexpr int NVOUT = 2;
static_assert(VOUT_WARP + NVOUT == 512 / 32, "warp roles fill the CTA");
constexpr int NTHREADS = 512;       // 4 warpgroups: consumers (2), aux, producer
// Register split (setmaxnreg): launched at 65536 / 512 = 128 per thread; the consumer warpgroups
// take 168 and the others give back down to 88 (2 x 128 x 168 + 2 x 128 x 88 = 65536).
constexpr int REGS_CONSUMER = 168, REGS_OTHER = 88;
static_assert(2 * 128 * REGS_CONSUMER + 2 * 128 * REGS_OTHER <= 65536, "register split over the launch total");
constexpr int MAX_OUTLIERS = 2048;  // per tile, on this path
constexpr float LOG2E_RSQRT_D = 1.4426950408889634f * 0.08838834764831845f;
// The running reference of a warp's softmax moves only when a score exceeds it by more than this
// (base-2 units): probabilities then stay below 2^8, so p * s of a token stays far inside fp16.
constexpr float RESCALE_SLACK = 8.0f;

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
  int rows_ph;            // partial rows per (b, query head): n_slots * NW range rows, then the tail row
  float* ws_m;
  float* ws_l;
  float* ws_o;
  int* status;
  const uint16_t* tail_k;  // fp tail (the call's inputs), attended by the idle warps
  const uint16_t* tail_v;
  int n_tail;
  long long tail_bh;       // elements between the tail rows of consecutive (b, h)
  long long tail_tok;      // elements between consecutive tokens of a tail row
};

// Per-stage operands the aux warps prepare for the consumer warps.
struct Ops {
  // Score B fragments: row n (0..7) holds, for each of the 16 k-groups, the pair (b0, b1) of the
  // lane that owns column n (X of pair n/2 for even n, Y for odd n): b0 = the column's two code
  // rows (q_b * s), b1 = its zero-point term (high, low). Row 8 stays zero (lanes holding no
  // part of B); rows are 36 words apart so that the 8 rows' 16-byte loads hit distinct banks.
  uint32_t b[9][36];
  float sk[T];         // key-outlier score term per token
};

struct Smem {
  Ops op[NB];
  float2 rope_a[8][64];      // (cos, sin) of 16a * theta_i, a = 0..7 (in-block angles, coarse)
  float2 rope_b[16][64];     // (cos, sin) of b * theta_i, b = 0..15 (fine): t = 16a + b
  float qb[2][D];            // per aux group: q rotated back by the block's start angle
  float outv[NW][D + 32];    // value outliers weighted by p, per consumer warp (+ a slot per lane)
  int own[NW][D + 32];       // owner table per (consumer warp, channel) for the value-outlier batches (32: none)
  float pub[NB][T];          // per stage: each token's probability p (relative to its warp's reference)
  float alw[NB][NW];         // per stage and consumer warp: the factor its reference moved by (1: none)
  uint64_t rec_full[NB];     // record landed (bulk copies)
  uint64_t ops_full[NB];     // score operands, key-outlier terms and outlier tags ready (AUX_GROUP arrivals)
  uint64_t empty[NB];        // the stage is free again (NW consumer + NVOUT value-outlier warp arrivals)
  uint64_t p_full[NB];       // the block's probabilities are published (NW arrivals)
  uint64_t vdone[NB];        // the block's value outliers are in outv (NVOUT arrivals)
  // followed by NB x rows_stride bytes, per stage: the token of each key outlier [round16(n)] and the
  // run index of each value outlier [round16(n)] (token for CSR value tiles, channel for CSC ones);
  // then per aux group round16(n) floats (the score term of each key outlier)
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

__device__ __forceinline__ uint32_t stage_bytes(const Geo& g) { return (uint32_t)g.rec_bytes; }

// 2^x on the special-function unit (x <= 0 here; -inf gives 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Per-stage outlier area (after the ring and Smem): the token tag of each key outlier
// [round16(n)] and the run index of each value outlier [round16(n)] (its token for CSR value tiles,
// its channel for CSC ones).
__host__ __device__ inline int rows_stride_of(int n_out) { return 2 * (int)round16((uint64_t)n_out); }

// (the memory clobber keeps loads of the role code below the register split)
template <uint32_t R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(R) : "memory");
}
template <uint32_t R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(R) : "memory");
}

#ifndef KVQ_NUQ_HELPER_SUSPEND
#define KVQ_NUQ_HELPER_SUSPEND 1  // measured 89.7 vs 91.1 us per decode, 1.6% fewer instructions
#endif
// Waits of the warps that run ahead of the consumers (producer, aux): a sleeping probe loop, or
// (KVQ_NUQ_HELPER_SUSPEND) the barrier's own suspending wait. Both bounded.
__device__ __forceinline__ bool helper_wait(uint64_t* bar, uint32_t parity, int* status, long long max_cycles) {
  if (KVQ_NUQ_HELPER_SUSPEND) return mbar_wait_bounded(bar, parity, status, max_cycles);
  return mbar_wait_backoff(bar, parity, status, max_cycles);
}

// Producer warp: copies block p of the range into stage p % NBS once the consumer warps have
// released the stage's previous block (NW arrivals on empty). A block's two copies (K half; V
// half with the CSR) go out as one instruction from two lanes, and the lane pair rotates over
// blocks: a thread services its own bulk copies one after another, a few hundred cycles each
// whatever their size, so copies from distinct lanes overlap. (Every further copy per block
// costs the same again: the block's RoPE start row, 512 bytes, comes through the aux warps'
// plain loads instead.) Before leaving it waits (bounded) for the last copies it issued.
template <int NBS>
__device__ void producer(const Args& a, Smem* sm, uint8_t* ring, long long x0, int n, int lane) {
  const Geo& g = a.g;
  const uint32_t rec = (uint32_t)g.rec_bytes, khalf = g.codes_off[1], sb = stage_bytes(g);
  long long u = x0 / a.nb;
  int blk = (int)(x0 - u * a.nb);
  int pb = (int)(u / g.H), ph = (int)(u - (long long)pb * g.H);  // (b, h) of block p
  if (g.dbg_stall) return;  // test switch: no copies, so every stage wait of the others runs out
  int issued = 0;
  for (int p = 0; p < n; ++p) {
    const int s = p % NBS;
    if (p >= NBS) {
      const bool got = helper_wait(&sm->empty[s], (uint32_t)(((p / NBS) - 1) & 1), a.status, g.wait_cycles);
      if (__any_sync(0xffffffffu, !got)) break;
    }
    const int set = 2 * (p & 15), part = lane - set;  // lanes set, set+1 copy this block
    if (lane == set) mbar_arrive_expect_tx(&sm->rec_full[s], rec);
    __syncwarp();
    if (part >= 0 && part < 2) {
      fence_proxy_async();
      const uint32_t off = part == 0 ? 0u : khalf;
      const uint32_t bytes = part == 0 ? khalf : rec - khalf;
      bulk_g2s(ring + (size_t)s * sb + off, a.base + record_offset(g, pb, ph, blk, a.status) + off, bytes,
               &sm->rec_full[s]);
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
// The value-outlier warps add p_t * v for the value outliers, with the tags written here.
template <int NBS, bool CSC>
__device__ void aux_warps(const Args& a, Smem* sm, uint8_t* ring, uint8_t* rows, int rows_stride, long long x0,
                          int n, int ax) {
  const Geo& g = a.g;
  const uint32_t sb = stage_bytes(g);
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
  const float2* rope_blk = reinterpret_cast<const float2*>(a.base + g.rope_off);
  // (cos, sin) of the block's start angle for pair j, from the RoPE table (L2-resident), loaded one
  // block of the group ahead so that its latency is hidden
  float2 cs_next = grp < n ? __ldg(rope_blk + (size_t)blk * 64 + j) : make_float2(1.0f, 0.0f);
  float* qb = sm->qb[grp];
  float* kterm = reinterpret_cast<float*>(rows + (size_t)NBS * rows_stride) + grp * tag_bytes;  // per group
  const int tA = j, tB = j + 64;
  for (int p = grp; p < n; p += 2) {
    if (u != cur_u) {
      cur_u = u;
      qv = load_q_pair(a, u, j);
    }
    const int s = p % NBS;
    const float2 cs = cs_next;
    {
      int nb2 = blk + 2;
      while (nb2 >= a.nb) nb2 -= a.nb;
      if (p + 2 < n) cs_next = __ldg(rope_blk + (size_t)nb2 * 64 + j);
    }
    const bool got = helper_wait(&sm->rec_full[s], (uint32_t)((p / NBS) & 1), a.status, g.wait_cycles);
    if (bar_or_group(grp, !got)) break;  // the consumers time out on their own waits
    const uint8_t* st = ring + (size_t)s * sb;
    Ops& op = sm->op[s];
    {
      const float qb0 = cs.x * qv.x + cs.y * qv.y, qb1 = -cs.y * qv.x + cs.x * qv.y;
      const uint16_t* km = reinterpret_cast<const uint16_t*>(st + g.meta_off[0]);
      const int kg = j >> 2, tqp = j & 3;
      const float s0 = h2f(km[2 * j]), s1 = h2f(km[2 * j + 1]);
      const float z0 = h2f(km[T + 2 * j]), z1 = h2f(km[T + 2 * j + 1]);
      const uint32_t bx = pack_h2(qb0 * s0, qb1 * s1);   // X column of pair j
      const uint32_t by = pack_h2(qb1 * s0, -qb0 * s1);  // Y column
      const float zx = qb0 * z0 + qb1 * z1, zy = qb1 * z0 - qb0 * z1;
      const __half zxh = __float2half_rn(zx), zyh = __float2half_rn(zy);
      *reinterpret_cast<uint2*>(&op.b[2 * tqp][2 * kg]) = make_uint2(bx, pack_h2(zx, zx - __half2float(zxh)));
      *reinterpret_cast<uint2*>(&op.b[2 * tqp + 1][2 * kg]) = make_uint2(by, pack_h2(zy, zy - __half2float(zyh)));
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
      }
      bar_group(grp);  // q_b and the key tags visible
      const uint16_t* val = reinterpret_cast<const uint16_t*>(csr);
      const uint8_t* col = csr + 2 * n_out + 2 * (T + 1);
      const int n_k = min((int)rp[T], n_out);
      auto key_term = [&](int e) {  // score term of key-outlier entry e < n_k
        const int c = col[e] & (D - 1), t = ktag[e] & (T - 1);
        // (cos, sin) of t * theta_pi from the coarse and fine tables (t = 16a + b)
        const float2 ca = sm->rope_a[t >> 4][c >> 1], cb = sm->rope_b[t & 15][c >> 1];
        const float cr = ca.x * cb.x - ca.y * cb.y, sr = ca.y * cb.x + ca.x * cb.y;
        const float qa = qb[c & ~1], qc = qb[c | 1];
        const float qq = (c & 1) ? (-sr * qa + cr * qc) : (cr * qa + sr * qc);
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

// ---- shared-memory accesses of the consumer warps, through 32-bit shared-window addresses (the
// stage, operand and outlier areas are all addressed from a few per-lane base registers)
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) { asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v)); }
// the same loads at a compile-time offset from a base register ([base + OFF] addressing)
template <int OFF>
__device__ __forceinline__ uint32_t lds_u16_at(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ float lds_f32_at(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 lds_v2_at(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint4 lds_v4_at(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a), "n"(OFF));
  return v;
}
template <int U>
__device__ __forceinline__ uint4 lds_v4_u(uint32_t a) { return lds_v4_at<16 * U>(a); }

constexpr uint32_t OPS_B = 0, OPS_ROW = 36 * 4, OPS_SK = 9 * 36 * 4;  // byte offsets in Ops
static_assert(sizeof(Ops) == OPS_SK + T * 4, "Ops layout");

// Scores of a consumer warp's 16 tokens in one block (after the reduction over the 4 lanes of a
// token and the key-outlier terms): s0 for token 16w + gq, s1 for token 16w + gq + 8.
// The m16n8k16 per k-group: A = the codebook values of 16 tokens x the group's 8 channels (k 0..7)
// and ones (k 8..15); B = the code rows and, at k 8 + 2(n/2) and 9 + 2(n/2), the zero-point term
// (high, low) of column n. ka: the lane's 24 code bytes; ba: its B row; ska: sk[t0].
__device__ __forceinline__ void block_scores(uint32_t ka, uint32_t ba, uint32_t ska, uint32_t ones,
                                             uint32_t tl0, uint32_t tl1, uint32_t th0, uint32_t th1,
                                             const float2 (&w)[2][16], float& s0, float& s1) {
  const uint2 k0 = lds_v2_at<0>(ka), k1 = lds_v2_at<8>(ka), k2 = lds_v2_at<16>(ka);
  const uint32_t cw[6] = {k0.x, k0.y, k1.x, k1.y, k2.x, k2.y};
  const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float2 acc[2][2] = {{{0.0f, 0.0f}, {0.0f, 0.0f}}, {{0.0f, 0.0f}, {0.0f, 0.0f}}};
#pragma unroll
  for (int uu = 0; uu < 8; ++uu) {
    const uint4 bq = uu == 0 ? lds_v4_u<0>(ba) : uu == 1 ? lds_v4_u<1>(ba) : uu == 2 ? lds_v4_u<2>(ba)
                   : uu == 3 ? lds_v4_u<3>(ba) : uu == 4 ? lds_v4_u<4>(ba) : uu == 5 ? lds_v4_u<5>(ba)
                   : uu == 6 ? lds_v4_u<6>(ba) : lds_v4_u<7>(ba);  // (b0, b1) of k-groups 2uu and 2uu + 1
    const uint32_t nw = nibble_word(cw, uu);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int kg = 2 * uu + hf;
      uint32_t a0, a1;
      lookup4(hf ? (nw >> 16) : nw, tl0, tl1, th0, th1, a0, a1);
      float d[4];
      mma16816(d, a0, a1, ones, ones, hf ? bq.z : bq.x, hf ? bq.w : bq.y, zero4);  // X, Y of pair 4kg+tq
      acc[0][hf] = __ffma2_rn(w[0][kg], make_float2(d[0], d[1]), acc[0][hf]);
      acc[1][hf] = __ffma2_rn(w[1][kg], make_float2(d[2], d[3]), acc[1][hf]);
    }
  }
  s0 = (acc[0][0].x + acc[0][1].x) + (acc[0][0].y + acc[0][1].y);
  s1 = (acc[1][0].x + acc[1][1].x) + (acc[1][0].y + acc[1][1].y);
  s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
  s0 += __shfl_xor_sync(0xffffffffu, s0, 2) + lds_f32_at<0>(ska);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 2) + lds_f32_at<32>(ska);
}

// Value product of one block for a consumer warp: p' = p * s_token as high/low B columns, the
// zero-point sum and 8 m16n8k16 over the V codes. va: the lane's 24 code bytes; vma: s_t0 of the
// value metadata (s_t1 = +16, zp_t0 = +256, zp_t1 = +272).
__device__ __forceinline__ void block_values(uint32_t va, uint32_t vma, int src_a, uint32_t xsel, uint32_t ysel,
                                             float p0, float p1, uint32_t tl0, uint32_t tl1, uint32_t th0,
                                             uint32_t th1, float& z_w, float (&acc)[8][4]) {
  uint32_t vb0, vb1;
  {
    const float pp0 = p0 * h2f((uint16_t)lds_u16_at<0>(vma)), pp1 = p1 * h2f((uint16_t)lds_u16_at<16>(vma));
    z_w = fmaf(p0, h2f((uint16_t)lds_u16_at<256>(vma)), fmaf(p1, h2f((uint16_t)lds_u16_at<272>(vma)), z_w));
    const __half h0 = __float2half_rn(pp0), h1 = __float2half_rn(pp1);
    const uint32_t hi = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
    const uint32_t lo = pack_h2(pp0 - __half2float(h0), pp1 - __half2float(h1));
    const uint32_t x = (hi & xsel) | (lo & ysel);
    vb0 = __shfl_sync(0xffffffffu, x, src_a);
    vb1 = __shfl_sync(0xffffffffu, x, src_a + 16);
  }
  const uint2 v0 = lds_v2_at<0>(va), v1 = lds_v2_at<8>(va), v2 = lds_v2_at<16>(va);
  const uint32_t cw[6] = {v0.x, v0.y, v1.x, v1.y, v2.x, v2.y};
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const uint32_t nw = nibble_word(cw, mt);
    uint32_t a0, a1, a2, a3;
    lookup4(nw, tl0, tl1, th0, th1, a0, a1);
    lookup4(nw >> 16, tl0, tl1, th0, th1, a2, a3);
    mma16816(acc[mt], a0, a1, a2, a3, vb0, vb1, acc[mt]);
  }
}

// CSR value tiles: the span [e0, e1) of the entries of consumer warp `warp`'s tokens (16w..16w+15)
// in one block, from the tile's row pointers.
__device__ __forceinline__ void value_outlier_span(uint32_t sa, const Geo& g, int warp, int& e0, int& e1) {
  const int n_out = g.n_out;
  const uint32_t rp = sa + g.csr_off[1] + 2 * n_out;
  e0 = min((int)lds_u16(rp + 32 * warp), n_out);
  e1 = min((int)lds_u16(rp + 32 * warp + 32), n_out);
}

// Entry k of [e0, e1) of a block's value outliers (k >= e1: none) for value-outlier warp `half`
// (consumer warps 4 half .. 4 half + 3, tokens 64 half .. 64 half + 63): the offset of its outv /
// owner-table slot (consumer warp t / 16 of its token t, its channel; a lane without an entry gets
// a scratch slot of its own, `scratch`) and x = p_t * v with p read from the probabilities the
// consumer warps published for the stage (pubs). rw: the stage's run index of each entry, written
// by the aux warps (CSR: its token; CSC: its channel). CSR tiles give each warp a contiguous run of
// entries; a CSC tile is read whole, in its (channel, token) order, by both warps, each keeping
// the entries of its own tokens.
template <bool CSC>
__device__ __forceinline__ void value_outlier_entry(uint32_t sa, uint32_t rw, const Geo& g, int k, int e1, int half,
                                                    uint32_t pubs, uint32_t scratch, uint32_t& slot, float& x) {
  const int n_out = g.n_out;
  const int kk = k < e1 ? k : 0;
  const uint32_t csr = sa + g.csr_off[1], idx = csr + 2 * n_out + 2 * (T + 1);  // idx: CSR channel, CSC token
  int t, ch;
  if (CSC) {
    t = (int)lds_u8(idx + kk);
    ch = (int)lds_u8(rw + kk);
  } else {
    t = (int)lds_u8(rw + kk);
    ch = (int)lds_u8(idx + kk);
  }
  const float v = h2f((uint16_t)lds_u16(csr + 2 * kk));
  t &= T - 1;
  const bool valid = k < e1 && (!CSC || (t >> 6) == half);
  slot = valid ? 4u * (uint32_t)((t >> 4) * (D + 32) + (ch & (D - 1))) : scratch;
  x = lds_f32(pubs + 4 * (uint32_t)t) * v;  // (lanes without an entry of their own add into scratch)
}

// The first token a consumer lane's probabilities belong to: 16w + gq (and that + 8).
__device__ __forceinline__ int t0_of(int warp, int lane) { return 16 * warp + (lane >> 2); }

// Value-outlier warps (NVOUT of them): for every block of the range, once the consumer warps have
// published its probabilities, they add the block's value outliers (x = p_t * v per entry) to the
// outv of the consumer warp that owns each token, in the consumers' place. Warp VOUT_WARP + i takes
// the entries of consumer warps 4i..4i+3 (tokens 64i..64i+63: a contiguous run of a CSR tile; a
// CSC tile is read whole, keeping those tokens), 32 entries per batch, blocks in order. In a batch the lanes post their ids to the owner table at their (consumer warp,
// channel) slot (a shared-memory atomic minimum) and read it back: the lowest lane of each slot
// adds its entry with no branch (a lane without an entry updates a scratch slot of its own) and
// resets the slot; the others (a slot hit twice or more) follow one after another in lane order.
// Within a slot the lanes' entries are in token order (CSR: (token, channel) order; CSC: (channel,
// token) order), so every channel's sum is the same sequence of fp32 additions, in token order, for
// both value-outlier layouts and whatever the thread timing.
// A consumer warp's reference move at block j reaches its outv first (scaled by the published
// factor), so outv stays relative to the consumer's current reference. A consumer reads its outv
// at the end of a segment after vdone of the segment's last block. These warps hold each stage
// until they are done with it (arrivals on empty).
template <int NBS, bool CSC>
__device__ void vout_warps(const Args& a, Smem* sm, uint8_t* ring, uint8_t* rows, int rows_stride, int n, int wi,
                           int lane) {
  const Geo& g = a.g;
  const int n_out = g.n_out;
  const uint32_t sb = stage_bytes(g);
  const uint32_t ring_sa = smem_u32(ring), rows_sa = smem_u32(rows);
  const uint32_t vtag_ofs = (uint32_t)round16((uint64_t)n_out);
  const uint32_t outv0 = smem_u32(&sm->outv[0][0]), own0 = smem_u32(&sm->own[0][0]);
  constexpr int WPV = NW / NVOUT;  // consumer warps per value-outlier warp
  // a slot of this lane's own past the channels of its first consumer warp (lanes without an entry)
  const uint32_t scratch = 4u * (uint32_t)(WPV * wi * (D + 32) + D + lane);
  for (int i = 0; i < n; ++i) {
    const int s = i % NBS;
    const bool got = helper_wait(&sm->p_full[s], (uint32_t)((i / NBS) & 1), a.status, g.wait_cycles);
    if (__any_sync(0xffffffffu, !got)) return;  // the consumers time out on their own waits
    const uint32_t sa = ring_sa + (uint32_t)s * sb;
    const uint32_t rw = rows_sa + (uint32_t)s * (uint32_t)rows_stride + vtag_ofs;
    const uint32_t pubs = smem_u32(&sm->pub[s][0]);
#pragma unroll
    for (int k = 0; k < WPV; ++k) {  // reference moves first
      const int w = WPV * wi + k;
      const float al = sm->alw[s][w];
      if (al != 1.0f) {  // warp-uniform
        const uint32_t outv = outv0 + 4u * (uint32_t)(w * (D + 32));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t o = outv + 4 * (lane + 32 * q);
          sts_f32(o, lds_f32(o) * al);
        }
      }
    }
    __syncwarp();
    int e0, e1;
    if (CSC) {  // the whole tile, in column order
      e0 = 0;
      e1 = min((int)lds_u16(sa + g.csr_off[1] + 2 * n_out + 2 * T), n_out);
    } else {    // the run of consumer warps WPV wi .. WPV wi + WPV - 1
      int d0, d1;
      value_outlier_span(sa, g, WPV * wi, e0, d0);
      value_outlier_span(sa, g, WPV * wi + WPV - 1, d1, e1);
    }
    for (int kb = e0; kb < e1; kb += 32) {  // batches of 32, each finished before the next
      uint32_t slot;
      float x;
      value_outlier_entry<CSC>(sa, rw, g, kb + lane, e1, wi, pubs, scratch, slot, x);
      const uint32_t os = own0 + slot, vs = outv0 + slot;
      asm volatile("red.shared.min.s32 [%0], %1;" ::"r"(os), "r"(lane));
      __syncwarp();
      int o;
      asm volatile("ld.shared.s32 %0, [%1];" : "=r"(o) : "r"(os));
      const bool first = o == lane;  // always for a lane without an entry (its own slot)
      const uint32_t addr = first ? vs : outv0 + scratch;
      sts_f32(addr, lds_f32(addr) + x);
      __syncwarp();
      asm volatile("st.shared.s32 [%0], %1;" ::"r"(os), "r"(32));
      const uint32_t rest = __ballot_sync(0xffffffffu, !first);
      for (uint32_t m = rest; m; m &= m - 1) {  // a slot hit twice or more: in lane order
        __syncwarp();
        if (lane == __ffs(m) - 1) sts_f32(vs, lds_f32(vs) + x);
      }
      __syncwarp();
    }
    if (lane == 0) {
      mbar_arrive(&sm->vdone[s]);
      mbar_arrive(&sm->empty[s]);
    }
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
  // (cos, sin) of the lane's (token, pair) cells: tokens 16w + gq + 8r, pairs 4kg + tq, from the
  // cache's in-block angle table (L2-resident)
  const float2* rope_loc = reinterpret_cast<const float2*>(a.base + g.rope_off) + (size_t)(g.max_blocks + 1) * 64;
  float2 wcs[2][16];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int kg = 0; kg < 16; ++kg) wcs[r][kg] = __ldg(rope_loc + (16 * warp + gq + 8 * r) * 64 + 4 * kg + tq);
  const int brow = (gq >> 1) == tq ? gq : 8;             // lanes holding a part of the score B operand
  const uint32_t ones = 0x3c003c00u;                     // A columns 8..15 = 1.0 (fp16)
  const int src_a = 4 * tq + (gq < 2 ? gq : 2);          // value B: (high, low, zero) source lanes
  const uint32_t xsel = tq == 0 ? 0xffffffffu : 0u;      // this lane sends p' high (tq 0) ...
  const uint32_t ysel = tq == 1 ? 0xffffffffu : 0u;      // ... or low (tq 1) or zero
  const int t0 = 16 * warp + gq;
  // shared-window addresses: stage bases and the lane's fixed offsets in a stage / operand block
  const uint32_t ring_sa = smem_u32(ring), ops_sa = smem_u32(&sm->op[0]);
  const uint32_t rows_sa = smem_u32(rows);
  const uint32_t outv = smem_u32(&sm->outv[warp][0]);
  const uint32_t pub0 = smem_u32(&sm->pub[0][t0_of(warp, lane)]), alw0 = smem_u32(&sm->alw[0][warp]);
  float alf = 1.0f;  // the factor the warp's reference moved by in this block
  const uint32_t vtag_ofs = (uint32_t)round16((uint64_t)g.n_out);
  const uint32_t kofs = g.codes_off[0] + warp * 768 + lane * 24, vofs = g.codes_off[1] + warp * 768 + lane * 24;
  const uint32_t vmofs = g.meta_off[1] + 2 * t0;
  const uint32_t bofs = OPS_B + brow * OPS_ROW, skofs = OPS_SK + 4 * t0;
  auto stage_sa = [&](int i) { return ring_sa + (uint32_t)(i % NBS) * sb; };
  auto ops_of = [&](int i) { return ops_sa + (uint32_t)(i % NBS) * (uint32_t)sizeof(Ops); };

  auto ready_now = [&](int i) -> bool {  // the stage of range block i is ready (no waiting)
    const int s = i % NBS;
    const uint32_t par = (uint32_t)((i / NBS) & 1);
    return mbar_test_wait(&sm->ops_full[s], par) & mbar_test_wait(&sm->rec_full[s], par);
  };
  const bool vout = g.n_out > 0;
  auto wait_stage = [&](int i) -> bool {  // false when a wait gave up
    const int s = i % NBS;
    const uint32_t par = (uint32_t)((i / NBS) & 1);
    const bool got = mbar_wait_bounded(&sm->ops_full[s], par, a.status, g.wait_cycles) &&
                     mbar_wait_bounded(&sm->rec_full[s], par, a.status, g.wait_cycles);
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
    for (int k = 0; k < 4; ++k) sts_f32(outv + 4 * (lane + 32 * k), 0.0f);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
    float m_w = -INFINITY, l_w = 0.0f, z_w = 0.0f;
    __syncwarp();
    if (!wait_stage(i)) return;
    bool ahead = i + 1 < iend ? ready_now(i + 1) : true;
    // software pipeline: the scores of block j + 1 are issued first (they do not depend on the
    // softmax), then block j's softmax and value product, whose dependency chain the score work
    // covers; block j + 1's scores are only needed in the next iteration
    float sv0, sv1;
    block_scores(stage_sa(i) + kofs, ops_of(i) + bofs, ops_of(i) + skofs, ones, tl0, tl1, th0, th1, wcs, sv0, sv1);
    for (int j = i; j < iend; ++j) {
      const int s = j % NBS;
      const uint32_t sa = stage_sa(j);
      const bool more = j + 1 < iend;  // warp-uniform
      // stage j + 1 was probed during the previous block (no waiting); only when that probe
      // failed does the warp wait for it here
      if (!__all_sync(0xffffffffu, ahead)) {
        if (more && !wait_stage(j + 1)) return;
      }
      float nv0 = 0.0f, nv1 = 0.0f;
      if (more) {
        const uint32_t sa1 = stage_sa(j + 1), op1 = ops_of(j + 1);
        block_scores(sa1 + kofs, op1 + bofs, op1 + skofs, ones, tl0, tl1, th0, th1, wcs, nv0, nv1);
      }
      // probe stage j + 2 (its latency overlaps the work below)
      ahead = j + 2 < iend ? ready_now(j + 2) : true;
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
        const float al = fast_exp2(m_w - mloc);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          acc[mt][0] *= al; acc[mt][1] *= al; acc[mt][2] *= al; acc[mt][3] *= al;
        }
        l_w *= al;
        z_w *= al;
        alf = al;
        m_w = mloc;
      }
      const float p0 = fast_exp2(sv0 - m_w), p1 = fast_exp2(sv1 - m_w);
      l_w += p0 + p1;
      if (vout) {  // publish the block's probabilities and reference move for the value-outlier warps
        if (tq == 0) {
          sts_f32(pub0 + (uint32_t)s * (T * 4), p0);
          sts_f32(pub0 + (uint32_t)s * (T * 4) + 32, p1);
        }
        if (lane == 0) sts_f32(alw0 + (uint32_t)s * (NW * 4), alf);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->p_full[s]);
        alf = 1.0f;
      }
      block_values(sa + vofs, sa + vmofs, src_a, xsel, ysel, p0, p1, tl0, tl1, th0, th1, z_w, acc);
      release(s);
      sv0 = nv0;
      sv1 = nv1;
    }
    // the segment's partial row (its value outliers are in outv once vdone of its last block passed)
    if (vout) {
      const int jl = iend - 1;
      const bool got = mbar_wait_bounded(&sm->vdone[jl % NBS], (uint32_t)((jl / NBS) & 1), a.status, g.wait_cycles);
      if (__any_sync(0xffffffffu, !got)) return;
    }
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
        const uint64_t row = ((uint64_t)(b * g.Hq + h)) * a.rows_ph + (uint64_t)slot * NW + warp;
        if (tq == 0) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int c0 = 16 * mt + gq, c1 = c0 + 8;
            a.ws_o[row * D + c0] = acc[mt][0] + acc[mt][1] + zt + lds_f32(outv + 4 * c0);
            a.ws_o[row * D + c1] = acc[mt][2] + acc[mt][3] + zt + lds_f32(outv + 4 * c1);
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

// The idle warps (IDLE of them per CTA): attention over the fp tail, the n_tail < 128 tokens past the
// cached blocks (positions n0 + t, n0 = nb * 128), one warp per (b, query head), written as the
// last partial row (m, l, o) of that head for the combine to merge with the cached part. The keys
// are stored before RoPE like the cache's: the score is (R(n0)^T q) . (R(t) k_t), the in-block
// angles from the cache's table. Lane l holds channel pairs l and l + 32. It reads only the call's
// inputs and the angle tables, so it runs beside the ring without waiting on it.
constexpr int IDLE = 1;  // warps per CTA that attend the tail
constexpr int TCH = 6;  // tail tokens per chunk (the idle warps run with 88 registers)
__device__ void tail_warp(const Args& a, int wi, int lane) {
  const Geo& g = a.g;
  const int nt = a.n_tail;
  if (nt <= 0) return;
  const int n_heads = g.B * g.Hq;
  const float2* rope_blk = reinterpret_cast<const float2*>(a.base + g.rope_off);
  const float2* rope_loc = rope_blk + (size_t)(g.max_blocks + 1) * 64;
  for (int hidx = (int)blockIdx.x * IDLE + wi; hidx < n_heads; hidx += a.n_ranges * IDLE) {
    const int b = hidx / g.Hq, h = hidx - b * g.Hq;  // one query head per KV head
    const uint16_t* qp = a.q + (uint64_t)hidx * D;
    float q0[2][2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int pr = lane + 32 * k;
      const float x0 = load_in(qp + 2 * pr, g.in_bf16), x1 = load_in(qp + 2 * pr + 1, g.in_bf16);
      const float2 cs = __ldg(rope_blk + (size_t)a.nb * 64 + pr);
      q0[k][0] = cs.x * x0 + cs.y * x1;
      q0[k][1] = -cs.y * x0 + cs.x * x1;
    }
    const uint16_t* tk = a.tail_k + ((uint64_t)b * g.H + h) * a.tail_bh;
    const uint16_t* tv = a.tail_v + ((uint64_t)b * g.H + h) * a.tail_bh;
    float m = -INFINITY, l = 0.0f, o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    // TCH tokens at a time, every load of a chunk issued before any is used (tokens past the
    // tail read the last one again and get probability 0)
    for (int t0 = 0; t0 < nt; t0 += TCH) {
      uint32_t kw[TCH][2];
      float2 cs[TCH][2];
#pragma unroll
      for (int i = 0; i < TCH; ++i) {
        const int t = min(t0 + i, nt - 1);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int pr = lane + 32 * k;
          kw[i][k] = __ldg(reinterpret_cast<const unsigned int*>(tk + (uint64_t)t * a.tail_tok + 2 * pr));
          cs[i][k] = __ldg(rope_loc + (size_t)t * 64 + pr);
        }
      }
      float sc[TCH];
#pragma unroll
      for (int i = 0; i < TCH; ++i) {
        float acc = 0.0f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float k0 = in_bits_to_f32((uint16_t)(kw[i][k] & 0xffffu), g.in_bf16);
          const float k1 = in_bits_to_f32((uint16_t)(kw[i][k] >> 16), g.in_bf16);
          acc = fmaf(q0[k][0], cs[i][k].x * k0 - cs[i][k].y * k1, fmaf(q0[k][1], cs[i][k].y * k0 + cs[i][k].x * k1, acc));
        }
        sc[i] = acc;
      }
      uint32_t vw[TCH][2];
#pragma unroll
      for (int i = 0; i < TCH; ++i) {
        const int t = min(t0 + i, nt - 1);
#pragma unroll
        for (int k = 0; k < 2; ++k)
          vw[i][k] = __ldg(reinterpret_cast<const unsigned int*>(tv + (uint64_t)t * a.tail_tok + 2 * (lane + 32 * k)));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int i = 0; i < TCH; ++i) sc[i] += __shfl_xor_sync(0xffffffffu, sc[i], off);
      float cm = -INFINITY;
#pragma unroll
      for (int i = 0; i < TCH; ++i) {  // the same values in every lane
        sc[i] = t0 + i < nt ? sc[i] * LOG2E_RSQRT_D : -INFINITY;
        cm = fmaxf(cm, sc[i]);
      }
      if (cm > m) {
        const float al = exp2f(m - cm);
        l *= al;
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] *= al;
        m = cm;
      }
#pragma unroll
      for (int i = 0; i < TCH; ++i) {
        const float pt = exp2f(sc[i] - m);
        l += pt;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          o[2 * k] = fmaf(pt, in_bits_to_f32((uint16_t)(vw[i][k] & 0xffffu), g.in_bf16), o[2 * k]);
          o[2 * k + 1] = fmaf(pt, in_bits_to_f32((uint16_t)(vw[i][k] >> 16), g.in_bf16), o[2 * k + 1]);
        }
      }
    }
    const uint64_t row = (uint64_t)hidx * a.rows_ph + (uint64_t)(a.rows_ph - 1);
#pragma unroll
    for (int k = 0; k < 2; ++k)
      *reinterpret_cast<float2*>(a.ws_o + row * D + 2 * (lane + 32 * k)) = make_float2(o[2 * k], o[2 * k + 1]);
    if (lane == 0) {
      a.ws_m[row] = m;
      a.ws_l[row] = l;
    }
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
  const int rows_stride = rows_stride_of(a.g.n_out);
  const long long R = blockIdx.x;
  if (R >= a.n_ranges) return;
  const long long x0 = R * a.total / a.n_ranges, x1 = (R + 1) * a.total / a.n_ranges;
  const int n = (int)(x1 - x0);
  if (n <= 0) return;
  {  // the in-block angle tables of the key outliers: t * theta_i = 16a * theta_i + b * theta_i
    const float2* loc = reinterpret_cast<const float2*>(a.base + a.g.rope_off) + (size_t)(a.g.max_blocks + 1) * 64;
    for (int e = tid; e < 8 * 64; e += NTHREADS) sm->rope_a[e >> 6][e & 63] = __ldg(loc + (size_t)(16 * (e >> 6)) * 64 + (e & 63));
    for (int e = tid; e < 16 * 64; e += NTHREADS) sm->rope_b[e >> 6][e & 63] = __ldg(loc + e);
  }
  for (int e = tid; e < NBS * 36; e += NTHREADS) sm->op[e / 36].b[8][e % 36] = 0u;
  for (int e = tid; e < NW * (D + 32); e += NTHREADS) (&sm->own[0][0])[e] = 32;
  if (tid == 0) {
    for (int s = 0; s < NBS; ++s) {
      mbar_init(&sm->rec_full[s], 1);
      mbar_init(&sm->ops_full[s], AUX_GROUP);
      mbar_init(&sm->empty[s], NW + (a.g.n_out > 0 ? NVOUT : 0));
      mbar_init(&sm->p_full[s], NW);
      mbar_init(&sm->vdone[s], NVOUT);
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
    else if (warp == TAIL_WARP) tail_warp(a, 0, lane);
    else if (a.g.n_out > 0) vout_warps<NBS, CSC>(a, sm, ring, rows, rows_stride, n, warp - VOUT_WARP, lane);
  }
}

size_t smem_bytes(const Geo& g) {
  return (size_t)NB * (size_t)g.rec_bytes + sizeof(Smem) + (size_t)NB * rows_stride_of(g.n_out) +
         2 * sizeof(float) * round16((uint64_t)g.n_out);
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

// slots: range slots per (b, query head); the workspace holds, per (b, query head), slots * NW
// partial rows of the cached blocks and then one row for the fp tail (rows_ph in all).
cudaError_t kvq_launch_decode_nuq(const kvq::Geo& g, const uint8_t* base, const float* codebook, const uint16_t* q,
                                  int n_blocks, long long ranges, long long slots, long long rows_ph, float* ws_m,
                                  float* ws_l, float* ws_o, int* status, const uint16_t* tail_k,
                                  const uint16_t* tail_v, int n_tail, long long tail_bh, long long tail_tok,
                                  cudaStream_t st) {
  using namespace kvq::nuqdec;
  const size_t smem = smem_bytes(g);
  auto fn = g.v_csc ? decode_nuq_kernel<NB, true> : decode_nuq_kernel<NB, false>;
  cudaError_t e = kvq::ensure_smem_attr((const void*)fn, smem);
  if (e != cudaSuccess) return e;
  Args a;
  a.g = g; a.base = base; a.codebook = codebook; a.q = q; a.nb = n_blocks;
  a.total = (long long)g.B * g.H * n_blocks; a.n_ranges = (int)ranges; a.n_slots = (int)slots;
  a.ws_m = ws_m; a.ws_l = ws_l; a.ws_o = ws_o; a.status = status;
  a.rows_ph = (int)rows_ph;
  a.tail_k = tail_k; a.tail_v = tail_v; a.n_tail = n_tail; a.tail_bh = tail_bh; a.tail_tok = tail_tok;
  fn<<<(int)ranges, NTHREADS, smem, st>>>(a);
  return cudaGetLastError();
}
