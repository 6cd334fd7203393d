/*
 * kvq.h - C ABI of libkvq: low-bit KV-cache quantization in 128-token blocks and
 * decode attention that reads the packed cache directly (sm_103a, one GPU).
 *
 * Sources (cited by page and section):
 *   [KVQ] "KVQuant: Towards 10 Million Context Length LLM Inference with KV Cache
 *         Quantization" reading notes (zhongzhuzhou.org).
 *   [KVN] "KVarN: Variance-Normalized KV-Cache Quantization Mitigates Error Accumulation
 *         in Reasoning Tasks" summary (paper.rainbus.top).
 *   [TQ]  TurboQuant KV-cache reproduction blog (pwwt.cn).
 *
 * Conventions shared by every call
 *   - All tensors live in device memory owned by the caller; the library allocates
 *     nothing (no cudaMalloc, no host buffers beyond its arguments).
 *   - Calls are asynchronous on the given stream. The returned kvq_status covers argument
 *     checks and launch errors only. Errors found on the device (a bounded wait that gave
 *     up, an index out of range) are written to the caller's device status word
 *     (kvq_cache.dev_status, first error wins); read it after a synchronize.
 *   - Pointers passed to the library must be 16-byte aligned; the cache base must be
 *     128-byte aligned. Violations return KVQ_ERR_ALIGNMENT and launch nothing.
 *   - head_dim and block are both 128. A "tile" is one (batch b, KV head h, block) slab
 *     of 128 tokens x 128 channels of K or of V.
 *   - K, V, q and tail inputs are in cfg.in_dtype (fp16 or bf16), contiguous, layout
 *     given per call. Outputs are fp32.
 *   - Nothing here falls back to the CPU: without a usable CUDA device every call that
 *     launches work returns KVQ_ERR_CUDA.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_FORMAT_VERSION 2u
#define KVQ_BLOCK 128
#define KVQ_HEAD_DIM 128
#define KVQ_MAX_GROUP 16      /* n_q_heads / n_kv_heads supported by decode */

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,   /* a NULL pointer, a size out of range, an inconsistent config */
  KVQ_ERR_UNSUPPORTED = 2,   /* a valid but unimplemented combination (e.g. INT4 with bits 2) */
  KVQ_ERR_CAPACITY = 3,      /* an append past cfg.max_blocks, or a buffer smaller than needed */
  KVQ_ERR_ALIGNMENT = 4,     /* a pointer that breaks the alignment rules above */
  KVQ_ERR_CUDA = 5,          /* a CUDA runtime error (launch failure, no device) */
  KVQ_ERR_TIMEOUT = 6,       /* device side: a bounded wait gave up (written to dev_status) */
  KVQ_ERR_PAGE = 7           /* device side: a block-table entry outside [0, n_pages) was read
                                (written to dev_status; that block used page 0 instead) */
} kvq_status;

/* Quantization method of a cache (fixed for its lifetime). */
typedef enum {
  KVQ_RTN = 0,   /* KIVI-style asymmetric round-to-nearest: keys per channel over the 128 tokens
                    of a block, values per token over the 128 channels; x_dq = (q + z) * s
                    ([KVN] preliminaries; [KVQ] §1.2, §3.1). bits 2..4. */
  KVQ_NUQ = 1,   /* KVQuant: per-channel keys (optionally pre-RoPE) and per-token values normalised
                    to [-1, 1] by the non-outlier centre/half-range, nearest entry of a per-KV-head
                    2^bits codebook, and the ceil(outlier_frac * 16384) largest-|x| entries of each
                    tile kept in fp16 as CSR ([KVQ] §3.2-3.4, §3.8 Algorithm 1). bits 2..4. */
  KVQ_VARN = 2,  /* KVarN: FWHT-128 on channels, Sinkhorn-style variance normalisation, RTN
                    (keys per channel, values per token) and a second fp16 scale s1 (keys: per
                    token, values: per channel); x_dq = (q + z) * s * s1 ([KVN] method steps 1-5).
                    bits 2..4. */
  KVQ_INT4 = 3   /* TurboQuant-style symmetric absmax integers: one fp16 scale s = absmax/(2^(b-1)-1)
                    per block of scale_group contiguous channels of a token (128: the whole head
                    vector; 64: two blocks per token), q = clamp(rne(x/s), -2^(b-1), 2^(b-1)-1)
                    stored as b-bit two's complement ([TQ] §2.1, §4.2). bits 4 (int4 nibbles)
                    or 8 (the 8-bit precision [TQ] §5.1 keeps for sensitive layers). */
} kvq_method;

typedef enum { KVQ_F16 = 0, KVQ_BF16 = 1 } kvq_dtype;

/* Layout of the code words of a tile (see kvq_layout_t).
 *   KVQ_LAYOUT_ROWS: one row per token for keys and values, each row's 128 codes in
 *                    floor(32/b)-code words ([KVQ] §9.3 bit layout; 3-bit rows are 13 words).
 *   KVQ_LAYOUT_MMA : the tensor-core decode's format: 2- and 4-bit value tiles hold one row per
 *                    channel; 3-bit tiles are bit planes in matrix-fragment order, 48 bytes per
 *                    128 codes ([KVQ] §9.3 byte count). The tensor-core decodes need this layout;
 *                    with KVQ_LAYOUT_ROWS every decode runs on the CUDA cores (~12 instructions
 *                    per element, several times slower). KVQ_LAYOUT_ROWS stays the default (0)
 *                    because it is the pages' byte layout; a caller who wants decode speed creates
 *                    its caches with KVQ_LAYOUT_MMA. Of the nuq caches only 3-bit ones with
 *                    pre-RoPE keys and one query head per KV head have a tensor-core decode. */
typedef enum { KVQ_LAYOUT_ROWS = 0, KVQ_LAYOUT_MMA = 1 } kvq_code_layout;

/* Cache configuration. All fields are read by kvq_layout / kvq_cache_init. */
typedef struct {
  int32_t method;        /* kvq_method */
  int32_t bits;          /* code width: 2, 3 or 4 (INT4: 4 or 8) */
  int32_t batch;         /* B >= 1 */
  int32_t n_kv_heads;    /* H_kv >= 1 */
  int32_t n_q_heads;     /* H_q, a multiple of H_kv, H_q / H_kv <= KVQ_MAX_GROUP */
  int32_t head_dim;      /* must be 128 */
  int32_t block;         /* must be 128 */
  int32_t max_blocks;    /* capacity per (b, h) in blocks of 128 tokens, >= 1 */
  int32_t in_dtype;      /* kvq_dtype of K, V, q and the tail */
  int32_t pre_rope;      /* NUQ only: keys are stored before RoPE; decode rotates them at their
                            absolute position after dequantisation ([KVQ] §3.2). 0 otherwise. */
  double rope_theta;     /* RoPE base (10000): angle of channel pair i at position n is
                            n * theta^(-2i/128) ([KVQ] §1.3) */
  float outlier_frac;    /* NUQ: fraction of each tile kept as fp16 outliers (0.01); 0 disables */
  int32_t varn_iters;    /* VARN: variance-normalisation iterations (8); 0..64 */
  int32_t hadamard;      /* VARN: 1 applies the FWHT-128 (the decode transforms q and o too) */
  int32_t layout;        /* kvq_code_layout of the code words (0: KVQ_LAYOUT_ROWS) */
  int32_t n_pages;       /* 0: the records of (b, h) are contiguous, [B][H_kv][max_blocks].
                            > 0: paged cache. The record pool holds n_pages pages; a page holds
                            the records of all H_kv heads of one 128-token block, and a block
                            table (kvq_cache.block_table) maps block blk of sequence b to its
                            page (the paged KV cache the KVQuant and TurboQuant pages' serving
                            sections use, vLLM-style). */
  int32_t key_calib;     /* NUQ only. 0: key statistics per block (centre/half-range of each
                            channel, the tile's top outlier_frac entries as outliers). 1: offline
                            statistics per (KV head, channel) from kvq_calibrate_keys ([KVQ]
                            §3.6, Algorithm 1): entries with |k| > tau_c are outliers (at most
                            n_outliers per tile, the largest first), the rest normalised with the
                            calibrated centre and half-range. Values stay per token, online. */
  int32_t sink;          /* NUQ only. 1: the first token of every sequence is kept in the input
                            precision ([KVQ] §3.5 attention sink): block 0's tiles hold zeros in
                            its place and decode attends the kept K and V rows at position 0. */
  int32_t scale_group;   /* INT4 only: channels per absmax scale, 128 (also 0) or 64 ([TQ] §2.1:
                            a smaller block doubles the scale overhead). Other methods: 0 or 128.
                            Tiles with bits 8 or groups of 64 decode on the CUDA cores. */
  int32_t v_csc;         /* NUQ only. 0: value outliers in CSR like the keys (rows = tokens).
                            1: value outliers in CSC (columns = channels), the value storage of
                            [KVQ] §3.4 ("by column"). Same region size and outlier set; decode
                            results are bitwise those of the CSR cache. */
} kvq_config;

/* Byte layout of a cache, from kvq_layout. One record per (b, h, block), at
 *   base + ((b * n_kv_heads + h) * max_blocks + block) * record_bytes            (n_pages = 0)
 *   base + (block_table[b * max_blocks + block] * n_kv_heads + h) * record_bytes  (n_pages > 0),
 * holding the K tile then the V tile; every region starts 16-byte aligned:
 *   codes : KVQ_LAYOUT_ROWS: 128 rows x words_per_row uint32, one row per token (K and V);
 *           code i of a row at bits [b*(i%n)+b-1 : b*(i%n)] of word i/n, n = floor(32/b),
 *           unused high bits zero ([KVQ] §9.3 layout, generalised; 3-bit: 13 words per row).
 *           KVQ_LAYOUT_MMA, 2 and 4 bits: the same rows, but a V tile has one row per channel
 *           (its codes for the 128 tokens).
 *           KVQ_LAYOUT_MMA, 3 bits: 1536 uint32 (48 bytes per 128 codes, the count of [KVQ] §9.3),
 *           bit planes in matrix-fragment order. Segment s = t/16 (t = token in the block)
 *           holds 32 groups of 6 words (group base word s*192 + 6*grp); in a group, slot k
 *           (0..7) of nibble word u (0..7) keeps a code's two low bits in word u/2 at bit
 *           4k + 2(u%2) and its high bit in word 4 + u/4 at bit 4k + {2,3,0,1}[u%4].
 *           K tile, code (t, channel c): grp = 4(t%8) + (c/2)%4, u = c/16,
 *             k = 4((c/8)%2) + 2((t%16)/8) + c%2.
 *           V tile, code (t, c): grp = 4(c%8) + t%4, u = c/16,
 *             k = 4(((t%16)/4)%2) + 2((c/8)%2) + (t%16)/8.
 *           words_per_row is 12 for 3-bit KVQ_LAYOUT_MMA caches (the tile holds 128 x 12 words).
 *   meta  : fp16 vectors of 128. RTN and VARN: s, z (keys: per channel; values: per token),
 *           VARN adds s1 (keys: per token; values: per channel). NUQ: s (half-range),
 *           zp (centre). INT4: s (per token); with scale_group 64 two vectors, the scales
 *           of channels 0..63 of every token, then those of channels 64..127.
 *   csr   : NUQ only: val fp16[n_outliers], row_ptr uint16[129] (row = token),
 *           col uint8[n_outliers] (channel), zero padded; entries in (token, channel) order.
 *           A V tile of a v_csc cache holds the same arrays by column instead: val,
 *           col_ptr uint16[129] (column = channel), row uint8[n_outliers] (token), entries in
 *           (channel, token) order.
 * After the records, for pre-RoPE caches: a table of (cos, sin) fp32 pairs of
 * block*128*theta_i for block = 0..max_blocks, then of t*theta_i for t = 0..127 (64 pairs each),
 * written by kvq_cache_init. */
typedef struct {
  uint64_t record_bytes;
  uint64_t codes_off[2], codes_bytes[2];   /* [0] = K, [1] = V, offsets within a record */
  uint64_t meta_off[2], meta_bytes[2];
  uint64_t csr_off[2], csr_bytes[2];
  uint64_t records_bytes;                  /* B * H_kv * max_blocks * record_bytes */
  uint64_t rope_off, rope_bytes;           /* from base; rope_bytes = 0 without pre-RoPE keys */
  uint64_t total_bytes;                    /* bytes the caller must provide at base */
  int32_t words_per_row;
  int32_t n_outliers;                      /* NUQ: outliers per tile; 0 otherwise */
  uint32_t format_version;                 /* KVQ_FORMAT_VERSION */
  int32_t reserved;
  uint64_t calib_off, calib_bytes;         /* key_calib: float tau[H_kv][128], then fp16
                                              s[H_kv][128], then fp16 zp[H_kv][128]; else 0 */
  uint64_t sink_off, sink_bytes;           /* sink: per (b, h), the first token's K row then V
                                              row, 128 values each in cfg.in_dtype; else 0 */
} kvq_layout_t;

/* A cache handle: plain data owned by the caller. kvq_cache_init fills it. */
typedef struct {
  kvq_config cfg;
  kvq_layout_t lay;
  void* base;              /* device, lay.total_bytes, caller-owned */
  const float* codebook;   /* device fp32 [n_kv_heads][2^bits], NUQ only (else NULL), caller-owned */
  int32_t* dev_status;     /* device int32, caller-owned; 0 = no device-side error */
  int32_t n_blocks;        /* blocks appended so far, per (b, h) */
  int32_t device;          /* CUDA device ordinal the cache was initialised on */
  const int32_t* block_table; /* paged caches (cfg.n_pages > 0): device int32 [B][max_blocks],
                            caller-owned and caller-filled: entry (b, blk) is the page of block
                            blk of sequence b. kvq_cache_init sets it to NULL; set it before the
                            first append. Decode and dequant read the entries of blocks
                            [0, n_blocks), append those of the new blocks and writes their pages
                            (sequences may share a page for reading, e.g. a common prefix, but an
                            append must not write a page that another block uses). An entry
                            outside [0, n_pages) is reported as KVQ_ERR_PAGE in dev_status and
                            that block uses page 0 instead. NULL for contiguous caches.
                            4-byte aligned. */
  int32_t calibrated;      /* key_calib caches: set by kvq_calibrate_keys; append refuses until then */
} kvq_cache;

/* Human-readable name of a status code (static string). */
const char* kvq_status_str(kvq_status s);

/* Dense KV-cache size 2*n*h*d*e*b*l bytes ([KVQ] §1.1; [TQ] §1.1). Pure. */
uint64_t kvq_dense_kv_bytes(int64_t n_layers, int64_t n_heads, int64_t head_dim,
                            int64_t elem_bytes, int64_t batch, int64_t seq_len);

/* Checks cfg and computes its layout. Host only, pure; *out is written only on KVQ_OK. */
kvq_status kvq_layout(const kvq_config* cfg, kvq_layout_t* out);

/* Binds caller memory to a cache: checks cfg, the size (bytes >= lay.total_bytes) and the
 * alignment, records the pointers and sets n_blocks = 0. For pre-RoPE caches it launches one
 * kernel on `stream` that writes the RoPE tables (fp64 angles rounded to fp32). It also sets
 * *dev_status = 0 on `stream`. codebook: NUQ only, device fp32 [n_kv_heads][2^bits], read by
 * every append and decode (keep it alive and unchanged). No allocation. */
kvq_status kvq_cache_init(kvq_cache* cache, const kvq_config* cfg, void* dev_base, size_t bytes,
                          const float* dev_codebook, int32_t* dev_status, cudaStream_t stream);

/* Offline key calibration of a key_calib cache ([KVQ] §3.6 and Algorithm 1 offline steps 3-4,
 * the first token excluded as §3.5 asks). For every KV head h and channel c, over tokens
 * 1 .. n_tokens-1 of k_calib[h]:
 *   tau     = the ceil((1 - f) * (n_tokens - 1))-th smallest |k| (f = cfg.outlier_frac as fp32,
 *             computed in fp64; f = 0: tau = +inf, no outliers),
 *   zp, s   = centre and half-range of the entries with |k| <= tau (fp32, stored fp16).
 * k_calib : device [H_kv][n_tokens][128] in cfg.in_dtype (pre-RoPE keys for pre-RoPE caches),
 *           n_tokens >= 2, 16-byte aligned. Writes the cache's calibration table on `stream`
 * and sets cache->calibrated. KVQ_ERR_INVALID_ARG if the cache has no key_calib. */
kvq_status kvq_calibrate_keys(kvq_cache* cache, const void* k_calib, int32_t n_tokens, cudaStream_t stream);

/* Quantizes n_blocks new blocks of 128 tokens for every (b, h) and stores them at block
 * positions cache->n_blocks .. cache->n_blocks + n_blocks - 1; on success cache->n_blocks
 * grows by n_blocks ([KVQ] §3.8 Algorithm 1 inference steps 1-4; [KVN] method steps 1-4;
 * [TQ] §4.2 quantize_kv_block).
 *   k, v            : device [B][H_kv][n_blocks*128][128] in cfg.in_dtype (pre-RoPE keys for
 *                     pre-RoPE caches). Partial blocks are not accepted: fewer than 128 new
 *                     tokens stay in the caller's fp tail.
 *   dbg_varn_scales : VARN only, nullable: device fp32 [B][H_kv][n_blocks][2 (K, V)][2 (r, c)][128]
 *                     receives the unrounded VarN token scales r and channel scales c.
 * Returns KVQ_ERR_CAPACITY (nothing written) if cache->n_blocks + n_blocks > max_blocks. */
kvq_status kvq_append_block(kvq_cache* cache, const void* k, const void* v, int32_t n_blocks,
                            float* dbg_varn_scales, cudaStream_t stream);

/* Drops the newest blocks: sets cache->n_blocks = n_blocks (0 <= n_blocks <= current).
 * Host only; the dropped records are overwritten by later appends. */
kvq_status kvq_truncate(kvq_cache* cache, int32_t n_blocks);

/* kvq_truncate(cache, 0). */
kvq_status kvq_reset(kvq_cache* cache);

/* Test switch for the failure path of the bounded device waits (not part of the method; no
 * counterpart on the pages). With enable = 1, every later decode of this process that runs on the
 * 3-bit nuq tensor-core kernel launches it with its copy-issuing warp idle and its stage waits
 * bounded at ~2 million SM clocks (about 1 ms): the waits run out, the kernel records
 * KVQ_ERR_TIMEOUT in dev_status, every thread returns, and out is written as NaN. Nothing faults
 * and the context stays usable. enable = 0 restores normal decodes; the caller clears dev_status.
 * Other decode kernels ignore the switch. Returns KVQ_ERR_INVALID_ARG for other values. */
kvq_status kvq_debug_stall_decode(int32_t enable);

/* Number of sequence splits the decode uses for n_blocks cached blocks (a pure function of
 * the config and n_blocks). */
int32_t kvq_decode_splits(const kvq_config* cfg, int32_t n_blocks);

/* Device workspace kvq_decode_attn needs for n_blocks cached blocks, in bytes. Pure. */
kvq_status kvq_decode_workspace_bytes(const kvq_config* cfg, int32_t n_blocks, size_t* out);

/* Packed-cache bytes one decode step reads for n_blocks blocks per (b, h): code words plus
 * metadata plus CSR records, K and V (the algorithmic byte count of the decode). Pure. */
uint64_t kvq_decode_bytes(const kvq_config* cfg, int32_t n_blocks);

/* Decode attention of one new query per head over the packed cache plus an fp tail
 * ([KVQ] §3.7 fused matvec kernels and Algorithm 1 dequantisation; [TQ] §5.2 fused dequant
 * inside attention): out = softmax(q . k_n / sqrt(128)) weighted sum of v_n over the n_blocks*128
 * cached tokens then the n_tail tail tokens, where k_n and v_n are dequantised in registers
 * (never written to memory), pre-RoPE keys are rotated at their absolute position n, and KVarN
 * caches are read in the Hadamard domain (q is transformed, the output transformed back).
 * Query head j attends with KV head j / (H_q / H_kv).
 *   q        : device [B][H_q][128] in cfg.in_dtype (already position-encoded for pre-RoPE caches)
 *   tail_k/v : device [B][H_kv][n_tail][128] in cfg.in_dtype, tokens at positions
 *              n_blocks*128 + j (pre-RoPE keys are rotated there); NULL when n_tail == 0
 *   n_tail   : 0..127
 *   out      : device fp32 [B][H_q][128]
 *   workspace: device scratch of at least kvq_decode_workspace_bytes(cfg, n_blocks) bytes
 * At least one token must be attended (n_blocks > 0 or n_tail > 0). Every device-side wait is
 * bounded (about one second); a decode whose wait gives up records KVQ_ERR_TIMEOUT in
 * dev_status and writes NaN to out. */
kvq_status kvq_decode_attn(const kvq_cache* cache, const void* q, const void* tail_k,
                           const void* tail_v, int32_t n_tail, float* out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/* kvq_decode_attn over tail buffers laid out by two strides (in elements): channel c of tail
 * token t of (b, h) is at ((b * H_kv + h) * tail_bh_stride + t * tail_token_stride + c). A caller
 * that keeps its tail in a buffer of fixed capacity, [B][H_kv][capacity][128] (bh stride
 * capacity * 128, token stride 128) or token-major [capacity][B][H_kv][128] (bh stride 128, token
 * stride B * H_kv * 128, so that each new token is one contiguous copy), decodes without
 * repacking it. Both strides are multiples of 8 (KVQ_ERR_ALIGNMENT otherwise), the token stride
 * is at least 128, both at most 2^40; rows must not overlap. kvq_decode_attn is this call with
 * the packed strides (n_tail * 128, 128). */
kvq_status kvq_decode_attn_ex(const kvq_cache* cache, const void* q, const void* tail_k,
                              const void* tail_v, int32_t n_tail, int64_t tail_bh_stride,
                              int64_t tail_token_stride, float* out, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* Size of the decode scratch that the library itself holds for kvq_decode_attn_static:
 * one copy per GPU that loads the library, kept until the process exits. */
#define KVQ_STATIC_WORKSPACE_BYTES (8u << 20)

/* kvq_decode_attn without a workspace argument, for callers that cannot allocate device
 * memory or hand the library a scratch buffer. Examples: an engine whose whole device memory
 * pool is owned by another allocator, or a latency-critical loop where a cudaMalloc (which
 * may synchronise the device) is not acceptable. The pages have no counterpart: this is a
 * deployment convenience, not part of the method.
 *
 * Same arguments, results and checks as kvq_decode_attn, minus the workspace. The split
 * partials go to a fixed device array of KVQ_STATIC_WORKSPACE_BYTES inside the library; a
 * decode that would need more (see kvq_decode_workspace_bytes) returns KVQ_ERR_CAPACITY and
 * launches nothing. No memory is allocated on any call: the first call on a device looks up
 * the array's device address (make that first call before any stream capture), later calls
 * reuse it. Nothing in the array needs to start at zero: every call writes each partial
 * before reading it. All calls on a device share the one array and it keeps the last call's
 * contents, so calls that may overlap on the GPU (other streams, other host threads) race
 * and give wrong results: order them on one stream or synchronise between them. A decode
 * whose bounded wait runs out (KVQ_ERR_TIMEOUT in dev_status) leaves its partials unwritten;
 * its output is then NaN, never a merge of an earlier call's partials. The looked-up address
 * belongs to the device's context as it was at the first call: do not call this entry again
 * after cudaDeviceReset (or any teardown of that context) in the same process. */
kvq_status kvq_decode_attn_static(const kvq_cache* cache, const void* q, const void* tail_k,
                                  const void* tail_v, int32_t n_tail, float* out, cudaStream_t stream);

/* Dequantises blocks [first_block, first_block + n_blocks) of every (b, h) to fp32, for
 * checking only (never on the decode path: [TQ] §4.2 and §5.2 warn that materialising costs
 * more than it saves).
 *   domain 0: the stored representation (pre-RoPE keys un-rotated, KVarN in the Hadamard domain)
 *   domain 1: the input domain (inverse Hadamard for KVarN; same as 0 otherwise)
 *   out_k, out_v: device fp32 [B][H_kv][n_blocks*128][128]; either may be NULL to skip. */
kvq_status kvq_dequant(const kvq_cache* cache, int32_t first_block, int32_t n_blocks,
                       int32_t domain, float* out_k, float* out_v, cudaStream_t stream);

/* ---------------------------------------------------------------- error diagnostics
 * [KVN] splits the squared reconstruction error of a token into a norm part and a direction
 * part, |x - x_dq|^2 = E_M + E_D with E_M = (|x| - |x_dq|)^2 and E_D = 2|x||x_dq|(1 - cos theta)
 * (key innovation; Figure 1a plots sum E_M / sum E_T over the largest errors, Figure 1b the
 * token-norm deviation). These two calls compute both on the GPU for cached blocks. */

/* Per-token error statistics of blocks [first_block, first_block + n_blocks) of every (b, h)
 * against the inputs they were appended from. For each token row (its 128 channels, in the
 * input domain: KVarN rows are transformed back from the Hadamard domain; pre-RoPE keys stay
 * un-rotated) four fp32 values:
 *   [0] |x|,  [1] |x_dq| - |x| (the token-norm deviation; E_M is its square),
 *   [2] E_T = |x - x_dq|^2,  [3] E_D (0 when |x| or |x_dq| is 0).
 * [1] and [3] are evaluated without cancellation: [1] = sum (x_dq - x)(x_dq + x) / (|x_dq| + |x|),
 * [3] = |x||x_dq| |x/|x| - x_dq/|x_dq||^2. For caches with the attention sink, token 0 of block 0
 * is the kept row (decode attends it instead of the tile's row).
 *   k, v           : device [B][H_kv][n_blocks*128][128] in cfg.in_dtype: the rows given to
 *                    kvq_append_block for those blocks (pre-RoPE keys for pre-RoPE caches)
 *   stats_k/stats_v: device fp32 [B][H_kv][n_blocks*128][4]; either pair (k, stats_k) or
 *                    (v, stats_v) may be NULL to skip that kind.
 * Fails (KVQ_ERR_INVALID_ARG) outside the cached range. Inputs 16-byte aligned. */
kvq_status kvq_error_stats(const kvq_cache* cache, const void* k, const void* v, int32_t first_block,
                           int32_t n_blocks, float* stats_k, float* stats_v, cudaStream_t stream);

/* ---------------------------------------------------------------- codebook fitting
 * Sensitivity-weighted nuq codebook ([KVQ] §3.3, Algorithm 2), per KV head h: Lloyd iterations
 * on normalised calibration samples a[h][0..n) with Fisher weights w[h][0..n). Samples are
 * clamped to [-1, 1] and weights to [0, 1]. The k = 2^bits centres start evenly spaced over
 * [-1, 1] (c_j = -1 + 2j/(k-1), fp64 rounded to fp32). An iteration assigns every sample to its
 * nearest centre (|a - c_j| in fp32, the lowest j on ties); when no assignment changed the head
 * stops, else each centre whose members weigh more than zero moves to their weighted mean. The
 * sums are exact: w*a and w are scaled by 2^32, rounded half-even to 64-bit integers and added
 * as integers; a centre is the fp64 quotient of its two sums rounded to fp32. So the codebook
 * does not depend on thread order, and the CPU model reproduces it bit for bit. (The kernels
 * stop a head when an update leaves its centres unchanged, one pass after the rule above at most,
 * with the same centres; so the result is the same for every max_iter.) Inputs must be finite.
 *   a, w     : device fp32 [n_heads][n], 4-byte aligned; 1 <= n <= 2^30
 *   bits     : 1..4;  max_iter: 1..10000 iterations at most
 *   codebook : device fp32 [n_heads][2^bits] (written; usable as kvq_cache_init's codebook)
 *   workspace: device scratch of kvq_fit_codebook_workspace_bytes(n_heads, n) bytes (16-byte
 *              aligned; 272 bytes per head, whatever n)
 * Every step runs on `stream` with no host synchronisation. */
size_t kvq_fit_codebook_workspace_bytes(int32_t n_heads, int64_t n);
kvq_status kvq_fit_codebook(const float* a, const float* w, int32_t n_heads, int64_t n, int32_t bits,
                            int32_t max_iter, float* codebook, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* Most fractions kvq_error_topk takes in one call. */
#define KVQ_TOPK_MAX_FRACS 8

/* Workspace kvq_error_topk needs, in bytes. Pure. */
size_t kvq_error_topk_workspace_bytes(void);

/* Shares of the largest errors ([KVN] Figure 1a). For each fraction f (host array, 0 < f <= 1):
 * the k = ceil(f * n_rows) rows (k computed in fp64) of `stats` with the largest E_T (column 2;
 * equal values: the lower row first) and, summed in fp64 over them,
 *   out[i] = { k, sum E_T, sum E_M (column 1 squared), sum E_D }  (device fp64 [n_fracs][4]).
 * stats: device fp32 [n_rows][4] as kvq_error_stats writes them (finite, E_T >= 0).
 * The selection is a radix select on (E_T, row) keys; every step runs on `stream` with no host
 * synchronisation and the sums come out in a fixed order (bitwise reproducible).
 * 1 <= n_fracs <= KVQ_TOPK_MAX_FRACS, n_rows >= 1 and < 2^32. */
kvq_status kvq_error_topk(const float* stats, int64_t n_rows, const double* fracs, int32_t n_fracs,
                          double* out, void* workspace, size_t workspace_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
