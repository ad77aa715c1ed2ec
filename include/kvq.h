/*
 * kvq.h -- C ABI of the quantized-KV decode library (libkvq.so), sm_103a.
 *
 * Two operations make up the decode hot path:
 *   kvq_append  quantize-on-write of new key/value vectors into a paged cache
 *   kvq_decode  fused dequantize-on-load split attention for one decode step
 * plus kvq_dequant (reads the stored cache back for tests) and a few helpers.
 *
 * Sources (page title, section):
 *   [P1] "KV Cache Quantization Perturbs Attention Through Stored Keys and Values"
 *   [P2] "KV Cache Quantization Reduces Cache Bytes with Separate Accuracy and Kernel Costs"
 *   [P3] "KV Cache Quantization and Per-Token Scale Placement"
 *
 * Conventions shared by every entry point
 *   - All buffers are caller-owned.  "device" pointers must be CUDA device
 *     memory of the current device; "host" pointers are plain host memory.
 *   - Calls are stream-ordered and asynchronous on `stream` (a cudaStream_t
 *     passed as void*; NULL = legacy default stream).  The library never
 *     allocates, frees or synchronizes.
 *   - Arguments are validated on the host; a bad argument returns a status and
 *     launches nothing.  Problems that only the device can see (a block-table
 *     entry out of range, a length beyond the table's capacity, a pipeline wait
 *     that gave up) set bits in the caller's device word *err_word (nullable)
 *     with atomicOr and skip the offending item: kernels never trap.
 *   - Head dimension D = 128 and block size 16 tokens are fixed.
 *
 * Cache layout (device memory, all pools 16-byte aligned)
 *   Codes pool  : [num_kv_heads][num_blocks][block_bytes] (head-major, so the
 *                 consecutive blocks of one head are adjacent in memory), with
 *                 block_bytes = 16 * 128 * bits / 8 (int2 512, int4 1024, int8 2048,
 *                 bf16 4096).
 *                 Inside a block the bytes are ordered so that each lane of a
 *                 warp reads its tensor-core operand with one 16-byte load per
 *                 512-byte chunk ("fragment-native" order).  Let lane = 4*g + t.
 *     Keys, element (token i in block, dim d):
 *         g = i & 7, hi = i >> 3, t = d >> 5, e = d & 31
 *         int8 : chunk = 2*hi + (e >> 4), byte = e & 15
 *         int4 : chunk = hi, word = e >> 3, nibble = ((e & 7) >> 1) + 4*(e & 1)
 *         bf16 : chunk = 4*hi + (e >> 3), element = e & 7 (2 bytes each)
 *         int2 : chunk = 0, word = e >> 3, field bit = 16*(e & 1) + 8*((e >> 2) & 1)
 *                + 2*(hi + 2*((e & 3) >> 1))
 *     Values, element (token i, dim d):
 *         mt = d >> 4, r = d & 15, g = r & 7, hi = r >> 3,
 *         t = (i & 7) >> 1, j = 2*(i & 1) + (i >> 3)
 *         int8 : chunk = mt >> 1, word = 2*(mt & 1) + hi, byte j of the word
 *         int4 : chunk = mt >> 2, word = mt & 3, nibble = 2*hi + (j >> 1) + 4*(j & 1)
 *         bf16 : chunk = mt, word = 2*hi + (j >> 1), element j & 1 of the word
 *         int2 : chunk = 0, word = mt >> 1, field bit = 16*(j & 1) + 8*(mt & 1)
 *                + 2*(hi + 2*(j >> 1))
 *     Byte offset = chunk*512 + lane*16 + word*4 + (byte or nibble/2 or 2*element
 *     or field bit/8); for int8 keys "byte" is the offset inside the lane's 16
 *     bytes.  Nibble n of a little-endian 32-bit word occupies bits 4n..4n+3; a
 *     2-bit field at "field bit" b occupies bits b..b+1 of the word.  Codes are
 *     stored offset-binary: an int8 code c in [-127,127] is the byte c + 128, an
 *     int4 code c in [-8,7] (-8 never produced) is the nibble c + 8, an int2
 *     code c in [-2,1] (-2 never produced) is the field c + 2.  In the
 *     asymmetric format the unsigned code u (int8: 0..255, int4: 0..15, int2:
 *     0..3) is stored as the byte, nibble or field u itself.
 *   Metadata pool: float [num_kv_heads][num_blocks][M], one record of M floats
 *                 per block (absent for a bf16 cache), tokens in natural order:
 *                 symmetric M = 32: the block's 16 key scales, then its 16
 *                 value scales; asymmetric M = 64: key scales, key zero points,
 *                 value scales, value zero points.  A block's record is one
 *                 128-byte (256-byte) read.  Keys under per-channel scales only
 *                 leave the key-scale entries unused.  2-bit blocks (token-group
 *                 scales) M = 4: the block's key scale, key zero point, value
 *                 scale, value zero point (zero points 0 when symmetric), one
 *                 16-byte read.
 *   Window ring : bf16 [window_batch][num_kv_heads][window / 16][4096 bytes]:
 *                 window / 16 blocks per (sequence, head) for keys and for
 *                 values, each in the bf16 key / value block order above;
 *                 position p of sequence b lives in slot p % window, which is
 *                 token (slot % 16) of ring block slot / 16.
 *   Block table : int32 [batch][max_blocks_per_seq]; logical block j of
 *                 sequence b is physical block block_table[b*max_blocks_per_seq+j].
 *                 Position p of a sequence is token p % 16 of logical block p / 16.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,  /* null / negative / inconsistent argument            */
  KVQ_ERR_UNSUPPORTED = 2,  /* valid but not implemented (D != 128, G > 8, ...)    */
  KVQ_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned                      */
  KVQ_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required            */
  KVQ_ERR_CUDA = 5          /* a CUDA runtime call or launch failed                  */
} kvq_status;

/* Bits of the device error word. */
#define KVQ_DEVERR_BLOCK_ID 1u  /* block-table entry outside [0, num_blocks)        */
#define KVQ_DEVERR_SEQ_LEN 2u   /* length < 0 or beyond the block table's capacity  */
#define KVQ_DEVERR_TIMEOUT 4u   /* a pipeline wait gave up (the CTA skipped work)   */
#define KVQ_DEVERR_RANGE 8u     /* reserved: no longer raised (any value scale is   */
                                /* decoded; the weights are kept in fp16 range)     */
#define KVQ_DEVERR_POSITION 16u /* append: sequence index or position out of range  */

/* kvq_append modes */
#define KVQ_APPEND_QUANT 0 /* quantize the new vectors into the block store at pos      */
#define KVQ_APPEND_RING 1  /* copy the new bf16 vectors into window slot pos % window   */
#define KVQ_APPEND_STEP 2  /* decode step with a window: the token at pos - window (if  */
                           /* pos >= window) leaves the ring and is quantized into the  */
                           /* block store, then the new token enters the ring           */

/* kvq_prefill: stream_ctas value that selects the query-tile path */
#define KVQ_PREFILL_TILES (-1)

/* Description of one layer's cache.  Every pointer is caller-owned device memory. */
typedef struct {
  int32_t num_kv_heads;   /* H_kv >= 1                                              */
  int32_t head_dim;       /* must be 128                                            */
  int32_t block_size;     /* must be 16                                             */
  int32_t num_blocks;     /* physical blocks in each pool                           */
  int32_t k_bits;         /* 8 or 4 (quantized), 2 together with v_bits = 2 (token- */
                          /* group scales, see kvq_append), or 16 together with     */
                          /* v_bits = 16 (plain bf16 cache)                         */
  int32_t v_bits;         /* 8 or 4, 2 with k_bits = 2, or 16 with k_bits = 16      */
  void* k_codes;          /* codes pool for keys (see layout above)                 */
  void* v_codes;          /* codes pool for values                                  */
  float* meta;            /* metadata pool (layout above); NULL for a bf16 cache    */
  /* Asymmetric format ([P1] "Quantization granularity defines which values
   * share a scale": a scale and, depending on the scheme, a zero point; [P3]
   * "Per-token scales and where they can live": a scale and zero point cost
   * twice the metadata).  0: symmetric codes.  1 (8-, 4- or 2-bit blocks): per
   * token per head (2-bit blocks: per 16-token group per head, over all the
   * group's values) m = min(x), s = RN32((max(x) - min(x)) / (2^bits - 1))
   * (difference and quotient in double; a constant vector stores s = 1), u =
   * clamp(round_half_even((x - m) / s), 0, 2^bits - 1) with the difference and
   * quotient in double, x_hat = u * s + m; K and V both. */
  int32_t asym;
  const float* k_channel_factor; /* [num_kv_heads][128] positive, or NULL           */
  int32_t window;         /* recent-token bf16 window W: 0 = none, or 16..128 in    */
                          /* steps of 16                                            */
  int32_t window_batch;   /* first dimension of the ring buffers (sequences)        */
  void* k_window;         /* bf16 ring (layout above), or NULL if W == 0            */
  void* v_window;
  /* Query format of kvq_decode against this cache ([P3] "Precision floors and
   * mixed cache formats": an 8-bit query meets the integer key codes, the dot
   * product accumulates in integers and is converted to float before the
   * exponential).  0 or 16: the bf16 query, carried into the code contraction
   * as fp16 scaled by a power of two (11 significant bits), and the value
   * weights p * s_v as fp16 (default).  32 (two-part mode): the query and the
   * value weights each carried as an fp16 high part plus an fp16 low part
   * (about 22 significant bits; one more MMA per k-slice of each contraction:
   * 6-15 % more time measured), for scores large enough that 11 bits of query
   * cost more than the output tolerance, and so that results do not depend on
   * how the token range is split beyond fp32 rounding.  8: each query row, after
   * the per-channel key factor is multiplied onto it in float32, is quantized
   * per row with the symmetric int8 rule of kvq_append (s_q = RN32(max|x| /
   * 127), q_int = clamp(round_half_even(x / s_q))) and the score is
   * s_q * s_k * (q_int . k_int) / sqrt(D), the integer dot exact; bf16 window
   * keys see q_int * s_q.  Needs 8-, 4- or 2-bit blocks; not combined with both a
   * per-channel key factor and a window (KVQ_ERR_UNSUPPORTED). */
  int32_t q_bits;
  /* Per-channel key scales only ([P3] "The axis choice is a kernel decision":
   * per-channel key scales are moved onto the query).  0: the per-channel key
   * factor (if any) divides the keys before the per-token quantizer.  1: the
   * keys carry no per-token scale: code_j = clamp(round_half_even(k_j / c_j))
   * with c = k_channel_factor as the per-channel scale (required; the clamp
   * binds for values beyond qmax * c_j), k_hat_j = c_j * code_j; the key-scale
   * entries of the metadata pool are not read or written.  Symmetric 8- or
   * 4-bit keys only. */
  int32_t k_per_channel;
} kvq_cache_desc;

/* Human-readable name of a status code (static string, never NULL). */
const char* kvq_status_string(kvq_status status);

/* Bytes of one 16-token block of one KV head for a code width (2, 4, 8 or 16). */
kvq_status kvq_block_bytes(int32_t bits, size_t* bytes);

/*
 * kvq_append -- quantize-on-write.
 * [P3] "Per-token scales and where they can live": the scale is computed from
 * the vector being written, at write time, and stored alongside it, one scale
 * per token per head.  [P2] "Quantization needs a scale convention" and the
 * listing in [P3] "The axis choice is a kernel decision": s = max|x| / qmax
 * (stored as float32, RN), code = clamp(round_half_even(x / s)), all-zero
 * vector -> codes 0 and s = 1.  qmax = 127 (int8) or 7 (int4).  With a
 * per-channel key factor c, keys are first divided by c (float32, RN) and then
 * quantized per token ([P3] "The axis choice is a kernel decision"); with
 * k_per_channel = 1 a key's codes are clamp(round_half_even(k_j / c_j)) and no
 * key scale is stored.  Codes are the correctly rounded quotient of the exact
 * x / s.  With asym = 1 the
 * asymmetric quantizer of kvq_cache_desc is used instead and the zero point is
 * stored beside the scale.
 * 2-bit caches ([P3] "Per-token scales and where they can live": several
 * tokens under one scale): the unit of quantization is the 16-token block of
 * one head.  The same rule (qmax = 1, codes in [-1, 1]; asymmetric u in
 * [0, 3]) is applied to all of a block's present values as one vector, after
 * the per-channel key factor division; absent tokens of a block (the tail of a
 * sequence) store code 0 and are never read.  KVQ_APPEND_QUANT writes a block
 * whole: the rows of one call at positions 16j, 16j+1, ... of one sequence
 * must follow each other in the call, led by the row at 16j (up to 16 rows); a
 * row that is not part of such a run sets KVQ_DEVERR_POSITION and is skipped.
 * KVQ_APPEND_STEP is refused (KVQ_ERR_UNSUPPORTED): a growing 2-bit cache keeps
 * its recent tokens in the bf16 window (RING) and quantizes whole blocks.
 *   k_new, v_new : device bf16 [n][num_kv_heads][128]
 *   n            : number of new tokens (0 is a no-op)
 *   seq_idx, pos : device int32 [n]; token r belongs to sequence seq_idx[r] at
 *                  position pos[r].  Within one call the positions of one
 *                  sequence must be distinct, and in KVQ_APPEND_STEP mode they
 *                  must span fewer than `window` positions.
 *   mode         : KVQ_APPEND_QUANT / RING / STEP (RING and STEP need window > 0)
 *   block_table  : device int32 [batch][max_blocks_per_seq] (unused by RING)
 *   err_word     : device uint32 or NULL (POSITION / BLOCK_ID bits)
 */
kvq_status kvq_append(const kvq_cache_desc* cache, const void* k_new, const void* v_new, int32_t n,
                      const int32_t* seq_idx, const int32_t* pos, int32_t mode,
                      const int32_t* block_table, int32_t batch, int32_t max_blocks_per_seq,
                      uint32_t* err_word, void* stream);

/* Work decomposition of kvq_decode (host-only arithmetic, no CUDA calls). */
typedef struct {
  int32_t stream_ctas;    /* CTAs sharing the token blocks of all (seq, kv_head) units */
  int32_t window_ctas;    /* one CTA per unit for the bf16 window (0 without a window) */
  int32_t units;          /* batch * num_kv_heads                                       */
  int32_t partial_slots;  /* partial-result records in the workspace                    */
  size_t workspace_bytes; /* bytes kvq_decode needs for this plan                       */
} kvq_decode_plan;

/* Plan for `num_sms` SMs with `ctas_per_sm` resident decode CTAs each, or an
 * explicit `stream_ctas` (> 0 overrides the SM-based count). */
kvq_status kvq_make_decode_plan(int32_t batch, int32_t q_heads, int32_t num_kv_heads, int32_t window,
                                int32_t num_sms, int32_t ctas_per_sm, int32_t stream_ctas,
                                kvq_decode_plan* plan);

/* The plan kvq_decode uses on the current device: stream CTAs = SMs x resident
 * decode CTAs per SM (occupancy of this cache format) minus the window CTAs,
 * or the explicit stream_ctas (> 0). */
kvq_status kvq_decode_device_plan(const kvq_cache_desc* cache, int32_t batch, int32_t q_heads,
                                  int32_t stream_ctas, kvq_decode_plan* plan);

/* Workspace bytes kvq_decode needs on the current device (stream_ctas 0 = automatic). */
kvq_status kvq_decode_workspace_size(const kvq_cache_desc* cache, int32_t batch, int32_t q_heads,
                                     int32_t stream_ctas, size_t* bytes);

/* Zero a decode workspace.  Its merge counters (the first 4 * batch *
 * num_kv_heads bytes) must start at zero; a kvq_decode that completes leaves
 * them at zero again, including one that flagged KVQ_DEVERR_BLOCK_ID,
 * KVQ_DEVERR_SEQ_LEN or KVQ_DEVERR_RANGE.  A call that flagged
 * KVQ_DEVERR_TIMEOUT may leave counters of the units it gave up on non-zero:
 * after that bit, call kvq_workspace_init again before the workspace's next
 * kvq_decode (otherwise later merges would combine the wrong records).  Call it
 * once after allocating the workspace. */
kvq_status kvq_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * kvq_decode -- one decode step of attention over the quantized cache.
 * [P1] "Key error acts before the softmax" and [P2] "Keys and values need not
 * have identical error sensitivity": score_i = q . k_hat_i / sqrt(D),
 * o = sum_i softmax(score)_i v_hat_i.  [P3] "The axis choice is a kernel
 * decision": the per-token key scale multiplies the score after the integer
 * dot product; the per-channel key factor is applied to the query once.
 * [P3] "Per-token scales and where they can live": dequantization happens as
 * the kernel loads (codes and scales are two read streams).  [P1] "Cache growth
 * changes the serving trade": the last min(W, L) positions are read from the
 * bf16 window, older ones from the quantized blocks.  Query head hq reads KV
 * head hq / (q_heads / num_kv_heads).  In the asymmetric format the scores and
 * outputs use x_hat = u * s + m (the zero-point terms are added to the code
 * contractions: m * sum(q) per score, sum(p * m) per output).
 *   q          : device bf16 [batch][q_heads][128]
 *   seq_lens   : device int32 [batch], tokens attended per sequence (0 allowed:
 *                out = 0, lse = -inf)
 *   out        : device [batch][q_heads][128], bf16 (out_fp32 = 0) or float32
 *   lse        : device float [batch][q_heads] natural-log log-sum-exp of the
 *                scores, or NULL
 *   workspace  : device, >= kvq_decode_workspace_size bytes, zeroed once by
 *                kvq_workspace_init (again after a KVQ_DEVERR_TIMEOUT); one
 *                workspace per concurrently running call
 *   stream_ctas: 0 = one wave on all SMs, > 0 = explicit count (tests)
 * Requirements: q_heads % num_kv_heads == 0, q_heads / num_kv_heads <= 8.
 */
kvq_status kvq_decode(const kvq_cache_desc* cache, const void* q, int32_t batch, int32_t q_heads,
                      const int32_t* seq_lens, const int32_t* block_table, int32_t max_blocks_per_seq,
                      void* out, int32_t out_fp32, float* lse, void* workspace, size_t workspace_bytes,
                      int32_t stream_ctas, uint32_t* err_word, void* stream);

/* kvq_decode_ex flag: seq_lens and block_table hold their final values before
 * the kernel that precedes this call on the stream ends -- they are written by
 * host copies or by kernels that completed before that kernel started, never
 * by it (nor by a kernel it overlaps).  The usual decode step qualifies: the
 * scheduler writes lengths and tables before the step; the kernels just ahead
 * of attention (projections, kvq_append) write queries and cache entries.  The
 * decode kernel then reads the lengths, and works out its split, while that
 * kernel finishes, instead of after it (0.5-1 us per call on GB300). */
#define KVQ_DECODE_GEOMETRY_READY 1u

/*
 * kvq_decode_ex -- kvq_decode with flags (0 or KVQ_DECODE_GEOMETRY_READY; any
 * other bit: KVQ_ERR_INVALID_ARG).  Same arguments, results and errors
 * otherwise; kvq_decode is kvq_decode_ex with flags 0.  With the flag the
 * results are identical (the same arithmetic); only the order of the loads
 * changes.  A device error found in the lengths or the table is reported the
 * same way.
 */
kvq_status kvq_decode_ex(const kvq_cache_desc* cache, const void* q, int32_t batch, int32_t q_heads,
                         const int32_t* seq_lens, const int32_t* block_table, int32_t max_blocks_per_seq,
                         void* out, int32_t out_fp32, float* lse, void* workspace, size_t workspace_bytes,
                         int32_t stream_ctas, uint32_t flags, uint32_t* err_word, void* stream);

/* Size of the fixed device scratch behind kvq_decode_static_scratch (bytes). */
#define KVQ_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * kvq_decode_static_scratch -- kvq_decode for callers that cannot allocate.
 * The pages have no counterpart to this entry point: it is a library
 * integration variant of kvq_decode with identical arguments and results,
 * minus the workspace.
 * Some callers cannot call cudaMalloc on their decode path: code embedded in a
 * host runtime that owns every device allocation (a plugin or custom operator
 * given only input and output buffers), or loops that must not pay the
 * implicit device synchronisation and allocator locking of cudaMalloc.  For
 * them the split-attention scratch (partial records and merge counters) lives
 * in one file-scope device array of KVQ_STATIC_SCRATCH_BYTES that every GPU
 * loading the library holds until the process exits.  The caller still passes
 * all inputs and outputs.
 *   - A call whose plan (kvq_decode_device_plan) needs more than
 *     KVQ_STATIC_SCRATCH_BYTES returns KVQ_ERR_WORKSPACE and launches nothing.
 *   - The first call on each device does the set-up: it looks up the array's
 *     device address (with that device current) and caches it with the CUDA
 *     context it belongs to; make that first call before any stream capture.
 *     A call under a different context (after cudaDeviceReset, for example)
 *     repeats the set-up, which then also must not fall inside a capture.
 *   - Every call clears the merge counters with cudaMemsetAsync on `stream`
 *     (no allocation) and then runs kvq_decode on the shared array.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents: calls that overlap on the GPU (different streams, or several
 *     host threads) race and corrupt each other's results.  Serialise them.
 */
kvq_status kvq_decode_static_scratch(const kvq_cache_desc* cache, const void* q, int32_t batch, int32_t q_heads,
                                     const int32_t* seq_lens, const int32_t* block_table,
                                     int32_t max_blocks_per_seq, void* out, int32_t out_fp32, float* lse,
                                     int32_t stream_ctas, uint32_t* err_word, void* stream);

/*
 * kvq_prefill -- chunked-prefill attention over the quantized cache, with the
 * chunk's own quantize-on-write.  The cache is written incrementally and read
 * repeatedly ("KV Cache Quantization and Per-Token Scale Placement", opening
 * section): a chunk of n new positions is first quantized into the block
 * store (exactly kvq_append in KVQ_APPEND_QUANT mode, when k_new and v_new
 * are given), and then every new position attends causally to the stored
 * cache of its sequence, itself included:
 *   for row r, query head hq:  o = sum_{i <= pos[r]} softmax(score)_i v_hat_i,
 *   score_i = q[r][hq] . k_hat_i / sqrt(D), over positions 0..pos[r] of
 *   sequence seq_idx[r], read from the quantized blocks as kvq_decode reads them.
 * The write and the attention are two launches in stream order (the second
 * starts under programmatic dependent launch and waits for the first).  Two
 * attention paths, chosen by stream_ctas:
 *   KVQ_PREFILL_TILES (-1): query tiles.  A CTA takes 16 / G consecutive rows
 *     x the G query heads of one KV head (16 query vectors, one tensor-core
 *     row tile) and streams the blocks of their sequence once for all of
 *     them; rows of one tile that belong to different sequences are taken in
 *     turn.  Quantized caches (8-, 4- or 2-bit, symmetric or asymmetric, any
 *     q_bits); a bf16 cache gives KVQ_ERR_UNSUPPORTED.  Needs no workspace
 *     (NULL accepted).
 *   > 0: split rows.  Every row is one query group of the decode kernel's
 *     split over that many stream CTAs, so rows of one sequence read
 *     overlapping prefixes (mostly from L2 when they run together).  Every
 *     cache format.
 *   0: the tile path when the cache format allows it and the (tile, KV head)
 *     pairs number at least 9/16 of the SMs; split rows otherwise.
 * Both paths compute the same attention within the output tolerance (they
 * differ in rounding order only).
 *   q          : device bf16 [n][q_heads][128]
 *   seq_idx,pos: device int32 [n] (as kvq_append); a row with a sequence outside
 *                [0, batch) sets KVQ_DEVERR_POSITION and gets out = 0, lse = -inf
 *   k_new,v_new: device bf16 [n][num_kv_heads][128] to write first, or both NULL
 *                when the chunk is already in the cache; for 2-bit caches the
 *                chunk's positions must start at a block boundary (blocks are
 *                written whole)
 *   block_table: device int32 [batch][max_blocks_per_seq]
 *   out, lse   : device [n][q_heads][128] (bf16 or float32), float [n][q_heads] or NULL
 *   workspace  : >= kvq_prefill_workspace_size bytes, zeroed once by kvq_workspace_init
 *                (the split-rows path; unused by the tile path)
 * Requirements: window == 0 (KVQ_ERR_UNSUPPORTED otherwise), n <= 4096, the
 * kvq_decode requirements on q_heads.
 */
kvq_status kvq_prefill(const kvq_cache_desc* cache, const void* q, int32_t n, int32_t q_heads,
                       const int32_t* seq_idx, const int32_t* pos, const void* k_new, const void* v_new,
                       const int32_t* block_table, int32_t batch, int32_t max_blocks_per_seq, void* out,
                       int32_t out_fp32, float* lse, void* workspace, size_t workspace_bytes, int32_t stream_ctas,
                       uint32_t* err_word, void* stream);

/* Workspace bytes kvq_prefill needs for n rows on the current device with
 * this stream_ctas (0 for KVQ_PREFILL_TILES; with 0 the split-rows size, since
 * the automatic choice may take that path). */
kvq_status kvq_prefill_workspace_size(const kvq_cache_desc* cache, int32_t n, int32_t q_heads, int32_t stream_ctas,
                                      size_t* bytes);

/*
 * kvq_dequant -- read the block store back: x_hat = RN32(code * s)
 * ([P2] "Quantization needs a scale convention"), without the per-channel key
 * factor; in the asymmetric format x_hat = RN32(u * s + m) (one fused
 * multiply-add); keys under per-channel scales only give RN32(code * c_j).
 * For a bf16 cache the stored values are widened.  For tests.
 *   slots : device int32 [n], physical slot = physical_block * 16 + token
 *   k_out, v_out : device float [n][num_kv_heads][128]
 */
kvq_status kvq_dequant(const kvq_cache_desc* cache, const int32_t* slots, int32_t n, float* k_out,
                       float* v_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
