/*
 * tq.h -- C ABI of the rotated-codebook KV-cache library (sm_103a / GB300).
 *
 * The library compresses attention keys and values into a paged cache and
 * runs single-token decode attention directly over the compressed pages.
 *
 *   Keys   (turbo-attn, "How it works", steps 1-3; 0xsero/turboquant,
 *           "Compression Pipeline"): store ||k|| as bf16, rotate the unit key
 *           with a seeded random orthogonal matrix Pi, quantise every scaled
 *           coordinate z = sqrt(d) (Pi k / ||k||)_j against a Lloyd-Max codebook
 *           for N(0,1), and -- when k_bits <= 3 -- keep the QJL sign sketch
 *           sign(S r) of the residual r plus ||r|| as bf16.
 *   Values (0xsero/turboquant, "Value Compression"; tiny-turboquant,
 *           "Measured quality"): per group of `group` channels, an fp16
 *           (scale, zero) pair and round-half-up codes, bit-packed.
 *   Decode (turbo-attn, "How it works" and TKV_DECODE_SPLITS under
 *           "Configuration"): queries are pre-rotated once; a split-K paged
 *           kernel scores them against the packed key codes (plus the QJL
 *           correction), runs an online softmax, accumulates dequantised
 *           values, and the splits are merged by a log-sum-exp combine.
 *
 * Conventions for every call:
 *   - Pointers named `*_dev` or documented "device" are CUDA device pointers
 *     owned by the caller; the library never frees or retains them.
 *   - bf16 data crosses the ABI as uint16_t bit patterns; fp16 likewise.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every call except tq_init / tq_destroy / tq_get_status / tq_export_params
 *     is asynchronous on `stream`, never synchronises and never allocates, so
 *     it may be captured in a CUDA graph.
 *   - Arguments are validated on the host before any launch; a non-OK status
 *     means nothing was launched, and tq_last_error() describes why.
 *   - Out-of-range slot or block ids found on the device are skipped and set
 *     bits in a per-handle device status word (see tq_get_status); kernels
 *     never trap.
 *
 * Supported parameters: head_dim in {128, 256}; k_bits, v_bits in {2, 3, 4};
 * group in {32, 64, 128} dividing head_dim; page_size in {16, 32}.  QJL is on
 * exactly when k_bits <= 3 (m = head_dim projection rows, one bit each).
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tq_ctx *tq_handle;

typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, negative size, bad handle */
    TQ_ERR_UNSUPPORTED = 2,  /* parameter outside the supported set above */
    TQ_ERR_CUDA = 3,         /* a CUDA runtime call failed (message in tq_last_error) */
    TQ_ERR_OOM = 4           /* tq_init could not allocate its parameter tables */
} tq_status;

/* Device status bits accumulated by kernels (read with tq_get_status). */
#define TQ_DEVERR_SLOT_RANGE  0x1u  /* compress: slot >= num_blocks * page_size (token skipped)   */
#define TQ_DEVERR_BLOCK_RANGE 0x2u  /* decode/dequant: block id < 0 or >= num_blocks (page skipped) */
#define TQ_DEVERR_SEQ_RANGE   0x4u  /* decode: seq_len > max_blocks_per_seq * page_size (clamped)  */
#define TQ_DEVERR_TIMEOUT     0x8u  /* a barrier wait ran past the handle's wait limit (tq_set_wait_limit):
                                       compress -- a tensor-core completion or hand-off wait; the CTA stops
                                       and the rows of its unfinished tiles are left unwritten;
                                       decode -- a page-copy wait; the CTA stops issuing copies, waits
                                       (bounded) for those in flight and drops its split from the result */

/*
 * tq_init -- build the codec parameters for one (head_dim, k_bits, v_bits,
 * group, seed) and upload them to the current CUDA device.
 *
 * Pi (d x d) is the Q factor, with a positive-diagonal R, of the QR
 * decomposition of a d x d matrix of standard Gaussians (Haar measure); S
 * (d x d) is a second matrix of standard Gaussians (0xsero/turboquant,
 * "Compression Pipeline": rotation state and QJL projection).  Gaussians come
 * from SplitMix64 stream s started at seed XOR (0x9E3779B97F4A7C15 * (s + 1)),
 * s = 0 for Pi and 1 for S, through Box-Muller, filled row-major.  The codebook
 * is the Lloyd-Max quantiser of N(0,1) with 2^k_bits levels (brightcoding blog,
 * "What is TurboQuant-GPU?").
 *
 * Allocates device memory for the tables (this is the only allocating call).
 * On success *out receives a handle; on failure *out is set to NULL.
 */
tq_status tq_init(int head_dim, int k_bits, int v_bits, int group, uint64_t seed, tq_handle *out);

/*
 * tq_init_ex -- tq_init with options, flags = bitwise OR of:
 *   TQ_ROTATION_HADAMARD  Pi is a randomized Hadamard rotation H D / sqrt(d)
 *     (turbo-attn, "How it works", step 1: a fast Walsh-Hadamard transform), with
 *     H the Sylvester Hadamard matrix, H[i][j] = (-1)^popcount(i & j), and
 *     D = diag(s), s_j = -1 when the top bit of the j-th output of SplitMix64
 *     stream 0 (the stream the dense rotation draws from) is set, else +1.
 *     S, the codebook and the records are unchanged; the rotation runs as
 *     butterflies where that pays (key compression at head_dim 256).
 *     Without this flag Pi is the dense Haar rotation described above.
 *   TQ_VALUES_MSE  values are coded like keys without the QJL sketch
 *     (brightcoding blog, "What is TurboQuant-GPU?" and "Example 4": 3-bit MSE
 *     values; normalize -> rotate -> Lloyd-Max quantize -> pack): the value's
 *     norm is stored as bf16 and every coordinate of z = sqrt(d) Pi v / ||v||
 *     is coded against the v_bits-bit Lloyd-Max codebook of N(0,1); `group` is
 *     then unused (it must still be a supported value).  The V record becomes
 *     codes [P][d*v_bits/8] | norms [P] bf16, and dequant / decode use
 *     V~ = n Pi^T c[code] / sqrt(d) (decode accumulates in the rotated space and
 *     rotates the output back once per query head).
 * tq_init(...) is tq_init_ex(..., 0, ...).
 */
#define TQ_ROTATION_HADAMARD 1u
#define TQ_VALUES_MSE 2u
tq_status tq_init_ex(int head_dim, int k_bits, int v_bits, int group, uint64_t seed, unsigned flags,
                     tq_handle *out);

/* Frees the handle's device tables.  Accepts NULL. */
tq_status tq_destroy(tq_handle h);

/*
 * tq_cache_layout -- bytes of one page record for one (block, kv head).
 * The record size does not depend on the number of kv heads, so unlike the
 * pool sizes it takes no head count: a pool holds num_blocks * num_kv_heads
 * records.
 *
 * The K pool is laid out [num_blocks][num_kv_heads][k_page_bytes] and the V
 * pool [num_blocks][num_kv_heads][v_page_bytes].  Token slot s lives in block
 * s / page_size at offset o = s % page_size.  Inside a record (P = page_size):
 *   K: codes [P][d*k_bits/8] | signs [P][d/8] (QJL) | norms [P] bf16 | gammas [P] bf16 (QJL)
 *   V: codes [P][d*v_bits/8] | meta  [P][d/group][2] fp16 (scale, zero)
 *      (with TQ_VALUES_MSE: codes [P][d*v_bits/8] | norms [P] bf16)
 * Codes are LSB-first bitstreams (code j in bits [b*j, b*j+b)); sign bit i is
 * bit i%8 of byte i/8.  Every sub-array is a multiple of 16 bytes.
 */
tq_status tq_cache_layout(tq_handle h, int page_size, size_t *k_page_bytes, size_t *v_page_bytes);

/*
 * tq_compress_kv -- write T tokens of K and V into the paged pools.
 *
 * k, v: device bf16, token t / kv head h at k + t*k_stride_tok + h*head_dim
 *       (strides in elements; each head row contiguous, 16-byte aligned).
 * slot_mapping: device int64 [T]; -1 skips the token; a slot >= num_blocks *
 *       page_size is skipped and sets TQ_DEVERR_SLOT_RANGE.
 * k_cache, v_cache: device pools sized num_blocks * num_kv_heads * page bytes
 *       (tq_cache_layout), 16-byte aligned.  Only the bytes of written slots
 *       change.  Two tokens mapped to one slot race (caller error).
 * One or two kernel launches on `stream` (one with QJL keys at head_dim 128 and
 * with the Hadamard rotation and 4-bit keys at 256; otherwise the keys and the
 * values are coded by separate kernels, MSE-coded values by a second keys-only
 * pass); T == 0 launches nothing.
 */
tq_status tq_compress_kv(tq_handle h, const uint16_t *k, const uint16_t *v, int64_t T, int num_kv_heads,
                         int64_t k_stride_tok, int64_t v_stride_tok, const int64_t *slot_mapping,
                         uint8_t *k_cache, uint8_t *v_cache, int page_size, int64_t num_blocks, void *stream);

/*
 * tq_dequant_kv -- reconstruct bf16 K and V for a list of slots, so that any
 * third-party attention can consume them (turbo-attn, "Two independently-
 * usable pieces": codec -> any attention backend).
 *
 * Keys come back in the ORIGINAL (unrotated) space:
 *   K~ = n Pi^T ( c[code]/sqrt(d) + [QJL] sqrt(pi/2)/d * gamma * S^T (2 sigma - 1) ),
 *   V~ = code * scale + zero.
 * slots: device int64 [T] (-1 -> the output rows are left untouched).
 * k_out, v_out: device bf16 [T][num_kv_heads][head_dim], contiguous.
 */
tq_status tq_dequant_kv(tq_handle h, const uint8_t *k_cache, const uint8_t *v_cache, int page_size,
                        int64_t num_blocks, int num_kv_heads, const int64_t *slots, int64_t T,
                        uint16_t *k_out, uint16_t *v_out, void *stream);

/*
 * tq_decode_splits -- the split count tq_decode_attention uses when called
 * with splits = 0: about eight (sequence, kv head, split) work units per SM,
 * raised to fill whole waves of resident decode CTAs (4 per SM at d = 128, 2 at
 * d = 256) when the last wave would be less than half full, at least one page
 * per split, at most 64 splits.  Reads no device memory.
 */
int tq_decode_splits(tq_handle h, int batch, int num_kv_heads, int max_blocks_per_seq, int page_size);

/* Workspace bytes tq_decode_attention needs for `splits` splits (0 = auto is
 * not accepted here: pass the value tq_decode_splits returned). */
size_t tq_decode_workspace_bytes(tq_handle h, int batch, int num_q_heads, int splits);

/*
 * tq_decode_attention -- one query token per sequence against its paged,
 * compressed context (no mask: the token attends to all seq_lens[b] tokens).
 *
 * q: device bf16 [B][Hq][d]; query head qh reads kv head qh / (Hq / Hkv).
 * block_table: device int32 [B][max_blocks_per_seq]; position t of sequence b
 *   is slot block_table[b][t / P] * P + t % P.
 * seq_lens: device int32 [B]; 0 gives a zero output row.
 * sm_scale: score scale (usually 1/sqrt(d)).
 * splits: split-K count, 0 = tq_decode_splits(...).
 * workspace: device scratch of ws_bytes >= tq_decode_workspace_bytes(splits),
 *   256-byte aligned; holds rotated queries and per-split partial outputs.  It
 *   starts with the outputs in fp32 before their bf16 rounding, float
 *   [B][Hq][d] at offset 0, which the caller may read after the call.
 * out: device bf16 [B][Hq][d].
 * Three launches on `stream` (query rotation, split-K decode, combine).
 */
tq_status tq_decode_attention(tq_handle h, const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                              const int32_t *block_table, const int32_t *seq_lens, int batch, int num_q_heads,
                              int num_kv_heads, int page_size, int max_blocks_per_seq, int64_t num_blocks,
                              float sm_scale, int splits, void *workspace, size_t ws_bytes, uint16_t *out,
                              void *stream);

/*
 * tq_prefill_attention -- chunked prefill over the compressed cache (turbo-attn,
 * "How it works": the prefill path dequantises the codec inline in the
 * attention mainloop, with no decompress buffer): the last q_tokens positions of
 * every sequence attend causally to its compressed context, their own (already
 * compressed) keys and values included.
 *
 * q: device bf16 [B][q_tokens][Hq][d]; query token i of sequence b sits at
 *   position seq_lens[b] - q_tokens + i and attends to positions 0 .. that one
 *   (positions below 0 -- a sequence shorter than q_tokens -- see nothing and
 *   give zero rows).  Query head qh reads kv head qh / (Hq / Hkv).
 * block_table, seq_lens, pools, sm_scale, splits, status bits: as in
 *   tq_decode_attention; splits = 0 picks tq_prefill_splits(...).
 * workspace: ws_bytes >= tq_decode_workspace_bytes(h, B * q_tokens, Hq, splits),
 *   256-byte aligned; it starts with the fp32 outputs [B][q_tokens][Hq][d].
 * out: device bf16 [B][q_tokens][Hq][d].
 * A CTA takes tq_prefill_queries_per_cta consecutive query tokens of one
 * sequence and kv head; their (token, head) pairs are the columns of its
 * tensor-core products, so every key and value operand decoded from the codes
 * serves all of them, and each column keeps its own causal limit and online
 * softmax.  head_dim 128: 128 columns per CTA (128 / G query tokens), the pages
 * of each 64-token tile decoded once into shared-memory operand tiles, scores
 * and P.V on tcgen05.mma with the accumulators in tensor memory.  head_dim 256:
 * the decode's split-K kernel with 8 columns per CTA (8 / G query tokens).
 * Three launches on `stream` (query rotation, split-K, combine).
 *
 * tq_prefill_queries_per_cta: query tokens per CTA for this handle and G.
 * tq_prefill_splits: the split count tq_prefill_attention picks for splits = 0
 *   (from the sizes only: it never reads seq_lens).
 */
int tq_prefill_queries_per_cta(tq_handle h, int num_q_heads, int num_kv_heads);
int tq_prefill_splits(tq_handle h, int batch, int q_tokens, int num_q_heads, int num_kv_heads,
                      int max_blocks_per_seq, int page_size);
tq_status tq_prefill_attention(tq_handle h, const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                               const int32_t *block_table, const int32_t *seq_lens, int batch, int q_tokens,
                               int num_q_heads, int num_kv_heads, int page_size, int max_blocks_per_seq,
                               int64_t num_blocks, float sm_scale, int splits, void *workspace, size_t ws_bytes,
                               uint16_t *out, void *stream);

/*
 * tq_decode_attention_static -- tq_decode_attention without a workspace, for
 * callers that cannot allocate device memory or own no memory to lend (code
 * inside another runtime's fixed memory budget, plug-ins in a host process that
 * owns every allocation, schedulers that must not touch an allocator on their
 * launch path).  The pages describe no such entry point; it is a deployment
 * convenience of this library.
 *
 * Same arguments and results as tq_decode_attention minus workspace/ws_bytes.
 * The scratch lives in one file-scope device array of TQ_STATIC_SCRATCH_BYTES
 * that every GPU loading the library holds until exit.  A call whose scratch
 * need (tq_decode_workspace_bytes) exceeds it returns TQ_ERR_UNSUPPORTED and
 * launches nothing.  Allocates nothing.  tq_init looks up the array's device
 * address (cudaGetSymbolAddress) in the context current when the handle is
 * created and keeps it in the handle, so use the handle in that context.  All
 * calls share the array: calls that overlap on the GPU (other streams, other
 * handles) race.
 */
#define TQ_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
tq_status tq_decode_attention_static(tq_handle h, const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                     const int32_t *block_table, const int32_t *seq_lens, int batch, int num_q_heads,
                                     int num_kv_heads, int page_size, int max_blocks_per_seq, int64_t num_blocks,
                                     float sm_scale, int splits, uint16_t *out, void *stream);

/*
 * tq_decode_attention_bf16 -- the bypass decode: the same split-K paged decode
 * (splits, workspace, combine, status bits and outputs as tq_decode_attention)
 * over an ordinary bf16 paged KV cache instead of the compressed one
 * (turbo-attn, "Two independently-usable pieces", item 2: a bypass loader that
 * reads plain bf16 pages in the same decode kernel).  It serves as the
 * bandwidth control of the compressed decode on identical shapes.
 *
 * k_pool, v_pool: device bf16 [num_blocks][num_kv_heads][page_size][head_dim]
 *   (head_dim from the handle), 16-byte aligned; token position t of sequence b
 *   is row t % page_size of block block_table[b][t / page_size].
 * The scores are sm_scale * <q, k> with exact bf16 products and fp32 sums; the
 * probabilities enter the value product as two bf16 terms (~16 bits).
 * Two launches on `stream` (decode, combine); the pools are read through tensor
 * maps encoded on the host for each call (no allocation, no synchronisation).
 */
tq_status tq_decode_attention_bf16(tq_handle h, const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                   const int32_t *block_table, const int32_t *seq_lens, int batch, int num_q_heads,
                                   int num_kv_heads, int page_size, int max_blocks_per_seq, int64_t num_blocks,
                                   float sm_scale, int splits, void *workspace, size_t ws_bytes, uint16_t *out,
                                   void *stream);

/*
 * tq_set_wait_limit -- the number of SM clock cycles a kernel of this handle
 * polls one barrier (a tensor-core completion, a page copy, a hand-off between
 * warps) before it gives up, sets TQ_DEVERR_TIMEOUT and winds its CTA down.
 * The default, TQ_DEFAULT_WAIT_LIMIT, is about one second at the maximum
 * clock; no correct run comes near it.  A limit of 0 makes every wait test its
 * barrier once without blocking and give up if it has not completed, so that
 * the error path can be exercised on purpose without any real hang (the waits
 * for work already in flight keep a fixed bound of their own).  Host-only;
 * affects later launches of this handle.
 */
#define TQ_DEFAULT_WAIT_LIMIT 2000000000LL
tq_status tq_set_wait_limit(tq_handle h, int64_t cycles);

/*
 * tq_get_status -- synchronises `stream`, returns the device status bits
 * accumulated since the last call (TQ_DEVERR_*), and clears them.
 */
tq_status tq_get_status(tq_handle h, uint32_t *device_error_bits, void *stream);

/*
 * tq_export_params -- host copies of the handle's tables (fp32, as used by the
 * kernels): Pi [d][d] row-major, S [d][d], centroids [2^k_bits] and
 * thresholds [2^k_bits - 1] (N(0,1) units).  Any pointer may be NULL.
 * Synchronous.
 */
tq_status tq_export_params(tq_handle h, float *Pi, float *S, float *centroids, float *thresholds);

/* Message describing the last non-OK status returned on this thread. */
const char *tq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
