/*
 * tq.h -- C ABI of the quantized-KV decode-attention library (libtq.so).
 *
 * The library implements single-step (decode) attention over a TurboQuant-style
 * quantized KV cache and the encode/append that fills that cache, as hand-written
 * CUDA kernels for sm_103a (GB300).
 *
 * What the operations compute (sources: turboquant_plus "SMEM Pre-Dequant
 * Experiment", sections "What Was Changed" and "What Would Actually Work
 * (Hypotheses)"; mlxcel pull request #369 "route Turbo4Asym decode through
 * dequant-SDPA", sections Problem, Change and Result):
 *
 *   Each 128-dim K or V head vector x is stored as
 *     n16   = fp16(||x||_2)                          (round to nearest even)
 *     u     = Rot(x) / ||x||,  Rot(x) = H (s * x) / sqrt(128)
 *     idx_i = nearest entry of a symmetric b-bit codebook to u_i (ties: lower)
 *   with s a seeded +-1 sign vector and H the Sylvester Hadamard matrix.
 *   Attention over such a cache equals attention over the fully dequantized
 *   vectors Rot^-1(n16 * c[idx]); because Rot is orthogonal the library scores
 *   with Rot(q) against n16*c[idx], accumulates P.V in the rotated basis, and
 *   inverse-rotates only the [B, Hq, Tq, 128] output (the rotated-basis identity
 *   rotate(SDPA(q,k,v)) == SDPA(q,k,rotate(v)) of the mlxcel pull request).
 *
 * Conventions for every call:
 *   - Return 0 on success, a negative TQ_ERR_* code on failure.  Argument errors
 *     are detected on the host before any launch; nothing is launched then.
 *   - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *     void*, NULL = legacy default stream) and never synchronize, except
 *     tq_get_status (its context's latest stream) and tq_get_kernel_time.
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees them.  The library owns only the context (workspace, status
 *     word, cached tables), created lazily when *ctx == NULL and released by
 *     tq_free.  A context is bound to the device that was current when it was
 *     created.  Its workspace and counters serve one call at a time: calls on
 *     one context that could overlap on the GPU (different streams without an
 *     ordering between them) must be ordered by the caller or use separate
 *     contexts.
 *   - CUDA graphs: after one eager call on a context (which sizes its
 *     workspace), tq_encode_append and tq_decode_attention can be captured
 *     and replayed; device-side counters and the status word reset
 *     themselves, tensor maps are built at capture, and the decode grid is
 *     fixed by the max_len_hint given at capture (it must cover the lengths
 *     every replay sees).
 *   - Conditions only the GPU can see (a sequence whose append passes the
 *     capacity, a norm that overflows fp16, a sequence shorter than the query
 *     block, a pipeline wait that timed out) never trap: the kernels OR a bit
 *     into the context's device status word, read by tq_get_status.
 */
#ifndef TQ_H
#define TQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* error codes */
#define TQ_OK                0
#define TQ_ERR_INVALID_ARG  (-1)
#define TQ_ERR_UNSUPPORTED  (-2)
#define TQ_ERR_CAPACITY     (-3)
#define TQ_ERR_CUDA         (-4)
#define TQ_ERR_NOMEM        (-5)

/* modes: (K format, V format).  Turbo4Asym = fp16 K + 4-bit rotated V
 * (mlxcel pull request #369, Problem); turbo3 / turbo4 = K and V both 3- or
 * 4-bit rotated ("4-mag LUT" turbo3 of the smem-dequant experiment);
 * turbo3-asym = fp16 K + 3-bit rotated V (the memory-extremis mode of the
 * mlxcel advisor commit); turbo4k-3v = 4-bit K + 3-bit V, the remaining
 * pairing of the two codecs. */
#define TQ_TURBO4_ASYM  0
#define TQ_TURBO3       1
#define TQ_TURBO4       2
#define TQ_TURBO3_ASYM  3
#define TQ_TURBO4K_3V   4
/* turbo3 K and V in the centroid x norm table format (turboquant_plus
 * smem-dequant experiment, "What Would Actually Work" item 1): each 64-byte
 * record is the 48-byte 3-bit code layout followed by eight fp16 values
 * fp16(c_j * n16), j = 0..7 in ascending codebook order, in place of the norm
 * (k_norm and v_norm are not used and may be NULL). */
#define TQ_TURBO3_TABLE 5

/* device status bits (tq_get_status) */
#define TQ_STATUS_CAPACITY        1u  /* an append would pass `capacity`; that sequence was skipped */
#define TQ_STATUS_NORM_OVERFLOW   2u  /* a vector norm overflowed fp16; stored as +inf */
#define TQ_STATUS_SHORT_CONTEXT   4u  /* a query row saw no token (length < Tq); its output is 0 */
#define TQ_STATUS_PIPELINE_STALL  8u  /* a bounded in-kernel wait gave up; results are invalid */

typedef struct tq_ctx tq_ctx;

/*
 * The packed cache (caller-owned device memory).
 *
 *   k_data  TQ_TURBO4_ASYM / TQ_TURBO3_ASYM: fp16 [batch, num_kv_heads,
 *           capacity, 128], unrotated.  Otherwise: uint8 [batch, num_kv_heads,
 *           capacity, rb_k] packed codes, rb_k = tq_record_bytes(bits_k) (48
 *           for 3-bit, 64 for 4-bit; 64 for TQ_TURBO3_TABLE records).
 *   k_norm  fp16 [batch, num_kv_heads, capacity] (NULL for the fp16-K modes
 *           and TQ_TURBO3_TABLE).
 *   v_data  uint8 [batch, num_kv_heads, capacity, rb_v] packed codes.
 *   v_norm  fp16 [batch, num_kv_heads, capacity] (NULL for TQ_TURBO3_TABLE).
 *   lengths int32 [batch]: visible tokens per sequence; tq_encode_append
 *           advances it on the device.
 *   Code layout of one record (dimension d, code kappa = sign<<(b-1) | rank,
 *   sign = 1 for the negative half of the codebook, rank 0 = smallest |c|):
 *     4-bit: sixteen little-endian 32-bit words, word k = dims 8k..8k+7; bits
 *            4j..4j+2 = rank of dim 8k+j; bit 8j+7 = sign of dim 8k+j and bit
 *            8j+3 = sign of dim 8k+4+j (j = 0..3).
 *     3-bit: four 12-byte quarters; quarter q = dims 32q..32q+31 as three
 *            little-endian 32-bit words w0..w2 at bytes 12q+4k; bits 4j..4j+2
 *            of wk = kappa(32q+8k+j), bit 4j+3 of wk = bit k of kappa(32q+24+j).
 *   Every pointer must be 16-byte aligned and capacity a multiple of 16.
 *
 *   codebook_k / codebook_v: HOST pointers to 2^bits fp32 values, strictly
 *   ascending and exactly symmetric (c[j] == -c[2^bits-1-j]); codebook_k is
 *   ignored for TQ_TURBO4_ASYM.  tq_lloyd_max_codebook gives the standard one.
 *   rot_seed: seed of the sign vector (s_i = -1 iff bit 63 of the i-th
 *   splitmix64 output is set).  v_rescale: scalar applied to V (its effect on
 *   the output is a plain scale).
 */
typedef struct {
    int32_t mode;
    int32_t batch;
    int32_t num_kv_heads;
    int32_t head_dim;        /* must be 128 */
    int32_t capacity;        /* tokens per (batch, kv head) row; multiple of 16 */
    void *k_data;
    void *k_norm;
    void *v_data;
    void *v_norm;
    int32_t *lengths;
    const float *codebook_k;
    int32_t codebook_k_size;
    const float *codebook_v;
    int32_t codebook_v_size;
    uint64_t rot_seed;
    float v_rescale;
} tq_cache;

/*
 * Append t_new tokens per sequence: the cache update that precedes the
 * attention of a decode step (mlxcel pull request #369, Change: the decode
 * path updates the packed cache exactly as the plain update does, then
 * attends over the visible prefix).
 *   k_new, v_new: fp16 [batch, num_kv_heads, t_new, 128] device pointers.
 *   Token j of sequence b is written at position lengths[b] + j; afterwards
 *   lengths[b] += t_new.  A sequence with lengths[b] + t_new > capacity is left
 *   untouched and TQ_STATUS_CAPACITY is raised.  t_new == 0 is a no-op.
 *   More than 4096 vectors per stream (batch * num_kv_heads * t_new) take the
 *   tensor-core encode, which reads k_new / v_new through tensor maps built
 *   on the host in this call; fewer take a warp per vector.  Both give the
 *   same records except for elements within ~1e-6 of a decision midpoint.
 */
int tq_encode_append(tq_ctx **ctx, const tq_cache *cache, const void *k_new,
                     const void *v_new, int32_t t_new, void *stream);

/*
 * Decode attention over the visible cache (scores, online softmax, rotated-
 * basis P.V, split-K combine, inverse rotation of the output).
 *   q:   fp16 [batch, num_q_heads, tq, 128] device pointer.
 *   out: fp16 [batch, num_q_heads, tq, 128] device pointer.
 *   num_q_heads must be a multiple of num_kv_heads; q head h reads kv head
 *   h / (num_q_heads / num_kv_heads).  Query j (0 <= j < tq) of sequence b
 *   attends to tokens [0, lengths[b] - tq + j] (causal within the block).
 *   max_len_hint: an upper bound of every lengths[b] (sizes the split-K grid);
 *   it must not exceed capacity; tokens past it are not read.
 *   scale: softmax scale, 0 selects 1/sqrt(128).
 *   The call uses context workspace; it grows (cudaMalloc) when a larger
 *   problem arrives, so warm up before capturing a CUDA graph.
 */
int tq_decode_attention(tq_ctx **ctx, const tq_cache *cache, const void *q,
                        int32_t num_q_heads, int32_t tq, int32_t max_len_hint,
                        float scale, void *out, void *stream);

/*
 * Chunked-prefill attention: the same result as tq_decode_attention (query j
 * of the Tq block attends to tokens [0, lengths[b] - tq + j]) for blocks of
 * many queries, typically a prompt chunk just appended with tq_encode_append.
 * The scores and P.V run on the 5th-generation tensor cores (tcgen05, fp32
 * accumulators in tensor memory) over K/V tiles dequantised once per 128
 * query rows.  (The pages' second workload: the 8K-prefill leg of the mlxcel
 * measurement sweep, advisor commit of pull request #369.)
 *   Arguments and layouts as tq_decode_attention; any tq >= 1 and any group
 *   size up to 128 (num_q_heads / num_kv_heads); batch * num_kv_heads at most
 *   65535.  TQ_TURBO3_TABLE, and a K codebook whose entries are not all fp16
 *   values, are not supported (TQ_ERR_UNSUPPORTED).
 *   The call allocates nothing beyond the context created on first use.
 */
int tq_prefill_attention(tq_ctx **ctx, const tq_cache *cache, const void *q,
                         int32_t num_q_heads, int32_t tq, int32_t max_len_hint,
                         float scale, void *out, void *stream);

/*
 * Sparse-V decode: tq_decode_attention, except that a token whose softmax
 * weight is below tau adds nothing to the weighted sum of V (its weight still
 * counts in the normaliser).  This is the V skip of turboquant_plus
 * (smem-dequant-experiment.md, "What Would Actually Work" item 2: V dequant is
 * skipped for negligible weights), which the mlxcel ADR 0002 commit ("Turbo KV
 * split-dequant vs fused, sparse-V study") finds exact at tau = 1e-6 and
 * places inside a fused kernel.
 *   tau: finite, >= 0 (TQ_ERR_INVALID_ARG otherwise); 0 gives exactly the
 *        plain decode.
 * The kernel skips the V dequant and P.V of a 16-token tile when, for every
 * query row of the tile's row group, each token's weight taken against the
 * running maximum of its split is below tau.  That weight is never below the
 * final normalised one, so a skipped token is always one the definition
 * skips; a token the definition skips may still be kept.  Hence the result
 * differs from the full decode by at most the sum, over the tokens with weight
 * below tau, of weight * |v| per output element.
 */
int tq_decode_attention_sparse_v(tq_ctx **ctx, const tq_cache *cache, const void *q,
                                 int32_t num_q_heads, int32_t tq, int32_t max_len_hint,
                                 float scale, float tau, void *out, void *stream);

/*
 * No-allocation decode (this entry point has no counterpart on the pages; it
 * exists for callers that cannot allocate device memory on the decode path,
 * e.g. a server that owns all device memory through its own pools, or a
 * process under a hard memory budget, and that therefore cannot let
 * tq_decode_attention create a context and grow its workspace).
 *
 * Same computation and arguments as tq_decode_attention, without a context:
 * the split-K scratch lives in a fixed TQ_NOALLOC_SCRATCH_BYTES array that the
 * library's CUDA module reserves on every GPU where it is loaded, until the
 * process exits.  The call allocates nothing (no cudaMalloc/cudaFree).
 *   status: device pointer to a caller-owned uint32 into which the kernels OR
 *           TQ_STATUS_* bits (the caller clears it), or NULL to drop them.
 *   Returns TQ_ERR_CAPACITY when the problem needs more scratch than the
 *   array holds: one 8320-byte slot per decode CTA and one per (batch, kv
 *   head, row group) unit must fit (a row group is 8 query rows, or 16 when a
 *   kv head has more than 8); the CTA count is reduced to fit when possible.
 * The first call on a device, with that device current, looks up the array's
 * address (cudaGetSymbolAddress, once per device); make that first call before
 * any stream capture.  All calls share the one array and it keeps the last
 * call's contents: calls that overlap on the GPU (other streams, other host
 * threads) race and must be serialised by the caller.
 */
#define TQ_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int tq_decode_attention_noalloc(const tq_cache *cache, const void *q, int32_t num_q_heads,
                                int32_t tq, int32_t max_len_hint, float scale, void *out,
                                uint32_t *status, void *stream);

/* Self-test of the failure path, for tests: launches one CTA that waits, with
 * the kernels' own bounded wait and a limit of limit_us microseconds (1 ..
 * 1000000), on an mbarrier nothing arrives on.  The wait gives up and the
 * next tq_get_status reports TQ_STATUS_PIPELINE_STALL; the context stays
 * usable (no fault, no trap).  Allocates the context on first use. */
int tq_selftest_bounded_wait(tq_ctx **ctx, int32_t limit_us, void *stream);

/* Release a context (device memory included).  tq_free(NULL) is a no-op. */
void tq_free(tq_ctx *ctx);

/* Return the device status bits in *status and clear them.  The read is
 * ordered on the stream of the context's most recent call and waits for that
 * stream only (not the whole device); bits that work still running on other
 * streams sets later show in a later read.  Returns TQ_ERR_CUDA if the stream
 * reported an error. */
int tq_get_status(tq_ctx *ctx, uint32_t *status);

/* Host-only: the standard codebook: the Lloyd-Max levels of N(0, 1/128) with
 * 2^bits levels (bits in 1..4), iterated in double precision to a fixed point
 * and rounded to the nearest fp16 value (the half-precision centroid tables of
 * the smem-dequant experiment and of the mlxcel dequant), ascending, as fp32
 * values into out[0 .. 2^bits-1].  Any other strictly ascending, exactly
 * symmetric fp32 codebook is accepted by the calls too; one whose entries are
 * not all fp16 values takes a slower decode path that adds the entries'
 * fp16 rounding residuals to every score. */
int tq_lloyd_max_codebook(int32_t bits, float *out);

/* Host-only: bytes of one packed record: 48 (bits 3), 64 (bits 4), 256 (16 = fp16). */
int tq_record_bytes(int32_t bits);

/* Host-only: the decode grid tq_decode_attention would launch when every
 * sequence is max_len_hint long.  The grid is waves of CTAs (two or, for
 * large contexts, three for row groups of up to 8 rows; one for 16-row
 * groups) that split the
 * context's 32-token chunks over all (batch, kv head, row group) units evenly
 * (the split follows the actual lengths on the device):
 *   *num_splits   = number of decode CTAs;
 *   *split_tokens = tokens each CTA streams at that length (a multiple of 32). */
int tq_plan_splits(int32_t mode, int32_t batch, int32_t num_kv_heads,
                   int32_t rows_per_kv_head, int32_t max_len_hint,
                   int32_t *split_tokens, int32_t *num_splits);

/* The sparse-V decode's tile counts since the last read, then cleared:
 * *skipped = 16-token tiles (of one row group) whose V work was skipped,
 * *judged = tiles judged.  Ordered on the stream of the context's latest
 * call; waits for that stream only.  (32-bit device counters: read them at
 * least every 2^32 tiles.) */
int tq_get_sparse_v_tiles(tq_ctx *ctx, uint64_t *skipped, uint64_t *judged);

/* Benchmark hook: when enabled, tq_decode_attention (and its sparse-V form)
 * records CUDA events around its main (split-K) kernel and
 * tq_prefill_attention around its kernel; tq_get_kernel_time synchronizes on
 * the last event and returns the summed milliseconds and the number of timed
 * launches since the last read (and resets both). */
int tq_set_kernel_timing(tq_ctx *ctx, int32_t enable);
int tq_get_kernel_time(tq_ctx *ctx, float *ms_total, int32_t *launches);

/* Human-readable text of an error code. */
const char *tq_error_string(int32_t code);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
