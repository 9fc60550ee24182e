/*
 * qs.h -- C ABI of libqs: the QuantSpec hierarchical quantized KV cache hot
 * path on one NVIDIA GB300 (sm_103a).
 *
 * What it computes (sources named by page title and section):
 *  - "QuantSpec: Self-Speculative Decoding with Hierarchical Quantized KV
 *    Cache" (Pith review), "What carries the argument": each key or value group
 *    of size G is stored once as an upper INT4 tensor C_U and a lower INT4
 *    residual C_L sharing one scale and zero-point, C_INT8 = 2^4 C_U + C_L;
 *    the draft pass dequantizes C_U only, the target (verify) pass the INT8
 *    reconstruction; a double full-precision buffer of two halves of G tokens
 *    takes new tokens, rejected speculative tokens are dropped before
 *    quantization, and a half is quantized once every G decoding steps.
 *  - same page, Figure 7 caption and Appendix D: keys are quantized per
 *    channel (a group = G tokens of one channel), values per token (a group =
 *    G channels of one token); asymmetric quantization.
 *  - same page, Appendix E: the buffer design is compatible with Flash
 *    Decoding (split-KV partial softmax plus a log-sum-exp combine).
 *  - "QuantSpec Guide: Self-Speculative Decoding & Quantized KV", sections
 *    "1. Hierarchical Two-Level Quantization with Bit-Sharing" (draft loads only
 *    the upper 4 bits from HBM) and the quantizer listing (min/max over the
 *    group, 255 levels, round, clamp, upper = q >> 4, lower = q & 15, draft
 *    reconstruction at the nibble midpoint).
 *
 * Rounding convention QS-RN-v1 (this library's reading; the pages print no
 * rule for the stored scale): for a group x_0..x_{G-1} of fp16 values
 *   r = fp32(max) - fp32(min), s = r == 0 ? 0 : fp16_round_up(r / 255.0f),
 *   z = min (a zero minimum is stored as +0),
 *   q_i = s == 0 ? 0 : clamp(rne((fp32(x_i) - fp32(z)) / fp32(s)), 0, 255)
 * (every fp32 step IEEE round-to-nearest-even), C_U = q >> 4, C_L = q & 15,
 *   verify: deq = s * (16 C_U + C_L) + z,   draft: deq = s * (16 C_U + 8) + z.
 *
 * Ownership: every array is caller-owned device memory; the library never
 * allocates and keeps no global state, except the fixed scratch array behind
 * qs_attn_decode_static_ws (see there).  Every call that launches work is
 * asynchronous on the given stream, except qs_get_errors, which synchronizes
 * it.  Calls on different caches may run concurrently; calls on one cache
 * must be ordered by the caller (one stream).
 *
 * Host-side errors are returned as qs_status before anything is launched.
 * Preconditions that depend on device-resident counters (overflow, rollback
 * beyond the pending tokens, flush without G committed tokens, capacity,
 * fewer buffered tokens than queries) are checked on the device: the
 * operation becomes a no-op for that sequence and a bit is set in the
 * sequence's error word (QS_DEV_*), read back with qs_get_errors.  No kernel
 * of this library traps or waits without a time limit.
 *
 * v1 supports D = G = 128 only (all workloads of the pages use head_dim 128
 * and G = 128); other values return QS_ERR_UNSUPPORTED.
 */
#ifndef QS_H_
#define QS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers */
typedef struct CUstream_st *qs_stream_t;

typedef enum {
  QS_OK = 0,
  QS_ERR_ARG = 1,         /* null pointer, bad count or mode */
  QS_ERR_SHAPE = 2,       /* inconsistent sizes */
  QS_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned */
  QS_ERR_CUDA = 4,        /* a CUDA call or launch failed */
  QS_ERR_UNSUPPORTED = 5, /* D or G other than 128 */
  QS_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required */
  QS_ERR_TOO_LARGE = 7    /* problem needs more scratch than qs_attn_decode_static_ws has */
} qs_status;

typedef enum {
  QS_DRAFT_UPPER4 = 0, /* the draft: keys/values from the top upper_bits bits of
                          the code only, at the middle of the codes sharing them:
                          s * (16 C_U + 8) + z (upper_bits 4), or
                          s * (64 C_U2 + 32) + z (upper_bits 2) */
  QS_VERIFY_INT8 = 1   /* keys/values from C_U and C_L: s * (16 C_U + C_L) + z */
} qs_mode;

/* Device-side error bits, one error word per sequence. */
enum {
  QS_DEV_OVERFLOW = 1,           /* append would exceed the 2G buffer */
  QS_DEV_OVER_ROLLBACK = 2,      /* n_drop < 0 or > pending tokens */
  QS_DEV_FLUSH_UNCOMMITTED = 4,  /* flush with fewer than G committed tokens */
  QS_DEV_CAPACITY = 8,           /* flush with n_groups == cap_groups */
  QS_DEV_NQ_GT_FILL = 16,        /* attention with n_q > buffered tokens */
  QS_DEV_TIMEOUT = 32,           /* a pipeline wait ran out of time (never
                                    expected; the call's results are invalid) */
  QS_DEV_PREFILL = 64            /* prefill of a non-empty cache, or a prompt
                                    length outside [0, T] */
};

/* Per-sequence counters: int32 state[B][QS_STATE_WORDS]. */
enum {
  QS_ST_N_GROUPS = 0,  /* quantized groups; quantized tokens Tq = n_groups * G */
  QS_ST_FILL = 1,      /* tokens in the fp16 buffer (committed + pending) */
  QS_ST_PENDING = 2,   /* speculative tokens at the end of the buffer */
  QS_ST_HALF_BASE = 3, /* 0/1: buffer half that holds logical token 0 */
  QS_ST_ERR = 4,       /* QS_DEV_* bits */
  QS_ST_TICKET = 5,    /* internal arrival counter; must start at 0 */
  QS_STATE_WORDS = 8
};

/* Rows of the per-group metadata block (fp16 [4][128] per group). */
enum { QS_META_K_SCALE = 0, QS_META_K_ZERO = 1, QS_META_V_SCALE = 2, QS_META_V_ZERO = 3 };

/*
 * The cache: one struct of device pointers, all caller-owned, 16-byte
 * aligned.  Logical buffer token i of sequence b lives in slot
 * (half_base * G + i) mod 2G.  Sizes for each array: qs_cache_bytes.
 *
 *  upper_bits  4 or 2: how many top bits of C_INT8 the draft reads (below).
 *  k_upper, k_lower  uint8 [B][H][cap][G tokens][D/2]: C_U / C_L of the keys,
 *      token-major; byte i of a token row holds channel 2i in bits 0-3 and
 *      channel 2i+1 in bits 4-7 (64 bytes per token).
 *  v_upper, v_lower  uint8 [B][H][cap][G/32][D][16]: C_U / C_L of the values,
 *      per group in four quarters of 32 tokens, channel-major inside a
 *      quarter: 16 bytes = 32 nibbles per (quarter u, channel d).  Nibble
 *      position p (byte p/2, bits 0-3 for even p, 4-7 for odd p) holds token
 *        32u + 16*((p>>1)&1) + 8*(p&1) + 2*(p>>3) + ((p>>2)&1)
 *      of the group.  This fixed permutation lets one 32-bit shared-memory
 *      word per lane feed tensor-core fragments without byte shuffles.
 *  meta  fp16 [B][H][cap][4][128]: per group, rows QS_META_*: key scale and
 *      zero per channel, value scale and zero per token, each row in a fixed
 *      order matched to the tensor-core fragments:
 *        key rows: position p holds channel
 *          32*((p>>3)&3) + 8*(p>>5) + 2*((p>>2)&1) + ((p>>1)&1) + 4*(p&1);
 *        value rows: position p holds token
 *          32*(p>>5) + ((p>>2)&7) + 16*((p>>1)&1) + 8*(p&1).
 *  With upper_bits = 2 (C_INT8 = 64 C_U2 + 16 M2 + C_L, the draft reading
 *      the top two bits only; source: Pith review page, "Editorial
 *      extensions", "Reading between the lines", which leaves drafts from
 *      other numbers of leading bits open) the 8 KB of k_upper / v_upper per group hold
 *      the same nibbles C_U = 4 C_U2 + M2 re-packed: regard the 4-bit plane
 *      above as a sequence of 32-bit words w_0, w_1, ... (8 nibbles each,
 *      nibble j in bits 4j..4j+3).  Word k of the first 4 KB (the C_U2 plane)
 *      holds, in nibble position j, C_U2 of w_2k's nibble j in bits 4j..4j+1
 *      and C_U2 of w_2k+1's nibble j in bits 4j+2..4j+3; word k of the second
 *      4 KB (the M2 plane) holds M2 the same way.  k_lower, v_lower and meta
 *      are the same for both.
 *  buf_k, buf_v  fp16 [B][H][2G][D]: the double full-precision buffer.
 *  state  int32 [B][QS_STATE_WORDS]: counters above; zero it (qs_state_reset)
 *      before first use.
 *  arrive  int32 [B][H]: arrival counters of qs_attn_decode (the CTA that
 *      finishes a head last merges its split partials).  Internal: zeroed by
 *      qs_state_reset and left at zero by every completed attention call, so
 *      at most one attention call may run on a cache at a time.
 */
typedef struct {
  int32_t B, H, D, G, cap_groups;
  int32_t upper_bits;     /* 4 or 2 */
  uint8_t *k_upper, *k_lower, *v_upper, *v_lower;
  uint16_t *meta;         /* fp16 bits */
  uint16_t *buf_k, *buf_v; /* fp16 bits */
  int32_t *state;
  int32_t *arrive;
} qs_cache;

typedef struct {
  size_t k_upper, k_lower, v_upper, v_lower, meta, buf_k, buf_v, state, arrive;
} qs_cache_bytes_t;

/* Byte size of every cache array for the given dimensions.  Pure host
 * function.  Errors: QS_ERR_ARG (null out, non-positive sizes),
 * QS_ERR_UNSUPPORTED (D or G != 128).  The sizes follow the layout above;
 * the pages fix the planes' contents (Pith review page, "What carries the
 * argument": C_U and C_L per group with a shared scale and zero-point; the
 * double buffer of two halves of G tokens), not a memory layout. */
qs_status qs_cache_bytes(int32_t B, int32_t H, int32_t D, int32_t G, int32_t cap_groups,
                         qs_cache_bytes_t *out);

/* Zero every sequence's counters (empty cache) and the attention arrival
 * counters.  Asynchronous memsets.  No counterpart on the pages: it is this
 * library's initialisation of its device-resident bookkeeping. */
qs_status qs_state_reset(const qs_cache *c, qs_stream_t stream);

/* Append n_new tokens per sequence to the fp16 buffer as pending tokens.
 * k_new, v_new: fp16 [B][H][n_new][D] device arrays, 1 <= n_new <= 2G.
 * Per sequence: needs fill + n_new <= 2G, else QS_DEV_OVERFLOW and no-op.
 * Source: Pith review page, "What carries the argument" (new tokens enter
 * the double full-precision buffer). */
qs_status qs_buffer_append(const qs_cache *c, const uint16_t *k_new, const uint16_t *v_new,
                           int32_t n_new, qs_stream_t stream);

/* Drop the last n_drop[b] pending tokens of each sequence and commit the
 * rest (pending becomes 0).  d_n_drop: int32 [B] device array.  n_drop < 0 or
 * > pending gives QS_DEV_OVER_ROLLBACK and a no-op.  The quantized cache is
 * never touched.  Source: Pith review page, "What carries the argument"
 * (rejected tokens dropped before quantization); "QuantSpec Guide",
 * "Zero-Overhead Rollback". */
qs_status qs_buffer_rollback(const qs_cache *c, const int32_t *d_n_drop, qs_stream_t stream);

/* d_mask[b] = 1 if appending n_next more tokens would exceed 2G, else 0.
 * d_mask: uint8 [B] device array, written by the call (caller-owned).
 * Feed it to qs_quantize_flush before the append.  Host errors: QS_ERR_ARG
 * (null mask, negative n_next).  Source: Pith review page, "What
 * carries the argument": a buffer half is quantized once every G decoding
 * steps.  The pages do not say at which point of a round; this library
 * flushes right before an append that would overflow the 2G buffer, when the
 * oldest half is fully committed as long as n_next <= G / 2. */
qs_status qs_need_flush(const qs_cache *c, int32_t n_next, uint8_t *d_mask, qs_stream_t stream);

/* Quantize-on-flush.  For every sequence with d_mask[b] != 0 (all when
 * d_mask is NULL): quantize the oldest buffer half (logical tokens 0..G-1,
 * which must be committed: fill - pending >= G) into group n_groups --
 * keys per channel over the G tokens, values per token over the D channels,
 * convention QS-RN-v1 -- then n_groups += 1, half_base ^= 1, fill -= G.
 * Failing preconditions give QS_DEV_FLUSH_UNCOMMITTED or QS_DEV_CAPACITY and a
 * no-op.  Source: Pith review page, "What carries the argument", Figure 7 and
 * Appendix D; "QuantSpec Guide", "Periodic Group Quantization". */
qs_status qs_quantize_flush(const qs_cache *c, const uint8_t *d_mask, qs_stream_t stream);

/* qs_need_flush(n_next) followed by qs_quantize_flush with that mask, in one
 * launch and without the mask array: every sequence whose buffer cannot take
 * n_next more tokens (fill + n_next > 2G) quantizes its oldest half, with the
 * same preconditions, results and error bits as qs_quantize_flush.  Host
 * errors: QS_ERR_ARG (n_next outside 0..2G).  Source: as qs_need_flush and
 * qs_quantize_flush. */
qs_status qs_quantize_flush_due(const qs_cache *c, int32_t n_next, qs_stream_t stream);

/* Bulk prefill: fill empty caches from a prompt in one call.  k, v: fp16
 * [B][H][T][D] device arrays (token t of head h of sequence b at
 * [b][h][t]); d_len: int32 [B] device array, the prompt length of each
 * sequence.  With L = d_len[b]: the first n_groups * G tokens become groups
 * 0..n_groups-1 (G tokens each, in order, convention QS-RN-v1 as in
 * qs_quantize_flush) and the remaining fill tokens become committed buffer
 * tokens 0..fill-1 in ring slots 0..fill-1, where
 *   n_groups = L > 2G ? ceil((L - 2G) / G) : 0,   fill = L - G * n_groups,
 * pending = 0 and half_base = 0.  These are the groups and the logical buffer
 * that appending the prompt in pieces of at most G tokens (qs_buffer_append,
 * commit, qs_quantize_flush whenever qs_need_flush asks) would leave.
 * Per sequence: a cache that is not empty (n_groups, fill or pending non-zero)
 * or L outside [0, T] gives QS_DEV_PREFILL, n_groups > cap_groups gives
 * QS_DEV_CAPACITY; either leaves the sequence unchanged.  Host errors:
 * QS_ERR_ARG (null pointers, T < 0 or T > 2^26), QS_ERR_ALIGN.  Ownership:
 * all arrays are the caller's; the call only reads k, v and d_len.
 * Source: "QuantSpec Guide", core architectural blueprint (the prefill
 * context is quantized once into the hierarchical cache); Pith review page,
 * "What carries the argument" (groups of G tokens, two buffer halves). */
qs_status qs_prefill(const qs_cache *c, const uint16_t *k, const uint16_t *v, int32_t T,
                     const int32_t *d_len, qs_stream_t stream);

/* Speculative-sampling acceptance for B sequences with gamma draft tokens
 * each (1 <= gamma <= 64), vocabulary V; all arrays are device arrays, read
 * or written only by this call, 4-byte aligned:
 *   p        float [B][gamma+1][V]  target probabilities at the gamma + 1
 *                                   positions (the last one for the bonus)
 *   q        float [B][gamma][V]    draft probabilities the draft tokens were
 *                                   sampled from
 *   draft    int32 [B][gamma]       the draft tokens
 *   u        float [B][gamma]       uniforms in [0, 1), one per draft token
 *   e        float [B][V]           Exp(1) variates for the one draw per
 *                                   sequence (positive)
 *   n_accept int32 [B] (out)        accepted draft tokens a
 *   token    int32 [B] (out)        the token emitted after them, or -1 if its
 *                                   weights are all zero
 *   n_drop   int32 [B] (out)        gamma - a: pass it to qs_buffer_rollback
 * Draft token i is accepted when u_i * q_i(x_i) < p_i(x_i) in fp32, i.e. with
 * probability min(1, p_i(x_i) / q_i(x_i)); the first rejection at position a
 * ends the round and the token is drawn from max(0, p_a - q_a) (from p_a if
 * that is zero everywhere); after gamma acceptances it is drawn from p_gamma.
 * A draft token outside [0, V) is rejected.  Draws: the index of the smallest
 * e_x / w_x over w_x > 0 (ties to the smaller index), which is distributed as
 * w / sum(w).  One cluster of 8 CTAs per sequence splits the vocabulary.
 * Errors: QS_ERR_ARG (null pointer, B outside 1..65535, gamma outside 1..64,
 * V < 1), QS_ERR_ALIGN.  Source: Pith review page, referee report on
 * Algorithm 1 (VERIFY / CORRECT as rejection sampling with acceptance
 * min(1, p/q) and residual (p - q)_+); "QuantSpec Guide", "The
 * Self-Speculative Verification Loop". */
qs_status qs_spec_accept(const float *p, const float *q, const int32_t *draft, const float *u,
                         const float *e, int32_t B, int32_t gamma, int32_t V, int32_t *n_accept,
                         int32_t *token, int32_t *n_drop, qs_stream_t stream);

/* Bytes of device workspace qs_attn_decode needs for n_q queries (1..8) on
 * the current device.  Pure host function (reads device attributes).  The
 * workspace holds the split-KV partials of Flash Decoding (Pith review page,
 * Appendix E); its size is this implementation's, not the pages'. */
qs_status qs_attn_workspace_size(const qs_cache *c, int32_t n_q, size_t *bytes);

/* Split-KV decode attention over the quantized groups and the fp16 buffer.
 *   q      fp16 [B][H][n_q][D] device, 1 <= n_q <= 8; query j of sequence b sits
 *          at buffer position fill - n_q + j and sees every token at or before
 *          it (all quantized tokens plus a causal prefix of the buffer);
 *   mode   QS_DRAFT_UPPER4 (reads the upper planes only: C_U, or with
 *          upper_bits 2 their C_U2 half) or QS_VERIFY_INT8;
 *   softmax_scale  multiplies q . k (usually 1/sqrt(D));
 *   out    fp16 [B][H][n_q][D] device: softmax-weighted sum of the values;
 *   lse    float [B][H][n_q] device or NULL: natural log of the softmax
 *          denominator of the scaled scores;
 *   workspace  device scratch of at least qs_attn_workspace_size bytes, 16-byte
 *          aligned; it holds split partials and is not read across calls.
 * Sequences with n_q > fill get QS_DEV_NQ_GT_FILL, zero output, lse = -inf.
 * One kernel launch: a persistent split-KV pass over a balanced partition of
 * all (sequence, head, group) units, whose log-sum-exp merge of the splits
 * runs in the same kernel.  Errors: QS_ERR_ARG (null q/out, n_q outside 1..8,
 * bad mode, non-positive or non-finite scale), QS_ERR_ALIGN, QS_ERR_WORKSPACE,
 * QS_ERR_CUDA.  Sources: "QuantSpec Guide", "Hierarchical Two-Level
 * Quantization with Bit-Sharing"; Pith review page, "What carries the
 * argument" and Appendix E (Flash Decoding). */
qs_status qs_attn_decode(const qs_cache *c, qs_mode mode, const uint16_t *q, int32_t n_q,
                         float softmax_scale, uint16_t *out, float *lse, void *workspace,
                         size_t workspace_bytes, qs_stream_t stream);

/* Grouped-query variant: `group` query heads share each KV head (query head
 * h*group + i attends KV head h; group = 1 is qs_attn_decode).  q and out are
 * fp16 [B][H*group][n_q][D], lse float [B][H*group][n_q]; group * n_q <= 24
 * query rows per KV head.  Every KV byte is read once for all the rows of its
 * group (the 5-query verify of a 4-way group is a 20-row tile).  Workspace:
 * qs_attn_workspace_size_gqa.  Errors as qs_attn_decode, plus QS_ERR_ARG for
 * group < 1 or group * n_q > 24.  Source: the pages name Llama-3.1-8B
 * ("QuantSpec Guide", speedup table); its grouped-query head layout is taken
 * from the model family (32 query heads on 8 KV heads), not from the pages. */
qs_status qs_attn_workspace_size_gqa(const qs_cache *c, int32_t n_q, int32_t group,
                                     size_t *bytes);
qs_status qs_attn_decode_gqa(const qs_cache *c, qs_mode mode, const uint16_t *q, int32_t n_q,
                             int32_t group, float softmax_scale, uint16_t *out, float *lse,
                             void *workspace, size_t workspace_bytes, qs_stream_t stream);

/* qs_buffer_append followed by qs_attn_decode_gqa, in one launch: n_new
 * tokens k_new, v_new (fp16 [B][H][n_new][D] device arrays, 16-byte aligned,
 * 1 <= n_new <= 2G; H counts KV heads) enter each sequence's buffer as pending
 * tokens, then the queries attend over the buffer including them -- the
 * speculative round's "append a draft token, then draft" and "append the
 * gamma + 1 target tokens, then verify" without a launch in between.  The
 * results, the buffer, the counters and the error words equal those of the
 * two separate calls: a sequence whose buffer cannot take the tokens gets
 * QS_DEV_OVERFLOW and attends over its buffer as it was.  The attention reads
 * the new rows from k_new / v_new while the same launch writes them into the
 * ring, so k_new and v_new must stay unchanged until the call completes.
 * Arguments, workspace and errors otherwise as qs_attn_decode_gqa (group = 1
 * is qs_attn_decode), plus QS_ERR_ARG for null k_new / v_new or n_new outside
 * 1..2G.  Sources: Pith review page, "What carries the argument" (new tokens
 * enter the double full-precision buffer; both passes attend over it);
 * "QuantSpec Guide", "The Self-Speculative Verification Loop". */
qs_status qs_attn_decode_append(const qs_cache *c, qs_mode mode, const uint16_t *k_new,
                                const uint16_t *v_new, int32_t n_new, const uint16_t *q,
                                int32_t n_q, int32_t group, float softmax_scale, uint16_t *out,
                                float *lse, void *workspace, size_t workspace_bytes,
                                qs_stream_t stream);

/* Size of the fixed scratch array behind qs_attn_decode_static_ws. */
#define QS_STATIC_WS_BYTES (8u << 20)

/* qs_attn_decode for callers that cannot allocate device memory.  No
 * counterpart on the pages: it exists for callers that cannot allocate
 * device memory -- a serving process whose device memory is fixed up front,
 * a foreign runtime without a CUDA allocator, a plug-in handed only its input
 * and output buffers.  Same arguments, results and errors as qs_attn_decode,
 * minus the workspace: the split partials go to a fixed array of
 * QS_STATIC_WS_BYTES (8 MiB) inside this library, which every GPU that loads
 * libqs holds until the process exits.  The caller still passes q, out and
 * lse.  The call allocates nothing (no cudaMalloc or cudaFree).  Limits and
 * sharing:
 *  - a problem whose qs_attn_workspace_size exceeds QS_STATIC_WS_BYTES returns
 *    QS_ERR_TOO_LARGE before launching anything;
 *  - the first call on a device looks up the array's device address (with
 *    that device current) and caches it together with the identity of the
 *    current CUDA context; make that first call before any stream capture.
 *    A call under another context of the same device (after cudaDeviceReset,
 *    or a context made current through the driver API) looks the address up
 *    again, so make its first call before capture too;
 *  - every call on a device uses the same array: calls that overlap on the
 *    GPU (other streams, other threads) race and corrupt each other's
 *    results; order them on one stream.  The array needs no clearing: every
 *    value a call reads is written earlier in the same call. */
qs_status qs_attn_decode_static_ws(const qs_cache *c, qs_mode mode, const uint16_t *q,
                                   int32_t n_q, float softmax_scale, uint16_t *out, float *lse,
                                   qs_stream_t stream);

/* Copy every sequence's error word to h_err (int32 [B], host memory) and
 * clear them on the device.  Synchronizes the stream.  No counterpart on the
 * pages: it reports the device-side precondition failures of the calls above. */
qs_status qs_get_errors(const qs_cache *c, int32_t *h_err, qs_stream_t stream);

/* Human-readable name of a status code (static string). */
const char *qs_status_string(qs_status s);

#ifdef __cplusplus
}
#endif
#endif /* QS_H_ */
