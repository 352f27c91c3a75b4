/*
 * h3gqa: bf16 causal grouped-query attention prefill for long sequences on
 * GB300 (sm_103a). C ABI.
 *
 * The operation. antirez/h3.c issue #47 ("Qwen layer 0 causal GQA failed:
 * causal attention sequence 10231 exceeds threadgroup memory"), sections
 * "Error" and "Suggested fix directions": the causal grouped-query attention
 * of the Qwen text encoder's prefill, whose Metal kernel keeps a query's whole
 * fp32 score row on chip and so refuses sequences above about 7700 tokens.
 * This library computes the same step with no bound on the sequence length
 * from on-chip memory:
 *
 *   for each packed sequence b (token rows [cu[b], cu[b+1])),
 *   for each query head h, key/value head g = h / (n_q_heads / n_kv_heads),
 *   for each query row i of b:
 *     z_j      = scale * <q[h,i,:], k[g,j,:]>    for keys j of b with j <= i
 *     o[h,i,:] = sum_j softmax_j(z) * v[g,j,:]
 *     lse[h,i] = ln sum_j exp(z_j)
 *
 * Layouts (all contiguous and head-major: head, then row, then dimension,
 * the attention order that the h3.c README describes in its "Profiling and
 * diagnostic paths" section):
 *   q, o : [n_q_heads][T][head_dim] bf16     T = cu_seqlens[n_seqs]
 *   k, v : [n_kv_heads][T][head_dim] bf16
 *   lse  : [n_q_heads][T] fp32 (natural log)
 *
 * Ownership and threading. The caller owns every buffer. Calls allocate no
 * device memory and keep no per-call state. Work is queued on `stream`, on
 * the calling thread's current CUDA device (ordinals 0-63), and the call
 * returns without waiting for it. Any number of host threads may call the
 * library at once; calls on different streams may run concurrently as long
 * as their outputs do not overlap. The first call on a device also does a
 * one-time setup that is not a stream operation (kernel attributes, the
 * driver's tensor-map entry point); after one such call, calls can be
 * captured into CUDA graphs and replayed.
 *
 * A device reset (cudaDeviceReset) drops the kernel attribute the setup
 * made; a launch that fails for that reason sets the device up again and is
 * retried once.
 *
 * Errors. Every entry point returns a status and never exits or aborts the
 * process. Argument checks run on the host before any CUDA call. A kernel
 * whose internal pipeline wait exceeds its time bound (2 s of wall clock)
 * stops, lets its in-flight copies finish, frees what it holds and raises a
 * device-side flag; h3gqa_sync_and_check reports it as H3GQA_ERR_TIMEOUT.
 * Rows of o and lse that such a kernel did not reach are left as they were.
 * The flag is one word per device shared by every call on it; for a result
 * that belongs to one call, pass h3gqa_options.status.
 *
 * Inputs must be finite. Keys a query must not see (later keys of its own
 * sequence, keys of the next packed sequence in the same 128-key tile) get
 * probability 0, but their value rows still enter the P.V product as 0 * v,
 * so an infinite or NaN value anywhere in v[g][0..T) can reach rows that do
 * not attend to it.
 */
#ifndef H3GQA_H_
#define H3GQA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; 0 is the legacy default stream. */
typedef struct CUstream_st *h3gqa_stream_t;

typedef enum {
    H3GQA_OK = 0,
    H3GQA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad cu_seqlens, bad scale, heads, options */
    H3GQA_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim != 128, too many sequences, T, device ordinal >= 64 */
    H3GQA_ERR_ARCH = 3,          /* current device is not compute capability 10.3 */
    H3GQA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    H3GQA_ERR_TIMEOUT = 5        /* a kernel gave up on a bounded internal wait */
} h3gqa_status;

/*
 * Causal GQA forward (the step of issue #47, "Error"; definition above).
 *
 *   q, k, v     device pointers, bf16, layouts above, 16-byte aligned.
 *   o           device pointer, bf16 [n_q_heads][T][head_dim], 16-byte aligned.
 *   lse         device pointer, fp32 [n_q_heads][T], 4-byte aligned.
 *   cu_seqlens  HOST pointer to n_seqs + 1 int32: cu[0] = 0, non-decreasing,
 *               cu[n_seqs] = T. Zero-length sequences are allowed. A single
 *               sequence of length S is {0, S}.
 *   n_seqs      number of packed sequences (>= 0; at most 1024 non-empty).
 *   n_q_heads, n_kv_heads   n_q_heads = G * n_kv_heads for any G >= 1
 *               (query head h reads KV head h / G; G = 1 is plain multi-head
 *               attention). Each 128-row MMA tile packs the query heads of
 *               one KV head: all G of them when G <= 128 (else the largest
 *               divisor of G that is <= 128) times floor(128 / heads) tokens,
 *               so when 128 is not a multiple of G a few of its rows go
 *               unused.
 *   head_dim    must be 128.
 *   scale       multiplies the logits; finite and > 0 (e.g. 1/sqrt(128)).
 *   stream      stream to queue the kernel on.
 *
 * Returns H3GQA_OK once the kernel is queued (T = 0 queues nothing).
 * Invalid arguments return before any CUDA call; an o that shares a byte
 * with q, k, v or lse is one (o is written while other work units of the
 * same call still read the inputs). There is no limit on the
 * sequence length other than T < 2^31 - 256 (TMA coordinates are int32).
 * Rows of o/lse are written only for tokens inside some sequence, i.e. all
 * of [0, T).
 */
h3gqa_status h3gqa_causal_fwd(const void *q, const void *k, const void *v,
                              void *o, float *lse,
                              const int32_t *cu_seqlens, int n_seqs,
                              int n_q_heads, int n_kv_heads, int head_dim,
                              float scale, h3gqa_stream_t stream);

/*
 * Options of h3gqa_attention_fwd: the bidirectional variant and the output
 * forms the out-projection consumes.
 *
 * causal = 0 is the same attention without the causal rule (every query of a
 * sequence sees every key of that sequence): the long bidirectional
 * attention of H3's DiT, whose 19316- and 34121-row forwards appear in
 * tgo-app-dev/vpipe issue #10, and which the h3.c README ("Metal 4 and
 * TensorOps paths") keeps on MPSGraph at those sizes.
 *
 * out_layout = H3GQA_LAYOUT_TOKEN_MAJOR writes o as [T][Hq][head_dim], the
 * row-major order the out-projection reads, instead of leaving it in
 * head-major order for a separate gather (h3.c README, "Profiling
 * and diagnostic paths", which gathers and int8-quantizes the SDPA output on
 * its way into the out-projection).
 *
 * out_int8 = 1 writes o as int8 codes with one fp32 scale per (token, head)
 * row of head_dim values: scale = max|o_row| / 127 (1 for an all-zero row),
 * code = round-to-nearest-even(o / scale) clamped to [-127, 127], so
 * o ~= code * scale. A row whose max|o_row| is at most 3.75e-37 (where
 * 127 / max|o_row| would overflow fp32) gets all-zero codes, its scale still
 * max|o_row| / 127. o then holds 1 byte per element (16-byte aligned) and
 * o_scale is laid out like o without the last dimension.
 */
typedef enum {
    H3GQA_LAYOUT_HEAD_MAJOR = 0,     /* [Hq][T][head_dim] */
    H3GQA_LAYOUT_TOKEN_MAJOR = 1     /* [T][Hq][head_dim] */
} h3gqa_layout;

typedef struct {
    int32_t causal;        /* 1: key j visible to query i iff j <= i; 0: every key of the sequence */
    int32_t out_layout;    /* h3gqa_layout of o (and of o_scale) */
    int32_t out_int8;      /* 0: o is bf16; 1: o is int8 codes plus o_scale */
    int32_t kv_head_begin; /* head shard: first KV head this call computes (0 = the first) */
    float *o_scale;        /* device fp32 [Hq][T] or [T][Hq], 4-byte aligned; required iff out_int8 */
    /* Q/K prologue (see below); all null = inputs are used as given. */
    const void *q_norm_weight;   /* device bf16 [head_dim], 16-byte aligned, or null */
    const void *k_norm_weight;   /* device bf16 [head_dim], 16-byte aligned, or null */
    const float *rope_cos;       /* device fp32 [T][head_dim/2], 16-byte aligned, or null */
    const float *rope_sin;       /* same shape; given together with rope_cos */
    void *k_out;                 /* device bf16 [Hkv][T][head_dim], 16-byte aligned: receives the
                                    prepared keys; required iff k is prepared; may equal k (then
                                    k is overwritten, and a second such call prepares it again),
                                    must not overlap q, v or part of k */
    float norm_eps;              /* added to the mean square; finite and >= 0 */
    int32_t kv_head_count;       /* head shard: KV heads this call computes; 0 = all from kv_head_begin */
    uint32_t *status;            /* optional device word, 4-byte aligned, zeroed by the caller: a
                                    kernel of this call that gives up on a bounded wait ORs a
                                    non-zero bit into it (read it once the stream has finished) */
} h3gqa_options;

/*
 * Head shard (kv_head_begin, kv_head_count). The KV heads, and with them
 * their query heads, are independent: a call may compute only KV heads
 * [kv_head_begin, kv_head_begin + kv_head_count) and the query heads that
 * read them, so that several calls (on one GPU or one per GPU) together
 * cover all heads with no exchange between them. Such a call writes only its
 * heads' rows of o, lse and o_scale (the buffers keep their full shapes) and
 * prepares only its heads' rows of k_out; every other row is left as it
 * was. 0 <= kv_head_begin < n_kv_heads and kv_head_begin + kv_head_count <=
 * n_kv_heads, else H3GQA_ERR_INVALID_ARG. The default (0, 0) is every head.
 */

/*
 * Q/K prologue (h3.c README, "Profiling and diagnostic paths" and
 * "Checkpoint layout and media pipeline": the fused Q/K normalisation and
 * rotary embedding that precedes attention). With a norm weight w, every
 * (head, token) row x of q (k) becomes x * rsqrt(mean(x^2) + norm_eps) * w;
 * with rope tables, then, for i < head_dim/2 and token t,
 *   (y_i, y_{i+D/2}) <- (y_i cos[t][i] - y_{i+D/2} sin[t][i],
 *                        y_{i+D/2} cos[t][i] + y_i sin[t][i])
 * (the rotate-half pairing; the tables carry any position scheme). The result
 * is rounded to bf16 once. The rotation applies to q and k; the norms to
 * whichever has a weight. q is transformed on the fly in the attention
 * kernel (q itself is not modified); k is transformed once into k_out, which
 * the attention then reads.
 */

/*
 * h3gqa_causal_fwd with options (NULL options = causal, head-major bf16 o,
 * i.e. exactly h3gqa_causal_fwd). Arguments and errors as for
 * h3gqa_causal_fwd; in addition an options value outside the ranges above,
 * out_int8 without a valid o_scale, a misaligned prologue pointer, rope_cos
 * without rope_sin (or the reverse), a prepared k without k_out, a k_out
 * that overlaps q, v or part of k, an o that overlaps k_out or o_scale, a
 * misaligned status word or a head shard outside [0, n_kv_heads) returns
 * H3GQA_ERR_INVALID_ARG. lse is always
 * [Hq][T].
 */
h3gqa_status h3gqa_attention_fwd(const void *q, const void *k, const void *v,
                                 void *o, float *lse,
                                 const int32_t *cu_seqlens, int n_seqs,
                                 int n_q_heads, int n_kv_heads, int head_dim,
                                 float scale, const h3gqa_options *options,
                                 h3gqa_stream_t stream);

/* Work plan of one h3gqa_causal_fwd call, computed on the host only (no GPU
 * needed). A unit is (sequence, block of 2 * floor(128 / heads_per_tile)
 * tokens, head group of heads_per_tile query heads); it owns two 128-row
 * query tiles (heads_per_tile heads x floor(128 / heads_per_tile) tokens
 * each) and visits every 128-key tile up to its last token. */
typedef struct {
    int64_t total_tokens;       /* T */
    int64_t n_units;            /* work units */
    int64_t n_kv_tiles;         /* sum over units of 128-key tiles visited */
    double tensor_flops;        /* FLOPs the MMAs execute: n_kv_tiles * 2 tiles * 2 GEMMs * 2*128^3 */
    double causal_flops;        /* needed FLOPs, 4*D per visible (query, key, head): causal sum_b 2*Hq*D*S_b*(S_b+1) */
    double metric_flops;        /* headline count: causal sum_b 2*Hq*D*S_b^2 */
    double exp2_count;          /* needed exponentials, one per visible pair: causal sum_b Hq*S_b*(S_b+1)/2 */
    double algorithmic_bytes;   /* q,k,v read once + o,lse written once */
    int32_t tokens_per_unit;    /* 2 * floor(128 / heads_per_tile) (256 / G for G a power of two) */
    int32_t max_kv_tiles;       /* most 128-key tiles any unit visits */
    int32_t heads_per_tile;     /* query heads packed in one tile: G if G <= 128 */
    int32_t rows_per_tile;      /* used MMA rows of a tile (128 when G divides 128) */
} h3gqa_plan;

/* Fills *plan for the given shape; same argument rules as h3gqa_causal_fwd
 * (pointers and scale are not involved). Returns the status that
 * h3gqa_causal_fwd would return for these sizes, without touching CUDA. */
h3gqa_status h3gqa_make_plan(const int32_t *cu_seqlens, int n_seqs,
                             int n_q_heads, int n_kv_heads, int head_dim,
                             h3gqa_plan *plan);

/* The plan of h3gqa_attention_fwd with the given causal flag. For causal = 0
 * every unit visits all key tiles of its sequence, causal_flops counts all
 * (query, key) pairs (4*Hq*D*S^2) and metric_flops equals it. */
h3gqa_status h3gqa_attention_plan(const int32_t *cu_seqlens, int n_seqs,
                                  int n_q_heads, int n_kv_heads, int head_dim,
                                  int32_t causal, h3gqa_plan *plan);

/* Waits for `stream`, then reads and clears the current device's timeout
 * flag. Returns H3GQA_ERR_TIMEOUT if any kernel of this library on this
 * device gave up on a bounded wait since the last check, H3GQA_ERR_CUDA if
 * the synchronisation failed, else H3GQA_OK. The flag is device-wide: the
 * timeout may belong to a call on another stream, and when two threads check
 * the same device at once the read and the clear of one may straddle the
 * other's, so one of them can miss a timeout. h3gqa_options.status gives
 * each call its own word instead. */
h3gqa_status h3gqa_sync_and_check(h3gqa_stream_t stream);

/* Static description of a status code. */
const char *h3gqa_status_string(h3gqa_status status);

/* Library version as 10000*major + 100*minor + patch. */
int h3gqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* H3GQA_H_ */
