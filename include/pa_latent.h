/*
 * pa_latent.h — C ABI of the paged LATENT (absorbed multi-head latent)
 * attention operator for NVIDIA GB300 (sm_103a).
 *
 * The operator is `com.microsoft::PagedAttention` v1 with
 * kv_cache_layout="LATENT" as the onnx-runtime-ep-cuda page
 * `src/kernels/paged_attention.rs` defines it (module doc, sections
 * "LATENT semantics" and "Capture safety"; input order in the PR #1978
 * review, "ORT v1.29 schema"). It has two phases, issued in this order on
 * one stream:
 *
 *   1. pa_latent_write   — partial RoPE on each new latent key row, then a
 *                          scatter into the paged cache at slot_mapping[t]
 *                          (slot -1 skips the token).
 *   2. pa_latent_decode  — causal attention of each query row (after
 *      pa_latent_prefill   partial RoPE) over the sequence's cached prefix,
 *                          read through block_table; one latent KV head of
 *                          head_size channels; V is its leading
 *                          v_head_size channels.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every buffer pointer is a DEVICE pointer owned by the caller. The
 *   library allocates nothing, never synchronises the host and never copies
 *   between host and device; each call only enqueues kernels on `stream`
 *   (a cudaStream_t passed as void*, NULL = the legacy default stream).
 *   Calls are therefore safe to record into a CUDA graph, provided the
 *   first call of each entry point on a device happened outside capture
 *   (that call configures kernel attributes once per device).
 * - Tensors are dense, row-major, with no padding between rows. Half
 *   precision tensors (query, key, key_cache, cos/sin, out) must be
 *   16-byte aligned; int32 tensors 4-byte aligned.
 * - Symbols: T = num_tokens (new tokens in the batch, all sequences),
 *   B = num_seqs, H = num_heads, hs = head_size, vhs = v_head_size,
 *   bs = block_size, rd = rotary_dim.
 * - Host-detectable errors return a status before anything is enqueued.
 *   Conditions only the device can see (an index read from device memory
 *   that is out of range) set a bit in the caller's int32 *err_flags
 *   (atomic OR, never cleared by the library) and the offending access is
 *   skipped: a cache row is not written, an output row is written as zeros.
 *   No kernel traps, asserts or waits without bound.
 */
#ifndef PA_LATENT_H
#define PA_LATENT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARGUMENT = 1, /* bad geometry, pointer, alignment or scale */
  PA_ERR_NOT_IMPLEMENTED = 2,  /* a valid mode this library does not run   */
  PA_ERR_CUDA = 3,             /* a CUDA runtime call failed               */
  PA_ERR_WORKSPACE = 4         /* workspace missing or smaller than needed */
} pa_status;

typedef enum pa_dtype {
  PA_DTYPE_F16 = 0,
  PA_DTYPE_BF16 = 1
} pa_dtype;

/* Element format of key_cache (pa_latent_params.cache_dtype). */
typedef enum pa_cache_dtype {
  PA_CACHE_DEFAULT = 0,  /* the query dtype (pa_latent_params.dtype)           */
  PA_CACHE_FP8_E4M3 = 1  /* OCP FP8 E4M3 ("e4m3fn") codes, one byte per channel,
                            with one dequantization scale k_scale for the cache */
} pa_cache_dtype;

/* Bits OR-ed into *err_flags by the device (see "Conventions"). */
#define PA_DEVERR_SLOT        0x01 /* slot_mapping[t] >= num_blocks*bs or < -1     */
#define PA_DEVERR_BLOCK       0x02 /* block_table entry read is not in [0, num_blocks) */
#define PA_DEVERR_POSITION    0x04 /* absolute position >= cos_rows (rotary on)    */
#define PA_DEVERR_CUMSEQ      0x08 /* cumseq not monotone, cumseq[0]!=0 or cumseq[B]!=T */
#define PA_DEVERR_DECODE_QLEN 0x10 /* pa_latent_decode saw a sequence with q_len != 1 */
#define PA_DEVERR_CONTEXT     0x20 /* past < 0 or context > max_blocks_per_seq*bs  */
#define PA_DEVERR_TIMEOUT     0x40 /* an internal pipeline wait exceeded its bound;
                                      the affected rows were not written          */
#define PA_DEVERR_RANGE       0x80 /* FP8 cache, bf16 query: a rotated query value
                                      exceeded 65504 (the fp16 operands of that
                                      read path) and was saturated to +-65504     */

/* pa_latent_params.flags */
#define PA_FLAG_PORTABLE 0x1 /* run the portable CUDA-core attention kernels even
                                where a tensor-core kernel exists (verification aid) */
/* PA_FLAG_AFTER_WRITE (read calls only; the write phase ignores it): the
 * caller promises that this call is enqueued on the same stream directly
 * after pa_latent_write of the same batch, with no other work in between.
 * The read kernel may then start while the write kernel runs: it loads the
 * query rows, sequence tables and rotary rows at once and waits for the
 * write only before its first cache read. Without the flag the read kernel
 * waits for all earlier work on the stream before touching any input. Set
 * it on the first read call after the write only (a second read call
 * follows a read, not the write). */
#define PA_FLAG_AFTER_WRITE 0x2
/* PA_FLAG_OWN_SLOTS (read calls, together with PA_FLAG_AFTER_WRITE): the
 * caller promises that every slot_mapping[t] >= 0 of the preceding write is
 * the cache row of token t's own position in its own sequence
 * (block_table[b][pos / bs] * bs + pos % bs), and that no sequence of this
 * read reads a row another sequence's token writes. The rows a sequence b
 * reads below its first new position past[b] are then untouched by the
 * write, and the read kernel loads them without waiting for the write
 * kernel; it waits only before the tiles at or after past[b]. */
#define PA_FLAG_OWN_SLOTS 0x4

/*
 * Operator attributes and cache geometry (the PagedAttention node
 * attributes num_heads, v_head_size, rotary_offset, do_rotary,
 * rotary_interleaved, softcap, local_window_size and scale; paged_attention.rs
 * PagedAttentionFactory::create and execute's geometry checks).
 */
typedef struct pa_latent_params {
  int32_t dtype;              /* pa_dtype of query, key, key_cache, cos/sin, out     */
  int32_t num_heads;          /* H >= 1 query heads (kv_num_heads is 1 in LATENT)    */
  int32_t head_size;          /* hs: latent row width, multiple of 16, 16..1024      */
  int32_t v_head_size;        /* vhs in 1..hs; 0 means hs                           */
  int32_t rotary_offset;      /* first rotary channel, multiple of 8                 */
  int32_t rotary_dim;         /* rd = 2 * cos_cache.dims[1]; 0 = no RoPE, else %16   */
  int32_t rotary_interleaved; /* 0 = half-split pairs, 1 = adjacent pairs            */
  int32_t cos_rows;           /* rows of cos/sin caches (largest position + 1)       */
  int32_t block_size;         /* bs: power of two >= 16                              */
  int32_t num_blocks;         /* physical blocks in key_cache                        */
  int32_t max_blocks_per_seq; /* columns of block_table                              */
  float scale;                /* > 0; 0 selects 1/sqrt(hs), allowed only if vhs==hs */
  float softcap;              /* <= 0: off; else s = softcap*tanh(s/softcap)         */
  int32_t local_window_size;  /* < 0: off; else keys with pos - j > window skipped   */
  int32_t flags;              /* PA_FLAG_*                                           */
  int32_t cache_dtype;        /* pa_cache_dtype of key_cache                         */
  float k_scale;              /* FP8 cache: a channel's value is code * k_scale; the
                                 write stores e4m3(v / k_scale) (f32 division,
                                 round to nearest even, saturated to +-448)          */
} pa_latent_params;

/* Checks the parameters alone (the first group of checks of every entry
 * point). Returns PA_OK, PA_ERR_INVALID_ARGUMENT or PA_ERR_NOT_IMPLEMENTED. */
pa_status pa_latent_validate(const pa_latent_params* p);

/*
 * Write phase — paged_attention.rs module doc "Write phase" and the device
 * function write_impl: for every token t with slot_mapping[t] >= 0, the row
 * key[t, :] gets partial RoPE on channels [rotary_offset, rotary_offset+rd)
 * at the token's absolute position past[b] + (t - cumseq[b]) (b: the
 * sequence with cumseq[b] <= t < cumseq[b+1]), is rounded to the dtype and
 * stored at key_cache[slot_mapping[t], :]. Other channels are copied bit
 * for bit; slot -1 skips the token.
 *
 *   key          [T, hs]                     input
 *   cos_cache    [cos_rows, rd/2]            input (ignored when rd == 0)
 *   sin_cache    [cos_rows, rd/2]            input (ignored when rd == 0)
 *   slot_mapping int32 [T]                   input, block*bs + offset or -1
 *   cumseq       int32 [B+1]                 input, cumseq[0]=0, cumseq[B]=T
 *   past         int32 [B]                   input, context length minus q_len
 *   key_cache    [num_blocks, bs, 1, hs]     updated in place
 *   err_flags    int32 [1]                   device error bits (may be NULL)
 * Two tokens naming the same slot race; the caller must not do that.
 */
pa_status pa_latent_write(const pa_latent_params* p, const void* key, int64_t num_tokens,
                          const void* cos_cache, const void* sin_cache,
                          const int32_t* slot_mapping, const int32_t* cumseq,
                          const int32_t* past, int32_t num_seqs, void* key_cache,
                          int32_t* err_flags, void* stream);

/*
 * Read phase for decode sequences — paged_attention.rs module doc "Read
 * phase" and the device function attn_impl: for every token t of the
 * sequences [seq_begin, seq_end) and every head h, q = RoPE(query[t,
 * h*hs:(h+1)*hs]) at the token's position pos; keys j = 0..pos (minus
 * those with pos - j > window when the window is on) are read from row
 * block_table[b, j/bs]*bs + j%bs of key_cache; s_j = scale * q.K_j, then
 * softcap*tanh(s_j/softcap) if softcap > 0; out[t, h*vhs:(h+1)*vhs] =
 * sum_j softmax(s)_j K_j[:vhs], rounded to the dtype.
 *
 * Arithmetic (default kernels): both products accumulate in f32 on the
 * tensor cores, the softmax runs in f32 (base 2, lazily rescaled), and the
 * probabilities are rounded to the dtype for the product with V. With head_size 576 one
 * token is handled by two SMs that each hold half of the latent channels
 * and exchange their f32 partial scores, so the split adds no rounding.
 *
 * Every sequence in [seq_begin, seq_end) must have exactly one new token
 * (cumseq[b+1]-cumseq[b] == 1); a sequence that does not sets
 * PA_DEVERR_DECODE_QLEN and its rows of `out` are left as they were.
 * Keys are split across SMs and merged with a log-sum-exp combine, which
 * uses the caller's workspace (pa_latent_workspace_size bytes, 256-byte
 * aligned, contents need not be initialised, must not be shared with a
 * concurrent call).
 *
 *   query        [T, H*hs]                   input
 *   key_cache    [num_blocks, bs, 1, hs]     input (written by pa_latent_write)
 *   block_table  int32 [B, max_blocks_per_seq] input, physical block ids
 *   out          [T, H*vhs]                  output rows of the covered tokens
 * Other arguments as for pa_latent_write.
 */
pa_status pa_latent_decode(const pa_latent_params* p, const void* query, int64_t num_tokens,
                           const void* key_cache, const void* cos_cache,
                           const void* sin_cache, const int32_t* cumseq,
                           const int32_t* past, const int32_t* block_table,
                           int32_t num_seqs, int32_t seq_begin, int32_t seq_end,
                           void* workspace, size_t workspace_bytes, void* out,
                           int32_t* err_flags, void* stream);

/*
 * Read phase for any sequences (same definition as pa_latent_decode, no
 * restriction on q_len): the chunked-prefill form of attn_impl, where the
 * new tokens of a sequence attend causally to each other through the cache
 * rows pa_latent_write stored for them. Arguments as for pa_latent_decode.
 */
pa_status pa_latent_prefill(const pa_latent_params* p, const void* query, int64_t num_tokens,
                            const void* key_cache, const void* cos_cache,
                            const void* sin_cache, const int32_t* cumseq,
                            const int32_t* past, const int32_t* block_table,
                            int32_t num_seqs, int32_t seq_begin, int32_t seq_end,
                            void* workspace, size_t workspace_bytes, void* out,
                            int32_t* err_flags, void* stream);

/*
 * Read phase for a whole mixed batch in one call: sequences [0,
 * num_decode_seqs) are decodes (one new token each, as pa_latent_decode)
 * and [num_decode_seqs, num_seqs) prefills (as pa_latent_prefill), the
 * serving batch the op receives. Where the single-CTA tensor-core kernel
 * runs (latent widths 64..256), both kinds of work are one grid: the decode
 * splits first, the prefill units after them on the SMs the decode tail
 * frees, then the split combine. Otherwise (576/512, PA_FLAG_PORTABLE) the
 * call is a pa_latent_decode followed by a pa_latent_prefill. Workspace as
 * pa_latent_decode (pa_latent_workspace_size for num_seqs sequences is
 * enough). PA_FLAG_AFTER_WRITE / PA_FLAG_OWN_SLOTS apply to this one call.
 */
pa_status pa_latent_mixed(const pa_latent_params* p, const void* query, int64_t num_tokens,
                          const void* key_cache, const void* cos_cache, const void* sin_cache,
                          const int32_t* cumseq, const int32_t* past,
                          const int32_t* block_table, int32_t num_seqs,
                          int32_t num_decode_seqs, void* workspace, size_t workspace_bytes,
                          void* out, int32_t* err_flags, void* stream);

/*
 * Allocation-free decode. The operator definition has no counterpart for
 * this call; it exists for callers that cannot allocate device memory and so
 * cannot hand pa_latent_decode a workspace: an execution provider whose host
 * framework owns every device allocation, a serving loop that must not touch
 * the allocator once running, or plain C code without a device allocator.
 *
 * Same arguments and results as pa_latent_decode, minus the workspace: the
 * split-KV partials go to a scratch array of 32 MiB in device global memory
 * that the library creates when it is loaded on a GPU and holds until the
 * process exits (on every GPU that loads it). A call whose sequence range
 * [seq_begin, seq_end) needs more than 32 MiB of workspace returns
 * PA_ERR_WORKSPACE: on the tensor-core kernels that is more than 127
 * sequences with head_size 576 / v_head_size 512, or more than 504 with
 * 192 / 128 (a larger batch can be decoded in ranges of that size). The call
 * allocates nothing.
 *
 * The first call on each device looks up the scratch address on that device
 * (with the device current); make that first call before any stream capture.
 * Every call shares the one scratch array and leaves its contents behind:
 * calls that overlap on the GPU (other streams, other threads) race on it,
 * so serialize them.
 */
pa_status pa_latent_decode_noalloc(const pa_latent_params* p, const void* query,
                                   int64_t num_tokens, const void* key_cache,
                                   const void* cos_cache, const void* sin_cache,
                                   const int32_t* cumseq, const int32_t* past,
                                   const int32_t* block_table, int32_t num_seqs,
                                   int32_t seq_begin, int32_t seq_end, void* out,
                                   int32_t* err_flags, void* stream);

/* Bytes of workspace pa_latent_decode / pa_latent_prefill need for these
 * parameters on the current device (0 if none). Host-only; returns 0 and
 * records an error message for invalid parameters. */
size_t pa_latent_workspace_size(const pa_latent_params* p, int32_t num_seqs,
                                int64_t num_tokens);

/* Which attention kernel family a decode (phase 0) or prefill (phase 1)
 * call with these parameters runs: 0 = portable CUDA-core kernels,
 * 1 = tcgen05/TMA tensor-core kernels, -1 = invalid parameters. */
int32_t pa_latent_kernel_family(const pa_latent_params* p, int32_t phase);

/* Static text for a status code. */
const char* pa_latent_status_string(pa_status s);

/* Message describing the last non-OK status returned on the calling thread
 * (empty string if none). */
const char* pa_latent_last_error(void);

/*
 * Paged streaming probe: a measurement aid, not part of the operator. It
 * reads every visible cache row of a decode batch (positions 0..past[b] of
 * sequence b, addressed through block_table exactly as the read phase
 * addresses them) with the tensor-core kernels' TMA boxes (64 channels x
 * min(block_size, tile_keys) rows) into a ring of `stages` shared-memory
 * stages of tile_keys rows, on num_SMs x ctas_per_sm CTAs, and does nothing
 * with the data. The caller times it (CUDA events on `stream`); the
 * visible rows x head_size x 2 bytes over that time is the ceiling of paged
 * TMA streaming that the decode kernels run against.
 *   p            geometry (dtype, head_size, block_size, num_blocks,
 *                max_blocks_per_seq are used; 16-bit caches only)
 *   key_cache    device, [num_blocks, block_size, 1, head_size], read only
 *   past         device int32 [num_seqs] (context of sequence b: past[b] + 1)
 *   block_table  device int32 [num_seqs, max_blocks_per_seq]
 *   num_seqs     1..4096; tile_keys 32, 64 or 128; stages 1..8;
 *   ctas_per_sm  1..4 (stages x tile must fit in 226 KB of shared memory)
 *   err_flags    device int32: PA_DEVERR_BLOCK / PA_DEVERR_CONTEXT as the
 *                read phase reports them
 * Returns PA_OK, PA_ERR_INVALID_ARGUMENT, PA_ERR_NOT_IMPLEMENTED (FP8 cache)
 * or PA_ERR_CUDA; enqueues one kernel and allocates nothing.
 */
pa_status pa_latent_gather_probe(const pa_latent_params* p, const void* key_cache,
                                 const int32_t* past, const int32_t* block_table,
                                 int32_t num_seqs, int32_t tile_keys, int32_t stages,
                                 int32_t ctas_per_sm, int32_t* err_flags, void* stream);

/* ======================================================================
 * SEPARATE layout — the op's other dense mode (kv_cache_layout="SEPARATE"):
 * grouped-query attention over separate key and value caches, with an
 * optional sink logit per query head and optional RMSNorm of the query and
 * key heads. The PR #1940 page lists it among the oracle's modes ("SEPARATE
 * (GQA, RoPE, softcap, local window, head_sink, q/k RMSNorm)", "num_heads %
 * kv_num_heads == 0"); the PR #1978 page gives the input order (value 2,
 * value_cache 4, head_sink 11, q_norm_weight 12, k_norm_weight 13). Where
 * the pages say no more, this library reads it as follows:
 *   - key_cache [num_blocks, bs, kvH, hs], value_cache [num_blocks, bs, kvH,
 *     vhs], slot-major like the LATENT cache (row slot*kvH + g);
 *   - query head h reads kv head g = h / (H / kvH);
 *   - RMSNorm: y = x / sqrt(mean(x^2) + rms_eps) * w over a head's hs
 *     channels, one weight vector [hs] for all heads, in f32, before RoPE;
 *   - head_sink[h] is a raw logit (no scale, no softcap) that joins the
 *     softmax denominator only: out = sum_j e^(s_j-m) V_j / (sum_j e^(s_j-m)
 *     + e^(z_h-m)), m = max(max_j s_j, z_h); values get no norm or RoPE.
 * Conventions (ownership, errors, err_flags, streams) as for the LATENT
 * entry points above. Kernels: tcgen05 tensor cores for head_size and
 * v_head_size in 64..256 and up to 128 query heads per kv head (others:
 * PA_ERR_NOT_IMPLEMENTED).
 * ====================================================================== */
typedef struct pa_separate_params {
  int32_t dtype;              /* pa_dtype of every half-precision tensor             */
  int32_t num_heads;          /* H query heads                                       */
  int32_t kv_num_heads;       /* kvH >= 1, dividing H                                */
  int32_t head_size;          /* hs, multiple of 16                                  */
  int32_t v_head_size;        /* vhs in 1..hs; 0 means hs                            */
  int32_t rotary_offset;      /* as pa_latent_params                                 */
  int32_t rotary_dim;
  int32_t rotary_interleaved;
  int32_t cos_rows;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  float scale;                /* 0 selects 1/sqrt(hs)                                */
  float softcap;
  int32_t local_window_size;
  float rms_eps;              /* RMSNorm epsilon (used when a norm weight is given)  */
  int32_t flags;              /* PA_FLAG_AFTER_WRITE / PA_FLAG_OWN_SLOTS             */
} pa_separate_params;

pa_status pa_separate_validate(const pa_separate_params* p);

/* Write phase: for every token t with slot_mapping[t] >= 0 and kv head g,
 *   key_cache[slot, g]   = RoPE(RMSNorm(key[t, g]) * k_norm_weight)  (norm only
 *                          when k_norm_weight is not NULL), rounded to the dtype;
 *   value_cache[slot, g] = value[t, g].
 *   key [T, kvH*hs], value [T, kvH*vhs], k_norm_weight [hs] or NULL; the rest
 *   as pa_latent_write. head_size <= 256 and v_head_size a multiple of 8. */
pa_status pa_separate_write(const pa_separate_params* p, const void* key, const void* value,
                            int64_t num_tokens, const void* cos_cache, const void* sin_cache,
                            const void* k_norm_weight, const int32_t* slot_mapping,
                            const int32_t* cumseq, const int32_t* past, int32_t num_seqs,
                            void* key_cache, void* value_cache, int32_t* err_flags,
                            void* stream);

/* Read phase (decode: one new token per sequence, split-KV + combine with
 * the caller's workspace; prefill: any sequences), as defined above.
 *   query [T, H*hs], q_norm_weight [hs] or NULL, head_sink [H] or NULL,
 *   out [T, H*vhs]; the rest as pa_latent_decode. */
pa_status pa_separate_decode(const pa_separate_params* p, const void* query, int64_t num_tokens,
                             const void* key_cache, const void* value_cache,
                             const void* cos_cache, const void* sin_cache,
                             const void* q_norm_weight, const void* head_sink,
                             const int32_t* cumseq, const int32_t* past,
                             const int32_t* block_table, int32_t num_seqs, int32_t seq_begin,
                             int32_t seq_end, void* workspace, size_t workspace_bytes, void* out,
                             int32_t* err_flags, void* stream);
pa_status pa_separate_prefill(const pa_separate_params* p, const void* query,
                              int64_t num_tokens, const void* key_cache, const void* value_cache,
                              const void* cos_cache, const void* sin_cache,
                              const void* q_norm_weight, const void* head_sink,
                              const int32_t* cumseq, const int32_t* past,
                              const int32_t* block_table, int32_t num_seqs, int32_t seq_begin,
                              int32_t seq_end, void* workspace, size_t workspace_bytes,
                              void* out, int32_t* err_flags, void* stream);

/* Workspace bytes pa_separate_decode needs for num_seqs sequences (prefill
 * needs none); 0 for invalid parameters. */
size_t pa_separate_workspace_size(const pa_separate_params* p, int32_t num_seqs,
                                  int64_t num_tokens);

#ifdef __cplusplus
}
#endif

#endif /* PA_LATENT_H */
