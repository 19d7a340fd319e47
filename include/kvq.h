/*
 * kvq.h -- C ABI of a group-wise low-bit KV cache with fused dequant decode
 * attention, for one NVIDIA GB300 (sm_103a).
 *
 * The method (pages cited by short name, address and section):
 *  - [TurboQuant-3bit] "TurboQuant 3-bit KV-cache quantization"
 *    (dpshk.com/news/6341316): §2.1 KV footprint, §3.1 asymmetric min/max
 *    quantizer with offset = group minimum, §3.3 bit packing.
 *  - [KVQuant] "KVQuant: breaking the KV-cache memory wall"
 *    (cf-1.com/news/2306543): §2.2 per-channel keys, per-token values and
 *    the dense-and-sparse split with fp16 outliers, §3.3 outlier ratio ~1 %,
 *    §3.4 the decode-time kernel steps (quantize the new token, store codes
 *    and outliers, dequantize on read, attend).
 *  - [TurboQuant-mem] "TurboQuant: the KV cache as memory killer"
 *    (demingchina.com/news/57821): §2.3 group-wise scales and dequantization
 *    folded into the attention matmul, §1.3 / §4.2 decode is bound by the
 *    bytes of cache it reads.
 *  - [W4A8-FA3] (discosf.com/news/4854722) §2.4: per-head groups of 64
 *    positions, each with a scale and a zero point.
 *  - [NIAH-q8_0] (cf-1.com/news/5482713) §1.2: symmetric int8 codes with
 *    zero point 0; §2.2: only the newly written row is quantized.
 *
 * Conventions for every entry point:
 *  - Returns KVQ_OK or an error status; nothing aborts, traps or throws.
 *    Argument errors are detected on the host before any work is enqueued.
 *    kvq_last_error() returns a thread-local message for the last failure.
 *  - Every device call is asynchronous on `stream` (a cudaStream_t passed
 *    as void*; NULL = the legacy default stream).
 *  - The library never allocates device memory. The caller owns the cache
 *    buffer, every input, output and workspace; each must stay valid until
 *    the work enqueued on it has finished. Device pointers must be 16-byte
 *    aligned; the cache buffer 256-byte aligned.
 *  - fp16 means IEEE binary16. Layouts are C order (last index fastest).
 *  - One cache serves num_layers layers; a layer's lengths are uniform over
 *    the batch unless kvq_prefill_quantize_varlen gave each batch row its
 *    own. head_dim must be 128.
 *  - Calls that enqueue work (prefill, append, decode, status) need the
 *    device that holds the cache buffer to be current; otherwise they
 *    return KVQ_ERR_INVALID_ARG. Caches on several devices may be used from
 *    one process (kernel attributes are set per device).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, bad size, bad layer     */
  KVQ_ERR_UNSUPPORTED = 2,      /* valid but unsupported configuration              */
  KVQ_ERR_BUFFER_TOO_SMALL = 3, /* cache buffer or workspace smaller than required  */
  KVQ_ERR_CAPACITY = 4,         /* the layer would exceed max_seq tokens            */
  KVQ_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed             */
  KVQ_ERR_TIMEOUT = 6,          /* a bounded device-side wait gave up               */
  KVQ_ERR_DEVICE_STATUS = 7     /* the device status word reports an error          */
} kvq_status;

/* Grouping of one tensor (K or V).
 *  KVQ_SYM_PER_TOKEN    symmetric, zero point 0 ([NIAH-q8_0] §1.2): per token,
 *                       groups of `group` consecutive channels; one fp16 scale
 *                       = absmax / (2^(b-1) - 1); codes in [-(2^(b-1)-1), 2^(b-1)-1].
 *  KVQ_ASYM_PER_TOKEN   asymmetric ([TurboQuant-3bit] §3.1): per token, groups
 *                       of `group` channels; fp16 scale = (max-min)/(2^b-1) and
 *                       fp16 zero point = min; codes in [0, 2^b - 1].
 *  KVQ_ASYM_PER_CHANNEL asymmetric, per channel over `group` consecutive
 *                       tokens ([KVQuant] §2.2 item 1, [W4A8-FA3] §2.4); keys
 *                       only. The last (length mod group) keys stay in an fp16
 *                       residual until a whole block can be quantized.
 *  KVQ_CODEBOOK_PER_TOKEN  non-uniform 4-bit codes ([KVQuant] §2.2 item 2; the
 *                       4-bit minifloat of [TurboQuant-3bit] §3.3 is one such
 *                       codebook): per token, groups of `group` channels; one
 *                       fp16 scale = absmax / max_i |cb_i|, code = the index i
 *                       of the level cb_i nearest to x / s16 (fp32, lowest index
 *                       on ties), x_hat = cb[code] * s16. Keys and values both
 *                       use it or neither; no outliers.
 * In the integer modes code = clamp(rne((x - z16) / s16)) computed in fp32
 * from the stored fp16 scale s16 and zero point z16 (z16 = 0 for symmetric
 * groups); a group with s16 == 0 stores code 0 everywhere. */
typedef enum kvq_mode {
  KVQ_SYM_PER_TOKEN = 0,
  KVQ_ASYM_PER_TOKEN = 1,
  KVQ_ASYM_PER_CHANNEL = 2,
  KVQ_CODEBOOK_PER_TOKEN = 3
} kvq_mode;

typedef enum kvq_dtype { KVQ_F32 = 0, KVQ_F16 = 1 } kvq_dtype;

typedef struct kvq_config {
  int32_t num_layers;       /* >= 1                                                   */
  int32_t batch;            /* B >= 1                                                 */
  int32_t num_kv_heads;     /* H_kv >= 1                                              */
  int32_t head_dim;         /* D; must be 128                                         */
  int32_t max_seq;          /* token capacity per layer, >= 1                         */
  int32_t k_bits, v_bits;   /* 3, 4 or 8 (symmetric modes: 8 only)                    */
  int32_t k_mode, v_mode;   /* kvq_mode; v_mode may not be KVQ_ASYM_PER_CHANNEL        */
  int32_t k_group, v_group; /* per-token: 16, 32, 64 or 128 channels, and a multiple of
                               the codes per word (3-bit: 128 only);
                               per-channel: 64, 128 or 256 tokens                      */
  int32_t outliers_per_row; /* 0 = dense only; 1..8 fp16 outliers per (token, head)
                               row, chosen by |x| descending, ties to the lower channel
                               ([KVQuant] §2.2 item 3, §3.3)                             */
  uint16_t codebook[16];    /* fp16 bit patterns of the 16 levels of KVQ_CODEBOOK_PER_TOKEN
                               tensors (ignored otherwise); finite, max |level| > 0  */
  int32_t sink_tokens;      /* 0..64: the first sink_tokens tokens of every stream are
                               kept in fp16 for keys and values and take part in
                               attention as they are ("attention sinks", [KVQuant]
                               §4.1, which keeps the first 5-10); quantization (and
                               the per-channel key blocks) starts after them         */
} kvq_config;

/* Packed layout of one layer, for inspection (parity tests, checkpoints).
 * "Stream" = one (batch b, kv-head h) pair, index n = b * H_kv + h.
 * Every array below holds one slice per stream, `*_stream_bytes` apart.
 *  k_codes / v_codes : uint32 words [n][capacity][words_per_row]. Code j of a
 *      (token, head) row sits in word j / cpw at bit offset (j % cpw) * b,
 *      cpw = 32/b for b in {4, 8} and 10 for b = 3 (top two bits zero).
 *      Symmetric codes are b-bit two's complement.
 *  k_meta / v_meta : per-token modes: [n][capacity][D/group] entries;
 *      per-channel: [n][capacity/group][D] entries. An entry is one fp16
 *      scale (symmetric, 2 bytes) or an fp16 (scale, zero) pair (4 bytes,
 *      scale first).
 *  k_resid : fp16 [n][k_group][D] keys waiting for a whole block
 *      (per-channel keys only; the first k_resid_len rows are live).
 *  *_out_rowptr / *_out_col / *_out_val : CSR outliers per stream over the
 *      quantized rows: int32 row pointers [capacity + 4] (only the first
 *      rows+1 are meaningful), uint16 channel [capacity * k], fp16 value
 *      [capacity * k], entries of a row sorted by channel. The dense code at
 *      an outlier slot is 0. NULL when outliers_per_row == 0. */
typedef struct kvq_layout {
  int32_t capacity;           /* rows per stream (max_seq rounded up)              */
  int32_t length;             /* tokens cached in this layer (sinks included)      */
  int32_t k_quantized_len;    /* key rows held as codes                            */
  int32_t k_resid_len;        /* key rows held in the fp16 residual                */
  int32_t k_words_per_row, v_words_per_row;
  int32_t k_meta_entry_bytes, v_meta_entry_bytes;
  int64_t k_codes_stream_bytes, v_codes_stream_bytes;
  int64_t k_meta_stream_bytes, v_meta_stream_bytes;
  int64_t k_resid_stream_bytes;
  int64_t out_rowptr_stream_bytes, out_col_stream_bytes, out_val_stream_bytes;
  void* k_codes;
  void* k_meta;
  void* k_resid;
  void* v_codes;
  void* v_meta;
  void* k_out_rowptr;
  void* k_out_col;
  void* k_out_val;
  void* v_out_rowptr;
  void* v_out_col;
  void* v_out_val;
  /* attention sinks: fp16 keys and values [n][sink_tokens][D] each; the first
   * sink_len rows are live. The coded rows (k_quantized_len, k_resid_len and
   * the value rows, length - sink_len of them) start after the sinks. */
  int32_t sink_tokens;
  int32_t sink_len;
  int64_t sink_stream_bytes;
  void* k_sink;
  void* v_sink;
} kvq_layout;

typedef struct kvq_cache kvq_cache; /* opaque host-side handle */

/* Device bytes a cache of this configuration needs (all layers + a 256-byte
 * header holding the device status word). Host only. */
KVQ_API kvq_status kvq_cache_bytes(const kvq_config* cfg, size_t* bytes);

/* Validates `cfg`, lays the cache out in the caller-owned device buffer
 * `dev_buf` (256-byte aligned, at least kvq_cache_bytes bytes) and zeroes it
 * on `stream`. On success *out receives a new handle; all layers are empty.
 * The handle is a host object: use it from one host thread at a time. */
KVQ_API kvq_status kvq_cache_create(const kvq_config* cfg, void* dev_buf, size_t bytes,
                            void* stream, kvq_cache** out);

/* Per-layer code widths (mixed precision by layer: more bits for the layers
 * whose attention is most sensitive; [TurboQuant-mem] §5.3, [KVQuant] §4.2).
 * layer_bits: NULL (every layer uses cfg->k_bits / cfg->v_bits, as
 * kvq_cache_bytes / kvq_cache_create) or num_layers pairs (k_bits, v_bits),
 * layer by layer; each pair must be valid with cfg's modes and groups. The
 * array is read during the call only. Modes, groups, outliers and capacity
 * stay common to all layers; kvq_cache_get_layout reports each layer's own
 * word counts and strides. */
KVQ_API kvq_status kvq_cache_bytes_per_layer(const kvq_config* cfg, const int32_t* layer_bits,
                                             size_t* bytes);
KVQ_API kvq_status kvq_cache_create_per_layer(const kvq_config* cfg, const int32_t* layer_bits,
                                              void* dev_buf, size_t bytes, void* stream,
                                              kvq_cache** out);

/* Frees the host handle only; the device buffer stays the caller's. */
KVQ_API kvq_status kvq_cache_destroy(kvq_cache* cache);

/* Prefill: quantizes a whole prompt into layer `layer`, replacing what it
 * held. k, v: fp16 [B][H_kv][seq_len][D] device arrays. Per-token groups are
 * quantized row by row; per-channel keys are quantized in whole blocks of
 * k_group tokens and the last seq_len mod k_group keys are copied to the
 * fp16 residual; outliers (if enabled) are chosen per row before the group
 * statistics and left out of them. seq_len == 0 empties the layer.
 * Errors: KVQ_ERR_CAPACITY if seq_len > max_seq. */
KVQ_API kvq_status kvq_prefill_quantize(kvq_cache* cache, int32_t layer, const void* k,
                                const void* v, int32_t seq_len, void* stream);

/* Append: quantizes one new token per stream into layer `layer` (length += 1).
 * k, v: fp16 [B][H_kv][D]. The value row (and a per-token key row) is
 * quantized at once ([NIAH-q8_0] §2.2); a per-channel key joins the fp16
 * residual, and when the residual holds k_group keys the block is quantized
 * and the residual emptied. Codes already written are never requantized.
 * Errors: KVQ_ERR_CAPACITY when the layer is full. */
KVQ_API kvq_status kvq_append_quantize(kvq_cache* cache, int32_t layer, const void* k,
                               const void* v, void* stream);

/* Workspace bytes kvq_decode_attention needs for `num_q_heads` query heads
 * at any length up to max_seq (the split partials, and the attention over
 * the sink tokens when the cache keeps some). Host only. */
KVQ_API kvq_status kvq_decode_workspace_bytes(const kvq_cache* cache, int32_t num_q_heads,
                                      size_t* bytes);

/* Decode attention for one new query token per (batch, query head) over all
 * tokens cached in layer `layer` (codes, fp16 outliers and fp16 residual
 * keys), dequantizing in registers ([TurboQuant-mem] §2.3; [KVQuant] §3.4):
 *   e_t = softmax_scale * <q, k_hat_t>,  p = softmax(e),  o = sum_t p_t v_hat_t
 * q: fp16 [B][H_q][D]; out: [B][H_q][D] in out_dtype (kvq_dtype). Query head
 * h reads KV head h / (H_q / H_kv); H_q must be a multiple of H_kv with
 * H_q / H_kv in {1, 2, 4, 8}. workspace: device scratch of at least
 * kvq_decode_workspace_bytes bytes, not shared with concurrent calls.
 * Splits of the sequence are merged (log-sum-exp) inside the decode kernel by
 * the last CTA of each stream, which counts arrivals on per-layer counters
 * held in the cache buffer; every call leaves them at zero. Decode calls on
 * the same layer therefore must not overlap on the GPU (one stream per layer,
 * or ordered streams); calls on different layers may.
 * With 8 query heads per kv-head (per-channel keys, per-token values) the
 * decode is one persistent launch over all streams (stream-K: the key blocks
 * of all streams cut into one range per SM), otherwise one CTA per (split,
 * stream). When the layer holds sink tokens (cfg.sink_tokens), a first small
 * launch computes the attention over them and the decode merges it into its
 * output (log-sum-exp); with only sink tokens cached it writes the output.
 * Errors: KVQ_ERR_INVALID_ARG when the layer is empty;
 * KVQ_ERR_BUFFER_TOO_SMALL for a short workspace. */
KVQ_API kvq_status kvq_decode_attention(kvq_cache* cache, int32_t layer, const void* q,
                                int32_t num_q_heads, float softmax_scale, void* out,
                                int32_t out_dtype, void* workspace, size_t ws_bytes,
                                void* stream);

/* Decode attention exactly as kvq_decode_attention, but with no workspace
 * argument: for callers that cannot allocate device memory (host callbacks
 * and other code that may not call the CUDA allocator, plugins whose host
 * program owns every allocation, servers that forbid allocating after
 * start-up). The pages describe no counterpart of this call; it exists for
 * those callers only.
 * Scratch: the split partials go to a device array the library declares
 * itself, 4 MiB on every GPU that loads the library, kept until the process
 * exits. A call that would need more returns KVQ_ERR_BUFFER_TOO_SMALL (use
 * kvq_decode_attention with a workspace then). The first call on a device
 * looks up that array's address with the device current, so make that first
 * call before any stream capture. All calls share the one array and each
 * call overwrites it completely before reading it (nothing needs clearing);
 * calls that overlap on the GPU (several streams, or another thread) race on
 * it. q, out, num_q_heads, softmax_scale and out_dtype as in
 * kvq_decode_attention; the cache's device must be current. */
KVQ_API kvq_status kvq_decode_attention_static(kvq_cache* cache, int32_t layer, const void* q,
                                               int32_t num_q_heads, float softmax_scale,
                                               void* out, int32_t out_dtype, void* stream);

/* One decode step of every layer: for each layer l, the append of (k1[l],
 * v1[l]) and then the decode of q[l] into out[l], as kvq_append_quantize and
 * kvq_decode_attention (arrays of num_layers device pointers; one workspace
 * serves every layer's decode, in order on `stream`). With an `aux_stream`
 * (other than `stream`) the appends run there and layer l's decode waits
 * only for layer l's append, so the appends of later layers overlap the
 * decodes of earlier ones (the pages run quantization and attention on
 * separate streams: [NIAH-q8_0] §4.3); the appends start after everything
 * already enqueued on `stream`, and the decodes, on `stream`, end the step.
 * With aux_stream NULL everything runs on `stream` in order. Argument and
 * capacity errors of any layer are found before anything is enqueued. */
KVQ_API kvq_status kvq_decode_step(kvq_cache* cache, const void* const* q, const void* const* k1,
                                   const void* const* v1, int32_t num_q_heads, float softmax_scale,
                                   void* const* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                                   void* stream, void* aux_stream);

/* Prefill attention over the quantized cache: the queries of the last
 * `chunk` cached positions of layer `layer` (the chunk whose K/V were just
 * quantized into the cache, by kvq_prefill_quantize or appends) attend the
 * cache causally, as the decode reads it (fp16 sinks, codes with their
 * outliers, fp16 residual keys) -- the prefill whose time to first token the
 * pages measure ([NIAH-q8_0] §4.2) on the dequantized cache ([KVQuant] §3.4):
 *   query i (0 <= i < chunk) sits at position p_i = length - chunk + i;
 *   e_t = softmax_scale * <q_i, k_hat_t> for t = 0 .. p_i, p = softmax(e),
 *   o_i = sum_t p_t v_hat_t.
 * q: fp16 [B][chunk][H_q][D] (token-major, as a prefill's queries come);
 * out: [B][chunk][H_q][D] in out_dtype. Query head h reads KV head
 * h / (H_q / H_kv); H_q must be a multiple of H_kv. Every codec of the
 * cache is served. No workspace; one launch, one CTA per 128 (position,
 * head) rows of a stream. q and out must be 16-byte aligned; the cache's
 * device must be current.
 * With variable lengths (kvq_prefill_quantize_varlen) each batch row's
 * chunk is its own last `chunk` positions.
 * Errors: KVQ_ERR_INVALID_ARG for an empty layer, chunk outside
 * [1, length] (or above a batch row's length), NULL or misaligned pointers
 * or a bad out_dtype. */
KVQ_API kvq_status kvq_prefill_attention(kvq_cache* cache, int32_t layer, const void* q, int32_t chunk,
                                         int32_t num_q_heads, float softmax_scale, void* out,
                                         int32_t out_dtype, void* stream);

/* Variable per-sequence lengths in a batch. Prefills layer `layer` from a
 * padded batch (k, v as in kvq_prefill_quantize, seq_len rows per stream)
 * in which batch row b holds lens[b] tokens (host array of cfg.batch
 * entries, 1 <= lens[b] <= seq_len); the rows past lens[b] are ignored.
 * From then on every kvq_append_quantize of the layer appends each batch
 * row's new token at that row's own length, and kvq_decode_attention
 * attends each batch row's own tokens, until the next kvq_prefill_quantize
 * of the layer makes the lengths equal again. kvq_cache_length reports the
 * largest length; kvq_cache_seq_lengths the rows' own.
 * Every codec: per-token rows are coded on their own; per-channel key
 * blocks start at each row's first token (one prefill launch per batch row
 * then), so a row's fp16 key residual fills and flushes at its own appends.
 * Decodes of such a layer take the split-K kernels (not the stream-K one).
 * KVQ_ERR_UNSUPPORTED for caches with sink tokens and for more than 64
 * batch rows.
 * Errors: KVQ_ERR_INVALID_ARG for a NULL lens or a length out of range. */
KVQ_API kvq_status kvq_prefill_quantize_varlen(kvq_cache* cache, int32_t layer, const void* k, const void* v,
                                               int32_t seq_len, const int32_t* lens, void* stream);

/* The tokens of each batch row of layer `layer` (host array of cfg.batch
 * entries): the rows' own lengths after kvq_prefill_quantize_varlen, else
 * the layer's length for every row (host mirror, no sync). */
KVQ_API kvq_status kvq_cache_seq_lengths(const kvq_cache* cache, int32_t layer, int32_t* lens);

/* Forces the number of sequence splits of later decode calls (0 = automatic):
 * for the stream-K decode the number of persistent CTAs (at most one per SM),
 * otherwise the splits per stream. Results agree for every count up to
 * rounding; used by tests. */
KVQ_API kvq_status kvq_cache_set_decode_splits(kvq_cache* cache, int32_t splits);

/* Layout and device pointers of layer `layer` (host only, no sync). */
KVQ_API kvq_status kvq_cache_get_layout(const kvq_cache* cache, int32_t layer, kvq_layout* out);

/* Tokens currently cached in layer `layer` (host mirror, no sync). */
KVQ_API kvq_status kvq_cache_length(const kvq_cache* cache, int32_t layer, int32_t* len);

/* Synchronizes `stream`, reads the device status word and clears it.
 * Returns KVQ_OK, KVQ_ERR_TIMEOUT (a bounded device wait gave up) or
 * KVQ_ERR_DEVICE_STATUS (a device-side check failed); *word (optional)
 * receives the raw bits. After a nonzero word the split-merge counters of
 * every layer are cleared too (a decode that gave up may have left them set). */
KVQ_API kvq_status kvq_cache_status(kvq_cache* cache, void* stream, uint32_t* word);

/* Thread-local description of the last error ("" if none). */
KVQ_API const char* kvq_last_error(void);

/* Number of device kernels this process has enqueued through the library
 * (all caches, all threads), counted on the host at each successful
 * launch: prefill 1 (none when every token is a sink), append 1 (none for a
 * sink token: it is copied), decode 1 plus 1 for the sink attention when
 * the layer holds sink tokens (the split partials are merged by
 * the last CTA of each stream inside the decode kernel), except the generic
 * decode used for the rarer codec combinations (per-token keys with
 * outliers, sub-32-channel groups), which adds 1 for a combine launch;
 * each self-test call 1. Occupancy queries launch
 * nothing and are not counted. */
KVQ_API uint64_t kvq_kernel_launches(void);

/* Library version, major * 10000 + minor * 100 + patch. */
KVQ_API int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
