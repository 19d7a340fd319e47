// Internal structures shared by the host API and the kernel launchers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

#include "kvq.h"

namespace kvq {

constexpr int kHeadDim = 128;   // channels per (token, head) row
constexpr int kTile = 64;       // decode tile (tokens) and capacity granularity
constexpr int kMaxOutliers = 8; // per (token, head) row

// The dynamic shared memory a kernel may take beyond the default, set the
// first time the kernel launches on each device: the attribute belongs to the
// kernel's image in one device's context, so every device needs its own call.
// One instance per kernel; devices past ordinal 63 set it on every launch.
class SmemAttr {
 public:
  template <typename K>
  cudaError_t ensure(K* kern, size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done_.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && bit) done_.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }

 private:
  std::atomic<unsigned long long> done_{0};
};

// Device status bits (see kvq_cache_status).
constexpr uint32_t kStatusTimeout = 1u << 0;
constexpr uint32_t kStatusBadState = 1u << 1;

// One tensor (K or V) of one layer, device side.
struct TensorDev {
  int bits;
  int mode;             // kvq_mode
  int group;            // channels (per-token) or tokens (per-channel)
  int words;            // 32-bit words per (token, head) row
  int meta_bytes;       // 2 (symmetric scale) or 4 (scale, zero)
  uint32_t* codes;      // [n][cap][words]
  int64_t codes_sstride;  // words between streams
  unsigned char* meta;  // see kvq_layout
  int64_t meta_sstride;   // bytes between streams
  __half* resid;        // [n][group][D] (per-channel keys only)
  int64_t resid_sstride;  // halves between streams
  int32_t* rowptr;      // [n][cap + 4]
  int64_t rowptr_sstride; // ints between streams
  uint16_t* col;        // [n][cap * k]
  __half* val;          // [n][cap * k]
  int64_t out_sstride;  // entries between streams
};

struct LayerDev {
  TensorDev k, v;
  int n_streams;        // batch * num_kv_heads
  int num_kv_heads;
  int capacity;
  int outliers;         // per row
  uint32_t* status;
  uint32_t* counters;   // [n_streams] split-merge counters of the layer, zero between calls
  int in_rows;          // prefill: input rows per stream (0: the rows quantized)
  int sink_tokens;      // fp16 attention-sink tokens per stream (0: none)
  __half* sink_k;       // [n][sink_tokens][D]
  __half* sink_v;       // [n][sink_tokens][D]
  uint16_t codebook[16];  // fp16 levels of KVQ_CODEBOOK_PER_TOKEN tensors
  // The nearest-level decision as a search: y (= x / s16 in fp32) takes code
  // cb_code[p], p the number of entries of cb_thr (ascending, +inf padded)
  // that are <= y. Built on the host by codebook_search_table.
  float cb_thr[16];
  uint8_t cb_code[16];
};

// Builds cb_thr / cb_code from 16 fp16 levels: over the distinct levels in
// ascending order (equal levels, -0 and +0 among them, share the lowest
// index), cb_thr[k] is the smallest fp32 y that is coded as level k + 1
// rather than level k. Requires the distinct levels to be at least
// max|level| / 65536 apart, which check_config enforces.
void codebook_search_table(const uint16_t levels[16], float thr[16], uint8_t code[16]);

// Variable per-sequence lengths (per-token key codecs): each batch row b has
// its own number of cached tokens; kernels read it from a fixed array.
constexpr int kMaxVarlenBatch = 64;

// Per-batch-row positions of an append (on: the rows' own lengths).
struct VarPos {
  int on;
  int hkv;   // streams of a batch row: n / hkv is the row
  int rows;  // batch rows
  int32_t pos[kMaxVarlenBatch];
};

constexpr int kMaxSinkTokens = 64;

// Prefill attention over the cache (the last `chunk` positions' queries).
struct PrefillAttnArgs {
  const __half* q;  // [B][chunk][Hq][D]
  void* out;        // [B][chunk][Hq][D], fp32 or fp16
  int out_dtype;
  int num_q_heads;
  int G;            // query heads per kv-head
  int chunk;        // queries per stream: positions length - chunk .. length - 1
  int length;       // cached tokens (sinks included)
  int sink_len;     // fp16 sink tokens among them
  int kq;           // per-channel keys: coded rows held as codes (the rest are the fp16 residual)
  float scale_log2; // softmax scale * log2(e)
  int varlen;       // batch row b holds lens[b] tokens (its chunk: its last `chunk` positions)
  int32_t lens[kMaxVarlenBatch];
};
cudaError_t launch_prefill_attention(const LayerDev& L, const PrefillAttnArgs& a, cudaStream_t stream);

// Prefill of seq_len tokens: k, v fp16 [n][seq_len][D].
cudaError_t launch_prefill(const LayerDev& L, const __half* k, const __half* v, int seq_len,
                           cudaStream_t stream);

// Codebook tensors (KVQ_CODEBOOK_PER_TOKEN, keys and values): rows
// [row0, row0 + rows) of every stream from k, v fp16 [n][in_rows][D] (input
// row i is coded row row0 + i).
cudaError_t launch_codebook_rows(const LayerDev& L, const __half* k, const __half* v, int rows, int in_rows, const VarPos& vp,
                                 int row0, cudaStream_t stream);

// Append of one token at position pos (= length before the call): k1, v1
// fp16 [n][D].
cudaError_t launch_append(const LayerDev& L, const __half* k1, const __half* v1, int pos, const VarPos& vp,
                          cudaStream_t stream);

struct DecodeArgs {
  const __half* q;      // [B][Hq][D]
  const float* sink_part;  // [B*Hq][kSinkPartRow] attention over the sink tokens, or NULL
  void* out;            // [B][Hq][D]
  int out_dtype;
  int num_q_heads;
  int gqa;              // Hq / Hkv
  float scale_log2;     // softmax_scale * log2(e)
  int length;           // tokens cached
  int k_quant_len;      // key rows held as codes
  int splits;
  int tiles_per_split;
  float* part_o;        // [B*Hq][splits][D]
  float* part_ml;       // [B*Hq][splits][2]
  int* occupancy_out;   // non-null: report resident CTAs per SM of the kernel, launch nothing
  int varlen;           // lengths per batch row in lens (per-token keys only), else `length` for all
  int32_t lens[kMaxVarlenBatch];
};

cudaError_t launch_decode(const LayerDev& L, const DecodeArgs& a, cudaStream_t stream);

// Attention over the fp16 sink tokens of every (batch, query head) row: the
// unnormalised partial o[128], its running max m (log2 units) and sum l, for
// the decode kernels to merge into their output (part: [B*Hq][kSinkPartRow]);
// with `final_out` set, the normalised output itself (no other tokens).
constexpr int kSinkPartRow = 132;  // o[128], m, l, pad
cudaError_t launch_sink_attention(const LayerDev& L, const __half* q, int num_q_heads, float scale_log2,
                                  int sink_len, float* part, void* final_out, int out_dtype,
                                  cudaStream_t stream);

bool decode_supported(const LayerDev& L, int gqa);

// Stream-K decode (decode_pipe.cuh): per-channel keys and asymmetric per-token
// values at 3/3, 4/4, 4/8, 8/4 or 8/8 bits, 1, 2, 4 or 8 query heads per kv-head.
struct PipePlan {
  int ctas;             // persistent CTAs (at most one per SM)
  int jmax;             // partial rows per stream
  int cps;              // key blocks per stream
  long long n_chunks;   // key blocks of all streams
  int vex;              // empty virtual blocks after each stream (stream-switch cost)
  long long n_virtual;  // streams * (cps + vex)
  size_t ws_bytes;      // workspace: partials
};
bool decode_pipe_supported(const LayerDev& L, int gqa);
PipePlan plan_decode_pipe(const LayerDev& L, int len, int gqa, int sm_count, int ctas_override);
size_t decode_pipe_workspace_max(const LayerDev& L, int gqa, int sm_count);
cudaError_t launch_decode_pipe(const LayerDev& L, const DecodeArgs& a, const PipePlan& p, cudaStream_t stream);
bool decode_mha_supported(const LayerDev& L);
cudaError_t launch_decode_mha(const LayerDev& L, const DecodeArgs& a, cudaStream_t stream);
bool decode_gqa_supported(const LayerDev& L, int gqa);
cudaError_t launch_decode_gqa(const LayerDev& L, const DecodeArgs& a, cudaStream_t stream);

// Adds n to the process-wide count returned by kvq_kernel_launches().
void count_launches(int n);

// The device status word of a cache (its header), and the check that the
// current device holds the cache (KVQ_ERR_INVALID_ARG, with a message, if not).
uint32_t* cache_status_word(kvq_cache* h);
kvq_status cache_device_is_current(const kvq_cache* h);

// Replaces the thread-local message returned by kvq_last_error().
void set_error_message(const char* msg);

}  // namespace kvq
