// ds4x_internal.h — declarations shared by the kernels' host launchers and the C ABI layer.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/ds4x.h"

namespace ds4x {

// Launches `kernel` on `st` with programmatic stream serialization (see pdl_wait / pdl_trigger in
// ds4x_ptx.cuh): the launch overlaps the tail of the previous kernel on the stream.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Number of SMs of the current device (cached per device).
int device_sm_count();
// Launches issued by the current call (reset by the ABI layer at entry).
void count_launch(int n = 1);
// Launch accounting of one C-ABI call: call_begin() at entry, call_end(rc) on return (records the
// count for ds4x_last_launch_count when rc == DS4X_OK and passes rc through).
void call_begin();
int call_end(int rc);
// Device address of the library's status word on the current device (bounded waits that give
// up record DS4X_ERR_TIMEOUT there).
int* device_status_ptr();
// The driver's cuTensorMapEncodeTiled, looked up once per process (nullptr if the driver lacks it).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();
// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device.  The
// attribute belongs to the device, so it is recorded per device (under a lock) and set again on
// each device that launches the kernel for the first time.
cudaError_t ensure_dynamic_smem_raw(const void* func, int bytes);
template <typename... KArgs>
inline cudaError_t ensure_dynamic_smem(void (*kernel)(KArgs...), int bytes) {
  return ensure_dynamic_smem_raw(reinterpret_cast<const void*>(kernel), bytes);
}

struct ScoreArgs {
  const void* q;             // [T, H, D] fp16
  const void* w;             // [T, H] fp16
  const void* k;             // [S, D] fp16
  const int32_t* positions;  // [T]
  float* scores;             // [T, ld]
  int64_t ld;
  int T, H, D, S, ratio;
  int skip_k_top;     // >0: tokens with n_vis <= skip_k_top need no scores (fused path)
  int write_masked;   // 1: write -inf on masked rows, including whole masked tiles
  uint32_t* zero_words = nullptr;  // fused path: words the kernel zeroes once the previous kernel is done
  int n_zero = 0;                  // (the top-k's barrier counters, so no memset sits between the launches)
  // T = 1: per CTA a slot of 4 words (16-byte aligned): the min and max ordered key of the visible
  // scores it wrote, the fourth largest of its threads' maximum keys (0 when fewer than four threads
  // saw a visible row), 0
  uint32_t* range_slots = nullptr;
};
int launch_score(const ScoreArgs& a, cudaStream_t stream);
bool score_shape_supported(int H, int D);
// CTAs the scorer launches for T tokens of H heads over S rows (the range slots it writes).
int score_grid(int T, int H, int S);

struct TopkArgs {
  const float* scores;
  int64_t ld;
  const int32_t* positions;
  int T, S, ratio, k_top;
  int32_t* indices;
  int32_t* counts;
  void* workspace;
  size_t workspace_bytes;
  int counters_zeroed = 0;  // 1: the workspace's barrier counters were zeroed by the kernel before (fused path)
  // range mode (one token whose row the cooperative kernel splits): the scorer zeroed the token's
  // scratch and wrote n_range_slots slots of 4 words at range_slots (see ScoreArgs::range_slots)
  const uint32_t* range_slots = nullptr;
  int n_range_slots = 0;
};
size_t topk_workspace_bytes(int T, int S, int k_top);
int launch_topk(const TopkArgs& a, cudaStream_t stream);
// Range mode applies (T = 1, the row split into slices, one cooperative launch, a scorer of at
// most the supported number of CTAs): then the scorer zeroes the first topk_range_zero_words words
// of the top-k scratch and writes its n_slots range slots at byte offset topk_range_slots_offset.
bool topk_range_mode(int T, int S, int k_top, int n_slots);
size_t topk_range_zero_words(int T, int S);
size_t topk_range_slots_offset(int T, int S);

// The raw sliding window joined to the pooled rows (window = 0 or L = 0: none): a token at p also
// attends to kv_local row r for every position a = local_pos0 + r with p - window < a <= p.
struct LocalWindow {
  const void* kv_local = nullptr;  // [L, Dkv], kv dtype
  int local_pos0 = 0, L = 0, window = 0;
  bool active() const { return window > 0 && L > 0; }
};

struct AttnArgs {
  const void* q_attn;  // [T, Hq, Dkv]
  const void* kv;      // [S, Dkv]
  int bf16;            // 1 = bf16, 0 = fp16
  const int32_t* indices;
  int T, Hq, Dkv, S, k_top;
  float scale;
  void* out;
  float* lse;
  void* partial;         // scratch for the split mode (NULL: every token on one CTA)
  size_t partial_bytes;  // used only when >= attn_partial_bytes(T, k_top, window)
  const int32_t* positions = nullptr;  // [T], read only with an active window
  LocalWindow local = {};
};
int launch_sparse_attn(const AttnArgs& a, cudaStream_t stream);
bool attn_shape_supported(int Hq, int Dkv);
// Scratch the split mode wants for T tokens on the current device (0: no split at this T).
size_t attn_partial_bytes(int T, int k_top, int window);

struct CompressArgs {
  const void* x;       // [T, D] raw rows
  const void* g;       // [T, D] gate logits
  const float* bias;   // [ratio, D]
  const void* fx;      // [n_frontier, D] held-over raw rows
  const void* fg;      // [n_frontier, D] held-over gate logits
  void* rows;          // [(n_frontier + T) / ratio, D]
  void* fx_out;        // [(n_frontier + T) % ratio, D]
  void* fg_out;
  int bf16;
  int T, D, ratio, n_frontier;
};
int launch_compress(const CompressArgs& a, cudaStream_t stream);

// The fused path (score -> top-k -> attention, Hq = 64, Dkv = 512) on validated arguments, and
// the workspace it needs: [scores T x S fp32 | top-k scratch | split-attention scratch].
size_t fused_workspace_bytes(int T, int S, int k_top, int window = 0);
int run_index_and_attend(const void* q, const void* w, const void* k, const int32_t* positions, const void* q_attn,
                         const void* kv, int bf16, int T, int H, int D, int S, int ratio, int k_top, float scale,
                         int32_t* indices, void* out, float* lse, void* workspace, size_t workspace_bytes,
                         cudaStream_t st, const LocalWindow& local = LocalWindow());

}  // namespace ds4x
