// ds4x_internal.h — declarations shared by the kernels' host launchers and the C ABI layer.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ds4x.h"

namespace ds4x {

// Number of SMs of the current device (cached per device).
int device_sm_count();
// Launches issued by the current call (reset by the ABI layer at entry).
void count_launch(int n = 1);
// Device address of the library's status word on the current device (bounded waits that give
// up record DS4X_ERR_TIMEOUT there).
int* device_status_ptr();

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
};
int launch_score(const ScoreArgs& a, cudaStream_t stream);
bool score_shape_supported(int H, int D);

struct TopkArgs {
  const float* scores;
  int64_t ld;
  const int32_t* positions;
  int T, S, ratio, k_top;
  int32_t* indices;
  int32_t* counts;
  void* workspace;
  size_t workspace_bytes;
};
size_t topk_workspace_bytes(int T, int S, int k_top);
int launch_topk(const TopkArgs& a, cudaStream_t stream);

struct AttnArgs {
  const void* q_attn;  // [T, Hq, Dkv]
  const void* kv;      // [S, Dkv]
  int bf16;            // 1 = bf16, 0 = fp16
  const int32_t* indices;
  int T, Hq, Dkv, S, k_top;
  float scale;
  void* out;
  float* lse;
};
int launch_sparse_attn(const AttnArgs& a, cudaStream_t stream);
bool attn_shape_supported(int Hq, int Dkv);

}  // namespace ds4x
