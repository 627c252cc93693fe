// decode.cu — the decode loop: one query token per step, with a compressed row appended to k and
// kv whenever the step's position completes one.
//
// Source: "How I made DeepSeek 12x faster on a Mac Studio" (decode at long context is the wall the
// indexer work targets) and "How I turned one oversized DeepSeek optimization into three merged oMLX
// PRs", section "The three changes that merged" (one pooled row per `ratio` positions).  A row
// s is visible to position p iff (s+1)*ratio <= p+1, so position p needs floor((p+1)/ratio) rows:
// the loop appends the next staged rows before the step that first needs them.
//
// Per step the fused path runs with T = 1 (score -> top-k -> attention, the attention split over
// CTAs); the loop itself lives on the host and only issues launches, so a caller may capture a
// whole call into a CUDA graph once the library has been used on the device (first calls set
// kernel attributes).
#include <cuda_runtime.h>
#include <stdint.h>

#include "ds4x_internal.h"
#include "ds4x_ptx.cuh"

namespace ds4x {
namespace {

__global__ void fill_positions_kernel(int32_t* positions, int32_t pos0, int n) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) positions[i] = pos0 + i;
}

// Copies n rows of k_new / kv_new (row lengths k16 / kv16 in 16-byte units) to k / kv; the
// pointers already point at the first destination and source rows.
__global__ void append_rows_kernel(uint4* __restrict__ k, const uint4* __restrict__ k_new, int k16,
                                   uint4* __restrict__ kv, const uint4* __restrict__ kv_new, int kv16, int n) {
  pdl_wait();
  pdl_trigger();
  const int per_row = k16 + kv16;
  const int total = n * per_row;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int r = i / per_row, c = i - r * per_row;
    if (c < k16)
      k[(int64_t)r * k16 + c] = k_new[(int64_t)r * k16 + c];
    else
      kv[(int64_t)r * kv16 + (c - k16)] = kv_new[(int64_t)r * kv16 + (c - k16)];
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ds4x

using namespace ds4x;

extern "C" {

size_t ds4x_decode_workspace_bytes(int32_t capacity, int32_t k_top) {
  if (capacity <= 0 || k_top <= 0) return 0;
  return fused_workspace_bytes(1, capacity, k_top);
}

}  // extern "C"

namespace {
// The decode loop, with or without the raw window (raw: kv_raw rows are positions 0, 1, ...; the
// n_steps rows of kv_raw_new land at rows pos0 .. pos0 + n_steps - 1 before the first step, and
// step i attends to the raw rows of positions p - window + 1 .. p, p = pos0 + i).
int decode_impl(const void* q, const void* w, const void* q_attn, void* k, void* kv, ds4x_dtype kv_dtype,
                int32_t capacity, int32_t S0, const void* k_new, const void* kv_new, int32_t n_new, int32_t pos0,
                int32_t n_steps, int32_t H, int32_t D, int32_t ratio, int32_t k_top, int32_t Hq, int32_t Dkv,
                float scale, int32_t* positions, int32_t* indices, void* out, float* lse, void* workspace,
                size_t workspace_bytes, int32_t* S_final, void* stream, void* kv_raw, int32_t raw_capacity,
                const void* kv_raw_new, int32_t window) {
  call_begin();
  if (n_steps < 0 || capacity < 1 || S0 < 0 || S0 > capacity || n_new < 0 || H <= 0 || D <= 0 || Hq <= 0 ||
      Dkv <= 0 || ratio < 1 || k_top < 1 || pos0 < 0 || window < 0)
    return DS4X_ERR_INVALID;
  if ((int64_t)pos0 + n_steps > INT32_MAX) return DS4X_ERR_INVALID;
  if (kv_dtype != DS4X_F16 && kv_dtype != DS4X_BF16) return DS4X_ERR_INVALID;
  if (k_top > DS4X_MAX_KTOP || window > DS4X_MAX_WINDOW) return DS4X_ERR_UNSUPPORTED;
  if (!score_shape_supported(H, D) || !attn_shape_supported(Hq, Dkv)) return DS4X_ERR_UNSUPPORTED;
  const bool win = window > 0;
  if (win && (int64_t)pos0 + n_steps > raw_capacity) return DS4X_ERR_INVALID;  // every step's raw row has a place
  if (n_steps == 0) {
    if (S_final) *S_final = S0;
    return call_end(DS4X_OK);
  }
  if (!q || !w || !q_attn || !k || !kv || !positions || !indices || !out || !workspace ||
      (n_new > 0 && (!k_new || !kv_new)) || (win && (!kv_raw || !kv_raw_new)))
    return DS4X_ERR_INVALID;
  if (!aligned16(q) || !aligned16(w) || !aligned16(q_attn) || !aligned16(k) || !aligned16(kv) ||
      !aligned16(positions) || !aligned16(indices) || !aligned16(out) || (lse && !aligned16(lse)) ||
      !aligned16(workspace) || (k_new && !aligned16(k_new)) || (kv_new && !aligned16(kv_new)) ||
      (win && (!aligned16(kv_raw) || !aligned16(kv_raw_new))))
    return DS4X_ERR_INVALID;
  // per-step tensors must stay 16-byte aligned: w rows are H fp16, index rows k_top int32
  if ((H * 2) % 16 != 0 || (k_top * 4) % 16 != 0) return DS4X_ERR_UNSUPPORTED;
  if (workspace_bytes < fused_workspace_bytes(1, capacity, k_top, window)) return DS4X_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_pdl(fill_positions_kernel, dim3((n_steps + 255) / 256), dim3(256), 0, st, positions, pos0, n_steps) !=
      cudaSuccess)
    return DS4X_ERR_CUDA;
  count_launch();
  const int k16 = D * 2 / 16, kv16 = Dkv * 2 / 16;
  LocalWindow lw;
  if (win) {
    // every step's raw row into place at once: a step's window never reaches past its own position
    const int total = n_steps * kv16;
    const int blocks = (total + 255) / 256 < 256 ? (total + 255) / 256 : 256;
    if (launch_pdl(append_rows_kernel, dim3(blocks), dim3(256), 0, st, static_cast<uint4*>(kv_raw) + (int64_t)pos0 * kv16,
                   static_cast<const uint4*>(kv_raw_new), kv16, static_cast<uint4*>(nullptr),
                   static_cast<const uint4*>(nullptr), 0, n_steps) != cudaSuccess)
      return DS4X_ERR_CUDA;
    count_launch();
    lw.kv_local = kv_raw;
    lw.local_pos0 = 0;
    lw.L = pos0 + n_steps;
    lw.window = window;
  }
  const int bf16 = kv_dtype == DS4X_BF16 ? 1 : 0;
  int S = S0, appended = 0;
  for (int i = 0; i < n_steps; ++i) {
    const int64_t pos = (int64_t)pos0 + i;
    const int64_t need = (pos + 1) / ratio;  // rows this position may see
    if (need > S && appended < n_new && S < capacity) {
      int n = (int)((need - S) < (int64_t)(n_new - appended) ? (need - S) : (n_new - appended));
      if (n > capacity - S) n = capacity - S;
      const int total = n * (k16 + kv16);
      const int blocks = (total + 255) / 256 < 64 ? (total + 255) / 256 : 64;
      if (launch_pdl(append_rows_kernel, dim3(blocks), dim3(256), 0, st, static_cast<uint4*>(k) + (int64_t)S * k16,
                     static_cast<const uint4*>(k_new) + (int64_t)appended * k16, k16,
                     static_cast<uint4*>(kv) + (int64_t)S * kv16,
                     static_cast<const uint4*>(kv_new) + (int64_t)appended * kv16, kv16, n) != cudaSuccess)
        return DS4X_ERR_CUDA;
      count_launch();
      S += n;
      appended += n;
    }
    const int rc = run_index_and_attend(
        static_cast<const uint16_t*>(q) + (int64_t)i * H * D, static_cast<const uint16_t*>(w) + (int64_t)i * H, k,
        positions + i, static_cast<const uint16_t*>(q_attn) + (int64_t)i * Hq * Dkv, kv, bf16, 1, H, D, S, ratio,
        k_top, scale, indices + (int64_t)i * k_top, static_cast<uint16_t*>(out) + (int64_t)i * Hq * Dkv,
        lse ? lse + (int64_t)i * Hq : nullptr, workspace, workspace_bytes, st, lw);
    if (rc != DS4X_OK) return rc;
  }
  if (S_final) *S_final = S;
  return call_end(DS4X_OK);
}
}  // namespace

extern "C" {

int ds4x_decode(const void* q, const void* w, const void* q_attn, void* k, void* kv, ds4x_dtype kv_dtype,
                int32_t capacity, int32_t S0, const void* k_new, const void* kv_new, int32_t n_new, int32_t pos0,
                int32_t n_steps, int32_t H, int32_t D, int32_t ratio, int32_t k_top, int32_t Hq, int32_t Dkv,
                float scale, int32_t* positions, int32_t* indices, void* out, float* lse, void* workspace,
                size_t workspace_bytes, int32_t* S_final, void* stream) {
  return decode_impl(q, w, q_attn, k, kv, kv_dtype, capacity, S0, k_new, kv_new, n_new, pos0, n_steps, H, D, ratio,
                     k_top, Hq, Dkv, scale, positions, indices, out, lse, workspace, workspace_bytes, S_final, stream,
                     nullptr, 0, nullptr, 0);
}

size_t ds4x_decode_local_workspace_bytes(int32_t capacity, int32_t k_top, int32_t window) {
  if (capacity <= 0 || k_top <= 0 || window < 0 || window > DS4X_MAX_WINDOW) return 0;
  return fused_workspace_bytes(1, capacity, k_top, window);
}

int ds4x_decode_local(const void* q, const void* w, const void* q_attn, void* k, void* kv, ds4x_dtype kv_dtype,
                      int32_t capacity, int32_t S0, const void* k_new, const void* kv_new, int32_t n_new,
                      int32_t pos0, int32_t n_steps, int32_t H, int32_t D, int32_t ratio, int32_t k_top, int32_t Hq,
                      int32_t Dkv, float scale, void* kv_raw, int32_t raw_capacity, const void* kv_raw_new,
                      int32_t window, int32_t* positions, int32_t* indices, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, int32_t* S_final, void* stream) {
  return decode_impl(q, w, q_attn, k, kv, kv_dtype, capacity, S0, k_new, kv_new, n_new, pos0, n_steps, H, D, ratio,
                     k_top, Hq, Dkv, scale, positions, indices, out, lse, workspace, workspace_bytes, S_final, stream,
                     kv_raw, raw_capacity, kv_raw_new, window);
}

}  // extern "C"
