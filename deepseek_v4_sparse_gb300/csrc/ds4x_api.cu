// ds4x_api.cu — the C ABI of libds4x.so (declared in include/ds4x.h).
//
// Host-side argument validation happens here, before anything is launched; the kernels and
// their launchers live in score_tcgen05.cu, topk_stream.cu and sparse_mqa.cu.  The library
// allocates no device memory: the fused entry carves the caller's workspace.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "ds4x_internal.h"
#include "ds4x_ptx.cuh"

namespace ds4x {

// Status word written by bounded waits that give up (one per device that loads the library).
__device__ int g_status_word = 0;

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
int* g_status_ptr[kMaxDevices];
thread_local int t_launches = 0;
thread_local int t_last_launches = 0;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return 0;
  return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

void call_begin() { t_launches = 0; }
int call_end(int rc) {
  if (rc == DS4X_OK) t_last_launches = t_launches;
  return rc;
}

namespace {
struct CallScope {  // launch accounting for ds4x_last_launch_count()
  CallScope() { call_begin(); }
  int done(int rc) { return call_end(rc); }
};
}  // namespace

int device_sm_count() {
  const int d = current_device();
  if (g_sm_count[d] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 148;
    g_sm_count[d] = n;
  }
  return g_sm_count[d];
}

int* device_status_ptr() {
  const int d = current_device();
  if (g_status_ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess) g_status_ptr[d] = static_cast<int*>(p);
  }
  return g_status_ptr[d];
}

void count_launch(int n) { t_launches += n; }

namespace {
size_t round256(size_t n) { return (n + 255) & ~size_t(255); }
}  // namespace

// Workspace of the fused path: [scores T x S fp32 | top-k scratch | split-attention scratch].
size_t fused_workspace_bytes(int T, int S, int k_top) {
  if (T <= 0 || S <= 0 || k_top <= 0) return 0;
  return round256((size_t)T * (size_t)S * sizeof(float)) + round256(topk_workspace_bytes(T, S, k_top)) +
         attn_partial_bytes(T, k_top);
}

int run_index_and_attend(const void* q, const void* w, const void* k, const int32_t* positions, const void* q_attn,
                         const void* kv, int bf16, int T, int H, int D, int S, int ratio, int k_top, float scale,
                         int32_t* indices, void* out, float* lse, void* workspace, size_t workspace_bytes,
                         cudaStream_t st) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t score_bytes = round256((size_t)T * (size_t)S * sizeof(float));
  const size_t topk_bytes = S > 0 ? round256(topk_workspace_bytes(T, S, k_top)) : 0;
  int rc = DS4X_OK;
  if (S > 0) {
    // scores only for tokens that the shortcut does not cover; masked rows are never read
    ScoreArgs sa{q, w, k, positions, reinterpret_cast<float*>(ws), (int64_t)S, T, H, D, S, ratio, k_top, 0};
    rc = launch_score(sa, st);
  }
  if (rc == DS4X_OK) {
    TopkArgs ta{reinterpret_cast<float*>(ws), (int64_t)(S > 0 ? S : 1), positions, T, S, ratio, k_top, indices,
                nullptr, S > 0 ? ws + score_bytes : nullptr, S > 0 ? workspace_bytes - score_bytes : 0};
    rc = launch_topk(ta, st);
  }
  if (rc == DS4X_OK) {
    const size_t used = score_bytes + topk_bytes;
    const bool room = S > 0 && workspace_bytes > used;
    AttnArgs aa{q_attn, kv, bf16, indices, T, 64, 512, S, k_top, scale, out, lse,
                room ? ws + used : nullptr, room ? workspace_bytes - used : 0};
    rc = launch_sparse_attn(aa, st);
  }
  return rc;
}

namespace {
// One thread waits on a barrier that nothing completes; the bounded wait gives up.
__global__ void bounded_wait_selftest_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait_ns(&bar, 0, status, 0x7e, timeout_ns);
}
}  // namespace

}  // namespace ds4x

using namespace ds4x;

extern "C" {

const char* ds4x_status_string(int status) {
  switch (status) {
    case DS4X_OK: return "DS4X_OK";
    case DS4X_ERR_INVALID: return "DS4X_ERR_INVALID: invalid argument";
    case DS4X_ERR_UNSUPPORTED: return "DS4X_ERR_UNSUPPORTED: shape not supported by this build";
    case DS4X_ERR_CUDA: return "DS4X_ERR_CUDA: a CUDA call or kernel launch failed";
    case DS4X_ERR_WORKSPACE: return "DS4X_ERR_WORKSPACE: workspace too small";
    case DS4X_ERR_TIMEOUT: return "DS4X_ERR_TIMEOUT: a bounded device wait gave up";
    default: return "DS4X_ERR_UNKNOWN";
  }
}

int ds4x_last_launch_count(void) { return t_last_launches; }

size_t ds4x_topk_workspace_bytes(int32_t T, int32_t S, int32_t k_top) {
  if (T <= 0 || S <= 0 || k_top <= 0) return 0;
  return topk_workspace_bytes(T, S, k_top);
}

size_t ds4x_workspace_bytes(int32_t T, int32_t S, int32_t k_top) { return fused_workspace_bytes(T, S, k_top); }

int ds4x_indexer_score(const void* q, const void* w, const void* k, const int32_t* positions, int32_t T,
                       int32_t H, int32_t D, int32_t S, int32_t ratio, float* scores, int64_t ld_scores,
                       void* stream) {
  CallScope scope;
  if (T < 0 || S < 0 || H <= 0 || D <= 0 || ratio < 1 || ld_scores < S) return DS4X_ERR_INVALID;
  if (T == 0 || S == 0) return scope.done(DS4X_OK);
  if (!q || !w || !k || !positions || !scores) return DS4X_ERR_INVALID;
  if (!aligned16(q) || !aligned16(w) || !aligned16(k) || !aligned16(positions) || !aligned16(scores))
    return DS4X_ERR_INVALID;
  if (!score_shape_supported(H, D)) return DS4X_ERR_UNSUPPORTED;
  ScoreArgs a{q, w, k, positions, scores, ld_scores, T, H, D, S, ratio, 0, 1};
  return scope.done(launch_score(a, static_cast<cudaStream_t>(stream)));
}

int ds4x_topk(const float* scores, int64_t ld_scores, const int32_t* positions, int32_t T, int32_t S,
              int32_t ratio, int32_t k_top, int32_t* indices, int32_t* counts, void* workspace,
              size_t workspace_bytes, void* stream) {
  CallScope scope;
  if (T < 0 || S < 0 || ratio < 1 || ld_scores < S) return DS4X_ERR_INVALID;
  if (k_top < 1 || k_top > DS4X_MAX_KTOP) return k_top < 1 ? DS4X_ERR_INVALID : DS4X_ERR_UNSUPPORTED;
  if (T == 0) return scope.done(DS4X_OK);
  if (!scores || !positions || !indices) return DS4X_ERR_INVALID;
  if (!aligned16(scores) || !aligned16(positions) || !aligned16(indices) || (counts && !aligned16(counts)))
    return DS4X_ERR_INVALID;
  TopkArgs a{scores, ld_scores, positions, T, S, ratio, k_top, indices, counts, workspace, workspace_bytes};
  return scope.done(launch_topk(a, static_cast<cudaStream_t>(stream)));
}

int ds4x_sparse_attn(const void* q_attn, const void* kv, ds4x_dtype dtype, const int32_t* indices, int32_t T,
                     int32_t Hq, int32_t Dkv, int32_t S, int32_t k_top, float scale, void* out, float* lse,
                     void* stream) {
  CallScope scope;
  if (T < 0 || S < 0 || Hq <= 0 || Dkv <= 0 || k_top < 1) return DS4X_ERR_INVALID;
  if (dtype != DS4X_F16 && dtype != DS4X_BF16) return DS4X_ERR_INVALID;
  if (k_top > DS4X_MAX_KTOP) return DS4X_ERR_UNSUPPORTED;
  if (T == 0) return scope.done(DS4X_OK);
  if (!q_attn || !indices || !out || (S > 0 && !kv)) return DS4X_ERR_INVALID;
  if (!aligned16(q_attn) || (kv && !aligned16(kv)) || !aligned16(indices) || !aligned16(out) ||
      (lse && !aligned16(lse)))
    return DS4X_ERR_INVALID;
  if (!attn_shape_supported(Hq, Dkv)) return DS4X_ERR_UNSUPPORTED;
  AttnArgs a{q_attn, kv, dtype == DS4X_BF16 ? 1 : 0, indices, T, Hq, Dkv, S, k_top, scale, out, lse, nullptr, 0};
  return scope.done(launch_sparse_attn(a, static_cast<cudaStream_t>(stream)));
}

int ds4x_index_and_attend(const void* q, const void* w, const void* k, const int32_t* positions,
                          const void* q_attn, const void* kv, ds4x_dtype kv_dtype, int32_t T, int32_t H,
                          int32_t D, int32_t S, int32_t ratio, int32_t k_top, int32_t Hq, int32_t Dkv,
                          float scale, int32_t* indices, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream) {
  CallScope scope;
  if (T < 0 || S < 0 || H <= 0 || D <= 0 || Hq <= 0 || Dkv <= 0 || ratio < 1 || k_top < 1)
    return DS4X_ERR_INVALID;
  if (kv_dtype != DS4X_F16 && kv_dtype != DS4X_BF16) return DS4X_ERR_INVALID;
  if (k_top > DS4X_MAX_KTOP) return DS4X_ERR_UNSUPPORTED;
  if (T == 0) return scope.done(DS4X_OK);
  if (!q || !w || !positions || !q_attn || !indices || !out || (S > 0 && (!k || !kv))) return DS4X_ERR_INVALID;
  if (!aligned16(q) || !aligned16(w) || (k && !aligned16(k)) || !aligned16(positions) || !aligned16(q_attn) ||
      (kv && !aligned16(kv)) || !aligned16(indices) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (workspace && !aligned16(workspace)))
    return DS4X_ERR_INVALID;
  if (!score_shape_supported(H, D) || !attn_shape_supported(Hq, Dkv)) return DS4X_ERR_UNSUPPORTED;
  const size_t need = ds4x_workspace_bytes(T, S, k_top);
  if (S > 0 && (workspace == nullptr || workspace_bytes < need)) return DS4X_ERR_WORKSPACE;
  return scope.done(run_index_and_attend(q, w, k, positions, q_attn, kv, kv_dtype == DS4X_BF16 ? 1 : 0, T, H, D, S,
                                         ratio, k_top, scale, indices, out, lse, workspace, workspace_bytes,
                                         static_cast<cudaStream_t>(stream)));
}

int ds4x_device_status(void* stream, int clear) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* p = device_status_ptr();
  if (!p) return DS4X_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return DS4X_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DS4X_ERR_CUDA;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyAsync(p, &zero, sizeof(int), cudaMemcpyHostToDevice, st) != cudaSuccess) return DS4X_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DS4X_ERR_CUDA;
  }
  return v == 0 ? DS4X_OK : -(v & 0xff);
}

int ds4x_selftest_bounded_wait(int64_t timeout_ns, void* stream) {
  CallScope scope;
  if (timeout_ns < 1000 || timeout_ns > 2000000000ll) return DS4X_ERR_INVALID;
  int* st = device_status_ptr();
  if (!st) return DS4X_ERR_CUDA;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st, (unsigned long long)timeout_ns);
  count_launch();
  return scope.done(cudaGetLastError() == cudaSuccess ? DS4X_OK : DS4X_ERR_CUDA);
}

}  // extern "C"
