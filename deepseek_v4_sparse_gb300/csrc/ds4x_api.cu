// ds4x_api.cu — the C ABI of libds4x.so (declared in include/ds4x.h).
//
// Host-side argument validation happens here, before anything is launched; the kernels and
// their launchers live in score_tcgen05.cu, topk_stream.cu and sparse_mqa.cu.  The library
// allocates no device memory: the fused entry carves the caller's workspace, and the
// host-buffer entry the caller's device buffer.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

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

// Window arguments: local_pos0 >= 0, L >= 0, 0 <= window <= DS4X_MAX_WINDOW, and a buffer (16-byte
// aligned when it is device memory) whenever a row of it can be attended.
int check_window(const void* kv_local, int32_t local_pos0, int32_t L, int32_t window, bool device) {
  if (local_pos0 < 0 || L < 0 || window < 0) return DS4X_ERR_INVALID;
  if (window > DS4X_MAX_WINDOW) return DS4X_ERR_UNSUPPORTED;
  if (window > 0 && L > 0 && (!kv_local || (device && !aligned16(kv_local)))) return DS4X_ERR_INVALID;
  return DS4X_OK;
}

LocalWindow window_of(const void* kv_local, int32_t local_pos0, int32_t L, int32_t window) {
  LocalWindow lw;
  lw.kv_local = kv_local;
  lw.local_pos0 = local_pos0;
  lw.L = L;
  lw.window = window;
  return lw;
}

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
struct SmemAttr {
  const void* func;
  int bytes;
};
constexpr int kMaxAttrKernels = 64;
std::mutex g_attr_mutex;
SmemAttr g_attr[kMaxDevices][kMaxAttrKernels];
int g_attr_count[kMaxDevices];
}  // namespace

EncodeTiledFn encode_tiled_fn() {
  static const EncodeTiledFn fn = [] {  // a function-local static: initialised once, thread-safe
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

cudaError_t ensure_dynamic_smem_raw(const void* func, int bytes) {
  const int d = current_device();
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  SmemAttr* tab = g_attr[d];
  int i = 0;
  while (i < g_attr_count[d] && tab[i].func != func) ++i;
  if (i < g_attr_count[d] && tab[i].bytes >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (i < g_attr_count[d]) {
    tab[i].bytes = bytes;
  } else if (i < kMaxAttrKernels) {  // a full table only means the attribute is set on every call
    tab[i] = SmemAttr{func, bytes};
    g_attr_count[d] = i + 1;
  }
  return cudaSuccess;
}

namespace {
size_t round256(size_t n) { return (n + 255) & ~size_t(255); }
}  // namespace

// Workspace of the fused path: [scores T x S fp32 | top-k scratch | split-attention scratch].
size_t fused_workspace_bytes(int T, int S, int k_top, int window) {
  if (T <= 0 || k_top <= 0 || (S <= 0 && window <= 0)) return 0;
  const size_t front = S > 0 ? round256((size_t)T * (size_t)S * sizeof(float)) +
                                   round256(topk_workspace_bytes(T, S, k_top))
                             : 0;
  return front + attn_partial_bytes(T, k_top, window > 0 ? window : 0);
}

int run_index_and_attend(const void* q, const void* w, const void* k, const int32_t* positions, const void* q_attn,
                         const void* kv, int bf16, int T, int H, int D, int S, int ratio, int k_top, float scale,
                         int32_t* indices, void* out, float* lse, void* workspace, size_t workspace_bytes,
                         cudaStream_t st, const LocalWindow& local) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t score_bytes = round256((size_t)T * (size_t)S * sizeof(float));
  const size_t topk_bytes = S > 0 ? round256(topk_workspace_bytes(T, S, k_top)) : 0;
  int rc = DS4X_OK;
  // the long-row top-k's barrier counters sit at the start of its scratch; the scorer zeroes them.
  // One token over a long row (a decode step): the scorer zeroes the token's whole top-k scratch and
  // hands over the key range of the scores it wrote, so the top-k starts at its histogram phase.
  const bool zero_counters = S > 0 && topk_bytes > 0;
  const int n_slots = S > 0 ? score_grid(T, H, S) : 0;
  // (the range slots are written and read as 16-byte words)
  const bool range_mode = zero_counters && topk_range_mode(T, S, k_top, n_slots) &&
                          aligned16(ws + score_bytes + topk_range_slots_offset(T, S));
  uint32_t* range_slots = range_mode ? reinterpret_cast<uint32_t*>(ws + score_bytes + topk_range_slots_offset(T, S))
                                     : nullptr;
  if (S > 0) {
    // scores only for tokens that the shortcut does not cover; masked rows are never read
    ScoreArgs sa{q, w, k, positions, reinterpret_cast<float*>(ws), (int64_t)S, T, H, D, S, ratio, k_top, 0};
    if (zero_counters) {
      sa.zero_words = reinterpret_cast<uint32_t*>(ws + score_bytes);
      sa.n_zero = range_mode ? (int)topk_range_zero_words(T, S) : T;
    }
    sa.range_slots = range_slots;
    rc = launch_score(sa, st);
  }
  if (rc == DS4X_OK) {
    TopkArgs ta{reinterpret_cast<float*>(ws), (int64_t)(S > 0 ? S : 1), positions, T, S, ratio, k_top, indices,
                nullptr, S > 0 ? ws + score_bytes : nullptr, S > 0 ? workspace_bytes - score_bytes : 0};
    ta.counters_zeroed = zero_counters ? 1 : 0;
    ta.range_slots = range_slots;
    ta.n_range_slots = range_mode ? n_slots : 0;
    rc = launch_topk(ta, st);
  }
  if (rc == DS4X_OK) {
    const size_t used = S > 0 ? score_bytes + topk_bytes : 0;
    const bool room = ws != nullptr && workspace_bytes > used;
    AttnArgs aa{q_attn, kv, bf16, indices, T, 64, 512, S, k_top, scale, out, lse,
                room ? ws + used : nullptr, room ? workspace_bytes - used : 0, positions, local};
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

namespace {
// ------------------------------------------------------------- the host-buffer fused path
// Device staging of ds4x_index_and_attend_host: [k | kv | window rows | w, positions and lse of every
// token | fused workspace of one sub-chunk | kHostSlots slots of one sub-chunk's q, q_attn, indices
// and out], every part 256-byte aligned.  The small per-token arrays move in one copy each; the
// large ones by sub-chunk, rotating over the slots.
constexpr int kHostSlots = 3;
struct HostLayout {
  int n = 0, tc = 0, ns = 0;                         // sub-chunks, tokens a slot holds, slots in use
  int T = 0, ramp = 0, mid = 0;                      // tokens of the short first and last sub-chunks; of the others
  // sub-chunk j: its first token and its token count.  With a ramp, the first and last sub-chunks
  // are short (the first copy in and the last copy out overlap nothing) and the others even.
  void chunk(int j, size_t& t0, int& tn) const {
    if (ramp == 0) {
      t0 = (size_t)j * tc;
      tn = (int)((size_t)T - t0 < (size_t)tc ? (size_t)T - t0 : (size_t)tc);
    } else if (j == 0) {
      t0 = 0;
      tn = ramp;
    } else if (j == n - 1) {
      t0 = (size_t)T - ramp;
      tn = ramp;
    } else {
      t0 = (size_t)ramp + (size_t)(j - 1) * mid;
      const size_t end = (size_t)T - ramp, e = t0 + mid < end ? t0 + mid : end;
      tn = (int)(e - t0);
    }
  }
  size_t k = 0, kv = 0, kvl = 0, w = 0, pos = 0, lse = 0, ws = 0, ws_bytes = 0, slot0 = 0, slot = 0, total = 0;
  size_t q = 0, qa = 0, idx = 0, out = 0;            // offsets within a slot
};

int default_host_chunks(int T) {  // sub-chunks of about 512 tokens (plus the short first and last)
  const int n = T / 512;
  return n < 1 ? 1 : n > 8 ? 8 : n;
}

HostLayout host_layout(int T, int H, int D, int S, int k_top, int Hq, int Dkv, int n_chunks, int Lrows = 0,
                       int window = 0) {
  const bool win = window > 0 && Lrows > 0;
  HostLayout L;
  L.T = T;
  L.n = n_chunks > 0 ? (n_chunks < T ? n_chunks : T) : default_host_chunks(T);
  L.tc = (T + L.n - 1) / L.n;
  L.n = (T + L.tc - 1) / L.tc;  // no empty sub-chunk
  if (L.n >= 4 && L.tc >= 8) {
    // a quarter-size first and last sub-chunk, the rest in even sub-chunks of at most tc tokens
    L.ramp = L.tc / 4;
    const int middle = T - 2 * L.ramp;
    const int nm = (middle + L.tc - 1) / L.tc;
    L.mid = (middle + nm - 1) / nm;
    L.n = nm + 2;
  }
  L.ns = L.n < kHostSlots ? L.n : kHostSlots;
  const size_t tc = (size_t)L.tc, e16 = 2;
  size_t o = 0;
  L.k = o;
  o += round256((size_t)S * D * e16);
  L.kv = o;
  o += round256((size_t)S * Dkv * e16);
  L.kvl = o;
  o += win ? round256((size_t)Lrows * Dkv * e16) : 0;
  L.w = o;
  o += round256((size_t)T * H * e16);
  L.pos = o;
  o += round256((size_t)T * sizeof(int32_t));
  L.lse = o;
  o += round256((size_t)T * Hq * sizeof(float));
  L.ws = o;
  L.ws_bytes = fused_workspace_bytes(L.tc, S, k_top, win ? window : 0);
  o += round256(L.ws_bytes);
  size_t s = 0;
  L.q = s;
  s += round256(tc * H * D * e16);
  L.qa = s;
  s += round256(tc * Hq * Dkv * e16);
  L.idx = s;
  s += round256(tc * k_top * sizeof(int32_t));
  L.out = s;
  s += round256(tc * Hq * Dkv * e16);
  L.slot = s;
  L.slot0 = o;
  L.total = o + (size_t)L.ns * s;
  return L;
}

// Copy streams and events of the host-buffer path, one set per device, created on first use;
// a call holds the mutex while it enqueues (the work itself runs after it returns).
struct HostPipe {
  std::mutex m;
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, fin = nullptr, in_done[kHostSlots] = {}, work_done[kHostSlots] = {},
              out_done[kHostSlots] = {};
};
HostPipe g_host_pipe[kMaxDevices];

cudaError_t host_pipe_init(HostPipe& hp) {
  if (hp.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.fin, cudaEventDisableTiming);
  for (int i = 0; i < kHostSlots && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.work_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.out_done[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) hp.ready = true;
  return e;
}
}  // namespace

extern "C" {

const char* ds4x_status_string(int status) {
  switch (status) {
    case DS4X_OK: return "DS4X_OK";
    case DS4X_ERR_INVALID: return "DS4X_ERR_INVALID: invalid argument";
    case DS4X_ERR_UNSUPPORTED: return "DS4X_ERR_UNSUPPORTED: shape not supported by this library";
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

size_t ds4x_workspace_bytes_local(int32_t T, int32_t S, int32_t k_top, int32_t window) {
  if (window < 0 || window > DS4X_MAX_WINDOW) return 0;
  return fused_workspace_bytes(T, S, k_top, window);
}

int ds4x_local_pooled_attn(const void* q_attn, const void* kv, const void* kv_local, ds4x_dtype dtype,
                           const int32_t* indices, const int32_t* positions, int32_t T, int32_t Hq, int32_t Dkv,
                           int32_t S, int32_t k_top, int32_t local_pos0, int32_t L, int32_t window, float scale,
                           void* out, float* lse, void* stream) {
  CallScope scope;
  if (T < 0 || S < 0 || Hq <= 0 || Dkv <= 0 || k_top < 1) return DS4X_ERR_INVALID;
  if (dtype != DS4X_F16 && dtype != DS4X_BF16) return DS4X_ERR_INVALID;
  const int wrc = check_window(kv_local, local_pos0, L, window, true);
  if (wrc != DS4X_OK) return wrc;
  if (k_top > DS4X_MAX_KTOP) return DS4X_ERR_UNSUPPORTED;
  if (T == 0) return scope.done(DS4X_OK);
  if (!q_attn || !indices || !out || !positions || (S > 0 && !kv)) return DS4X_ERR_INVALID;
  if (!aligned16(q_attn) || (kv && !aligned16(kv)) || !aligned16(indices) || !aligned16(positions) ||
      !aligned16(out) || (lse && !aligned16(lse)))
    return DS4X_ERR_INVALID;
  if (!attn_shape_supported(Hq, Dkv)) return DS4X_ERR_UNSUPPORTED;
  AttnArgs a{q_attn, kv, dtype == DS4X_BF16 ? 1 : 0, indices, T, Hq, Dkv, S, k_top, scale, out, lse, nullptr, 0,
             positions, window_of(kv_local, local_pos0, L, window)};
  return scope.done(launch_sparse_attn(a, static_cast<cudaStream_t>(stream)));
}

int ds4x_index_and_attend_local(const void* q, const void* w, const void* k, const int32_t* positions,
                                const void* q_attn, const void* kv, const void* kv_local, ds4x_dtype kv_dtype,
                                int32_t T, int32_t H, int32_t D, int32_t S, int32_t ratio, int32_t k_top,
                                int32_t Hq, int32_t Dkv, int32_t local_pos0, int32_t L, int32_t window, float scale,
                                int32_t* indices, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                void* stream) {
  CallScope scope;
  if (T < 0 || S < 0 || H <= 0 || D <= 0 || Hq <= 0 || Dkv <= 0 || ratio < 1 || k_top < 1)
    return DS4X_ERR_INVALID;
  if (kv_dtype != DS4X_F16 && kv_dtype != DS4X_BF16) return DS4X_ERR_INVALID;
  const int wrc = check_window(kv_local, local_pos0, L, window, true);
  if (wrc != DS4X_OK) return wrc;
  if (k_top > DS4X_MAX_KTOP) return DS4X_ERR_UNSUPPORTED;
  if (T == 0) return scope.done(DS4X_OK);
  if (!q || !w || !positions || !q_attn || !indices || !out || (S > 0 && (!k || !kv))) return DS4X_ERR_INVALID;
  if (!aligned16(q) || !aligned16(w) || (k && !aligned16(k)) || !aligned16(positions) || !aligned16(q_attn) ||
      (kv && !aligned16(kv)) || !aligned16(indices) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (workspace && !aligned16(workspace)))
    return DS4X_ERR_INVALID;
  if (!score_shape_supported(H, D) || !attn_shape_supported(Hq, Dkv)) return DS4X_ERR_UNSUPPORTED;
  if (S > 0 && (workspace == nullptr || workspace_bytes < fused_workspace_bytes(T, S, k_top, window)))
    return DS4X_ERR_WORKSPACE;
  return scope.done(run_index_and_attend(q, w, k, positions, q_attn, kv, kv_dtype == DS4X_BF16 ? 1 : 0, T, H, D, S,
                                         ratio, k_top, scale, indices, out, lse, workspace, workspace_bytes,
                                         static_cast<cudaStream_t>(stream),
                                         window_of(kv_local, local_pos0, L, window)));
}

size_t ds4x_index_and_attend_host_bytes(int32_t T, int32_t H, int32_t D, int32_t S, int32_t k_top, int32_t Hq,
                                        int32_t Dkv, int32_t n_chunks) {
  if (T <= 0 || S < 0 || H <= 0 || D <= 0 || k_top <= 0 || Hq <= 0 || Dkv <= 0 || n_chunks < 0) return 0;
  return host_layout(T, H, D, S, k_top, Hq, Dkv, n_chunks).total;
}

}  // extern "C"

namespace {
// The host-buffer fused path with an optional raw window (kv_local is host memory, copied once).
int host_path(const void* q, const void* w, const void* k, const int32_t* positions, const void* q_attn,
              const void* kv, ds4x_dtype kv_dtype, int32_t T, int32_t H, int32_t D, int32_t S, int32_t ratio,
              int32_t k_top, int32_t Hq, int32_t Dkv, float scale, int32_t* indices, void* out, float* lse,
              int32_t n_chunks, void* device_buffer, size_t device_bytes, void* stream, const LocalWindow& lw) {
  CallScope scope;
  if (T < 0 || S < 0 || H <= 0 || D <= 0 || Hq <= 0 || Dkv <= 0 || ratio < 1 || k_top < 1 || n_chunks < 0)
    return DS4X_ERR_INVALID;
  if (kv_dtype != DS4X_F16 && kv_dtype != DS4X_BF16) return DS4X_ERR_INVALID;
  if (k_top > DS4X_MAX_KTOP) return DS4X_ERR_UNSUPPORTED;
  if (T == 0) return scope.done(DS4X_OK);
  if (!q || !w || !positions || !q_attn || !indices || !out || (S > 0 && (!k || !kv)) || !device_buffer)
    return DS4X_ERR_INVALID;
  if (!aligned16(device_buffer)) return DS4X_ERR_INVALID;
  if (!score_shape_supported(H, D) || !attn_shape_supported(Hq, Dkv)) return DS4X_ERR_UNSUPPORTED;
  const HostLayout L = host_layout(T, H, D, S, k_top, Hq, Dkv, n_chunks, lw.L, lw.window);
  if (device_bytes < L.total) return DS4X_ERR_WORKSPACE;
  LocalWindow dlw = lw;  // the window rows' device copy

  HostPipe& hp = g_host_pipe[current_device()];
  std::lock_guard<std::mutex> lock(hp.m);
  if (host_pipe_init(hp) != cudaSuccess) return DS4X_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(device_buffer);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
#define DS4X_CK(x) \
  if ((x) != cudaSuccess) return DS4X_ERR_CUDA
  // the copies start after everything enqueued on the caller's stream (an earlier call's
  // kernels may still use this device buffer)
  DS4X_CK(cudaEventRecord(hp.start, st));
  DS4X_CK(cudaStreamWaitEvent(hp.in, hp.start, 0));
  DS4X_CK(cudaStreamWaitEvent(hp.out, hp.start, 0));
  if (S > 0) {
    DS4X_CK(cudaMemcpyAsync(base + L.k, k, (size_t)S * D * 2, h2d, hp.in));
    DS4X_CK(cudaMemcpyAsync(base + L.kv, kv, (size_t)S * Dkv * 2, h2d, hp.in));
  }
  if (lw.active()) {
    DS4X_CK(cudaMemcpyAsync(base + L.kvl, lw.kv_local, (size_t)lw.L * Dkv * 2, h2d, hp.in));
    dlw.kv_local = base + L.kvl;
  }
  // every token's w and position, once
  DS4X_CK(cudaMemcpyAsync(base + L.w, w, (size_t)T * H * 2, h2d, hp.in));
  DS4X_CK(cudaMemcpyAsync(base + L.pos, positions, (size_t)T * sizeof(int32_t), h2d, hp.in));
  const size_t qt = (size_t)H * D * 2, at = (size_t)Hq * Dkv * 2, it = (size_t)k_top * sizeof(int32_t);
  float* lse_dev = reinterpret_cast<float*>(base + L.lse);
  for (int j = 0; j < L.n; ++j) {
    const int b = j % L.ns;
    size_t t0;
    int tn;
    L.chunk(j, t0, tn);
    uint8_t* sl = base + L.slot0 + b * L.slot;
    // inputs of sub-chunk j, once sub-chunk j - ns (same slot) has been computed
    if (j >= L.ns) DS4X_CK(cudaStreamWaitEvent(hp.in, hp.work_done[b], 0));
    DS4X_CK(cudaMemcpyAsync(sl + L.q, static_cast<const uint8_t*>(q) + t0 * qt, tn * qt, h2d, hp.in));
    DS4X_CK(cudaMemcpyAsync(sl + L.qa, static_cast<const uint8_t*>(q_attn) + t0 * at, tn * at, h2d, hp.in));
    DS4X_CK(cudaEventRecord(hp.in_done[b], hp.in));
    // the work, once the inputs are in and sub-chunk j - ns's outputs are out of the slot
    DS4X_CK(cudaStreamWaitEvent(st, hp.in_done[b], 0));
    if (j >= L.ns) DS4X_CK(cudaStreamWaitEvent(st, hp.out_done[b], 0));
    const int rc = run_index_and_attend(sl + L.q, base + L.w + t0 * H * 2, S > 0 ? base + L.k : nullptr,
                                        reinterpret_cast<const int32_t*>(base + L.pos) + t0, sl + L.qa,
                                        S > 0 ? base + L.kv : nullptr, kv_dtype == DS4X_BF16 ? 1 : 0, tn, H, D, S,
                                        ratio, k_top, scale, reinterpret_cast<int32_t*>(sl + L.idx), sl + L.out,
                                        lse ? lse_dev + t0 * Hq : nullptr, base + L.ws, L.ws_bytes, st, dlw);
    if (rc != DS4X_OK) return rc;
    DS4X_CK(cudaEventRecord(hp.work_done[b], st));
    // outputs of sub-chunk j
    DS4X_CK(cudaStreamWaitEvent(hp.out, hp.work_done[b], 0));
    DS4X_CK(cudaMemcpyAsync(indices + t0 * k_top, sl + L.idx, tn * it, d2h, hp.out));
    DS4X_CK(cudaMemcpyAsync(static_cast<uint8_t*>(out) + t0 * at, sl + L.out, tn * at, d2h, hp.out));
    DS4X_CK(cudaEventRecord(hp.out_done[b], hp.out));
  }
  // every token's lse, once, after the last sub-chunk's work (the copy stream waited for it)
  if (lse) DS4X_CK(cudaMemcpyAsync(lse, lse_dev, (size_t)T * Hq * sizeof(float), d2h, hp.out));
  // later work on the caller's stream (a synchronisation included) sees the outputs
  DS4X_CK(cudaEventRecord(hp.fin, hp.out));
  DS4X_CK(cudaStreamWaitEvent(st, hp.fin, 0));
#undef DS4X_CK
  return scope.done(DS4X_OK);
}
}  // namespace

extern "C" {

int ds4x_index_and_attend_host(const void* q, const void* w, const void* k, const int32_t* positions,
                               const void* q_attn, const void* kv, ds4x_dtype kv_dtype, int32_t T, int32_t H,
                               int32_t D, int32_t S, int32_t ratio, int32_t k_top, int32_t Hq, int32_t Dkv,
                               float scale, int32_t* indices, void* out, float* lse, int32_t n_chunks,
                               void* device_buffer, size_t device_bytes, void* stream) {
  return host_path(q, w, k, positions, q_attn, kv, kv_dtype, T, H, D, S, ratio, k_top, Hq, Dkv, scale, indices, out,
                   lse, n_chunks, device_buffer, device_bytes, stream, LocalWindow());
}

size_t ds4x_index_and_attend_local_host_bytes(int32_t T, int32_t H, int32_t D, int32_t S, int32_t k_top,
                                              int32_t Hq, int32_t Dkv, int32_t L, int32_t window,
                                              int32_t n_chunks) {
  if (T <= 0 || S < 0 || H <= 0 || D <= 0 || k_top <= 0 || Hq <= 0 || Dkv <= 0 || n_chunks < 0 || L < 0 ||
      window < 0 || window > DS4X_MAX_WINDOW)
    return 0;
  return host_layout(T, H, D, S, k_top, Hq, Dkv, n_chunks, L, window).total;
}

int ds4x_index_and_attend_local_host(const void* q, const void* w, const void* k, const int32_t* positions,
                                     const void* q_attn, const void* kv, const void* kv_local, ds4x_dtype kv_dtype,
                                     int32_t T, int32_t H, int32_t D, int32_t S, int32_t ratio, int32_t k_top,
                                     int32_t Hq, int32_t Dkv, int32_t local_pos0, int32_t L, int32_t window,
                                     float scale, int32_t* indices, void* out, float* lse, int32_t n_chunks,
                                     void* device_buffer, size_t device_bytes, void* stream) {
  const int rc = check_window(kv_local, local_pos0, L, window, false);
  if (rc != DS4X_OK) return rc;
  return host_path(q, w, k, positions, q_attn, kv, kv_dtype, T, H, D, S, ratio, k_top, Hq, Dkv, scale, indices, out,
                   lse, n_chunks, device_buffer, device_bytes, stream, window_of(kv_local, local_pos0, L, window));
}

int ds4x_compress(const void* x, const void* g, const float* bias, ds4x_dtype dtype, int32_t T, int32_t D,
                  int32_t ratio, const void* frontier_x, const void* frontier_g, int32_t n_frontier, void* rows,
                  void* frontier_x_out, void* frontier_g_out, void* stream) {
  CallScope scope;
  if (T < 0 || D < 8 || D % 8 != 0 || ratio < 1 || ratio > DS4X_MAX_RATIO || n_frontier < 0 || n_frontier >= ratio)
    return DS4X_ERR_INVALID;
  if (dtype != DS4X_F16 && dtype != DS4X_BF16) return DS4X_ERR_INVALID;
  const int64_t n = (int64_t)n_frontier + T;
  const int64_t n_out = n / ratio, rem = n % ratio;
  if (T > 0 && (!x || !g || !aligned16(x) || !aligned16(g))) return DS4X_ERR_INVALID;
  if (n_frontier > 0 && (!frontier_x || !frontier_g || !aligned16(frontier_x) || !aligned16(frontier_g)))
    return DS4X_ERR_INVALID;
  if (n_out > 0 && (!rows || !bias || !aligned16(rows) || !aligned16(bias))) return DS4X_ERR_INVALID;
  if (rem > 0 && (!frontier_x_out || !frontier_g_out || !aligned16(frontier_x_out) || !aligned16(frontier_g_out)))
    return DS4X_ERR_INVALID;
  if (n_out == 0 && rem == 0) return scope.done(DS4X_OK);
  CompressArgs a{x, g, bias, frontier_x, frontier_g, rows, frontier_x_out, frontier_g_out,
                 dtype == DS4X_BF16 ? 1 : 0, T, D, ratio, n_frontier};
  return scope.done(launch_compress(a, static_cast<cudaStream_t>(stream)));
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
