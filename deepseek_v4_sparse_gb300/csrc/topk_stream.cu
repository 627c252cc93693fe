// topk_stream.cu — exact per-token top-k of the visible scores, emitted in ascending row order.
//
// Source: "How I made DeepSeek 12x faster on a Mac Studio", section "1: the kernels", PR #832:
// instead of a padded bitonic sort plus merge cascade (O(n log n) while only 512 indices
// survive), one streaming pass keeps a running 512th-best threshold and compacts the
// survivors without atomics contention via simd_ballot; the output is byte-identical to the
// sort.  The shortcut (n_vis <= k_top: emit 0..n-1, read nothing) is item 3 of "The three
// changes that merged" on "How I turned one oversized DeepSeek optimization into three
// merged oMLX PRs".
//
// Order used for selection (total, so the result is unique): the composite
//     c(s) = ordered_key(score[s]) << 32 | ~s
// where ordered_key maps float order to unsigned order; larger c = better (higher score,
// then lower row).  The top k_top rows are exactly { s : c(s) >= c_thr } for the k_top-th
// largest c_thr.
//
// Per token, one CTA of 256 threads:
//   1. stream the row once (coalesced, 4 loads in flight per thread); an element survives if
//      c >= the running threshold; survivors are appended to a shared-memory buffer with a
//      warp ballot + popc prefix (one shared atomic per warp per step);
//   2. when the buffer could overflow, raise the threshold to the k_top-th best buffered
//      composite (radix select over the buffer, 8-bit digits, window starting at the highest
//      bit where the buffer's max and min differ) and compact the buffer in place;
//   3. at the end select once more, mark the winners in a bitmap over the row and emit them in
//      ascending order with a block scan of the bitmap's popcounts.
// A decode-sized row (one token, 262k rows) is split over many CTAs (same routine, each
// emitting its local top-k as (key, row) pairs into the workspace) and merged by a second
// kernel that runs the routine over the candidates.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ds4x_internal.h"
#include "ds4x_ptx.cuh"

namespace ds4x {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCap = 2048;                 // buffered survivors (>= k_top + kChunk)
constexpr int kChunk = kThreads * 4;       // elements streamed per step
constexpr int kSplitRows = 4096;           // rows per CTA when a row is split
constexpr uint32_t kNoRow = 0xFFFFFFFFu;   // padding of partial candidate lists

__device__ __forceinline__ uint32_t ordered_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t row) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~row);
}

constexpr int kBins = 2048;                // histogram of the fast path
constexpr int kStageMax = 32768;           // rows up to this long are staged in shared memory

struct Shared {
  uint32_t key[kCap];
  uint32_t row[kCap];
  uint32_t hist[256];
  uint32_t bins[kBins];
  uint32_t warp_sum[kWarps];
  uint64_t red64[2 * kWarps];
  int count;
  int chosen_bin;
  int chosen_above;
};

// Inclusive scan of v over the block (256 threads); returns the thread's inclusive prefix and
// stores the total in *total.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, Shared& sh, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) sh.warp_sum[warp] = v;
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t s = sh.warp_sum[w];
    before += (w < warp) ? s : 0;
    all += s;
  }
  __syncthreads();
  *total = all;
  return v + before;
}

// Block-wide max and min of 64-bit values.
__device__ __forceinline__ void block_minmax(uint64_t mx, uint64_t mn, Shared& sh, uint64_t* omax, uint64_t* omin) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t a = __shfl_xor_sync(0xffffffffu, mx, o);
    const uint64_t b = __shfl_xor_sync(0xffffffffu, mn, o);
    mx = a > mx ? a : mx;
    mn = b < mn ? b : mn;
  }
  if (lane == 0) {
    sh.red64[warp] = mx;
    sh.red64[kWarps + warp] = mn;
  }
  __syncthreads();
  uint64_t M = sh.red64[0], m = sh.red64[kWarps];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    M = sh.red64[w] > M ? sh.red64[w] : M;
    m = sh.red64[kWarps + w] < m ? sh.red64[kWarps + w] : m;
  }
  __syncthreads();
  *omax = M;
  *omin = m;
}

// The need-th largest composite among the cnt buffered elements (1 <= need <= cnt).
__device__ uint64_t select_kth(Shared& sh, int cnt, int need) {
  uint64_t mx = 0, mn = ~0ull;
  for (int j = threadIdx.x; j < cnt; j += kThreads) {
    const uint64_t c = composite(sh.key[j], sh.row[j]);
    mx = c > mx ? c : mx;
    mn = c < mn ? c : mn;
  }
  uint64_t cmax, cmin;
  block_minmax(mx, mn, sh, &cmax, &cmin);
  if (need == cnt) return cmin;
  if (need == 1) return cmax;
  // bits above the highest differing bit are shared by every buffered composite
  const int hb = 63 - __clzll(static_cast<long long>(cmax ^ cmin));
  uint64_t prefix = (hb == 63) ? 0ull : (cmax & ~((2ull << hb) - 1ull));
  uint64_t fixed = (hb == 63) ? 0ull : ~((2ull << hb) - 1ull);  // bits already decided
  int top = hb;
  while (true) {
    const int width = top + 1 < 8 ? top + 1 : 8;
    const int shift = top + 1 - width;
    const uint32_t dmask = (1u << width) - 1u;
    sh.hist[threadIdx.x] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < cnt; j += kThreads) {
      const uint64_t c = composite(sh.key[j], sh.row[j]);
      if ((c & fixed) == prefix) atomicAdd(&sh.hist[(uint32_t)(c >> shift) & dmask], 1u);
    }
    __syncthreads();
    // suffix sums: thread i looks at bin (255 - i)
    const int bin = 255 - threadIdx.x;
    const uint32_t h = sh.hist[bin];
    uint32_t total;
    const uint32_t suffix = block_scan(h, sh, &total);  // count in bins >= bin
    if (h > 0 && suffix >= (uint32_t)need && suffix - h < (uint32_t)need) {
      sh.chosen_bin = bin;
      sh.chosen_above = (int)(suffix - h);
    }
    __syncthreads();
    const int b = sh.chosen_bin;
    need -= sh.chosen_above;
    const uint32_t hb_count = sh.hist[b];
    __syncthreads();
    prefix |= static_cast<uint64_t>(b) << shift;
    if ((int)hb_count == need || shift == 0) return prefix;  // the whole bin is in
    fixed |= static_cast<uint64_t>(dmask) << shift;
    top = shift - 1;
  }
}

// Keep only the buffered elements with composite >= thr (order-preserving, in place).
__device__ void compact(Shared& sh, uint64_t thr) {
  const int cnt = sh.count;
  int out_base = 0;
  for (int base = 0; base < cnt; base += kThreads) {
    const int j = base + threadIdx.x;
    uint32_t k = 0, r = 0;
    bool keep = false;
    if (j < cnt) {
      k = sh.key[j];
      r = sh.row[j];
      keep = composite(k, r) >= thr;
    }
    uint32_t total;
    const uint32_t incl = block_scan(keep ? 1u : 0u, sh, &total);  // also syncs
    if (keep) {
      sh.key[out_base + incl - 1] = k;
      sh.row[out_base + incl - 1] = r;
    }
    out_base += (int)total;
    __syncthreads();
  }
  if (threadIdx.x == 0) sh.count = out_base;
  __syncthreads();
}

// Append the survivors of one step (up to 4 per thread) with ballot/popc compaction.
__device__ __forceinline__ void append(Shared& sh, const uint32_t (&k)[4], const uint32_t (&r)[4],
                                       const bool (&v)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t bal = __ballot_sync(0xffffffffu, v[i]);
    if (bal == 0) continue;
    int base = 0;
    if (lane == 0) base = atomicAdd(&sh.count, __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (v[i]) {
      const int pos = base + __popc(bal & ((1u << lane) - 1u));
      sh.key[pos] = k[i];
      sh.row[pos] = r[i];
    }
  }
}

__device__ __forceinline__ int n_visible(const int32_t* positions, int t, int ratio, int S) {
  const int pos = positions[t];
  if (pos < 0) return 0;
  const long long n = ((long long)pos + 1) / ratio;
  return n < S ? (int)n : S;
}

// Source of elements: a score row (row index = position) or a candidate list.
struct RowSource {
  const float* row;
  __device__ __forceinline__ void get(int j, uint32_t& key, uint32_t& r, bool& valid) const {
    key = ordered_key(__ldcs(row + j));
    r = (uint32_t)j;
    valid = true;
  }
};
struct CandSource {
  const uint32_t* key;
  const uint32_t* row;
  __device__ __forceinline__ void get(int j, uint32_t& k, uint32_t& r, bool& valid) const {
    k = __ldcs(key + j);
    r = __ldcs(row + j);
    valid = r != kNoRow;
  }
};

// Stream elements [lo, hi) of src.  Leaves in the buffer every survivor and returns the
// threshold composite: exactly the min(k_top, survivors) buffered elements with composite >=
// threshold are the best of the stream (0 = everything buffered is in).  The next step's
// loads are issued before the current step is filtered, so two steps are in flight.
template <class Src>
__device__ uint64_t stream_select(Shared& sh, const Src& src, int lo, int hi, int k_top) {
  if (threadIdx.x == 0) sh.count = 0;
  __syncthreads();
  uint64_t thr = 0;
  uint32_t k[4], r[4];
  bool v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = lo + i * kThreads + threadIdx.x;
    v[i] = false;
    k[i] = 0;
    r[i] = 0;
    if (j < hi) src.get(j, k[i], r[i], v[i]);
  }
  for (int base = lo; base < hi; base += kChunk) {
    uint32_t nk[4], nr[4];
    bool nv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = base + kChunk + i * kThreads + threadIdx.x;
      nv[i] = false;
      nk[i] = 0;
      nr[i] = 0;
      if (j < hi) src.get(j, nk[i], nr[i], nv[i]);
    }
    if (sh.count + kChunk > kCap) {
      thr = select_kth(sh, sh.count, k_top);
      compact(sh, thr);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = v[i] && composite(k[i], r[i]) >= thr;
    append(sh, k, r, v);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      k[i] = nk[i];
      r[i] = nr[i];
      v[i] = nv[i];
    }
  }
  if (sh.count > k_top) thr = select_kth(sh, sh.count, k_top);
  return thr;
}

// Emit the rows marked in a bitmap over [0, n) in ascending order, pad with -1.
__device__ void emit_bitmap(Shared& sh, const uint32_t* bitmap, int n, int k_top, int32_t* out, int32_t* count_out) {
  const int nw = (n + 31) >> 5;
  const int per = (nw + kThreads - 1) / kThreads;
  const int w0 = threadIdx.x * per;
  const int w1 = min(nw, w0 + per);
  uint32_t mine = 0;
  for (int i = w0; i < w1; ++i) mine += __popc(bitmap[i]);
  uint32_t total;
  const uint32_t incl = block_scan(mine, sh, &total);
  uint32_t pos = incl - mine;
  for (int i = w0; i < w1; ++i) {
    uint32_t bits = bitmap[i];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      out[pos++] = i * 32 + b;
    }
  }
  for (int i = (int)total + threadIdx.x; i < k_top; i += kThreads) out[i] = -1;
  if (count_out && threadIdx.x == 0) *count_out = (int)total;
}

// Emit the buffered rows with composite >= thr (all < n) in ascending order, pad with -1.
__device__ void emit_sorted(Shared& sh, uint32_t* bitmap, uint64_t thr, int n, int k_top, int32_t* out,
                            int32_t* count_out) {
  const int nw = (n + 31) >> 5;
  for (int i = threadIdx.x; i < nw; i += kThreads) bitmap[i] = 0;
  __syncthreads();
  const int cnt = sh.count;
  for (int j = threadIdx.x; j < cnt; j += kThreads) {
    const uint32_t r = sh.row[j];
    if (composite(sh.key[j], r) >= thr) atomicOr(&bitmap[r >> 5], 1u << (r & 31));
  }
  __syncthreads();
  emit_bitmap(sh, bitmap, n, k_top, out, count_out);
}

__device__ __forceinline__ void emit_shortcut(int n, int k_top, int32_t* out, int32_t* count_out) {
  for (int i = threadIdx.x; i < k_top; i += kThreads) out[i] = i < n ? i : -1;
  if (count_out && threadIdx.x == 0) *count_out = n;
}


// ------------------------------------------------------------------------ histogram path
// Monotone bucketing of the ordered keys of one row: bin(key) = umulhi(key - kmin, mult) with
// mult = floor(kBins * 2^32 / (kmax - kmin + 1)) (capped), so bin is non-decreasing in the key and
// equal keys share a bin; every row in a bin above the boundary bin is in the top-k, the boundary
// bin's rows are resolved exactly with the composite order.
__device__ __forceinline__ uint32_t bin_of(uint32_t key, uint32_t kmin, uint32_t mult) {
  return __umulhi(key - kmin, mult);
}

// Block-wide min and max of 32-bit keys.
__device__ __forceinline__ void block_minmax32(uint32_t mn, uint32_t mx, Shared& sh, uint32_t* omin, uint32_t* omax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sh.warp_sum[warp] = mn;
    sh.red64[warp] = mx;
  }
  __syncthreads();
  uint32_t a = sh.warp_sum[0], b = (uint32_t)sh.red64[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    a = min(a, sh.warp_sum[w]);
    b = max(b, (uint32_t)sh.red64[w]);
  }
  __syncthreads();
  *omin = a;
  *omax = b;
}

// One pass over a row staged in shared memory: thread t visits the 4-element vectors t, t+256, ...
// (16-byte shared loads) and calls f(j, keys[4], valid4) with j = the vector's first element.
template <class F>
__device__ __forceinline__ void smem_row_pass(const float* srow, int n, F&& f) {
  const int nv = (n + 3) >> 2;
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    const float4 x = reinterpret_cast<const float4*>(srow)[v];
    const int j = 4 * v;
    const uint32_t k4[4] = {ordered_key(x.x), ordered_key(x.y), ordered_key(x.z), ordered_key(x.w)};
    const bool v4[4] = {j < n, j + 1 < n, j + 2 < n, j + 3 < n};
    f(j, k4, v4);
  }
}

// Exact top-k of one visible score row (staged in shared memory) with the histogram path.
// Returns false (having written nothing but shared memory) when every key is equal or the
// boundary bin holds more rows than the candidate buffer (massive ties); the caller then runs
// the streaming path.
__device__ bool topk_row_hist(Shared& sh, uint32_t* bitmap, const float* srow, int n, int k_top, int32_t* out,
                              int32_t* count_out) {
  const int tid = threadIdx.x;
  // pass A: key range
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  smem_row_pass(srow, n, [&](int, const uint32_t (&k4)[4], const bool (&v4)[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (v4[c]) {
        mn = min(mn, k4[c]);
        mx = max(mx, k4[c]);
      }
  });
  uint32_t kmin, kmax;
  block_minmax32(mn, mx, sh, &kmin, &kmax);
  if (kmin == kmax) return false;  // one value everywhere: every row ties
  const uint64_t range = static_cast<uint64_t>(kmax - kmin) + 1;
  const uint64_t m64 = (static_cast<uint64_t>(kBins) << 32) / range;
  const uint32_t mult = m64 > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(m64);
  // pass B: histogram
  for (int i = tid; i < kBins; i += kThreads) sh.bins[i] = 0;
  __syncthreads();
  smem_row_pass(srow, n, [&](int, const uint32_t (&k4)[4], const bool (&v4)[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (v4[c]) atomicAdd(&sh.bins[bin_of(k4[c], kmin, mult)], 1u);
  });
  __syncthreads();
  // boundary bin: thread i owns bins [kBins - 8(i+1), kBins - 8i), scanned from the top
  constexpr int kPer = kBins / kThreads;
  const int b_hi = kBins - kPer * tid;  // exclusive
  uint32_t c[kPer], mine = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    c[q] = sh.bins[b_hi - 1 - q];
    mine += c[q];
  }
  uint32_t total;
  uint32_t above = block_scan(mine, sh, &total) - mine;  // rows in bins above this thread's range
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (above < (uint32_t)k_top && above + c[q] >= (uint32_t)k_top) {
      sh.chosen_bin = b_hi - 1 - q;
      sh.chosen_above = (int)above;
    }
    above += c[q];
  }
  __syncthreads();
  const uint32_t bstar = (uint32_t)sh.chosen_bin;
  const int above_b = sh.chosen_above;
  const int cnt_b = (int)sh.bins[bstar];
  if (cnt_b > kCap) return false;
  // pass C: mark rows above the boundary bin; buffer the boundary bin's rows
  const int nw = (n + 31) >> 5;
  for (int i = tid; i < nw; i += kThreads) bitmap[i] = 0;
  if (tid == 0) sh.count = 0;
  __syncthreads();
  const int nv = (n + 3) >> 2;
  const int nv_pad = (nv + kThreads - 1) / kThreads * kThreads;  // whole warps take part in append
  for (int v = tid; v < nv_pad; v += kThreads) {
    const int j = 4 * v;
    uint32_t k4[4] = {0, 0, 0, 0}, r4[4];
    bool b4[4] = {false, false, false, false};
    uint32_t nib = 0;
    if (v < nv) {
      const float4 x = reinterpret_cast<const float4*>(srow)[v];
      k4[0] = ordered_key(x.x);
      k4[1] = ordered_key(x.y);
      k4[2] = ordered_key(x.z);
      k4[3] = ordered_key(x.w);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool valid = j + q < n;
        const uint32_t b = bin_of(k4[q], kmin, mult);
        nib |= (valid && b > bstar) ? (1u << q) : 0u;
        b4[q] = valid && b == bstar;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) r4[q] = (uint32_t)(j + q);
    if (nib) atomicOr(&bitmap[j >> 5], nib << (j & 31));
    append(sh, k4, r4, b4);
  }
  __syncthreads();
  // the boundary bin contributes its (k_top - above_b) best rows in the composite order
  const int need = k_top - above_b;
  uint64_t cthr = 0;
  if (need < cnt_b) cthr = select_kth(sh, cnt_b, need);
  for (int j = tid; j < cnt_b; j += kThreads) {
    const uint32_t r = sh.row[j];
    if (composite(sh.key[j], r) >= cthr) atomicOr(&bitmap[r >> 5], 1u << (r & 31));
  }
  __syncthreads();
  emit_bitmap(sh, bitmap, n, k_top, out, count_out);
  return true;
}

// Copy row[0, n) into shared memory: one bulk copy for the 16-byte-aligned body (when the row
// start is aligned), plain loads for the rest.  Bounded wait; returns false on timeout.
__device__ bool stage_row(const float* row, int n, float* srow, uint64_t* bar, int* status) {
  const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int n_bulk = aligned ? (n & ~3) : 0;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)n_bulk * 4u);
    if (n_bulk > 0)
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_u32(srow)),
          "l"(row), "r"((uint32_t)n_bulk * 4u), "r"(smem_u32(bar))
          : "memory");
  }
  for (int j = n_bulk + threadIdx.x; j < n; j += kThreads) srow[j] = row[j];
  // pad to a whole vector so that 16-byte reads past n see defined values
  if (threadIdx.x < 4 && n + threadIdx.x < ((n + 3) & ~3)) srow[n + threadIdx.x] = 0.f;
  const bool ok = mbar_wait(bar, 0, status, 50);
  __syncthreads();
  return ok;
}

struct KParams {
  const float* scores;
  int64_t ld;
  const int32_t* positions;
  int T, S, ratio, k_top;
  int32_t* indices;
  int32_t* counts;
  uint32_t* cand_key;  // [T, nsplit, k_top] (split mode)
  uint32_t* cand_row;
  int nsplit;
  int* status;
};

// One CTA per token: the whole row.
__global__ void __launch_bounds__(kThreads) topk_row_kernel(const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem_raw + sizeof(Shared));
  const int t = blockIdx.x;
  const int n = n_visible(p.positions, t, p.ratio, p.S);
  int32_t* out = p.indices + (int64_t)t * p.k_top;
  int32_t* cnt_out = p.counts ? p.counts + t : nullptr;
  if (n <= p.k_top) {
    emit_shortcut(n, p.k_top, out, cnt_out);
    return;
  }
  const float* row = p.scores + (int64_t)t * p.ld;
  if (p.S <= kStageMax) {
    float* srow = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(bitmap + (p.S + 31) / 32) + 15) &
                                           ~uintptr_t(15));
    __shared__ uint64_t row_bar;
    if (!stage_row(row, n, srow, &row_bar, p.status)) return;
    if (topk_row_hist(sh, bitmap, srow, n, p.k_top, out, cnt_out)) return;
    __syncthreads();
  }
  RowSource src{row};
  const uint64_t thr = stream_select(sh, src, 0, n, p.k_top);
  emit_sorted(sh, bitmap, thr, n, p.k_top, out, cnt_out);
}

// Split mode, pass 1: CTA (t, part) keeps the k_top best of rows [part*kSplitRows, ...).
__global__ void __launch_bounds__(kThreads) topk_part_kernel(const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  const int t = blockIdx.y, part = blockIdx.x;
  const int n = n_visible(p.positions, t, p.ratio, p.S);
  if (n <= p.k_top) return;  // the merge kernel takes the shortcut
  const int lo = part * kSplitRows;
  const int hi = min(n, lo + kSplitRows);
  uint32_t* ck = p.cand_key + ((int64_t)t * p.nsplit + part) * p.k_top;
  uint32_t* cr = p.cand_row + ((int64_t)t * p.nsplit + part) * p.k_top;
  int have = 0;
  if (lo < hi) {
    RowSource src{p.scores + (int64_t)t * p.ld};
    const uint64_t thr = stream_select(sh, src, lo, hi, p.k_top);
    if (sh.count > p.k_top) compact(sh, thr);
    have = sh.count;
    for (int j = threadIdx.x; j < have; j += kThreads) {
      ck[j] = sh.key[j];
      cr[j] = sh.row[j];
    }
  }
  for (int j = have + threadIdx.x; j < p.k_top; j += kThreads) {
    ck[j] = 0;
    cr[j] = kNoRow;
  }
}

// Split mode, pass 2: one CTA per token over its nsplit * k_top candidates.
__global__ void __launch_bounds__(kThreads) topk_merge_kernel(const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem_raw + sizeof(Shared));
  const int t = blockIdx.x;
  const int n = n_visible(p.positions, t, p.ratio, p.S);
  int32_t* out = p.indices + (int64_t)t * p.k_top;
  int32_t* cnt_out = p.counts ? p.counts + t : nullptr;
  if (n <= p.k_top) {
    emit_shortcut(n, p.k_top, out, cnt_out);
    return;
  }
  const int m = p.nsplit * p.k_top;
  CandSource src{p.cand_key + (int64_t)t * m, p.cand_row + (int64_t)t * m};
  const uint64_t thr = stream_select(sh, src, 0, m, p.k_top);
  emit_sorted(sh, bitmap, thr, n, p.k_top, out, cnt_out);
}

// dynamic shared memory of the row and merge kernels: the work struct, the bitmap of the row
// and (row kernel, rows that are staged) 16 bytes of alignment slack plus the staged row
size_t bitmap_smem(int S) { return sizeof(Shared) + (size_t)((S + 31) / 32 + 1) * sizeof(uint32_t); }
size_t row_kernel_smem(int S) {
  if (S > kStageMax) return bitmap_smem(S);
  return bitmap_smem(S) + 16 + ((size_t)(S + 3) & ~size_t(3)) * sizeof(float);
}

cudaError_t set_smem_attrs(size_t row_smem, size_t merge_smem) {
  cudaError_t e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)row_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)merge_smem);
  return e;
}

int split_parts(int T, int S) {
  // few tokens with long rows cannot fill the GPU with one CTA per token
  const int sms = device_sm_count();
  if (S <= 2 * kSplitRows || T >= sms) return 1;
  const int parts = (S + kSplitRows - 1) / kSplitRows;
  return parts;
}

}  // namespace

size_t topk_workspace_bytes(int T, int S, int k_top) {
  const int parts = split_parts(T, S);
  if (parts <= 1) return 0;
  return (size_t)T * parts * k_top * 2 * sizeof(uint32_t);
}

int launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.T == 0) return DS4X_OK;
  const size_t smem = row_kernel_smem(a.S);
  const size_t msmem = bitmap_smem(a.S);
  if (smem > 220 * 1024 || msmem > 220 * 1024) return DS4X_ERR_UNSUPPORTED;
  if (set_smem_attrs(smem, msmem) != cudaSuccess) return DS4X_ERR_CUDA;
  KParams p;
  p.scores = a.scores;
  p.ld = a.ld;
  p.positions = a.positions;
  p.T = a.T;
  p.S = a.S;
  p.ratio = a.ratio;
  p.k_top = a.k_top;
  p.indices = a.indices;
  p.counts = a.counts;
  p.nsplit = split_parts(a.T, a.S);
  p.cand_key = nullptr;
  p.cand_row = nullptr;
  p.status = device_status_ptr();
  if (p.nsplit <= 1) {
    topk_row_kernel<<<a.T, kThreads, smem, stream>>>(p);
    count_launch();
  } else {
    const size_t need = topk_workspace_bytes(a.T, a.S, a.k_top);
    if (a.workspace == nullptr || a.workspace_bytes < need) return DS4X_ERR_WORKSPACE;
    p.cand_key = static_cast<uint32_t*>(a.workspace);
    p.cand_row = p.cand_key + (size_t)a.T * p.nsplit * a.k_top;
    topk_part_kernel<<<dim3(p.nsplit, a.T), kThreads, sizeof(Shared), stream>>>(p);
    topk_merge_kernel<<<a.T, kThreads, msmem, stream>>>(p);
    count_launch(2);
  }
  return cudaGetLastError() == cudaSuccess ? DS4X_OK : DS4X_ERR_CUDA;
}

}  // namespace ds4x

// -----------------------------------------------------------------------------------------
// Top-k for callers that cannot allocate device memory.
//
// ds4x_topk needs a caller-supplied workspace when one long row is split across CTAs (the
// candidate lists of the split pass).  Some callers cannot provide one: an inference server that
// hands all of HBM to its KV cache at start-up and forbids any later allocation, or a plugin that
// runs inside a host framework owning the device allocator.  For them this variant keeps the
// candidate lists in a fixed array compiled into the library.  The array is file-scope device
// memory: every GPU that loads the library holds DS4X_TOPK_STATIC_SCRATCH_BYTES of it until the
// process exits, and every call on that GPU shares it.
namespace ds4x {

static __device__ __align__(256) unsigned char g_topk_static_scratch[DS4X_TOPK_STATIC_SCRATCH_BYTES];

namespace {
std::mutex g_static_scratch_mutex;
void* g_static_scratch_addr[64];  // device address of g_topk_static_scratch, per device

// Host code only knows a stand-in for the array's name; the device address is looked up once
// per device, with that device current.
void* static_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_scratch_mutex);
  if (g_static_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_topk_static_scratch) != cudaSuccess) return nullptr;
    g_static_scratch_addr[dev] = ptr;
  }
  return g_static_scratch_addr[dev];
}
}  // namespace

}  // namespace ds4x

extern "C" int ds4x_topk_static_scratch(const float* scores, int64_t ld_scores, const int32_t* positions,
                                        int32_t T, int32_t S, int32_t ratio, int32_t k_top, int32_t* indices,
                                        int32_t* counts, void* stream) {
  using namespace ds4x;
  if (T < 0 || S < 0 || ratio < 1 || ld_scores < S) return DS4X_ERR_INVALID;
  if (k_top < 1 || k_top > DS4X_MAX_KTOP) return k_top < 1 ? DS4X_ERR_INVALID : DS4X_ERR_UNSUPPORTED;
  if (T == 0) return DS4X_OK;
  if (!scores || !positions || !indices) return DS4X_ERR_INVALID;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(scores) | reinterpret_cast<uintptr_t>(positions) |
                         reinterpret_cast<uintptr_t>(indices) | reinterpret_cast<uintptr_t>(counts)) & 15u;
  if (mis) return DS4X_ERR_INVALID;
  // the candidate lists must fit the fixed array
  if (topk_workspace_bytes(T, S, k_top) > (size_t)DS4X_TOPK_STATIC_SCRATCH_BYTES) return DS4X_ERR_WORKSPACE;
  void* scratch = static_scratch_address();
  if (scratch == nullptr) return DS4X_ERR_CUDA;
  const size_t smem = row_kernel_smem(S);
  const size_t msmem = bitmap_smem(S);
  if (smem > 220 * 1024 || msmem > 220 * 1024) return DS4X_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (set_smem_attrs(smem, msmem) != cudaSuccess) return DS4X_ERR_CUDA;
  KParams p;
  p.scores = scores;
  p.ld = ld_scores;
  p.positions = positions;
  p.T = T;
  p.S = S;
  p.ratio = ratio;
  p.k_top = k_top;
  p.indices = indices;
  p.counts = counts;
  p.nsplit = split_parts(T, S);
  p.cand_key = nullptr;
  p.cand_row = nullptr;
  p.status = device_status_ptr();
  if (p.nsplit <= 1) {
    topk_row_kernel<<<T, kThreads, smem, st>>>(p);
  } else {
    // every slot of the candidate lists is written by the split pass (rows or padding), so
    // nothing left by an earlier call is ever read
    p.cand_key = static_cast<uint32_t*>(scratch);
    p.cand_row = p.cand_key + (size_t)T * p.nsplit * k_top;
    topk_part_kernel<<<dim3(p.nsplit, T), kThreads, sizeof(Shared), st>>>(p);
    topk_merge_kernel<<<T, kThreads, msmem, st>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? DS4X_OK : DS4X_ERR_CUDA;
}
