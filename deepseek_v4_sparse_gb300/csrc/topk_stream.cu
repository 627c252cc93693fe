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
// Rows up to 32768 long are staged in shared memory and resolved with a histogram of the keys
// (one pass for min / max, one for the histogram, one to mark the bins above the boundary bin
// and collect the boundary bin, whose rows are then ranked exactly).
// A decode-sized row (few tokens, e.g. one token over 262k rows) is spread over many CTAs with
// the same histogram scheme run across the grid in three launches (see "long rows").
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

struct alignas(16) Shared {
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

// The multiplier of nb bins over `range` keys (range > nb): about nb * 2^32 / range, computed in
// fp32 (a few instructions where the 64-bit integer quotient is a long routine) and lowered by a
// relative 2^-20, well above the fp32 quotient's error (under 2^-22), so that it never exceeds
// the exact quotient: bin = umulhi(key - min, mult) then stays below nb.  Any multiplier keeps the
// bins monotone in the key, and every CTA computes the same value from the same range.
__device__ __forceinline__ uint32_t bin_mult(uint64_t range, uint32_t nb) {
  const float q = (float)nb * 4294967296.0f / (float)range;
  return (uint32_t)(q * 0.999999f);
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

// Exact top-k of one visible score row (staged in shared memory) with the histogram path.
// Returns false (having written nothing but shared memory) when every key is equal or the
// boundary bin holds more rows than the candidate buffer (massive ties); the caller then runs
// the streaming path.
__device__ bool topk_row_hist(Shared& sh, uint32_t* bitmap, float* srow, int n, int k_top, int32_t* out,
                              int32_t* count_out) {
  const int tid = threadIdx.x;
  const int nv = (n + 3) >> 2;  // 4-row vectors (the staged row is padded to a whole vector)
  // pass A: key range; the staged scores are replaced by their ordered keys, which the later
  // passes read as they are (the streaming fallback reads the row from global memory)
  uint4* skey = reinterpret_cast<uint4*>(srow);
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  for (int v = tid; v < nv; v += kThreads) {
    const float4 x = reinterpret_cast<const float4*>(srow)[v];
    const uint4 k = make_uint4(ordered_key(x.x), ordered_key(x.y), ordered_key(x.z), ordered_key(x.w));
    skey[v] = k;
    const int j = 4 * v;
    const uint32_t k4[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (j + c < n) {
        mn = min(mn, k4[c]);
        mx = max(mx, k4[c]);
      }
  }
  uint32_t kmin, kmax;
  block_minmax32(mn, mx, sh, &kmin, &kmax);
  if (kmin == kmax) return false;  // one value everywhere: every row ties
  const uint64_t range = static_cast<uint64_t>(kmax - kmin) + 1;
  // at most kBins key values: the capped multiplier 2^32 - 1 gives bin max(d - 1, 0), d = key - kmin,
  // still monotone and below kBins
  const uint32_t mult = range <= (uint64_t)kBins ? 0xFFFFFFFFu : bin_mult(range, kBins);
  // pass B: histogram
  for (int i = tid; i < kBins; i += kThreads) sh.bins[i] = 0;
  __syncthreads();
  for (int v = tid; v < nv; v += kThreads) {
    const uint4 k = skey[v];
    const int j = 4 * v;
    const uint32_t k4[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (j + c < n) atomicAdd(&sh.bins[bin_of(k4[c], kmin, mult)], 1u);
  }
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
  const int nv_pad = (nv + kThreads - 1) / kThreads * kThreads;  // whole warps take part in append
  for (int v = tid; v < nv_pad; v += kThreads) {
    const int j = 4 * v;
    uint32_t k4[4] = {0, 0, 0, 0}, r4[4];
    bool b4[4] = {false, false, false, false};
    uint32_t nib = 0;
    if (v < nv) {
      const uint4 k = skey[v];
      k4[0] = k.x;
      k4[1] = k.y;
      k4[2] = k.z;
      k4[3] = k.w;
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
    // the boundary bin holds few rows: most warps have none of them in a step and skip the ballots
    if (__any_sync(0xffffffffu, b4[0] || b4[1] || b4[2] || b4[3])) append(sh, k4, r4, b4);
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
  uint8_t* long_ws;     // long-row mode: one LongLayout block per token
  uint32_t* gbar;       // one-launch long-row mode: a barrier counter per token (zeroed before the launch)
  int nslice;           // long-row mode: CTAs per token
  int* status;
  // one-launch long-row mode, one token: n_range_slots slots of 4 words written by the scorer (the
  // min and max ordered key of the scores a CTA wrote, the fourth largest of its threads' maximum
  // keys, 0), which also zeroed the token's scratch (nullptr: the kernel zeroes it and finds the
  // key range itself)
  const uint32_t* range_slots;
  int n_range_slots;
};

// One CTA per token: the whole row.
__global__ void __launch_bounds__(kThreads) topk_row_kernel(const KParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem_raw[];
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
    // offsets from the (16-byte aligned) base, so that srow stays a shared-space pointer
    const size_t srow_off = (sizeof(Shared) + (size_t)((p.S + 31) / 32) * sizeof(uint32_t) + 15) & ~size_t(15);
    float* srow = reinterpret_cast<float*>(smem_raw + srow_off);
    __shared__ uint64_t row_bar;
    if (!stage_row(row, n, srow, &row_bar, p.status)) return;
    if (topk_row_hist(sh, bitmap, srow, n, p.k_top, out, cnt_out)) return;
    __syncthreads();
  }
  RowSource src{row};
  const uint64_t thr = stream_select(sh, src, 0, n, p.k_top);
  emit_sorted(sh, bitmap, thr, n, p.k_top, out, cnt_out);
}

// ------------------------------------------------------------- register-resident rows
// Rows of up to B * NPT scores (prefill chunks): one CTA per token, thread i holding the ordered
// keys of rows [i*NPT, (i+1)*NPT) in registers, read once from global memory with nothing
// staged.  Rounds of the monotone histogram narrow the undecided rows ("candidates"): rows in
// bins above the boundary bin are taken, rows below it dropped, and the boundary bin's rows are
// the next round's candidates, until the boundary bin is taken whole, holds few enough rows to
// rank directly by the composite order, or all its rows share one key (then the lowest rows
// win, the tie rule).  A round maps the candidates' key range [lo, hi] onto NB bins (identity
// when the range is that small), so each round shrinks the range by that factor: at most four
// rounds for 32-bit keys and 2048 bins, eight for 256.  The selected rows are written in ascending order by one
// block scan.  The result is the same set as every other path's: the composite order is total.
constexpr int kRegRank = 256;   // boundary bins of up to this many rows are ranked directly
constexpr int kRegRounds = 12;  // more than a 32-bit key range can need with 256 bins or more

template <int NB>
struct RegShared {
  uint32_t bins[NB];
  uint32_t wmin[32], wmax[32], wsum[32];
  uint64_t cand[kRegRank];
  uint64_t cthr;
  uint32_t ncand, bstar, above, cntb;
};

// Block min / max (one barrier; the caller keeps wmin / wmax unwritten until every thread has
// passed a later barrier).
template <int B, class Sh>
__device__ __forceinline__ void reg_minmax(uint32_t mn, uint32_t mx, Sh& sh, uint32_t& omin, uint32_t& omax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sh.wmin[warp] = mn;
    sh.wmax[warp] = mx;
  }
  __syncthreads();
  // every warp reduces the per-warp values itself: one shared load a lane, then shuffles
  mn = lane < B / 32 ? sh.wmin[lane] : 0xFFFFFFFFu;
  mx = lane < B / 32 ? sh.wmax[lane] : 0u;
#pragma unroll
  for (int o = B / 64; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  omin = __shfl_sync(0xffffffffu, mn, 0);  // lanes past the warp count reduced only identities
  omax = __shfl_sync(0xffffffffu, mx, 0);
}

// Inclusive block scan (one barrier; same rule for wsum).
template <int B, class Sh>
__device__ __forceinline__ uint32_t reg_scan(uint32_t v, Sh& sh, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) sh.wsum[warp] = v;
  __syncthreads();
  // every warp scans the per-warp totals itself: one shared load a lane, then shuffles
  uint32_t x = lane < B / 32 ? sh.wsum[lane] : 0u;
#pragma unroll
  for (int o = 1; o < B / 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += u;
  }
  total = __shfl_sync(0xffffffffu, x, B / 32 - 1);
  const uint32_t upto = __shfl_sync(0xffffffffu, x, warp);  // totals of warps 0..warp
  return v + upto - __shfl_sync(0xffffffffu, v, 31);
}

template <int B, int NPT, int NB>
__global__ void __launch_bounds__(B) topk_reg_kernel(const KParams p) {
  static_assert(B % 32 == 0 && B <= 1024 && NB % B == 0 && NB >= 256 && NPT % 4 == 0 && NPT <= 32, "shape");
  pdl_wait();
  pdl_trigger();
  __shared__ RegShared<NB> sh;
  const int t = blockIdx.x, tid = threadIdx.x;
  const int n = n_visible(p.positions, t, p.ratio, p.S);
  int32_t* out = p.indices + (int64_t)t * p.k_top;
  int32_t* cnt_out = p.counts ? p.counts + t : nullptr;
  if (n <= p.k_top) {
    for (int i = tid; i < p.k_top; i += B) out[i] = i < n ? i : -1;
    if (cnt_out && tid == 0) *cnt_out = n;
    return;
  }
  const float* row = p.scores + (int64_t)t * p.ld;
  const int r0 = tid * NPT;
  uint32_t key[NPT];
  uint32_t cand = 0;  // bit i: row r0 + i is undecided
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && r0 + NPT <= n) {
#pragma unroll
    for (int v = 0; v < NPT / 4; ++v) {
      const float4 x = __ldcs(reinterpret_cast<const float4*>(row + r0) + v);
      key[4 * v] = ordered_key(x.x);
      key[4 * v + 1] = ordered_key(x.y);
      key[4 * v + 2] = ordered_key(x.z);
      key[4 * v + 3] = ordered_key(x.w);
    }
    cand = NPT == 32 ? 0xFFFFFFFFu : ((1u << NPT) - 1u);
  } else {
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
      const bool valid = r0 + i < n;
      key[i] = valid ? ordered_key(__ldcs(row + r0 + i)) : 0u;
      cand |= valid ? (1u << i) : 0u;
    }
  }
  uint32_t sel = 0;
  int need = p.k_top;
  for (int i = tid; i < NB; i += B) sh.bins[i] = 0;
  bool done = false;
  for (int round = 0; round < kRegRounds && !done; ++round) {
    uint32_t mn = 0xFFFFFFFFu, mx = 0;
#pragma unroll
    for (int i = 0; i < NPT; ++i)
      if ((cand >> i) & 1u) {
        mn = min(mn, key[i]);
        mx = max(mx, key[i]);
      }
    uint32_t lo, hi;
    reg_minmax<B>(mn, mx, sh, lo, hi);  // its barrier also orders the bins' zeroing
    if (lo == hi) {
      // one key left: the need lowest candidate rows win
      const uint32_t c = __popc(cand);
      uint32_t total;
      uint32_t rank = reg_scan<B>(c, sh, total) - c;
#pragma unroll
      for (int i = 0; i < NPT; ++i)
        if ((cand >> i) & 1u) {
          if ((int)rank < need) sel |= 1u << i;
          ++rank;
        }
      done = true;
      break;
    }
    const uint64_t range = (uint64_t)(hi - lo) + 1u;
    const bool ident = range <= (uint64_t)NB;
    const uint32_t mult = ident ? 0u : bin_mult(range, NB);
#pragma unroll
    for (int i = 0; i < NPT; ++i)
      if ((cand >> i) & 1u) {
        const uint32_t d = key[i] - lo;
        atomicAdd(&sh.bins[ident ? d : __umulhi(d, mult)], 1u);
      }
    __syncthreads();
    // boundary bin, counted from the top: thread tid owns bins [NB - BPT(tid+1), NB - BPT tid)
    constexpr int BPT = NB / B;
    const int b_hi = NB - BPT * tid;
    uint32_t mine = 0;
#pragma unroll
    for (int q = 0; q < BPT; ++q) mine += sh.bins[b_hi - 1 - q];
    uint32_t total;
    uint32_t above = reg_scan<B>(mine, sh, total) - mine;
#pragma unroll 4
    for (int q = 0; q < BPT; ++q) {
      const uint32_t c = sh.bins[b_hi - 1 - q];
      if (above < (uint32_t)need && above + c >= (uint32_t)need) {
        sh.bstar = (uint32_t)(b_hi - 1 - q);
        sh.above = above;
        sh.cntb = c;
      }
      above += c;
    }
    if (tid == 0) sh.ncand = 0;
    __syncthreads();
    const uint32_t bstar = sh.bstar;
    const int cntb = (int)sh.cntb;
    need -= (int)sh.above;
    uint32_t inb = 0;
#pragma unroll
    for (int i = 0; i < NPT; ++i)
      if ((cand >> i) & 1u) {
        const uint32_t d = key[i] - lo;
        const uint32_t b = ident ? d : __umulhi(d, mult);
        if (b > bstar) sel |= 1u << i;
        else if (b == bstar) inb |= 1u << i;
      }
    cand = inb;
    if (cntb == need) {  // the boundary bin is taken whole
      sel |= cand;
      done = true;
      break;
    }
    if (cntb <= kRegRank) {
      // rank the boundary bin's rows directly: the need-th largest composite is the threshold
#pragma unroll
      for (int i = 0; i < NPT; ++i)
        if ((cand >> i) & 1u) sh.cand[atomicAdd(&sh.ncand, 1u)] = composite(key[i], (uint32_t)(r0 + i));
      __syncthreads();
      for (int j = tid; j < cntb; j += B) {
        const uint64_t cj = sh.cand[j];
        int greater = 0;
        for (int m = 0; m < cntb; ++m) greater += sh.cand[m] > cj ? 1 : 0;
        if (greater == need - 1) sh.cthr = cj;
      }
      __syncthreads();
      const uint64_t cthr = sh.cthr;
#pragma unroll
      for (int i = 0; i < NPT; ++i)
        if (((cand >> i) & 1u) && composite(key[i], (uint32_t)(r0 + i)) >= cthr) sel |= 1u << i;
      done = true;
      break;
    }
    // next round on the boundary bin's rows
    __syncthreads();  // every thread has read the bins and the broadcast values
    for (int i = tid; i < NB; i += B) sh.bins[i] = 0;
  }
  if (!done) {  // cannot happen (each round shrinks the key range by NB); reported, not hidden
    if (tid == 0) report_timeout(p.status, 60);
    return;
  }
  __syncthreads();  // wsum is rewritten below
  const uint32_t c = __popc(sel);
  uint32_t total;
  int pos = (int)(reg_scan<B>(c, sh, total) - c);
#pragma unroll
  for (int i = 0; i < NPT; ++i)
    if ((sel >> i) & 1u) out[pos++] = r0 + i;
  for (int i = (int)total + tid; i < p.k_top; i += B) out[i] = -1;
  if (cnt_out && tid == 0) *cnt_out = (int)total;
}

// ---------------------------------------------------------------------------- long rows
// A token's row is spread over P = ceil(S / kSliceRows) CTAs, one slice each, in three launches
// that run the histogram scheme of the staged path across the grid:
//   long_minmax_kernel  min and max of the slice's ordered keys into the token's slot table;
//                       zeroes the token's histogram, bitmap and counters
//   long_hist_kernel    the row's min / max from the slots, then a kGBins-bin monotone histogram
//                       of the slice (shared memory, then global atomics); the token's last CTA
//                       (atomic ticket, no waiting) finds the boundary bin b* holding the k_top-th
//                       largest key and the number of rows above it
//   long_mark_kernel    rows in bins above b* are set in the token's bitmap (a warp owns a word:
//                       plain stores), rows in b* are collected; the token's last CTA ranks the
//                       collected rows by the composite order, adds the k_top - above best to the
//                       bitmap and emits it in ascending row order (when more than kCandCap rows
//                       share b*, it runs the streaming routine over the whole row instead).
constexpr int kSliceRows = 2048;   // a multiple of 32: every bitmap word lies in one slice
constexpr int kSlicePer = kSliceRows / kThreads;  // rows of a slice per thread, all loaded at once
constexpr int kGBins = 1024;
constexpr int kCandCap = 8192;

struct LongCtl {
  uint32_t kmin, mult, bstar, above;
  uint32_t ncand, done2, done3, whole;  // whole: one-launch mode, slice 0 emitted the whole row
  uint32_t npre;                        // range mode: rows at or above the lower bound (prefilter)
};

struct LongLayout {  // byte offsets inside one token's block of the workspace
  size_t ctl, slots, scnt, hist, bitmap, ckey, crow, rslots, total;
};
constexpr int kMaxRangeSlots = 1024;  // scorer CTAs whose key ranges the one-token mode takes
constexpr int kPreCap = 2048;         // prefilter candidates every slice ranks (kept in ckey / crow)
constexpr int kPrePer = kPreCap / kThreads;
static_assert(kPreCap <= kCandCap && kPreCap % kThreads == 0, "prefilter candidates");

__host__ __device__ inline size_t align_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

__host__ __device__ inline LongLayout long_layout(int S) {
  const size_t P = (size_t)(S + kSliceRows - 1) / kSliceRows;
  const size_t W = (size_t)(S + 31) / 32;
  LongLayout L;
  size_t o = 0;
  L.ctl = o;
  o += sizeof(LongCtl);
  L.slots = o;
  o = align_up(o + P * 2 * sizeof(uint32_t), 16);
  L.scnt = o;  // rows each slice selects (one-launch mode)
  o = align_up(o + P * sizeof(uint32_t), 16);
  L.hist = o;
  o += (size_t)kGBins * sizeof(uint32_t);
  L.bitmap = o;
  o = align_up(o + W * sizeof(uint32_t), 16);
  L.ckey = o;
  o += (size_t)kCandCap * sizeof(uint32_t);
  L.crow = o;
  o += (size_t)kCandCap * sizeof(uint32_t);
  o = align_up(o, 16);
  L.rslots = o;  // outside the zeroed part [ctl, bitmap end): the scorer writes it while others zero
  o += (size_t)4 * kMaxRangeSlots * sizeof(uint32_t);
  L.total = align_up(o, 256);
  return L;
}

// bin of an ordered key over [kmin, kmax]: direct when the range has at most kGBins values
// (mult == 0), else umulhi(key - kmin, floor(kGBins 2^32 / range)); non-decreasing in the key.
// A key outside [kmin, kmax] lands in an end bin rather than past the table: the range can come
// from another kernel (the scorer's key ranges), and scores that do not match it (a buffer
// rewritten in between) must not index shared memory out of bounds.
__device__ __forceinline__ uint32_t long_bin(uint32_t key, uint32_t kmin, uint32_t mult) {
  const uint32_t d = key > kmin ? key - kmin : 0u;
  return min(mult == 0 ? d : __umulhi(d, mult), (uint32_t)(kGBins - 1));
}

// Block-wide reduction helpers on a few words of static shared memory.
__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, uint32_t* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  uint32_t r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = min(r, red[w]);
  return r;
}
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  uint32_t r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = max(r, red[w]);
  return r;
}

// Block-wide min and max together (two barriers; red_mn / red_mx stay unwritten until every
// thread has passed a later barrier).
__device__ __forceinline__ void block_minmax_u32(uint32_t& mn, uint32_t& mx, uint32_t* red_mn, uint32_t* red_mx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    red_mn[threadIdx.x >> 5] = mn;
    red_mx[threadIdx.x >> 5] = mx;
  }
  __syncthreads();
  mn = red_mn[0];
  mx = red_mx[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    mn = min(mn, red_mn[w]);
    mx = max(mx, red_mx[w]);
  }
}

// The block's values, one a thread, in descending order: thread i returns the i-th largest.
// A bitonic network; partners 32 or more apart trade through xs (2 x kThreads words, the halves
// taken in turn, so one barrier a step suffices: a half is rewritten only after the next barrier).
__device__ __forceinline__ uint32_t block_sort_desc(uint32_t v, uint32_t* xs) {
  const int i = threadIdx.x;
  int half = 0;
#pragma unroll
  for (int k = 2; k <= kThreads; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      uint32_t o;
      if (j >= 32) {
        uint32_t* x = xs + half * kThreads;
        x[i] = v;
        __syncthreads();
        o = x[i ^ j];
        half ^= 1;
      } else {
        o = __shfl_xor_sync(0xffffffffu, v, j);
      }
      v = (((i & k) == 0) == ((i & j) == 0)) ? max(v, o) : min(v, o);
    }
  }
  return v;
}

// the thread's rows lo + i * kThreads + threadIdx.x of the slice as ordered keys (all loads issued
// before any is used); rows at or past hi are flagged invalid
__device__ __forceinline__ void load_slice(const float* row, int lo, int hi, uint32_t (&k)[kSlicePer],
                                           bool (&v)[kSlicePer]) {
  float x[kSlicePer];
#pragma unroll
  for (int i = 0; i < kSlicePer; ++i) {
    const int j = lo + i * kThreads + threadIdx.x;
    v[i] = j < hi;
    x[i] = v[i] ? __ldcs(row + j) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < kSlicePer; ++i) k[i] = ordered_key(x[i]);
}

__global__ void __launch_bounds__(kThreads) long_minmax_kernel(const KParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t red[kWarps];
  const int t = blockIdx.y, part = blockIdx.x, P = gridDim.x;
  const LongLayout L = long_layout(p.S);
  uint8_t* blk = p.long_ws + (size_t)t * L.total;
  uint32_t* hist = reinterpret_cast<uint32_t*>(blk + L.hist);
  uint32_t* bm = reinterpret_cast<uint32_t*>(blk + L.bitmap);
  const int W = (p.S + 31) / 32;
  for (int i = part * kThreads + threadIdx.x; i < kGBins; i += P * kThreads) hist[i] = 0;
  for (int i = part * kThreads + threadIdx.x; i < W; i += P * kThreads) bm[i] = 0;
  if (part == 0 && threadIdx.x < (int)(sizeof(LongCtl) / 4)) reinterpret_cast<uint32_t*>(blk + L.ctl)[threadIdx.x] = 0;
  const int n = n_visible(p.positions, t, p.ratio, p.S);
  if (n <= p.k_top) return;
  const int lo = part * kSliceRows, hi = min(n, lo + kSliceRows);
  const float* row = p.scores + (int64_t)t * p.ld;
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  uint32_t k[kSlicePer];
  bool v[kSlicePer];
  load_slice(row, lo, hi, k, v);
#pragma unroll
  for (int i = 0; i < kSlicePer; ++i)
    if (v[i]) {
      mn = min(mn, k[i]);
      mx = max(mx, k[i]);
    }
  mn = block_min_u32(mn, red);
  mx = block_max_u32(mx, red);
  if (threadIdx.x == 0) {  // an empty slice leaves the neutral pair (~0, 0)
    uint32_t* slot = reinterpret_cast<uint32_t*>(blk + L.slots) + 2 * part;
    slot[0] = mn;
    slot[1] = mx;
  }
}

__global__ void __launch_bounds__(kThreads) long_hist_kernel(const KParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t sh_hist[kGBins];
  __shared__ uint32_t red[kWarps];
  __shared__ int sh_last;
  const int t = blockIdx.y, part = blockIdx.x, P = gridDim.x;
  const int n = n_visible(p.positions, t, p.ratio, p.S);
  if (n <= p.k_top) return;
  const LongLayout L = long_layout(p.S);
  uint8_t* blk = p.long_ws + (size_t)t * L.total;
  LongCtl* ctl = reinterpret_cast<LongCtl*>(blk + L.ctl);
  uint32_t* hist = reinterpret_cast<uint32_t*>(blk + L.hist);
  const uint32_t* slots = reinterpret_cast<const uint32_t*>(blk + L.slots);
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  for (int i = threadIdx.x; i < P; i += kThreads) {
    mn = min(mn, __ldcg(slots + 2 * i));
    mx = max(mx, __ldcg(slots + 2 * i + 1));
  }
  const int lo = part * kSliceRows, hi = min(n, lo + kSliceRows);
  const float* row = p.scores + (int64_t)t * p.ld;
  uint32_t k[kSlicePer];
  bool v[kSlicePer];
  load_slice(row, lo, hi, k, v);  // in flight while the slots are reduced
  const uint32_t kmin = block_min_u32(mn, red);
  const uint32_t kmax = block_max_u32(mx, red);
  const uint64_t range = (uint64_t)kmax - kmin + 1;
  const uint32_t mult = range <= (uint64_t)kGBins ? 0u : bin_mult(range, kGBins);
  for (int i = threadIdx.x; i < kGBins; i += kThreads) sh_hist[i] = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kSlicePer; ++i)
    if (v[i]) atomicAdd(&sh_hist[long_bin(k[i], kmin, mult)], 1u);
  __syncthreads();
  for (int i = threadIdx.x; i < kGBins; i += kThreads)
    if (sh_hist[i]) atomicAdd(&hist[i], sh_hist[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sh_last = atomicAdd(&ctl->done2, 1u) == (uint32_t)(P - 1);
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  // the token's last CTA: suffix counts from the top bin down; thread i owns the 16 bins
  // [kGBins - 16 (i+1), kGBins - 16 i)
  constexpr int kPer = kGBins / kThreads;
  uint32_t c[kPer], own = 0;
  const int top = kGBins - kPer * threadIdx.x;  // bins top-1 .. top-kPer
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    c[i] = __ldcg(hist + top - 1 - i);
    own += c[i];
  }
  // inclusive prefix over threads (thread 0 = highest bins)
  uint32_t incl = own;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  uint32_t before_w = 0;
  for (int w = 0; w < warp; ++w) before_w += red[w];
  incl += before_w;
  const uint32_t need = (uint32_t)p.k_top;
  uint32_t run = incl - own;  // rows in bins above this thread's range
  if (run < need && incl >= need) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (run + c[i] >= need) {
        ctl->kmin = kmin;
        ctl->mult = mult;
        ctl->bstar = (uint32_t)(top - 1 - i);
        ctl->above = run;
        break;
      }
      run += c[i];
    }
  }
}

__global__ void __launch_bounds__(kThreads) long_mark_kernel(const KParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  uint32_t* sbm = reinterpret_cast<uint32_t*>(smem_raw + sizeof(Shared));
  __shared__ int sh_last;
  const int t = blockIdx.y, part = blockIdx.x, P = gridDim.x;
  const int n = n_visible(p.positions, t, p.ratio, p.S);
  int32_t* out = p.indices + (int64_t)t * p.k_top;
  int32_t* cnt_out = p.counts ? p.counts + t : nullptr;
  if (n <= p.k_top) {
    if (part == 0) emit_shortcut(n, p.k_top, out, cnt_out);
    return;
  }
  const LongLayout L = long_layout(p.S);
  uint8_t* blk = p.long_ws + (size_t)t * L.total;
  LongCtl* ctl = reinterpret_cast<LongCtl*>(blk + L.ctl);
  uint32_t* bm = reinterpret_cast<uint32_t*>(blk + L.bitmap);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(blk + L.ckey);
  uint32_t* crow = reinterpret_cast<uint32_t*>(blk + L.crow);
  const int lo = part * kSliceRows, hi = min(n, lo + kSliceRows);
  const float* row = p.scores + (int64_t)t * p.ld;
  uint32_t ks[kSlicePer];
  bool vs[kSlicePer];
  load_slice(row, lo, hi, ks, vs);
  const uint32_t kmin = __ldcg(&ctl->kmin), mult = __ldcg(&ctl->mult), bstar = __ldcg(&ctl->bstar);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < kSlicePer; ++i) {
    const int base = lo + i * kThreads + warp * 32;  // row of lane 0: a multiple of 32
    if (base >= hi) break;
    const int j = base + lane;
    const bool valid = vs[i];
    const uint32_t key = ks[i];
    const uint32_t b = valid ? long_bin(key, kmin, mult) : 0u;
    const uint32_t word = __ballot_sync(0xffffffffu, valid && b > bstar);
    if (lane == 0) bm[base >> 5] = word;  // this warp owns the word (base is a multiple of 32)
    const bool inb = valid && b == bstar;
    const uint32_t bal = __ballot_sync(0xffffffffu, inb);
    if (bal) {
      uint32_t slot0 = 0;
      if (lane == 0) slot0 = atomicAdd(&ctl->ncand, (uint32_t)__popc(bal));
      slot0 = __shfl_sync(0xffffffffu, slot0, 0);
      if (inb) {
        const uint32_t slot = slot0 + __popc(bal & ((1u << lane) - 1u));
        if (slot < (uint32_t)kCandCap) {
          ckey[slot] = key;
          crow[slot] = (uint32_t)j;
        }
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sh_last = atomicAdd(&ctl->done3, 1u) == (uint32_t)(P - 1);
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  const int m = (int)__ldcg(&ctl->ncand);
  if (m > kCandCap) {  // too many rows share the boundary bin: rank the whole row
    const uint64_t thr = stream_select(sh, RowSource{row}, 0, n, p.k_top);
    emit_sorted(sh, sbm, thr, n, p.k_top, out, cnt_out);
    return;
  }
  const int need = p.k_top - (int)__ldcg(&ctl->above);
  const int nw = (n + 31) >> 5;
  {  // the token's bitmap into shared memory: 16-byte loads, eight in flight per thread
    const int nq = (nw + 3) >> 2;  // the bitmap's allocation is a multiple of 16 bytes
    const uint4* src = reinterpret_cast<const uint4*>(bm);
    uint4* dst = reinterpret_cast<uint4*>(sbm);
    for (int q0 = 0; q0 < nq; q0 += 8 * kThreads) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = q0 + i * kThreads + threadIdx.x;
        if (q < nq) v[i] = __ldcg(src + q);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = q0 + i * kThreads + threadIdx.x;
        if (q < nq) dst[q] = v[i];
      }
    }
  }
  const uint64_t thr = stream_select(sh, CandSource{ckey, crow}, 0, m, need);
  if (sh.count > need) compact(sh, thr);
  for (int j = threadIdx.x; j < sh.count; j += kThreads) {
    const uint32_t r = sh.row[j];
    atomicOr(&sbm[r >> 5], 1u << (r & 31));
  }
  __syncthreads();
  emit_bitmap(sh, sbm, n, p.k_top, out, cnt_out);
}

// ----------------------------------------------------------------- long rows, one launch
// When a token's slices can all be resident at once (a cooperative launch), the scheme above
// runs in one kernel: a per-token grid barrier (an atomic counter polled with a time limit)
// separates the phases, each slice keeps its keys in registers throughout, and the emission is
// parallel: after slice 0 has ranked the boundary bin, every slice writes its selected rows at
// the offset given by the counts of the slices before it.

// Arrive on the token's counter and wait until it reaches `target` (= slices x phase).
__device__ bool token_barrier(uint32_t* counter, uint32_t target, int* status, int site) {
  __shared__ int sh_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(counter, 1u);
    int ok = 1;
    const uint64_t t0 = global_timer_ns();
    while (true) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
      if (v >= target) break;
      if (global_timer_ns() - t0 > DS4X_WAIT_TIMEOUT_NS) {
        report_timeout(status, site);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    sh_ok = ok;
  }
  __syncthreads();
  return sh_ok != 0;
}

__global__ void __launch_bounds__(kThreads) long_coop_kernel(const KParams p) {
  pdl_wait();  // returns at once unless launched as a programmatic dependent of the scorer
  extern __shared__ uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  uint32_t* sbm = reinterpret_cast<uint32_t*>(smem_raw + sizeof(Shared));  // whole-row fallback only
  __shared__ uint32_t sh_hist[kGBins];
  __shared__ uint32_t red[kWarps];
  __shared__ uint32_t red2[kWarps];
  __shared__ uint32_t sh_b[3];
  constexpr int kSliceWords = kSliceRows / 32;
  __shared__ uint64_t cand[kThreads];  // boundary-bin candidates' composites
  __shared__ uint32_t add[kThreads];   // winners among the candidates, per slice
  __shared__ uint32_t words[kSliceWords];
  __shared__ uint32_t n_in_b;
  const int t = blockIdx.y, part = blockIdx.x, P = gridDim.x;
  const int n = n_visible(p.positions, t, p.ratio, p.S);
  int32_t* out = p.indices + (int64_t)t * p.k_top;
  int32_t* cnt_out = p.counts ? p.counts + t : nullptr;
  if (n <= p.k_top) {  // every slice of the token leaves here, before any barrier
    if (part == 0) emit_shortcut(n, p.k_top, out, cnt_out);
    return;
  }
  const LongLayout L = long_layout(p.S);
  uint8_t* blk = p.long_ws + (size_t)t * L.total;
  LongCtl* ctl = reinterpret_cast<LongCtl*>(blk + L.ctl);
  uint32_t* slots = reinterpret_cast<uint32_t*>(blk + L.slots);
  uint32_t* scnt = reinterpret_cast<uint32_t*>(blk + L.scnt);
  uint32_t* hist = reinterpret_cast<uint32_t*>(blk + L.hist);
  uint32_t* bm = reinterpret_cast<uint32_t*>(blk + L.bitmap);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(blk + L.ckey);
  uint32_t* crow = reinterpret_cast<uint32_t*>(blk + L.crow);
  uint32_t* counter = p.gbar + t;
  const int W = (p.S + 31) / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // range mode: the scorer zeroed this token's scratch and wrote the key ranges of what it scored,
  // so phase 1 and its grid barrier fall away (nb counts the grid barriers passed); with a bound on
  // the row's k_top-th key from those slots, the prefilter below usually replaces phases 2 to 5
  const bool given = p.range_slots != nullptr;
  uint32_t nb = 0;

  // phase 1: zero this slice's share of the scratch; the slice's keys; their min and max
  if (!given) {
    for (int i = part * kThreads + threadIdx.x; i < kGBins; i += P * kThreads) hist[i] = 0;
    for (int i = part * kThreads + threadIdx.x; i < W; i += P * kThreads) bm[i] = 0;
    if (part == 0 && threadIdx.x < (int)(sizeof(LongCtl) / 4)) reinterpret_cast<uint32_t*>(ctl)[threadIdx.x] = 0;
  }
  const int lo = part * kSliceRows, hi = min(n, lo + kSliceRows);
  const int w0 = lo >> 5;  // this slice's first bitmap word
  const bool my_word_in = threadIdx.x < kSliceWords && lo + 32 * (int)threadIdx.x < hi;
  const float* row = p.scores + (int64_t)t * p.ld;
  const int nrs = given ? p.n_range_slots : P;
  // range mode: the scorer's slots are loaded together with the slice (one round trip to L2); when
  // the prefilter runs (at most kThreads slots) a thread takes at most one slot and keeps its bound
  const int m_rep = (p.k_top + 3) / 4;  // slots whose fourth-largest keys bound the k_top-th key
  const bool prefilter = given && p.k_top > 0 && nrs <= kThreads && m_rep <= nrs;
  uint32_t gmn = 0xFFFFFFFFu, gmx = 0, rep = 0;
  if (given)
    for (int i = threadIdx.x; i < nrs; i += kThreads) {
      const uint4 sl = __ldcg(reinterpret_cast<const uint4*>(p.range_slots) + i);
      gmn = min(gmn, sl.x);
      gmx = max(gmx, sl.y);
      rep = sl.z;
    }
  uint32_t k[kSlicePer];
  bool v[kSlicePer];
  load_slice(row, lo, hi, k, v);
  for (int i = threadIdx.x; i < kGBins; i += kThreads) sh_hist[i] = 0;  // ordered by the next barrier
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  if (!given) {
#pragma unroll
    for (int i = 0; i < kSlicePer; ++i)
      if (v[i]) {
        mn = min(mn, k[i]);
        mx = max(mx, k[i]);
      }
    block_minmax_u32(mn, mx, red, red2);
    if (threadIdx.x == 0) {
      slots[2 * part] = mn;
      slots[2 * part + 1] = mx;
    }
    if (!token_barrier(counter, ++nb * (uint32_t)P, p.status, 60)) return;
    for (int i = threadIdx.x; i < nrs; i += kThreads) {
      gmn = min(gmn, __ldcg(slots + 2 * i));
      gmx = max(gmx, __ldcg(slots + 2 * i + 1));
    }
  }

  // Prefilter (range mode). Each of the scorer's CTAs reported the fourth largest of its threads'
  // maximum keys, so at least four of its visible scores are at or above that report. Take L, the
  // m_rep-th largest report (m_rep = ceil(k_top / 4)): at least 4 m_rep >= k_top visible scores
  // are at or above L, hence so is the k_top-th largest key, and every row of the top-k has a key
  // at or above L. The slices collect those rows (about twice k_top in a row of independent
  // scores) in one list, pass one grid barrier, and each slice then ranks the whole list itself:
  // a histogram of its keys over [L, max], the boundary bin's rows ranked exactly. Each slice
  // knows from the list alone how many selected rows lie before it and writes its own rows in
  // ascending order. Exactness rests on the count alone: whatever the reports, when the list holds
  // at least k_top rows, the k_top-th largest key is at or above L. When it holds fewer (scores
  // that do not match the reports), more than kPreCap, or the boundary bin more than kThreads
  // rows, every slice sees the same counts and all go on with the histogram phases below.
  if (prefilter) {
    block_minmax_u32(gmn, gmx, red, red2);
    const uint32_t srt = block_sort_desc(rep, sh.key);  // threads past the slots hold 0
    if ((int)threadIdx.x == m_rep - 1) sh_b[2] = srt;
    if (threadIdx.x == 0) n_in_b = 0;
    if (threadIdx.x < kSliceWords) words[threadIdx.x] = 0;
    __syncthreads();
    const uint32_t L = sh_b[2];
    {  // this slice's rows at or above L into the list: one atomic a warp
      uint32_t bal[kSlicePer], tot = 0;
#pragma unroll
      for (int i = 0; i < kSlicePer; ++i) {
        bal[i] = __ballot_sync(0xffffffffu, v[i] && k[i] >= L);
        tot += __popc(bal[i]);
      }
      if (tot) {
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&ctl->npre, tot);
        base = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int i = 0; i < kSlicePer; ++i) {
          if ((bal[i] >> lane) & 1u) {
            const uint32_t slot = base + __popc(bal[i] & lt);
            if (slot < (uint32_t)kPreCap) {
              ckey[slot] = k[i];
              crow[slot] = (uint32_t)(lo + i * kThreads + (int)threadIdx.x);
            }
          }
          base += __popc(bal[i]);
        }
      }
    }
    if (!token_barrier(counter, ++nb * (uint32_t)P, p.status, 64)) return;
    // the count and the whole list at once (entries past the count are not used)
    const int C = (int)__ldcg(&ctl->npre);
    uint32_t ck[kPrePer], cr[kPrePer];
#pragma unroll
    for (int i = 0; i < kPrePer; ++i) {
      ck[i] = __ldcg(ckey + threadIdx.x + i * kThreads);
      cr[i] = __ldcg(crow + threadIdx.x + i * kThreads);
    }
    if (C >= p.k_top && C <= kPreCap) {
      const uint64_t crange = (uint64_t)max(gmx, L) - L + 1;
      const uint32_t cmult = crange <= (uint64_t)kGBins ? 0u : bin_mult(crange, kGBins);
      uint32_t cb[kPrePer];
#pragma unroll
      for (int i = 0; i < kPrePer; ++i) {
        cb[i] = long_bin(ck[i], L, cmult);
        if ((int)threadIdx.x + i * kThreads < C) atomicAdd(&sh_hist[cb[i]], 1u);
      }
      __syncthreads();
      {  // the boundary bin: suffix counts from the top bin down
        constexpr int kPer = kGBins / kThreads;
        uint32_t c[kPer], own = 0;
        const int top = kGBins - kPer * threadIdx.x;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          c[i] = sh_hist[top - 1 - i];
          own += c[i];
        }
        uint32_t total;
        const uint32_t incl = block_scan(own, sh, &total);
        uint32_t run = incl - own;
        const uint32_t need = (uint32_t)p.k_top;
        if (run < need && incl >= need) {
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            if (run + c[i] >= need) {
              sh_b[0] = (uint32_t)(top - 1 - i);
              sh_b[1] = run;
              break;
            }
            run += c[i];
          }
        }
        __syncthreads();
      }
      const uint32_t bstar = sh_b[0], above = sh_b[1];
      const uint32_t nstar = sh_hist[bstar];
      if (nstar <= (uint32_t)kThreads) {
        pdl_trigger();  // this slice has passed its last barrier
        // a selected row: counted when it lies before this slice, marked when in it
        uint32_t before = 0;
        auto take = [&](uint32_t r) {
          if (r < (uint32_t)lo) ++before;
          else if (r < (uint32_t)hi) atomicOr(&words[(r - lo) >> 5], 1u << (r & 31));
        };
#pragma unroll
        for (int i = 0; i < kPrePer; ++i) {
          if ((int)threadIdx.x + i * kThreads >= C || cb[i] < bstar) continue;
          if (cb[i] > bstar) take(cr[i]);
          else cand[atomicAdd(&n_in_b, 1u)] = composite(ck[i], cr[i]);
        }
        __syncthreads();
        if (threadIdx.x < nstar) {  // in iff fewer than need boundary rows beat it
          const uint64_t mine = cand[threadIdx.x];
          int rank = 0;
          for (int j = 0; j < (int)nstar; ++j) rank += cand[j] > mine;
          if (rank < p.k_top - (int)above) take(~static_cast<uint32_t>(mine));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
        if (lane == 0) red[warp] = before;
        __syncthreads();
        uint32_t offset = 0;
        for (int w = 0; w < kWarps; ++w) offset += red[w];
        if (part == 0 && cnt_out && threadIdx.x == 0) *cnt_out = p.k_top;
        const uint32_t word = my_word_in ? words[threadIdx.x] : 0u;
        uint32_t total;
        const uint32_t incl = block_scan((uint32_t)__popc(word), sh, &total);
        uint32_t pos = offset + incl - (uint32_t)__popc(word);
        uint32_t bits = word;
        while (bits) {
          const int b = __ffs(bits) - 1;
          bits &= bits - 1;
          out[pos++] = (w0 + (int)threadIdx.x) * 32 + b;
        }
        return;
      }
      __syncthreads();  // every thread has read the histogram
      for (int i = threadIdx.x; i < kGBins; i += kThreads) sh_hist[i] = 0;  // ordered by phase 2's barriers
    }
  }

  // phase 2: the row's key range from the slots; histogram of the slice into the token's
  block_minmax_u32(gmn, gmx, red, red2);  // its barriers also order the zeroed sh_hist
  const uint32_t kmin = gmn, kmax = gmx;
  const uint64_t range = (uint64_t)kmax - kmin + 1;
  const uint32_t mult = range <= (uint64_t)kGBins ? 0u : bin_mult(range, kGBins);
#pragma unroll
  for (int i = 0; i < kSlicePer; ++i)
    if (v[i]) atomicAdd(&sh_hist[long_bin(k[i], kmin, mult)], 1u);
  __syncthreads();
  for (int i = threadIdx.x; i < kGBins; i += kThreads)
    if (sh_hist[i]) atomicAdd(&hist[i], sh_hist[i]);
  if (!token_barrier(counter, ++nb * (uint32_t)P, p.status, 61)) return;

  // phase 3: every slice finds the boundary bin b* from the token's histogram, writes its words
  // of the bitmap (rows in bins above b*) and collects its rows in b*
  {
    constexpr int kPer = kGBins / kThreads;
    uint32_t c[kPer], own = 0;
    const int top = kGBins - kPer * threadIdx.x;  // this thread's bins: top-1 .. top-kPer
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      c[i] = __ldcg(hist + top - 1 - i);
      own += c[i];
    }
    uint32_t total;
    const uint32_t incl = block_scan(own, sh, &total);  // rows in this thread's bins and above
    uint32_t run = incl - own;
    const uint32_t need = (uint32_t)p.k_top;
    if (run < need && incl >= need) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        if (run + c[i] >= need) {
          sh_b[0] = (uint32_t)(top - 1 - i);
          sh_b[1] = run;
          break;
        }
        run += c[i];
      }
    }
    __syncthreads();
  }
  const uint32_t bstar = sh_b[0], above = sh_b[1];
  uint32_t marked = 0;
#pragma unroll
  for (int i = 0; i < kSlicePer; ++i) {
    const int base = lo + i * kThreads + warp * 32;  // row of lane 0: a multiple of 32
    if (base >= hi) break;
    const int j = base + lane;
    const uint32_t b = v[i] ? long_bin(k[i], kmin, mult) : 0u;
    const uint32_t word = __ballot_sync(0xffffffffu, v[i] && b > bstar);
    if (lane == 0) {
      bm[base >> 5] = word;
      marked += __popc(word);
    }
    const bool inb = v[i] && b == bstar;
    const uint32_t bal = __ballot_sync(0xffffffffu, inb);
    if (bal) {
      uint32_t slot0 = 0;
      if (lane == 0) slot0 = atomicAdd(&ctl->ncand, (uint32_t)__popc(bal));
      slot0 = __shfl_sync(0xffffffffu, slot0, 0);
      if (inb) {
        const uint32_t slot = slot0 + __popc(bal & ((1u << lane) - 1u));
        if (slot < (uint32_t)kCandCap) {
          ckey[slot] = k[i];
          crow[slot] = (uint32_t)j;
        }
      }
    }
  }
  if (lane == 0) red[warp] = marked;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t sum = 0;
    for (int w = 0; w < kWarps; ++w) sum += red[w];
    scnt[part] = sum;
  }
  if (!token_barrier(counter, ++nb * (uint32_t)P, p.status, 62)) return;

  // every value the fast path reads from L2, loaded at once (one round trip instead of four):
  // the candidate count (the same in every slice of the token), the candidates as far as the
  // fast path takes them (kThreads <= kCandCap: the loads stay inside the buffer, entries past the
  // count go unused), the slices' counts and this slice's bitmap words
  const int m_cand = (int)__ldcg(&ctl->ncand);
  const uint32_t my_key = __ldcg(ckey + threadIdx.x), my_row = __ldcg(crow + threadIdx.x);
  const uint32_t my_scnt = (int)threadIdx.x < P ? __ldcg(scnt + threadIdx.x) : 0u;
  const uint32_t my_word = my_word_in ? __ldcg(bm + w0 + threadIdx.x) : 0u;
  if (m_cand <= kThreads && P <= kThreads) {
    // few boundary rows (the usual case): every slice ranks them itself (candidate j is in iff
    // fewer than `need` candidates beat it), so each knows every slice's count without another
    // barrier, adds its own winners to its words and writes its rows after the earlier slices'
    pdl_trigger();  // this slice has passed its last barrier
    static_assert(kThreads <= kCandCap, "speculative candidate loads");
    const int need = p.k_top - (int)above;
    add[threadIdx.x] = 0;
    if (threadIdx.x < kSliceWords) words[threadIdx.x] = 0;
    const uint64_t mine = composite(my_key, my_row);
    if ((int)threadIdx.x < m_cand) cand[threadIdx.x] = mine;
    __syncthreads();
    if ((int)threadIdx.x < m_cand) {
      int rank = 0;
      for (int j = 0; j < m_cand; ++j) rank += cand[j] > mine;
      if (rank < need) {
        atomicAdd(&add[my_row / kSliceRows], 1u);
        if ((int)my_row >= lo && (int)my_row < hi) atomicOr(&words[(my_row - lo) >> 5], 1u << (my_row & 31));
      }
    }
    __syncthreads();
    uint32_t before = (int)threadIdx.x < part ? my_scnt + add[threadIdx.x] : 0u;  // P <= kThreads
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    if (lane == 0) red[warp] = before;
    __syncthreads();
    uint32_t offset = 0;
    for (int w = 0; w < kWarps; ++w) offset += red[w];
    if (part == 0 && cnt_out && threadIdx.x == 0) *cnt_out = p.k_top;
    const uint32_t word = my_word_in ? (my_word | words[threadIdx.x]) : 0u;
    uint32_t total;
    const uint32_t incl = block_scan((uint32_t)__popc(word), sh, &total);
    uint32_t pos = offset + incl - (uint32_t)__popc(word);
    uint32_t bits = word;
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      out[pos++] = (w0 + (int)threadIdx.x) * 32 + b;
    }
    return;
  }

  // phase 4: slice 0 ranks the boundary bin's rows and adds the missing ones (or, when more than
  // kCandCap rows share the bin, ranks and emits the whole row itself)
  if (part == 0) {
    const int m = (int)__ldcg(&ctl->ncand);
    if (m > kCandCap) {
      const uint64_t thr = stream_select(sh, RowSource{row}, 0, n, p.k_top);
      emit_sorted(sh, sbm, thr, n, p.k_top, out, cnt_out);
      if (threadIdx.x == 0) ctl->whole = 1;
    } else if (m <= kThreads) {
      // few candidates: candidate j is in iff fewer than `need` candidates beat it
      const int need = p.k_top - (int)above;
      for (int j = threadIdx.x; j < m; j += kThreads) {
        sh.key[j] = __ldcg(ckey + j);
        sh.row[j] = __ldcg(crow + j);
      }
      __syncthreads();
      if ((int)threadIdx.x < m) {
        const uint64_t mine = composite(sh.key[threadIdx.x], sh.row[threadIdx.x]);
        int rank = 0;
        for (int j = 0; j < m; ++j) rank += composite(sh.key[j], sh.row[j]) > mine;
        if (rank < need) {
          const uint32_t r = sh.row[threadIdx.x];
          atomicOr(&bm[r >> 5], 1u << (r & 31));
          atomicAdd(&scnt[r / kSliceRows], 1u);
        }
      }
      if (cnt_out && threadIdx.x == 0) *cnt_out = p.k_top;
    } else {
      const int need = p.k_top - (int)above;
      const uint64_t thr = stream_select(sh, CandSource{ckey, crow}, 0, m, need);
      if (sh.count > need) compact(sh, thr);
      for (int j = threadIdx.x; j < sh.count; j += kThreads) {
        const uint32_t r = sh.row[j];
        atomicOr(&bm[r >> 5], 1u << (r & 31));
        atomicAdd(&scnt[r / kSliceRows], 1u);
      }
      if (cnt_out && threadIdx.x == 0) *cnt_out = p.k_top;
    }
  }
  if (!token_barrier(counter, ++nb * (uint32_t)P, p.status, 63)) return;
  // the next kernel may start its prologue now: every slice has passed its last barrier, so early
  // CTAs of that kernel can no longer keep one of these from being resident
  pdl_trigger();
  if (__ldcg(&ctl->whole)) return;

  // phase 5: this slice's selected rows, in ascending order, after those of the slices before it
  uint32_t before = 0;
  for (int i = threadIdx.x; i < part; i += kThreads) before += __ldcg(scnt + i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  __syncthreads();
  if (lane == 0) red[warp] = before;
  __syncthreads();
  uint32_t offset = 0;
  for (int w = 0; w < kWarps; ++w) offset += red[w];
  const uint32_t word = my_word_in ? __ldcg(bm + w0 + threadIdx.x) : 0u;  // phase 4 may have added bits
  uint32_t total;
  const uint32_t incl = block_scan((uint32_t)__popc(word), sh, &total);
  uint32_t pos = offset + incl - (uint32_t)__popc(word);
  uint32_t bits = word;
  while (bits) {
    const int b = __ffs(bits) - 1;
    bits &= bits - 1;
    out[pos++] = (w0 + (int)threadIdx.x) * 32 + b;
  }
}

// dynamic shared memory of the row and long-row mark kernels: the work struct, the bitmap of the
// row and (row kernel, rows that are staged) 16 bytes of alignment slack plus the staged row
// (the bitmap holds whole 16-byte groups: the long-row kernel copies it in with 16-byte stores)
size_t bitmap_smem(int S) {
  static_assert(sizeof(Shared) % 16 == 0, "the bitmap after Shared must be 16-byte aligned");
  return sizeof(Shared) + (((size_t)(S + 31) / 32 + 1 + 3) & ~size_t(3)) * sizeof(uint32_t);
}
size_t row_kernel_smem(int S) {
  if (S > kStageMax) return bitmap_smem(S);
  return bitmap_smem(S) + 16 + ((size_t)(S + 3) & ~size_t(3)) * sizeof(float);
}

// Per-device host state: the largest dynamic shared memory granted to each kernel so far (the
// attribute is raised only when a call needs more) and the last occupancy answer.
struct DeviceTopkState {
  size_t row_smem = 0, mark_smem = 0;
  size_t occ_smem = 0;
  int occ_blocks = -1;
};
std::mutex g_topk_state_mutex;
DeviceTopkState g_topk_state[64];

int current_device_index() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return 0;
  return d;
}

cudaError_t set_smem_attrs(size_t row_smem, size_t mark_smem) {
  std::lock_guard<std::mutex> lock(g_topk_state_mutex);
  DeviceTopkState& st = g_topk_state[current_device_index()];
  cudaError_t e = cudaSuccess;
  if (row_smem > st.row_smem) {
    e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)row_smem);
    if (e == cudaSuccess) st.row_smem = row_smem;
  }
  if (e == cudaSuccess && mark_smem > st.mark_smem) {
    e = cudaFuncSetAttribute(long_mark_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mark_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(long_coop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mark_smem);
    if (e == cudaSuccess) st.mark_smem = mark_smem;
  }
  return e;
}

// The long-row workspace: [a barrier counter per token | one LongLayout block per token].
size_t long_counters_bytes(int T) { return align_up((size_t)T * sizeof(uint32_t), 256); }

// One launch when all of the tokens' slices can be resident at once.
bool long_coop_fits(int T, int P, size_t smem) {
  int nb = 0;
  {
    std::lock_guard<std::mutex> lock(g_topk_state_mutex);
    DeviceTopkState& st = g_topk_state[current_device_index()];
    if (st.occ_blocks < 0 || st.occ_smem != smem) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, long_coop_kernel, kThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return false;
      }
      st.occ_smem = smem;
      st.occ_blocks = nb;
    }
    nb = st.occ_blocks;
  }
  return (long long)nb * device_sm_count() >= (long long)T * P;
}

// counters_zeroed: the kernel before it on the stream zeroed the barrier counters (the fused path's
// scorer does), so no memset separates the two launches and this one may start early (programmatic
// dependent launch: its CTAs wait in pdl_wait until the scorer's results are visible).
cudaError_t launch_long_coop(KParams& p, cudaStream_t st, size_t smem, bool counters_zeroed) {
  cudaError_t e = cudaSuccess;
  if (!counters_zeroed) e = cudaMemsetAsync(p.gbar, 0, (size_t)p.T * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nslice, p.T);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = counters_zeroed ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, long_coop_kernel, p);
  count_launch();
  return e;
}

// CTAs per token in long-row mode (1: one CTA per token).  Few tokens with long rows cannot
// fill the GPU with one CTA per token.
int long_slices(int T, int S) {
  const int sms = device_sm_count();
  if (S <= 4 * kSliceRows || T >= sms) return 1;
  return (S + kSliceRows - 1) / kSliceRows;
}

// the three long-row launches (workspace already checked)
cudaError_t launch_long(KParams& p, cudaStream_t st, size_t mark_smem) {
  const dim3 grid(p.nslice, p.T);
  cudaError_t e = launch_pdl(long_minmax_kernel, grid, dim3(kThreads), 0, st, p);
  if (e == cudaSuccess) e = launch_pdl(long_hist_kernel, grid, dim3(kThreads), 0, st, p);
  if (e == cudaSuccess) e = launch_pdl(long_mark_kernel, grid, dim3(kThreads), mark_smem, st, p);
  count_launch(3);
  return e;
}

// One CTA per token: rows of up to kRegMaxRows keep their keys in registers (threads x keys a
// thread by row length), longer ones are staged in shared memory or streamed.
constexpr int kRegMaxRows = 4096;
cudaError_t launch_one_cta_per_token(const KParams& p, size_t row_smem, cudaStream_t st) {
  const dim3 grid(p.T);
  if (p.S <= 2048) return launch_pdl(topk_reg_kernel<128, 16, 256>, grid, dim3(128), 0, st, p);
  if (p.S <= kRegMaxRows) return launch_pdl(topk_reg_kernel<256, 16, 2048>, grid, dim3(256), 0, st, p);
  return launch_pdl(topk_row_kernel, grid, dim3(kThreads), row_smem, st, p);
}

}  // namespace

size_t topk_workspace_bytes(int T, int S, int k_top) {
  (void)k_top;
  if (long_slices(T, S) <= 1) return 0;
  return long_counters_bytes(T) + (size_t)T * long_layout(S).total;
}

bool topk_range_mode(int T, int S, int k_top, int n_slots) {
  if (T != 1 || long_slices(T, S) <= 1 || n_slots <= 0 || n_slots > kMaxRangeSlots) return false;
  const size_t msmem = bitmap_smem(S);
  if (msmem > 220 * 1024 || set_smem_attrs(row_kernel_smem(S), msmem) != cudaSuccess) return false;
  (void)k_top;
  return long_coop_fits(T, long_slices(T, S), msmem);
}

// [barrier counters | the token's control block, slots, counts, histogram and bitmap]
size_t topk_range_zero_words(int T, int S) {
  const LongLayout L = long_layout(S);
  return (long_counters_bytes(T) + L.bitmap + (size_t)((S + 31) / 32) * sizeof(uint32_t)) / sizeof(uint32_t);
}

size_t topk_range_slots_offset(int T, int S) { return long_counters_bytes(T) + long_layout(S).rslots; }

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
  p.nslice = long_slices(a.T, a.S);
  p.long_ws = nullptr;
  p.gbar = nullptr;
  p.status = device_status_ptr();
  p.range_slots = nullptr;
  p.n_range_slots = 0;
  if (p.nslice <= 1) {
    if (launch_one_cta_per_token(p, smem, stream) != cudaSuccess) return DS4X_ERR_CUDA;
    count_launch();
  } else {
    const size_t need = topk_workspace_bytes(a.T, a.S, a.k_top);
    if (a.workspace == nullptr || a.workspace_bytes < need) return DS4X_ERR_WORKSPACE;
    p.gbar = static_cast<uint32_t*>(a.workspace);
    p.long_ws = static_cast<uint8_t*>(a.workspace) + long_counters_bytes(a.T);
    const bool coop = long_coop_fits(a.T, p.nslice, msmem);
    if (coop && a.T == 1 && a.range_slots && a.n_range_slots > 0 && a.n_range_slots <= kMaxRangeSlots) {
      p.range_slots = a.range_slots;  // the caller's scorer zeroed the scratch (counters_zeroed too)
      p.n_range_slots = a.n_range_slots;
    }
    const cudaError_t e = coop ? launch_long_coop(p, stream, msmem, a.counters_zeroed != 0) : launch_long(p, stream, msmem);
    if (e != cudaSuccess) return DS4X_ERR_CUDA;
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
  call_begin();  // launch accounting for ds4x_last_launch_count
  if (T < 0 || S < 0 || ratio < 1 || ld_scores < S) return call_end(DS4X_ERR_INVALID);
  if (k_top < 1 || k_top > DS4X_MAX_KTOP) return call_end(k_top < 1 ? DS4X_ERR_INVALID : DS4X_ERR_UNSUPPORTED);
  if (T == 0) return call_end(DS4X_OK);
  if (!scores || !positions || !indices) return call_end(DS4X_ERR_INVALID);
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(scores) | reinterpret_cast<uintptr_t>(positions) |
                         reinterpret_cast<uintptr_t>(indices) | reinterpret_cast<uintptr_t>(counts)) & 15u;
  if (mis) return call_end(DS4X_ERR_INVALID);
  // the candidate lists must fit the fixed array
  if (topk_workspace_bytes(T, S, k_top) > (size_t)DS4X_TOPK_STATIC_SCRATCH_BYTES) return call_end(DS4X_ERR_WORKSPACE);
  void* scratch = static_scratch_address();
  if (scratch == nullptr) return call_end(DS4X_ERR_CUDA);
  const size_t smem = row_kernel_smem(S);
  const size_t msmem = bitmap_smem(S);
  if (smem > 220 * 1024 || msmem > 220 * 1024) return call_end(DS4X_ERR_UNSUPPORTED);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (set_smem_attrs(smem, msmem) != cudaSuccess) return call_end(DS4X_ERR_CUDA);
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
  p.nslice = long_slices(T, S);
  p.long_ws = nullptr;
  p.gbar = nullptr;
  p.status = device_status_ptr();
  p.range_slots = nullptr;
  p.n_range_slots = 0;
  cudaError_t e;
  if (p.nslice <= 1) {
    e = launch_one_cta_per_token(p, smem, st);
    count_launch();
  } else {
    // the first launch zeroes every counter, histogram and bitmap the later ones read, so
    // nothing left in the array by an earlier call is ever read
    p.gbar = static_cast<uint32_t*>(scratch);
    p.long_ws = static_cast<uint8_t*>(scratch) + long_counters_bytes(T);
    e = long_coop_fits(T, p.nslice, msmem) ? launch_long_coop(p, st, msmem, false) : launch_long(p, st, msmem);
  }
  return call_end(e == cudaSuccess ? DS4X_OK : DS4X_ERR_CUDA);
}
