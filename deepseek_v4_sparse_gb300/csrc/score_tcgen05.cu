// score_tcgen05.cu — the lightning-indexer scorer on the 5th-generation tensor cores.
//
//   score[t,s] = sum_h w[t,h] * max(0, q[t,h,:] . k[s,:])     (s < n_vis(t); -inf beyond)
//
// Source of the operation: "How I made DeepSeek 12x faster on a Mac Studio", section
// "1: the kernels", PRs #830 (stage Q/K tiles on chip once instead of re-reading ~1 KB per
// scored pair) and #831 (register blocking: keep operand tiles resident so that each load
// feeds more MMAs).  On sm_103a both ideas become: TMA-staged, 128B-swizzled shared-memory
// tiles feeding tcgen05.mma, with a q tile resident across a run of k tiles and the
// accumulator in TMEM.  The full T x H x S product never leaves the SM.
//
// Mapping (one UMMA per 16-wide K step, M=128, N=TN, fp16 in, fp32 accumulate):
//   A = k tile    [128 rows s] x [D]       (M axis = compressed rows = TMEM lanes)
//   B = q tile    [TN = TPT tokens x H heads] x [D]    (N axis = TMEM columns)
//   D = TMEM      [128 lanes] x [TN columns] fp32, NACC buffers
// so each epilogue thread owns one row s and reduces the H head columns of a token in its
// own registers: relu, multiply by w[t,h] (from shared memory, broadcast), sum, mask, store.
//
// Two tile widths.  Wide (TN = 256, four tokens of 64 heads): prefill, where a k tile feeds
// as many tokens as one UMMA can take.  Narrow (TN = max(64, H)): when all tokens fit in one
// narrow tile (a decode step), so that no tensor-pipe time and no shared memory goes to
// padding tokens: the q tile shrinks from 64 KB to 16 KB and the k pipeline deepens from 6 to
// 12 stages, which is what a pass over a long k needs to keep enough bytes in flight.
//
// Warp roles (384 threads, one CTA per SM, persistent over a contiguous range of tiles):
//   warp 0      TMA producer of k tiles, one per (group, s-tile)
//   warp 1      MMA issuer + TMEM allocation
//   warp 2      TMA producer of q tiles, one per token group
//   (each a converged warp issuing through one elected lane)
//   warps 4..   epilogue, groups of four: warp%4 selects the 32-lane TMEM quadrant; the groups
//               split a tile's tokens or, when a tile holds fewer tokens than there are
//               groups, take turns over the tiles
// Eight epilogue warps (two groups): the single thread issuing the products shares a scheduler
// with two of them, and measured faster than with four (more of its issue slots are taken) or
// one (the reduction of a tile no longer hides behind its products).
// The k pipeline stage is one 128-row x 64-column block (16 KB) so that D=128 tiles stream
// as two stages; q is double-buffered so that a new token group loads while the previous
// group's MMAs drain.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "ds4x_internal.h"
#include "ds4x_ptx.cuh"

namespace ds4x {
namespace {

constexpr int kTileS = 128;   // compressed rows per tile (UMMA M)
constexpr int kTileWide = 256;  // token x head columns of a wide tile (UMMA N)
constexpr int kEpiWarps = 8;
constexpr int kGroups = kEpiWarps / 4;  // epilogue groups of four warps (one per TMEM quadrant)
constexpr int kWStage = 512 / kGroups;  // floats of w staged per epilogue group
constexpr int kThreads = 32 * (4 + kEpiWarps);
constexpr int kBlockBytes = kTileS * 128;  // one k stage: 128 rows x 64 fp16
constexpr int kSmemBudget = 227 * 1024;

constexpr int narrow_tile(int H) { return H > 64 ? H : 64; }

template <int H, int D, int TN>
struct Cfg {
  static constexpr int TPT = TN / H;                  // tokens per tile
  static constexpr int SPLIT = TPT >= kGroups ? kGroups : TPT;  // epilogue groups sharing a tile's tokens
  static constexpr int ROT = kGroups / SPLIT;         // sets of groups taking turns over tiles
  static constexpr int TOKW = TPT / SPLIT;            // tokens one epilogue warp reduces per tile
  static constexpr int NACC = TN >= 256 ? 2 : 512 / TN > 8 ? 8 : 512 / TN;  // TMEM accumulators
  static constexpr uint32_t TMEM_COLS = NACC * TN;    // 512
  static constexpr int KB = D / 64;                // 64-wide blocks along D
  static constexpr int Q_BYTES = TN * D * 2;       // one q tile
  static constexpr int QB_BYTES = TN * 128;        // one 64-wide block of the q tile
  static constexpr int NQ = 2;                        // q tile buffers
  static constexpr int FIXED = NQ * Q_BYTES + kGroups * kWStage * 4 + 640;  // q, w of the epilogue groups, barriers
  static constexpr int NK_FIT = (kSmemBudget - FIXED) / kBlockBytes;
  static constexpr int NK = NK_FIT < 12 ? NK_FIT : 12;  // k stages (one 64-wide block each)
  static constexpr int SMEM = FIXED + NK * kBlockBytes;
  static_assert(TPT >= 1 && TPT * H == TN, "H must divide the tile width");
  static_assert(SPLIT * ROT == kGroups && TOKW * SPLIT == TPT, "epilogue split");
  static_assert(TOKW * H <= kWStage, "w stage of an epilogue group");
  static_assert(NACC >= ROT, "every set of epilogue groups needs a buffer of its own");
  static_assert(D % 64 == 0, "D must be a multiple of 64");
  static_assert(NK >= 4 && SMEM <= kSmemBudget, "shared memory");
  static_assert(TMEM_COLS <= 512, "TMEM");
  // barriers, the TMEM address, the per-warp key ranges and four largest keys fit the 640 bytes
  // set aside for them
  static_assert((2 * NK + 2 * NQ + 2 * NACC + 2 * kGroups) * 8 + 16 + 6 * kEpiWarps * 4 <= 640, "barrier area");
};

struct Params {
  const __half* w;
  const int32_t* positions;
  float* scores;
  int64_t ld;
  int T, S, ratio;
  int n_stiles;
  long long total_items;
  int skip_k_top;
  int write_masked;
  int* status;
  uint32_t* zero_words;  // zeroed (by all CTAs) once the previous kernel is done
  int n_zero;
  // T = 1: [grid][4] per CTA the min and max ordered key of the visible scores it wrote, the fourth
  // largest of its epilogue threads' maximum keys, 0
  uint32_t* range_slots;
};

// The warp's values in descending order: lane i returns the i-th largest (bitonic network).
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
      v = (((lane & k) == 0) == ((lane & j) == 0)) ? max(v, o) : min(v, o);
    }
  }
  return v;
}

__device__ __forceinline__ int n_visible(const Params& p, int t) {
  const int pos = __ldg(p.positions + t);
  if (pos < 0) return 0;
  const uint32_t n = (uint32_t)(pos + 1u) / (uint32_t)p.ratio;  // pos + 1 <= 2^31
  return n < (uint32_t)p.S ? (int)n : p.S;
}


// Packed fp32 pairs (sm_100 family): d = a * b + c element-wise, round to nearest.
__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Rows a token group needs scored (the most any of its tokens needs), with the group's
// positions loaded one group ahead: load(g + 1) when group g starts, rows() when g + 1 starts,
// so that no role waits on global loads at a group change.
template <int TPT>
struct GroupRowsAhead {
  int pos[TPT];
  __device__ __forceinline__ void load(const Params& p, int g) {
#pragma unroll
    for (int j = 0; j < TPT; ++j) {
      const long long t = (long long)g * TPT + j;
      pos[j] = t < p.T ? __ldg(p.positions + t) : -1;
    }
  }
  __device__ __forceinline__ int rows(const Params& p) const {
    int m = 0;
#pragma unroll
    for (int j = 0; j < TPT; ++j) {
      int n = 0;
      if (pos[j] >= 0) {  // pos + 1 <= 2^31: a 32-bit unsigned division, not a 64-bit routine
        const uint32_t v = (uint32_t)(pos[j] + 1u) / (uint32_t)p.ratio;
        n = v < (uint32_t)p.S ? (int)v : p.S;
      }
      if (p.skip_k_top > 0 && n <= p.skip_k_top) n = 0;  // the shortcut covers this token
      m = max(m, n);
    }
    return m;
  }
};

template <int H, int D, int TN>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const Params p) {
  using C = Cfg<H, D, TN>;
  constexpr uint32_t kIdesc = idesc_f16(kTileS, TN, 0, 0, 0);
  // Declared aligned (and checked) rather than rounded up through an integer: pointers derived
  // from the array keep the shared address space, so the epilogue's w reads are LDS, not
  // generic loads.
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the 128B-swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) report_timeout(p.status, 0x7e);
    return;
  }
  uint8_t* sq = smem;                                   // 2 x Q_BYTES
  uint8_t* sk = sq + C::NQ * C::Q_BYTES;                // NK x kBlockBytes
  float* sw = reinterpret_cast<float*>(sk + C::NK * kBlockBytes);  // kGroups x kWStage
  uint64_t* bars = reinterpret_cast<uint64_t*>(sw + kGroups * kWStage);
  uint64_t* kfull = bars;
  uint64_t* kempty = kfull + C::NK;
  uint64_t* qfull = kempty + C::NK;
  uint64_t* qempty = qfull + C::NQ;
  uint64_t* afull = qempty + C::NQ;
  uint64_t* aempty = afull + C::NACC;
  uint64_t* wdone = aempty + C::NACC;  // [epilogue group] its 4 warps are done with the group's w
  uint64_t* wready = wdone + kGroups;  // [epilogue group] the next token group's w is written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wready + kGroups);
  uint32_t* red_s = tmem_slot + 4;  // [2][kEpiWarps] per-warp key range (range mode)
  uint32_t* red4 = red_s + 2 * kEpiWarps;  // [kEpiWarps][4] per-warp four largest thread maxima

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NK; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < C::NQ; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < kGroups; ++i) {
      mbar_init(&wdone[i], 4);
      mbar_init(&wready[i], 1);
    }
    for (int i = 0; i < C::NACC; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], C::SPLIT * 4);  // the warps that read the buffer
    }
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // everything above touched only this CTA's own resources
  pdl_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.n_zero; i += gridDim.x * blockDim.x) p.zero_words[i] = 0u;

  const long long beg = (long long)blockIdx.x * p.total_items / gridDim.x;
  const long long end = (long long)(blockIdx.x + 1) * p.total_items / gridDim.x;

  // Every role walks the same (group, s-tile) sequence; a group's q tile is loaded (and waited
  // for) before its first tile that is not past every token's visibility.
  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer: k tiles
    int cur_g = -1, rows = 0;
    int ks = 0;          // k stage
    uint32_t kph = 0;    // its phase
    int g = (int)(beg / p.n_stiles), st = (int)(beg % p.n_stiles) - 1;
    GroupRowsAhead<C::TPT> ahead;
    ahead.load(p, g);  // the first group of the range
    for (long long it = beg; it < end; ++it) {
      if (++st == p.n_stiles) {
        st = 0;
        ++g;
      }
      if (g != cur_g) {
        cur_g = g;
        rows = ahead.rows(p);
        ahead.load(p, g + 1);
      }
      if (st * kTileS >= rows) continue;
      bool ok = true;
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        if (!mbar_wait_warp(&kempty[ks], kph ^ 1, p.status, 2)) { ok = false; break; }
        mbar_arrive_expect_tx_elect(&kfull[ks], kBlockBytes);
        tma_load_2d_elect(sk + ks * kBlockBytes, &tm_k, &kfull[ks], kb * 64, st * kTileS);
        if (++ks == C::NK) {
          ks = 0;
          kph ^= 1;
        }
      }
      if (!ok) break;
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------- TMA producer: q tiles
    // On a warp of its own, so that the next group's q tile loads as soon as its buffer is
    // free (when the group before the current one has finished), not only when the k
    // producer reaches that group a few stages ahead of the products.
    int cur_g = -1, rows = 0;
    bool started = false;
    uint32_t q_it = 0;
    int g = (int)(beg / p.n_stiles), st = (int)(beg % p.n_stiles) - 1;
    GroupRowsAhead<C::TPT> ahead;
    ahead.load(p, g);  // the first group of the range
    for (long long it = beg; it < end; ++it) {
      if (++st == p.n_stiles) {
        st = 0;
        ++g;
      }
      if (g != cur_g) {
        cur_g = g;
        rows = ahead.rows(p);
        ahead.load(p, g + 1);
        started = false;
      }
      if (started || st * kTileS >= rows) continue;
      const int b = q_it % C::NQ;
      if (!mbar_wait_warp(&qempty[b], ((q_it / C::NQ) & 1) ^ 1, p.status, 1)) break;
      mbar_arrive_expect_tx_elect(&qfull[b], C::Q_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_2d_elect(sq + b * C::Q_BYTES + kb * C::QB_BYTES, &tm_q, &qfull[b], kb * 64, g * TN);
      ++q_it;
      started = true;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (converged, so that descriptors and addresses stay in uniform
    // registers) and one elected lane issues each product and commit.  Lean between products:
    // descriptors are built once and offset by constants, stage and buffer indices are running
    // counters.
    // descriptor address field = byte address >> 4 (bits 0..13); offsets below never carry out
    const uint64_t adesc0 = desc_sw128(smem_u32(sk), 16, 1024);
    const uint64_t bdesc0 = desc_sw128(smem_u32(sq), 16, 1024);
    int cur_g = -1, rows = 0, qb = -1;
    bool started = false;
    uint32_t q_it = 0;
    int ks = 0, ab = 0;
    uint32_t kph = 0, aph = 0;
    int g = (int)(beg / p.n_stiles), st = (int)(beg % p.n_stiles) - 1;
    GroupRowsAhead<C::TPT> ahead;
    ahead.load(p, g);  // the first group of the range
    for (long long it = beg; it < end; ++it) {
      if (++st == p.n_stiles) {
        st = 0;
        ++g;
      }
      if (g != cur_g) {
        cur_g = g;
        rows = ahead.rows(p);
        ahead.load(p, g + 1);
        started = false;
      }
      if (st * kTileS >= rows) continue;
      if (!started) {
        if (qb >= 0) tc_commit_elect(&qempty[qb]);  // previous group's q tile is free once its MMAs finish
        qb = q_it % C::NQ;
        if (!mbar_wait_warp(&qfull[qb], (q_it / C::NQ) & 1, p.status, 3)) break;
        ++q_it;
        started = true;
        tc_fence_after();
      }
      if (!mbar_wait_warp(&aempty[ab], aph ^ 1, p.status, 4)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + ab * TN;
      const uint64_t bq = bdesc0 + (uint64_t)((qb * C::Q_BYTES) >> 4);
      bool ok = true;
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        if (!mbar_wait_warp(&kfull[ks], kph, p.status, 5)) { ok = false; break; }
        tc_fence_after();
        const uint64_t a0 = adesc0 + (uint64_t)((ks * kBlockBytes) >> 4);
        const uint64_t b0 = bq + (uint64_t)((kb * C::QB_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 16 columns = 32 bytes = 2 address units per step
          tc_mma_f16_elect(d_tmem, a0 + 2 * kk, b0 + 2 * kk, kIdesc, (kb | kk) != 0);
        tc_commit_elect(&kempty[ks]);  // k stage is free once these MMAs complete
        if (++ks == C::NK) {
          ks = 0;
          kph ^= 1;
        }
      }
      if (!ok) break;
      tc_commit_elect(&afull[ab]);
      if (++ab == C::NACC) {
        ab = 0;
        aph ^= 1;
      }
    }
  } else if (warp >= 4) {
    // --------------------------------------------------------------------- epilogue
    const int e = warp - 4;
    const int quad = warp & 3;             // TMEM lanes 32*quad .. 32*quad+31
    const int grp = e >> 2;                // epilogue group 0..kGroups-1
    const int set = grp / C::SPLIT;        // the tiles of this group: the set's turns
    const int tok0 = (grp % C::SPLIT) * C::TOKW;  // first token of a tile this warp reduces
    float* my_w = sw + grp * kWStage;      // the group's w[t, h] for its tokens, fp32 (shared by its 4 warps)
    constexpr int NW = C::TOKW * H;        // w values a warp holds per token group
    constexpr int WPL = (NW + 31) / 32;    // ... per lane
    // the next group's w and visibility are loaded into registers one group ahead
    float w_next[WPL];
    int nvis_next[C::TOKW];
    auto prefetch = [&](int g) {
      const int t0 = g * C::TPT + tok0;
#pragma unroll
      for (int i = 0; i < WPL; ++i) {
        const int idx = lane + 32 * i;
        const int t = t0 + idx / H;
        w_next[i] = (idx < NW && t < p.T) ? __half2float(p.w[(int64_t)t * H + (idx % H)]) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < C::TOKW; ++j) nvis_next[j] = (t0 + j < p.T) ? n_visible(p, t0 + j) : 0;
    };
    int cur_g = -1, rows = 0;
    uint32_t a_it = 0, gc = 0;  // gc: group changes so far (the w barriers' phase)
    int nvis[C::TOKW];
    uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;  // range mode: ordered keys of the visible scores written
    if (beg < end) prefetch((int)(beg / p.n_stiles));
    int g = (int)(beg / p.n_stiles), st = (int)(beg % p.n_stiles) - 1;
    GroupRowsAhead<C::TPT> ahead;
    ahead.load(p, g);  // the first group of the range
    for (long long it = beg; it < end; ++it) {
      if (++st == p.n_stiles) {
        st = 0;
        ++g;
      }
      if (g != cur_g) {
        cur_g = g;
        rows = ahead.rows(p);
        ahead.load(p, g + 1);
        // one copy of w per epilogue group: its 4 warps say they are done with the previous
        // token group's, its first warp waits for that, writes the new one and says so
        __syncwarp();
        if (lane == 0) mbar_arrive(&wdone[grp]);
        if (quad == 0) {
          if (!mbar_wait(&wdone[grp], gc & 1, p.status, 7)) break;
#pragma unroll
          for (int i = 0; i < WPL; ++i)
            if (lane + 32 * i < NW) my_w[lane + 32 * i] = w_next[i];
          __syncwarp();
          if (lane == 0) mbar_arrive(&wready[grp]);
        }
        if (!mbar_wait(&wready[grp], gc & 1, p.status, 8)) break;
        ++gc;
#pragma unroll
        for (int j = 0; j < C::TOKW; ++j) nvis[j] = nvis_next[j];
        const long long next_group_item = (long long)(g + 1) * p.n_stiles;
        if (next_group_item < end) prefetch(g + 1);
      }
      const int row = st * kTileS + quad * 32 + lane;
      const int t0 = g * C::TPT + tok0;
      if (st * kTileS >= rows) {
        if (p.write_masked && row < p.S && (st % C::ROT) == set) {
#pragma unroll
          for (int j = 0; j < C::TOKW; ++j)
            if (t0 + j < p.T) p.scores[(int64_t)(t0 + j) * p.ld + row] = -INFINITY;
        }
        continue;
      }
      const uint32_t my_it = a_it++;
      if ((int)(my_it % C::ROT) != set) continue;  // another set's tile
      const int ab = my_it % C::NACC;
      if (!mbar_wait(&afull[ab], (my_it / C::NACC) & 1, p.status, 6)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + ab * TN;
#pragma unroll
      for (int j = 0; j < C::TOKW; ++j) {
        const uint32_t col = (tok0 + j) * H;
        // sum_h w[h] * max(0, acc[h]): ReLU in scalar, products in packed f32x2 pairs
        uint64_t a01 = 0, a23 = 0;  // two pair accumulators (bit pattern 0 = +0.0f, +0.0f)
        constexpr int CW = H < 32 ? H : 32;  // columns read per TMEM wait (register budget)
#pragma unroll
        for (int c = 0; c < H; c += CW) {
          float v[CW];
          if constexpr (CW == 64) {
            tmem_ld32(t_row + col + c, *reinterpret_cast<float(*)[32]>(&v[0]));
            tmem_ld32(t_row + col + c + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
          } else if constexpr (CW == 32) {
            tmem_ld32(t_row + col + c, v);
          } else {
            tmem_ld16(t_row + col + c, v);
          }
          tc_wait_ld();
#pragma unroll
          for (int h = 0; h < CW; h += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(&my_w[j * H + c + h]);
            a01 = ffma2(pack_f2(w4.x, w4.y), pack_f2(fmaxf(v[h], 0.f), fmaxf(v[h + 1], 0.f)), a01);
            a23 = ffma2(pack_f2(w4.z, w4.w), pack_f2(fmaxf(v[h + 2], 0.f), fmaxf(v[h + 3], 0.f)), a23);
          }
        }
        float x0, x1, x2, x3;
        unpack_f2(a01, x0, x1);
        unpack_f2(a23, x2, x3);
        const float acc = (x0 + x1) + (x2 + x3);
        if (t0 + j < p.T && row < p.S) p.scores[(int64_t)(t0 + j) * p.ld + row] = row < nvis[j] ? acc : -INFINITY;
        if (row < nvis[j]) {  // the top-k's key order: larger score, larger key
          const uint32_t u = __float_as_uint(acc);
          const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
          kmn = min(kmn, key);
          kmx = max(kmx, key);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[ab]);
    }
    if (p.range_slots) {
      // this CTA's key range, over the warp and then over the epilogue warps; and the fourth
      // largest of the threads' maximum keys (a thread without visible rows holds 0): the four
      // largest of each warp, then of those. At least four of this CTA's visible scores have a key
      // at or above it (four distinct threads' maxima), which lets the top-k bound the row's
      // k_top-th key from below before it reads a score.
      const uint32_t srt = warp_sort_desc(kmx);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, o));
        kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, o));
      }
      if (lane == 0) {
        red_s[e] = kmn;
        red_s[kEpiWarps + e] = kmx;
      }
      if (lane < 4) red4[4 * e + lane] = srt;
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
      if (e == 0) {
        static_assert(4 * kEpiWarps == 32, "one warp sorts the warps' four largest");
        const uint32_t r4 = __shfl_sync(0xffffffffu, warp_sort_desc(red4[lane]), 3);
        if (lane == 0) {
          uint32_t a = red_s[0], b = red_s[kEpiWarps];
          for (int i = 1; i < kEpiWarps; ++i) {
            a = min(a, red_s[i]);
            b = max(b, red_s[kEpiWarps + i]);
          }
          reinterpret_cast<uint4*>(p.range_slots)[blockIdx.x] = make_uint4(a, b, r4, 0u);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------- host side

// 2-D fp16 tensor [rows, cols] (cols contiguous), box = 64 columns x box_rows rows, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One persistent CTA per SM, or one per work item when there are fewer.
int grid_for(long long total_items) {
  const int sms = device_sm_count();
  return (int)(total_items < sms ? total_items : sms);
}

template <int H, int D, int TN>
int launch_impl(const ScoreArgs& a, cudaStream_t stream) {
  using C = Cfg<H, D, TN>;
  if (ensure_dynamic_smem(score_kernel<H, D, TN>, C::SMEM) != cudaSuccess) return DS4X_ERR_CUDA;
  CUtensorMap tq, tk;
  if (!make_map(&tq, a.q, (uint64_t)a.T * H, D, TN) || !make_map(&tk, a.k, (uint64_t)a.S, D, kTileS))
    return DS4X_ERR_CUDA;
  Params p;
  p.w = static_cast<const __half*>(a.w);
  p.positions = a.positions;
  p.scores = a.scores;
  p.ld = a.ld;
  p.T = a.T;
  p.S = a.S;
  p.ratio = a.ratio;
  p.n_stiles = (a.S + kTileS - 1) / kTileS;
  const long long n_groups = (a.T + C::TPT - 1) / C::TPT;
  p.total_items = n_groups * p.n_stiles;
  p.skip_k_top = a.skip_k_top;
  p.write_masked = a.write_masked;
  p.status = device_status_ptr();
  p.zero_words = a.zero_words;
  p.n_zero = a.zero_words ? a.n_zero : 0;
  p.range_slots = a.range_slots;
  const int grid = grid_for(p.total_items);
  const cudaError_t e = launch_pdl(score_kernel<H, D, TN>, dim3(grid), dim3(kThreads), (size_t)C::SMEM, stream, tq, tk, p);
  count_launch();
  return e == cudaSuccess ? DS4X_OK : DS4X_ERR_CUDA;
}

// Narrow tiles when every token fits in one (a decode step), wide ones otherwise.
template <int H, int D>
int launch_shape(const ScoreArgs& a, cudaStream_t stream) {
  constexpr int TN = narrow_tile(H);
  if ((int64_t)a.T * H <= TN) return launch_impl<H, D, TN>(a, stream);
  return launch_impl<H, D, kTileWide>(a, stream);
}

}  // namespace

int score_grid(int T, int H, int S) {
  if (T <= 0 || S <= 0 || H <= 0) return 0;
  const int TN = (int64_t)T * H <= narrow_tile(H) ? narrow_tile(H) : kTileWide;  // as launch_shape chooses
  const long long tpt = TN / H;
  const long long n_groups = (T + tpt - 1) / tpt;
  return grid_for(n_groups * ((S + kTileS - 1) / kTileS));
}

bool score_shape_supported(int H, int D) {
  return (H == 16 || H == 32 || H == 64 || H == 128) && (D == 64 || D == 128);
}

int launch_score(const ScoreArgs& a, cudaStream_t stream) {
  if (a.T == 0 || a.S == 0) return DS4X_OK;
#define DS4X_SCORE_CASE(HH, DD) \
  if (a.H == HH && a.D == DD) return launch_shape<HH, DD>(a, stream);
  DS4X_SCORE_CASE(16, 64)
  DS4X_SCORE_CASE(16, 128)
  DS4X_SCORE_CASE(32, 64)
  DS4X_SCORE_CASE(32, 128)
  DS4X_SCORE_CASE(64, 64)
  DS4X_SCORE_CASE(64, 128)
  DS4X_SCORE_CASE(128, 64)
  DS4X_SCORE_CASE(128, 128)
#undef DS4X_SCORE_CASE
  return DS4X_ERR_UNSUPPORTED;
}

}  // namespace ds4x
