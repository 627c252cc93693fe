// sparse_mqa.cu — multi-query attention of 64 heads over the rows chosen by the indexer.
//
//   out[t,h,:] = sum_j softmax_j( scale * q_attn[t,h,:] . kv[idx_j,:] ) * kv[idx_j,:]
//
// Source: "How I turned one oversized DeepSeek optimization into three merged oMLX PRs",
// section "The three changes that merged", item 1 (attention over pooled compressed rows picked
// by an index list, kv rows serving as both key and value), fed by the top-512 of "How I made
// DeepSeek 12x faster on a Mac Studio", section "1: the kernels".
//
// Local-plus-pooled (same page and item: the native kernel that takes local and pooled state in
// one pass): with a window W the row list of token t grows by the raw rows of positions
// p-W+1 .. p held in kv_local, as extra 64-row chunks after the pooled ones, in the same softmax.
// A pooled chunk gathers through the indices; a window chunk through the token's position.  The
// window code is a template branch (kWin): the pooled-only kernel carries none of it (its chunk
// tests measurably slowed that kernel when they were runtime branches).
//
// One CTA per SM, persistent over tokens.  A token's selected rows are processed in chunks of
// 64, double-buffered in shared memory (each row is gathered with 16-byte cp.async into the
// 128B-swizzled layout both products read: 8 slots of 64 dims per chunk).  Per chunk:
//   S   [64 heads x 64 rows] = Q . Ksel^T     tcgen05, M = 64 (heads on TMEM lanes), K-major
//   O^T [512 x 64 heads]    += Vsel^T . P^T   tcgen05, M = 128 (dims), A MN-major, B K-major
// S puts each head's 64 scores in one TMEM lane; a 16x256b load spreads them over 4 threads,
// so a head's max and sum take two shuffles.  The running max of a head is only raised when its logits exceed it by
// more than 2^8 (then O^T's column and the head's sum are rescaled), so the probabilities
// written as fp16/bf16 stay <= 256.
//
// Warps: 0-3 gather, 4-7 softmax (heads 16*(warp-4) .. +15, 4 threads a head), 8-11 output
// (O^T lanes by quadrant), 12 issues the S products, 13 the O^T products, 14 loads q_attn.
// The two MMA warps run converged and issue with elect.sync in straight runs, so S of chunk
// c+2 and O^T of chunk c+1 interleave in the tensor pipe.  Buffers are released in 128-dim
// pieces: a chunk's slot pair as its O^T product completes (the next gather starts early), a
// pair of q blocks as the token's last S product passes it, a d-block of O^T as soon as the
// output warps hold it in registers.  O^T rotates over six 64-column TMEM slots (a token uses
// four), so the next token's first products do not wait for the previous token's output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>

#include "ds4x_internal.h"
#include "ds4x_ptx.cuh"

namespace ds4x {
namespace {

constexpr int kHq = 64;
constexpr int kDkv = 512;
constexpr int kRows = 64;                       // rows per chunk
constexpr int kSlots = kDkv / 64;               // 8 slots of 64 dims
constexpr int kPairs = kSlots / 2;              // 128-dim blocks of O^T
constexpr int kSlotBytes = kRows * 128;         // 8 KB
constexpr int kBufBytes = kSlots * kSlotBytes;  // 64 KB per chunk buffer
constexpr int kQBlockBytes = kHq * 128;         // 8 KB (64 heads x 64 dims)
constexpr int kQBytes = kSlots * kQBlockBytes;  // 64 KB
constexpr int kPBytes = kHq * 128;              // 8 KB: P[h][j], 64 heads x 64 rows
constexpr int kOffKV = kQBytes;
constexpr int kOffP = kOffKV + 2 * kBufBytes;
constexpr int kOffAlpha = kOffP + 2 * kPBytes;  // float[64] rescale factors of one chunk
constexpr int kOffLM = kOffAlpha + kHq * 4;     // float[2 tokens][3 (l, m, 1/l)][64]
constexpr int kOffBars = kOffLM + 2 * 3 * kHq * 4;
constexpr int kOSlots = 6;                      // O^T slots of 64 columns (a token uses 4)
constexpr int kNumBars = 2 * kPairs + 2 * 2 * kPairs + 2 + 2 + 2 + 2 + 2 * kOSlots + 2 + 2;
constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr int kSmem = kOffTmemSlot + 16;
constexpr int kThreads = 15 * 32;
constexpr int kSWarp = 12;   // issues S, allocates TMEM
constexpr int kOWarp = 13;   // issues O^T
constexpr int kQWarp = 14;   // loads q_attn of each token by TMA
constexpr uint32_t kTmemCols = 512;
// TMEM: S in columns [0, 128) (two buffers of 64), O^T in six slots of 64 from column 128.  A
// token's 128-dim block db accumulates in slot (4 * token + db) % 6, so the next token's first
// two blocks start in slots the previous token does not use while its output is drained, and
// its last two reuse the slots drained first.
constexpr uint32_t kColO = 128;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kSoftBar = 1, kEpiBar = 2, kGroupThreads = 128;
constexpr int kMaxSplit = (DS4X_MAX_KTOP + kRows - 1) / kRows;  // items a token can be split into

struct Params {
  const uint16_t* q;         // q_attn [T, 64, 512]; read by TMA (and prefetched to L2 a token ahead)
  const uint16_t* kv;        // [S, 512]; never read through an invalid index
  const uint16_t* zero_src;  // any valid address: source of the zero-filled (size 0) copies
  const int32_t* indices;
  const uint16_t* kv_local;  // [L, 512] raw rows of the window, row r = position local_pos0 + r
  const int32_t* positions;  // [T], read for the window chunks only
  uint16_t* out;
  float* lse;
  int* status;
  uint16_t* part;  // split mode: per item, sum_j 2^(x_j - m) kv_j / l  [items, 64, 512] in the kv dtype
                   // (a convex combination of kv rows: it cannot leave the dtype's range)
  float* part_ml;  // split mode: per item, m [64] then l [64] (m in log2 units of the scaled logits)
  int T, S, k_top, nchunks;
  int npc;                      // chunks [0, npc) hold pooled rows, [npc, nchunks) the window's
  int L, local_pos0, window;
  int nsplit, cps, items;  // a token's chunks are spread over nsplit items of cps chunks each
  float scale_log2;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool named_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Transpose-reduction over the warp: v[c] of every lane -> lane c holds op over all lanes of
// column c (31 shuffles for 32 columns).
template <bool kMax>
__device__ __forceinline__ float warp_columns_reduce(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int step = 16; step >= 1; step >>= 1) {
    const bool upper = (lane & step) != 0;
#pragma unroll
    for (int i = 0; i < step; ++i) {
      const float send = upper ? v[i] : v[i + step];
      const float keep = upper ? v[i + step] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, step);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// 2^x with the hardware approximation (MUFU.EX2, flushes subnormal results to zero); 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float a, float b, float& ra, float& rb) {
  if constexpr (kBf16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    ra = __low2float(h);
    rb = __high2float(h);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(a, b);
    ra = __low2float(h);
    rb = __high2float(h);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

template <bool kBf16>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (kBf16) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t*>(&h);
  } else {
    const __half h = __float2half_rn(x);
    return *reinterpret_cast<const uint16_t*>(&h);
  }
}

template <bool kBf16, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mqa_kernel(const __grid_constant__ CUtensorMap tm_q, const Params p) {
  constexpr uint32_t kIdescS = idesc_f16(64, kHq, kBf16 ? 1 : 0, 0, 0);
  constexpr uint32_t kIdescO = idesc_f16(128, kHq, kBf16 ? 1 : 0, 1, 0);
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) report_timeout(p.status, 0x7f);
    return;
  }
  uint8_t* sq = smem;
  uint8_t* skv = smem + kOffKV;
  uint8_t* sp = smem + kOffP;
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* lm = reinterpret_cast<float*>(smem + kOffLM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* qfull = bars;                   // [pair of 64-dim blocks]
  uint64_t* qempty = bars + kPairs;         // [pair]
  uint64_t* kvfull = bars + 2 * kPairs;     // [buffer][pair]
  uint64_t* kvempty = kvfull + 2 * kPairs;  // [buffer][pair]
  uint64_t* sfull = kvempty + 2 * kPairs;
  uint64_t* sempty = sfull + 2;
  uint64_t* pfull = sempty + 2;
  uint64_t* pempty = pfull + 2;
  uint64_t* ofull = pempty + 2;             // [O^T slot]
  uint64_t* oempty = ofull + kOSlots;       // [O^T slot]
  uint64_t* lready = oempty + kOSlots;           // [token parity] l, m of a token written
  uint64_t* lfree = lready + 2;             // [token parity] ... and read by the output warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nch = p.nchunks;
  auto oslot = [](uint32_t tok_i, int db) { return (int)((4u * (tok_i % 3u) + (uint32_t)db) % kOSlots); };
  // work item it: token it / nsplit, chunks [c0, c1) of it (all of them when nsplit = 1)
  auto item_of = [&](int it, int& t, int& c0, int& c1) {
    t = it / p.nsplit;
    c0 = (it - t * p.nsplit) * p.cps;
    c1 = min(nch, c0 + p.cps);
  };
  // the chunk after (t, c) in this CTA's sequence: the next chunk of the item, else the first
  // chunk of the CTA's next item (token p.T when there is none)
  auto next_chunk = [&](int it, int t, int c, int c1, int& nt, int& nc) {
    if (c + 1 < c1) {
      nt = t;
      nc = c + 1;
    } else {
      const int nit = it + (int)gridDim.x;
      int d1;
      item_of(nit, nt, nc, d1);
      if (nit >= p.items) nt = p.T;
    }
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPairs; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < kOSlots; ++i) {
      mbar_init(&ofull[i], 1);
      mbar_init(&oempty[i], 4);
    }
    for (int i = 0; i < 2 * kPairs; ++i) {
      mbar_init(&kvfull[i], 128);
      mbar_init(&kvempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 4);
      mbar_init(&pfull[i], 4);
      mbar_init(&pempty[i], 1);
      mbar_init(&lready[i], 4);
      mbar_init(&lfree[i], 4);
    }
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_q);
  }
  if (warp == kSWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // everything above touched only this CTA's own resources
  pdl_trigger();

  if (warp < 4) {
    // ------------------------------------------------------------------------ gather
    // thread pt copies 16-byte column chunk `ch` of rows (pt>>3) + 16 i, i = 0..3, in every slot
    const int pt = threadIdx.x;
    const int ch = pt & 7;
    uint32_t dst_off[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (pt >> 3) + 16 * i;
      dst_off[i] = r * 128 + ((ch ^ (r & 7)) << 4);
    }
    // a chunk's row sources, loaded a chunk ahead: a pooled chunk's indices, a window chunk's
    // token position (in idx[0])
    auto load_idx = [&](int t, int c, int32_t (&idx)[4]) {
      if (!kWin || c < p.npc) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = c * kRows + (pt >> 3) + 16 * i;
          idx[i] = (t < p.T && j < p.k_top) ? __ldg(p.indices + (int64_t)t * p.k_top + j) : -1;
        }
      } else {
        idx[0] = t < p.T ? __ldg(p.positions + t) : INT_MIN;
      }
    };
    uint32_t gc = 0;
    bool ok = true;
    int32_t idx[4];
    {
      int t0, a0, a1;
      item_of(blockIdx.x, t0, a0, a1);
      load_idx(blockIdx.x < p.items ? t0 : p.T, a0, idx);
    }
    for (int it = blockIdx.x; it < p.items && ok; it += gridDim.x) {
      int t, c0, c1;
      item_of(it, t, c0, c1);
      for (int c = c0; c < c1 && ok; ++c, ++gc) {
        const char* src[4];
        if (!kWin || c < p.npc) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            src[i] = (idx[i] >= 0 && idx[i] < p.S)
                         ? reinterpret_cast<const char*>(p.kv + (int64_t)idx[i] * kDkv) + ch * 16
                         : nullptr;
        } else {
          // window row jl of the token sits at position p - W + 1 + jl, buffer row that - local_pos0
          const int lc = (c - p.npc) * kRows;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int jl = lc + (pt >> 3) + 16 * i;
            const int64_t a = (int64_t)idx[0] - p.window + 1 + jl, r = a - p.local_pos0;
            src[i] = (jl < p.window && a >= 0 && r >= 0 && r < p.L)
                         ? reinterpret_cast<const char*>(p.kv_local + r * kDkv) + ch * 16
                         : nullptr;
          }
        }
        // the next chunk's indices are on their way while this chunk is issued
        {
          int nt, nc;
          next_chunk(it, t, c, c1, nt, nc);
          load_idx(nt, nc, idx);
        }
        const int b = gc & 1;
        uint8_t* buf = skv + b * kBufBytes;
        for (int pr = 0; pr < kPairs; ++pr) {
          if (!mbar_wait(&kvempty[b * kPairs + pr], ((gc >> 1) & 1) ^ 1, p.status, 21)) { ok = false; break; }
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int kb = 2 * pr + h2;
            const uint32_t base = smem_u32(buf + kb * kSlotBytes);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              cp_async16(base + dst_off[i], src[i] ? src[i] + kb * 128 : reinterpret_cast<const char*>(p.zero_src),
                         src[i] ? 16u : 0u);
          }
          cp_async_arrive(&kvfull[b * kPairs + pr]);
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------------ S = Q Ksel^T
    uint32_t gc = 0, tok_i = 0;
    bool ok = true;
    const uint32_t q_addr = smem_u32(sq);
    const uint32_t kv_addr = smem_u32(skv);
    for (int it = blockIdx.x; it < p.items && ok; it += gridDim.x, ++tok_i) {
      int t, c0, c1;
      item_of(it, t, c0, c1);
      for (int c = c0; c < c1; ++c, ++gc) {
        const int sb = gc & 1, b = gc & 1;
        if (!mbar_wait(&sempty[sb], ((gc >> 1) & 1) ^ 1, p.status, 31)) { ok = false; break; }
        for (int pr = 0; pr < kPairs; ++pr) {
          if (c == c0 && !mbar_wait(&qfull[pr], tok_i & 1, p.status, 30)) { ok = false; break; }
          if (!mbar_wait(&kvfull[b * kPairs + pr], (gc >> 1) & 1, p.status, 32)) { ok = false; break; }
          fence_proxy_async();  // gathered rows -> visible to the tensor core
          tc_fence_after();
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int kb = 2 * pr + h2;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = desc_sw128(q_addr + kb * kQBlockBytes + kk * 32, 16, 1024);
              const uint64_t bd = desc_sw128(kv_addr + b * kBufBytes + kb * kSlotBytes + kk * 32, 16, 1024);
              tc_mma_f16_elect(tmem + sb * kHq, a, bd, kIdescS, (kb | kk) != 0);
            }
          }
          if (c == c1 - 1) tc_commit_elect(&qempty[pr]);  // the next item's q may replace this pair
        }
        if (!ok) break;
        tc_commit_elect(&sfull[sb]);
      }
    }
  } else if (warp == kOWarp) {
    // --------------------------------------------------------------- O^T += V^T P^T
    uint32_t gc = 0, tok_i = 0;
    uint32_t o_ph = 0;  // bit s: phase of O^T slot s's empty barrier (uses completed, mod 2)
    bool ok = true;
    const uint32_t kv_addr = smem_u32(skv);
    const uint32_t p_addr = smem_u32(sp);
    for (int it = blockIdx.x; it < p.items && ok; it += gridDim.x, ++tok_i) {
      int t, c0, c1;
      item_of(it, t, c0, c1);
      for (int c = c0; c < c1; ++c, ++gc) {
        const int pb = gc & 1, b = gc & 1;
        if (!mbar_wait(&pfull[pb], (gc >> 1) & 1, p.status, 33)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int db = 0; db < kPairs; ++db) {
          const int os = oslot(tok_i, db);
          // an item's first product overwrites its O^T slot: the output that last read it is done
          if (c == c0) {
            if (!mbar_wait(&oempty[os], ((o_ph >> os) & 1u) ^ 1u, p.status, 34)) { ok = false; break; }
            o_ph ^= 1u << os;
            tc_fence_after();
          }
#pragma unroll
          for (int ks = 0; ks < kRows / 16; ++ks) {
            const uint64_t a = desc_sw128(kv_addr + b * kBufBytes + (2 * db) * kSlotBytes + ks * 2048, kSlotBytes, 1024);
            const uint64_t bd = desc_sw128(p_addr + pb * kPBytes + ks * 32, 16, 1024);
            tc_mma_f16_elect(tmem + kColO + os * kHq, a, bd, kIdescO, (c > c0 || ks > 0));
          }
          tc_commit_elect(&kvempty[b * kPairs + db]);  // this 128-dim slice of the chunk is free
          if (c == c1 - 1) tc_commit_elect(&ofull[os]);
        }
        if (!ok) break;
        tc_commit_elect(&pempty[pb]);
      }
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------------- softmax
    // S holds head 16q + i on TMEM lane 32q + i (i < 16).  The 16x256b load gives thread
    // (g = lane/4, e = lane%4) the heads hA = 16q + g and hB = hA + 8 and, of each, the
    // columns 8r + 2e + {0, 1}, r = 0..7: every head's 64 scores are spread over 4 threads.
    const int quad = warp - 4;
    const int g = lane >> 2, e = lane & 3;
    const int hA = 16 * quad + g, hB = hA + 8;
    const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
    const float c = p.scale_log2;
    uint32_t gc = 0, tok_i = 0;
    bool ok = true;
    // validity of the 64 rows of a chunk: two ballots over per-lane index loads, one chunk ahead
    // (a window chunk loads the token's position into i0 instead)
    auto load_valid = [&](int t, int ci, int32_t& i0, int32_t& i1) {
      if (!kWin || ci < p.npc) {
        const int j0 = ci * kRows + lane, j1 = j0 + 32;
        i0 = (t < p.T && ci < nch && j0 < p.k_top) ? __ldg(p.indices + (int64_t)t * p.k_top + j0) : -1;
        i1 = (t < p.T && ci < nch && j1 < p.k_top) ? __ldg(p.indices + (int64_t)t * p.k_top + j1) : -1;
      } else {
        i0 = t < p.T ? __ldg(p.positions + t) : INT_MIN;
        i1 = 0;
      }
    };
    auto window_row_valid = [&](int32_t pos, int ci, int j) {
      const int jl = (ci - p.npc) * kRows + j;
      const int64_t a = (int64_t)pos - p.window + 1 + jl, r = a - p.local_pos0;
      return jl < p.window && a >= 0 && r >= 0 && r < p.L;
    };
    int32_t ni0, ni1;
    {
      int t0, a0, a1;
      item_of(blockIdx.x, t0, a0, a1);
      load_valid(blockIdx.x < p.items ? t0 : p.T, a0, ni0, ni1);
    }
    for (int it = blockIdx.x; it < p.items && ok; it += gridDim.x, ++tok_i) {
      int t, c0, c1;
      item_of(it, t, c0, c1);
      float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;  // running max (scaled, log2) and sum
      for (int ci = c0; ci < c1; ++ci, ++gc) {
        const bool pooled = !kWin || ci < p.npc;
        const bool ok0 = pooled ? (ni0 >= 0 && ni0 < p.S) : window_row_valid(ni0, ci, lane);
        const bool ok1 = pooled ? (ni1 >= 0 && ni1 < p.S) : window_row_valid(ni0, ci, lane + 32);
        const uint32_t v0 = __ballot_sync(0xffffffffu, ok0) >> (2 * e);
        const uint32_t v1 = __ballot_sync(0xffffffffu, ok1) >> (2 * e);
        {
          int nt, nc;
          next_chunk(it, t, ci, c1, nt, nc);
          load_valid(nt, nc, ni0, ni1);
        }
        const int sb = gc & 1;
        ok = named_and(kSoftBar, kGroupThreads, mbar_wait(&sfull[sb], (gc >> 1) & 1, p.status, 40));
        if (!ok) break;
        tc_fence_after();
        float x[32];
        tmem_ld_16x256b_x8(tmem + t_lane + sb * kHq, x);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[sb]);
        float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t bits = (r < 4 ? v0 : v1) >> (8 * (r & 3));
          const bool ok0 = (bits & 1u) != 0, ok1 = (bits & 2u) != 0;
          x[4 * r] = ok0 ? x[4 * r] : -INFINITY;
          x[4 * r + 2] = ok0 ? x[4 * r + 2] : -INFINITY;
          x[4 * r + 1] = ok1 ? x[4 * r + 1] : -INFINITY;
          x[4 * r + 3] = ok1 ? x[4 * r + 3] : -INFINITY;
          mxA = fmaxf(mxA, fmaxf(x[4 * r], x[4 * r + 1]));
          mxB = fmaxf(mxB, fmaxf(x[4 * r + 2], x[4 * r + 3]));
        }
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2)) * c;
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2)) * c;
        // lazy running max: raised only when a logit exceeds it by more than 2^8 (or the head
        // saw its first valid row; alpha = 0 then, and nothing was accumulated for it yet)
        float aA = 1.f, aB = 1.f;
        bool needA = false, needB = false;
        if (mxA > mA + kRescaleLog2) {
          needA = mA != -INFINITY;
          aA = needA ? ex2_approx(mA - mxA) : 0.f;
          mA = mxA;
        }
        if (mxB > mB + kRescaleLog2) {
          needB = mB != -INFINITY;
          aB = needB ? ex2_approx(mB - mxB) : 0.f;
          mB = mxB;
        }
        if (named_or(kSoftBar, kGroupThreads, needA || needB)) {
          if (e == 0) {
            alpha_s[hA] = needA ? aA : 1.f;
            alpha_s[hB] = needB ? aB : 1.f;
          }
          named_sync(kSoftBar, kGroupThreads);
          // O^T must hold all of the previous chunk before its columns are rescaled
          const uint32_t prev = gc - 1;
          ok = named_and(kSoftBar, kGroupThreads, mbar_wait(&pempty[prev & 1], (prev >> 1) & 1, p.status, 41));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int q2 = 0; q2 < 2 * kPairs; ++q2) {  // 4 d-blocks x 2 halves of 32 heads
            float v[32];
            const uint32_t ta = tmem + t_lane + kColO + oslot(tok_i, q2 >> 1) * kHq + (q2 & 1) * 32;
            tmem_ld32(ta, v);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha_s[(q2 & 1) * 32 + i];
            tmem_st32(ta, v);
          }
          tc_wait_st();
          named_sync(kSoftBar, kGroupThreads);
        }
        lA *= aA;
        lB *= aB;
        // p = 2^(x c - m), rounded to the kv dtype; the sums use the rounded values
        const float nA = (mA == -INFINITY) ? 0.f : -mA;
        const float nB = (mB == -INFINITY) ? 0.f : -mB;
        uint32_t pkA[8], pkB[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          float r0, r1, r2, r3;
          pkA[r] = pack2<kBf16>(ex2_approx(fmaf(x[4 * r], c, nA)), ex2_approx(fmaf(x[4 * r + 1], c, nA)), r0, r1);
          pkB[r] = pack2<kBf16>(ex2_approx(fmaf(x[4 * r + 2], c, nB)), ex2_approx(fmaf(x[4 * r + 3], c, nB)), r2, r3);
          lA += r0 + r1;
          lB += r2 + r3;
        }
        const int pb = gc & 1;
        ok = named_and(kSoftBar, kGroupThreads, mbar_wait(&pempty[pb], ((gc >> 1) & 1) ^ 1, p.status, 42));
        if (!ok) break;
        {
          // P[h][j], K-major with the 128-byte swizzle: 16-byte chunk r of line h at (r ^ (h & 7))
          uint8_t* lineA = sp + pb * kPBytes + hA * 128 + 4 * e;
          uint8_t* lineB = sp + pb * kPBytes + hB * 128 + 4 * e;
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            *reinterpret_cast<uint32_t*>(lineA + ((r ^ (hA & 7)) << 4)) = pkA[r];
            *reinterpret_cast<uint32_t*>(lineB + ((r ^ (hB & 7)) << 4)) = pkB[r];
          }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[pb]);
        if (ci == c1 - 1) {
          lA += __shfl_xor_sync(0xffffffffu, lA, 1);
          lB += __shfl_xor_sync(0xffffffffu, lB, 1);
          lA += __shfl_xor_sync(0xffffffffu, lA, 2);
          lB += __shfl_xor_sync(0xffffffffu, lB, 2);
          // the slot of this item's parity was last read by the output of item tok_i - 2
          ok = named_and(kSoftBar, kGroupThreads,
                         mbar_wait(&lfree[tok_i & 1], ((tok_i >> 1) & 1) ^ 1, p.status, 45));
          if (!ok) break;
          if (e == 0) {
            float* row = lm + (tok_i & 1) * 3 * kHq;
            row[hA] = lA;
            row[kHq + hA] = mA;
            row[2 * kHq + hA] = lA > 0.f ? 1.f / lA : 0.f;
            row[hB] = lB;
            row[kHq + hB] = mB;
            row[2 * kHq + hB] = lB > 0.f ? 1.f / lB : 0.f;
            if (p.nsplit > 1) {
              float* ml = p.part_ml + (int64_t)it * 2 * kHq;
              ml[hA] = mA;
              ml[hB] = mB;
              ml[kHq + hA] = lA;
              ml[kHq + hB] = lB;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&lready[tok_i & 1]);
        }
      }
    }
  } else if (warp < 12) {
    // ----------------------------------------------------------------------- output
    // O^T lanes 32q + lane (dims) of each 128-dim block; every d-block is released to the next
    // token's products as soon as it is in registers
    const int quad = warp - 8;
    const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t tok_i = 0;
    uint32_t f_ph = 0;  // bit s: phase of O^T slot s's full barrier
    bool ok = true;
    const bool odd = lane & 1;
    for (int it = blockIdx.x; it < p.items && ok; it += gridDim.x, ++tok_i) {
      const int t = it / p.nsplit;
      const int par = tok_i & 1;
      ok = named_and(kEpiBar, kGroupThreads, mbar_wait(&lready[par], (tok_i >> 1) & 1, p.status, 43));
      if (!ok) break;
      const float* lrow = lm + par * 3 * kHq;
      if (quad == 0 && p.nsplit == 1) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int hh = lane + 32 * k;
          const float l = lrow[hh];
          if (p.lse) p.lse[(int64_t)t * kHq + hh] = l > 0.f ? (lrow[kHq + hh] + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
      }
      // an item of a split token writes its normalized part, in the output's layout and dtype
      uint32_t* orow = reinterpret_cast<uint32_t*>(p.nsplit > 1 ? p.part + (int64_t)it * kHq * kDkv
                                                                 : p.out + (int64_t)t * kHq * kDkv);
#pragma unroll 1
      for (int db = 0; db < kPairs; ++db) {
        const int os = oslot(tok_i, db);
        ok = __all_sync(0xffffffffu, mbar_wait(&ofull[os], (f_ph >> os) & 1u, p.status, 44));
        if (!ok) break;
        f_ph ^= 1u << os;
        tc_fence_after();
        float v[64];
        {
          float va[32], vb[32];
          tmem_ld32(tmem + t_lane + kColO + os * kHq, va);
          tmem_ld32(tmem + t_lane + kColO + os * kHq + 32, vb);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = va[i];
            v[i + 32] = vb[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&oempty[os]);
        const int d_even = db * 128 + quad * 32 + (lane & ~1);
#pragma unroll
        for (int h0 = 0; h0 < kHq; h0 += 2) {
          const float a0 = v[h0] * lrow[2 * kHq + h0];
          const float a1 = v[h0 + 1] * lrow[2 * kHq + h0 + 1];
          const float give = odd ? a0 : a1;
          const float got = __shfl_xor_sync(0xffffffffu, give, 1);
          const int hw = h0 + (odd ? 1 : 0);
          const uint32_t pair = odd ? (uint32_t)to16<kBf16>(got) | ((uint32_t)to16<kBf16>(a1) << 16)
                                    : (uint32_t)to16<kBf16>(a0) | ((uint32_t)to16<kBf16>(got) << 16);
          orow[((int64_t)hw * kDkv + d_even) >> 1] = pair;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&lfree[par]);
    }
  } else if (warp == kQWarp) {
    // ------------------------------------------------------------------------- q loader
    if (lane == 0) {
      uint32_t tok_i = 0;
      for (int it = blockIdx.x; it < p.items; it += gridDim.x, ++tok_i) {
        const int t = it / p.nsplit;
        const int nit = it + (int)gridDim.x;  // the next item's q (64 KB, contiguous) moves to L2 now
        if (nit < p.items) prefetch_l2(p.q + (int64_t)(nit / p.nsplit) * kHq * kDkv, kQBytes);
        bool ok = true;
        for (int pr = 0; pr < kPairs; ++pr) {
          if (!mbar_wait(&qempty[pr], (tok_i & 1) ^ 1, p.status, 20)) { ok = false; break; }
          mbar_arrive_expect_tx(&qfull[pr], 2 * kQBlockBytes);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int kb = 2 * pr + h2;
            tma_load_2d(sq + kb * kQBlockBytes, &tm_q, &qfull[pr], kb * 64, t * kHq);
          }
        }
        if (!ok) break;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge of a token's split items (one block per (token, head), 4 dims a thread): item i holds
// P_i = O_i / l_i, O_i = sum_j 2^(x_j - m_i) kv_j and l_i = sum_j 2^(x_j - m_i) over its rows, so
//   out = sum_i 2^(m_i - M) l_i P_i / L,  L = sum_i 2^(m_i - M) l_i,  M = max_i m_i,  lse = ln 2 (M + log2 L).
template <bool kBf16>
__device__ __forceinline__ float4 load4_16(const uint16_t* src) {
  const uint2 u = *reinterpret_cast<const uint2*>(src);
  if constexpr (kBf16) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x), b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
    return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
  } else {
    const __half2 a = *reinterpret_cast<const __half2*>(&u.x), b = *reinterpret_cast<const __half2*>(&u.y);
    return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(128) combine_kernel(const uint16_t* __restrict__ part,
                                                      const float* __restrict__ part_ml, int nsplit,
                                                      uint16_t* __restrict__ out, float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x / kHq, h = blockIdx.x - t * kHq;
  const float* ml = part_ml + (int64_t)t * nsplit * 2 * kHq;
  // every part's statistics and partial row are loaded before any is used (nsplit <= kMaxSplit)
  float m[kMaxSplit], l[kMaxSplit];
  float4 o[kMaxSplit];
#pragma unroll
  for (int i = 0; i < kMaxSplit; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
    o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < nsplit) {
      m[i] = ml[i * 2 * kHq + h];
      l[i] = ml[i * 2 * kHq + kHq + h];
      o[i] = load4_16<kBf16>(part + (((int64_t)t * nsplit + i) * kHq + h) * kDkv + 4 * threadIdx.x);
    }
  }
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMaxSplit; ++i) mx = fmaxf(mx, m[i]);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kMaxSplit; ++i) {
    const float wgt = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - mx) * l[i];
    L += wgt;
    acc.x += wgt * o[i].x;
    acc.y += wgt * o[i].y;
    acc.z += wgt * o[i].z;
    acc.w += wgt * o[i].w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float r0, r1;
  const uint32_t lo = pack2<kBf16>(acc.x * inv, acc.y * inv, r0, r1);
  const uint32_t hi = pack2<kBf16>(acc.z * inv, acc.w * inv, r0, r1);
  *reinterpret_cast<uint2*>(out + ((int64_t)t * kHq + h) * kDkv + 4 * threadIdx.x) = make_uint2(lo, hi);
  if (threadIdx.x == 0 && lse)
    lse[(int64_t)t * kHq + h] = L > 0.f ? (mx + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

// Chunks of one token: the pooled rows', then the window's.
int chunks_of(int k_top, int window) { return (k_top + kRows - 1) / kRows + (window + kRows - 1) / kRows; }

// Split plan: when the tokens fill less than half of the SMs, a token's nch chunks are spread over
// up to sms / T items (at least one chunk each, at most kMaxSplit) and merged by combine_kernel.
void split_plan(int T, int nch, int sms, int& nsplit, int& cps) {
  nsplit = 1;
  cps = nch;
  if (T <= 0 || 2 * T > sms || nch < 2) return;
  int want = sms / T;
  if (want > nch) want = nch;
  if (want > kMaxSplit) want = kMaxSplit;
  cps = (nch + want - 1) / want;
  nsplit = (nch + cps - 1) / cps;
}

size_t partial_bytes_for(int T, int nsplit) {
  if (nsplit <= 1) return 0;
  return (size_t)T * nsplit * ((size_t)kHq * kDkv * 2 + 2 * kHq * 4);
}


template <bool kBf16>
int launch_impl(const AttnArgs& a, cudaStream_t stream) {
  if (ensure_dynamic_smem(sparse_mqa_kernel<kBf16, false>, kSmem) != cudaSuccess ||
      ensure_dynamic_smem(sparse_mqa_kernel<kBf16, true>, kSmem) != cudaSuccess)
    return DS4X_ERR_CUDA;
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return DS4X_ERR_CUDA;
  CUtensorMap tq;
  cuuint64_t dims[2] = {(cuuint64_t)kDkv, (cuuint64_t)a.T * kHq};
  cuuint64_t strides[1] = {(cuuint64_t)kDkv * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kHq};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&tq, kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
         const_cast<void*>(a.q_attn), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return DS4X_ERR_CUDA;
  Params p;
  p.q = static_cast<const uint16_t*>(a.q_attn);
  p.kv = static_cast<const uint16_t*>(a.kv);
  p.zero_src = static_cast<const uint16_t*>(a.q_attn);
  p.indices = a.indices;
  const bool win = a.local.active();
  p.kv_local = win ? static_cast<const uint16_t*>(a.local.kv_local) : nullptr;
  p.positions = win ? a.positions : nullptr;
  p.L = win ? a.local.L : 0;
  p.local_pos0 = win ? a.local.local_pos0 : 0;
  p.window = win ? a.local.window : 0;
  p.out = static_cast<uint16_t*>(a.out);
  p.lse = a.lse;
  p.status = device_status_ptr();
  p.T = a.T;
  p.S = a.S;
  p.k_top = a.k_top;
  p.npc = (a.k_top + kRows - 1) / kRows;
  p.nchunks = chunks_of(a.k_top, p.window);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const int sms = device_sm_count();
  p.nsplit = 1;
  p.cps = p.nchunks;
  p.part = nullptr;
  p.part_ml = nullptr;
  if (a.partial) {
    int ns, cps;
    split_plan(a.T, p.nchunks, sms, ns, cps);
    const size_t need = partial_bytes_for(a.T, ns);
    if (ns > 1 && a.partial_bytes >= need) {
      p.nsplit = ns;
      p.cps = cps;
      p.part = static_cast<uint16_t*>(a.partial);
      p.part_ml = reinterpret_cast<float*>(p.part + (size_t)a.T * ns * kHq * kDkv);
    }
  }
  p.items = a.T * p.nsplit;
  const int grid = p.items < sms ? p.items : sms;
  if (launch_pdl(win ? sparse_mqa_kernel<kBf16, true> : sparse_mqa_kernel<kBf16, false>, dim3(grid), dim3(kThreads),
                 (size_t)kSmem, stream, tq, p) != cudaSuccess)
    return DS4X_ERR_CUDA;
  count_launch();
  if (p.nsplit > 1) {
    if (launch_pdl(combine_kernel<kBf16>, dim3(a.T * kHq), dim3(kDkv / 4), 0, stream, p.part, p.part_ml, p.nsplit,
                   static_cast<uint16_t*>(a.out), a.lse) != cudaSuccess)
      return DS4X_ERR_CUDA;
    count_launch();
  }
  return DS4X_OK;
}

}  // namespace

bool attn_shape_supported(int Hq, int Dkv) { return Hq == kHq && Dkv == kDkv; }

size_t attn_partial_bytes(int T, int k_top, int window) {
  int ns, cps;
  split_plan(T, chunks_of(k_top, window), device_sm_count(), ns, cps);
  return partial_bytes_for(T, ns);
}

int launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  if (a.T == 0) return DS4X_OK;
  return a.bf16 ? launch_impl<true>(a, stream) : launch_impl<false>(a, stream);
}

}  // namespace ds4x
