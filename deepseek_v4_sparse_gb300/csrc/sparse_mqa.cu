// sparse_mqa.cu — multi-query attention of 64 heads over the rows chosen by the indexer.
//
//   out[t,h,:] = sum_j softmax_j( scale * q_attn[t,h,:] . kv[idx_j,:] ) * kv[idx_j,:]
//
// Source: "How I turned one oversized DeepSeek optimization into three merged oMLX PRs",
// section "The three changes that merged", item 1 (attention over pooled compressed rows picked
// by an index list, kv rows serving as both key and value), fed by the top-512 of "How I made
// DeepSeek 12x faster on a Mac Studio", section "1: the kernels".
//
// One CTA per SM, persistent over tokens; per token the 512 selected rows are processed in
// chunks of 128.  Both products run on tcgen05 with M = 128 by putting the selected rows /
// the value dimension on the M axis:
//   logits^T [128 rows x 64 heads]  = Ksel [128 x 512] . Q^T           (A, B K-major)
//   O^T      [512 dims x 64 heads] += Vsel^T [512 x 128] . P^T [128 x 64] (A, B MN-major)
// with the fp32 accumulators in TMEM (logits double-buffered in columns 0..127, O^T in
// columns 256..511).  The softmax runs over TMEM lanes (the rows), so the per-head max and sum
// are cross-lane: each warp does a 31-shuffle transpose-reduction of its 32 rows x 32 heads,
// then four warps combine through shared memory.  The running max is only raised when a
// head's max grows by more than 2^8 (then O^T and the partial sums are rescaled in place),
// so the probabilities written as fp16/bf16 stay <= 256.
//
// Rows are gathered with 16-byte cp.async (zero-filled for invalid indices) straight into the
// 128B-swizzled layout both products read: row j of a chunk occupies one 128-byte line in
// each of 8 slots (slot = 64 consecutive dims); a slot is refilled as soon as the O^T product
// that reads it has completed.
//
// Warps: 0-3 gather (128 threads; thread 0 also loads Q by TMA), 4-11 softmax and output
// (warp%4 = TMEM lane quadrant, (warp-4)/4 = which 32 heads), 12 MMA issue + TMEM allocation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "ds4x_internal.h"
#include "ds4x_ptx.cuh"

namespace ds4x {
namespace {

constexpr int kHq = 64;
constexpr int kDkv = 512;
constexpr int kRows = 128;                      // rows per chunk
constexpr int kSlots = kDkv / 64;               // 8 slots of 64 dims
constexpr int kSlotBytes = kRows * 128;         // 16 KB
constexpr int kQBlockBytes = kHq * 128;         // 8 KB (64 heads x 64 dims)
constexpr int kQBytes = kSlots * kQBlockBytes;  // 64 KB
constexpr int kPBytes = kRows * 128;            // 16 KB (128 rows x 64 heads)
constexpr int kOffKV = kQBytes;
constexpr int kOffP = kOffKV + kSlots * kSlotBytes;
constexpr int kOffRed = kOffP + 2 * kPBytes;          // float[4][64]
constexpr int kOffM = kOffRed + 4 * kHq * 4;          // float[64] running max (log2 units)
constexpr int kOffAlpha = kOffM + kHq * 4;            // float[64] rescale factors / 1/l
constexpr int kOffBars = kOffAlpha + kHq * 4;
constexpr int kNumBars = 2 + 2 * kSlots + 2 + 2 + 2 + 2 + 2;
constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr int kSmem = kOffTmemSlot + 16;
constexpr int kThreads = 13 * 32;
constexpr int kMmaWarp = 12;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kSoftBar = 2;      // named barrier of the 8 softmax warps
constexpr int kSoftThreads = 256;

struct Params {
  const uint16_t* kv;        // [S, 512]; never read through an invalid index
  const uint16_t* zero_src;  // any valid address: source of the zero-filled (size 0) copies
  const int32_t* indices;
  uint16_t* out;
  float* lse;
  int* status;
  int T, S, k_top, nchunks;
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

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mqa_kernel(const __grid_constant__ CUtensorMap tm_q, const Params p) {
  constexpr uint32_t kIdescS = idesc_f16(128, kHq, kBf16 ? 1 : 0, 0, 0);
  constexpr uint32_t kIdescO = idesc_f16(128, kHq, kBf16 ? 1 : 0, 1, 1);
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) report_timeout(p.status, 0x7f);
    return;
  }
  uint8_t* sq = smem;
  uint8_t* skv = smem + kOffKV;
  uint8_t* sp = smem + kOffP;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* m_run = reinterpret_cast<float*>(smem + kOffM);
  float* alpha = reinterpret_cast<float*>(smem + kOffAlpha);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* qfull = bars;
  uint64_t* qempty = bars + 1;
  uint64_t* slot_full = bars + 2;
  uint64_t* slot_empty = slot_full + kSlots;
  uint64_t* sfull = slot_empty + kSlots;
  uint64_t* sempty = sfull + 2;
  uint64_t* pfull = sempty + 2;
  uint64_t* pempty = pfull + 2;
  uint64_t* ofull = pempty + 2;
  uint64_t* oempty = ofull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    mbar_init(qempty, 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&slot_full[i], 128);
      mbar_init(&slot_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 8);
      mbar_init(&pfull[i], 8);
      mbar_init(&pempty[i], 1);
    }
    mbar_init(ofull, 1);
    mbar_init(oempty, 8);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_q);
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------------------ gather
    const int pt = threadIdx.x;  // 0..127
    const int ch = pt & 7;       // 16-byte column chunk within a 128-byte line
    uint32_t gc = 0, tok_i = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.T && ok; t += gridDim.x, ++tok_i) {
      if (pt == 0) {
        if (!mbar_wait(qempty, (tok_i & 1) ^ 1, p.status, 20)) { ok = false; }
        if (ok) {
          mbar_arrive_expect_tx(qfull, kQBytes);
          for (int kb = 0; kb < kSlots; ++kb) tma_load_2d(sq + kb * kQBlockBytes, &tm_q, qfull, kb * 64, t * kHq);
        }
      }
      for (int c = 0; c < p.nchunks && ok; ++c, ++gc) {
        // this thread copies 16-byte column chunk `ch` of rows (pt>>3) + 16 i, i = 0..7, in every
        // slot: the source row offsets and the swizzled destinations are fixed for the chunk
        const char* src_row[8];
        uint32_t dst_off[8], src_bytes[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = (pt >> 3) + 16 * i;
          const int j = c * kRows + r;
          int32_t idx = -1;
          if (j < p.k_top) idx = __ldg(p.indices + (int64_t)t * p.k_top + j);
          const bool valid = idx >= 0 && idx < p.S;
          src_row[i] = valid ? reinterpret_cast<const char*>(p.kv + (int64_t)idx * kDkv) + ch * 16
                             : reinterpret_cast<const char*>(p.zero_src);
          src_bytes[i] = valid ? 16u : 0u;
          dst_off[i] = r * 128 + ((ch ^ (r & 7)) << 4);
        }
        for (int kb = 0; kb < kSlots; ++kb) {
          if (!mbar_wait(&slot_empty[kb], (gc & 1) ^ 1, p.status, 21)) { ok = false; break; }
          const uint32_t base = smem_u32(skv + kb * kSlotBytes);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            cp_async16(base + dst_off[i], src_row[i] + (src_bytes[i] ? kb * 128 : 0), src_bytes[i]);
          cp_async_arrive(&slot_full[kb]);
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------------------- MMA
    if (lane == 0) {
      uint32_t gc = 0, tok_i = 0;
      bool ok = true;
      const uint32_t q_addr = smem_u32(sq);
      const uint32_t kv_addr = smem_u32(skv);
      const uint32_t p_addr = smem_u32(sp);
      for (int t = blockIdx.x; t < p.T && ok; t += gridDim.x, ++tok_i) {
        if (!mbar_wait(qfull, tok_i & 1, p.status, 30)) break;
        tc_fence_after();
        for (int c = 0; c < p.nchunks; ++c, ++gc) {
          const int sb = gc & 1;
          if (!mbar_wait(&sempty[sb], ((gc >> 1) & 1) ^ 1, p.status, 31)) { ok = false; break; }
          tc_fence_after();
          for (int kb = 0; kb < kSlots && ok; ++kb) {
            if (!mbar_wait(&slot_full[kb], gc & 1, p.status, 32)) { ok = false; break; }
            fence_proxy_async();  // cp.async data -> visible to the tensor core
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = desc_sw128(kv_addr + kb * kSlotBytes + kk * 32, 16, 1024);
              const uint64_t b = desc_sw128(q_addr + kb * kQBlockBytes + kk * 32, 16, 1024);
              tc_mma_f16(tmem + sb * kHq, a, b, kIdescS, (kb | kk) != 0);
            }
          }
          if (!ok) break;
          tc_commit(&sfull[sb]);
          if (c == p.nchunks - 1) tc_commit(qempty);
          const int pb = gc & 1;
          if (!mbar_wait(&pfull[pb], (gc >> 1) & 1, p.status, 33)) { ok = false; break; }
          if (c == 0 && !mbar_wait(oempty, (tok_i & 1) ^ 1, p.status, 34)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int db = 0; db < kDkv / 128; ++db) {
#pragma unroll
            for (int ks = 0; ks < kRows / 16; ++ks) {
              const uint64_t a = desc_sw128(kv_addr + (2 * db) * kSlotBytes + ks * 2048, kSlotBytes, 1024);
              const uint64_t b = desc_sw128(p_addr + pb * kPBytes + ks * 2048, kSlotBytes, 1024);
              tc_mma_f16(tmem + kColO + db * kHq, a, b, kIdescO, (c > 0 || ks > 0));
            }
            tc_commit(&slot_empty[2 * db]);
            tc_commit(&slot_empty[2 * db + 1]);
          }
          tc_commit(&pempty[pb]);
        }
        if (!ok) break;
        tc_commit(ofull);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------- softmax and output
    const int quad = warp & 3;
    const int hh = (warp - 4) >> 2;  // heads 32*hh .. 32*hh+31
    const int hcol = hh * 32;
    const bool owner = (quad == 0);  // lane l of warps 4 and 8 owns head hcol + l
    const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t gc = 0, tok_i = 0;
    float lpart[32];
    bool ok = true;
    // validity of this thread's row in the next chunk, loaded one chunk ahead
    auto row_valid = [&](int t, int c) {
      const int j = c * kRows + quad * 32 + lane;
      if (t >= p.T || c >= p.nchunks || j >= p.k_top) return false;
      const int32_t idx = __ldg(p.indices + (int64_t)t * p.k_top + j);
      return idx >= 0 && idx < p.S;
    };
    bool next_valid = row_valid(blockIdx.x, 0);
    for (int t = blockIdx.x; t < p.T && ok; t += gridDim.x, ++tok_i) {
#pragma unroll
      for (int i = 0; i < 32; ++i) lpart[i] = 0.f;
      for (int c = 0; c < p.nchunks; ++c, ++gc) {
        const bool valid = next_valid;
        next_valid = (c + 1 < p.nchunks) ? row_valid(t, c + 1) : row_valid(t + gridDim.x, 0);
        const int sb = gc & 1;
        ok = named_and(kSoftBar, kSoftThreads, mbar_wait(&sfull[sb], (gc >> 1) & 1, p.status, 40));
        if (!ok) break;
        tc_fence_after();
        float x[32];
        tmem_ld32(tmem + t_lane + sb * kHq + hcol, x);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[sb]);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = valid ? x[i] * p.scale_log2 : -INFINITY;
        // The running max of a head only has to keep every logit within 2^8 of it (so the
        // probabilities stay <= 256); the exact column max is taken on a token's first chunk and
        // again only when some logit overshoots the running max by more than that.
        bool over = (c == 0);
        if (c > 0) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(&m_run[hcol + i]);
            over |= (x[i] > m4.x + kRescaleLog2) | (x[i + 1] > m4.y + kRescaleLog2) |
                    (x[i + 2] > m4.z + kRescaleLog2) | (x[i + 3] > m4.w + kRescaleLog2);
          }
        }
        const bool rescan = named_or(kSoftBar, kSoftThreads, over);
        bool rescale = false;
        if (rescan) {
          float tmp[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) tmp[i] = x[i];
          red[quad * kHq + hcol + lane] = warp_columns_reduce<true>(tmp);
          named_sync(kSoftBar, kSoftThreads);
          bool need = false;
          if (owner) {
            const int h = hcol + lane;
            const float cm = fmaxf(fmaxf(red[h], red[kHq + h]), fmaxf(red[2 * kHq + h], red[3 * kHq + h]));
            const float mo = (c == 0) ? -INFINITY : m_run[h];
            float a = 1.f;
            if (cm > mo + kRescaleLog2 || (mo == -INFINITY && cm > -INFINITY)) {
              a = (mo == -INFINITY) ? 0.f : ex2_approx(mo - cm);
              m_run[h] = cm;
              need = (c > 0) && (mo != -INFINITY);
            } else if (c == 0) {
              m_run[h] = mo;  // -inf: nothing visible yet
            }
            alpha[h] = a;
          }
          rescale = named_or(kSoftBar, kSoftThreads, need);
        }
        if (rescale) {
          // O^T and the partial sums were built with the old max: scale them first, once the
          // previous chunk's O^T product has completed.
          const uint32_t prev = gc - 1;
          ok = named_and(kSoftBar, kSoftThreads, mbar_wait(&pempty[prev & 1], (prev >> 1) & 1, p.status, 41));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int db = 0; db < kDkv / 128; ++db) {
            float v[32];
            const uint32_t ta = tmem + t_lane + kColO + db * kHq + hcol;
            tmem_ld32(ta, v);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha[hcol + i];
            tmem_st32(ta, v);
          }
          tc_wait_st();
#pragma unroll
          for (int i = 0; i < 32; ++i) lpart[i] *= alpha[hcol + i];
        }
        // probabilities, rounded to the kv dtype (the sums use the rounded values)
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 m4 = *reinterpret_cast<const float4*>(&m_run[hcol + i]);
          // a head with no visible row yet has m = -inf and only -inf logits: use 0 instead
          m4.x = m4.x == -INFINITY ? 0.f : m4.x;
          m4.y = m4.y == -INFINITY ? 0.f : m4.y;
          m4.z = m4.z == -INFINITY ? 0.f : m4.z;
          m4.w = m4.w == -INFINITY ? 0.f : m4.w;
          float r0, r1, r2, r3;
          packed[(i >> 1) + 0] = pack2<kBf16>(ex2_approx(x[i] - m4.x), ex2_approx(x[i + 1] - m4.y), r0, r1);
          packed[(i >> 1) + 1] = pack2<kBf16>(ex2_approx(x[i + 2] - m4.z), ex2_approx(x[i + 3] - m4.w), r2, r3);
          lpart[i] += r0;
          lpart[i + 1] += r1;
          lpart[i + 2] += r2;
          lpart[i + 3] += r3;
        }
        const int pb = gc & 1;
        ok = named_and(kSoftBar, kSoftThreads, mbar_wait(&pempty[pb], ((gc >> 1) & 1) ^ 1, p.status, 42));
        if (!ok) break;
        {
          const int r = quad * 32 + lane;
          uint8_t* line = sp + pb * kPBytes + r * 128;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = (hh * 4 + q4) ^ (r & 7);
            *reinterpret_cast<uint4*>(line + chunk * 16) =
                make_uint4(packed[q4 * 4 + 0], packed[q4 * 4 + 1], packed[q4 * 4 + 2], packed[q4 * 4 + 3]);
          }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[pb]);
      }
      if (!ok) break;
      // ------------------------------------------------------------ token epilogue
      ok = named_and(kSoftBar, kSoftThreads, mbar_wait(ofull, tok_i & 1, p.status, 43));
      if (!ok) break;
      tc_fence_after();
      red[quad * kHq + hcol + lane] = warp_columns_reduce<false>(lpart);
      named_sync(kSoftBar, kSoftThreads);
      if (owner) {
        const int h = hcol + lane;
        const float l = (red[h] + red[kHq + h]) + (red[2 * kHq + h] + red[3 * kHq + h]);
        alpha[h] = l > 0.f ? 1.f / l : 0.f;
        if (p.lse) p.lse[(int64_t)t * kHq + h] = l > 0.f ? (m_run[h] + log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
      named_sync(kSoftBar, kSoftThreads);
      // out[t, h, d]: lane = d within the 32-row quadrant of a 128-wide d-block.  Lanes pair up
      // (d, d+1) so that each store writes two values: the even lane stores the even heads, the
      // odd lane the odd heads.
      uint32_t* orow = reinterpret_cast<uint32_t*>(p.out + (int64_t)t * kHq * kDkv);
      const bool odd = lane & 1;
#pragma unroll 1
      for (int db = 0; db < kDkv / 128; ++db) {
        float v[32];
        tmem_ld32(tmem + t_lane + kColO + db * kHq + hcol, v);
        tc_wait_ld();
        const int d_even = db * 128 + quad * 32 + (lane & ~1);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float a0 = v[i] * alpha[hcol + i];          // head hcol+i, this lane's d
          const float a1 = v[i + 1] * alpha[hcol + i + 1];  // head hcol+i+1
          // even lane needs the odd lane's value of head i; odd lane needs the even lane's of i+1
          const float give = odd ? a0 : a1;
          const float got = __shfl_xor_sync(0xffffffffu, give, 1);
          const int h = hcol + i + (odd ? 1 : 0);
          const uint32_t pair = odd ? (uint32_t)to16<kBf16>(got) | ((uint32_t)to16<kBf16>(a1) << 16)
                                    : (uint32_t)to16<kBf16>(a0) | ((uint32_t)to16<kBf16>(got) << 16);
          orow[((int64_t)h * kDkv + d_even) >> 1] = pair;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(oempty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

template <bool kBf16>
int launch_impl(const AttnArgs& a, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(sparse_mqa_kernel<kBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
      return DS4X_ERR_CUDA;
    attr_set = true;
  }
  EncodeTiledFn fn = encode_fn();
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
  p.kv = static_cast<const uint16_t*>(a.kv);
  p.zero_src = static_cast<const uint16_t*>(a.q_attn);
  p.indices = a.indices;
  p.out = static_cast<uint16_t*>(a.out);
  p.lse = a.lse;
  p.status = device_status_ptr();
  p.T = a.T;
  p.S = a.S;
  p.k_top = a.k_top;
  p.nchunks = (a.k_top + kRows - 1) / kRows;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const int sms = device_sm_count();
  const int grid = a.T < sms ? a.T : sms;
  sparse_mqa_kernel<kBf16><<<grid, kThreads, kSmem, stream>>>(tq, p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? DS4X_OK : DS4X_ERR_CUDA;
}

}  // namespace

bool attn_shape_supported(int Hq, int Dkv) { return Hq == kHq && Dkv == kDkv; }

int launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  if (a.T == 0) return DS4X_OK;
  return a.bf16 ? launch_impl<true>(a, stream) : launch_impl<false>(a, stream);
}

}  // namespace ds4x
