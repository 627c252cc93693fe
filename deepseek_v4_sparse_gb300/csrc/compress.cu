// compress.cu — the compressor: one pooled row per `ratio` positions, the partial block carried.
//
//   rows[j,d] = sum_i a_i x_i[d],   a_i = softmax_i(g_i[d] + bias[i,d]),   i over block j's positions
//
// Source: "How I turned one oversized DeepSeek optimization into three merged oMLX PRs", section
// "The three changes that merged", item 3 (the skip path still advances the indexer compressor and
// its cache; one pooled row per `ratio` positions) and the ds4.c overview, disk-cache layout (the
// "compressor frontier" tensors kept with the compressed rows).  The pages give no formula: the
// gated pooling above is this library's definition (equal gates give the block mean).
//
// Streaming and HBM-bound: a thread owns 8 channels (16-byte loads of x and g), or 4 (8-byte loads,
// more threads) when the blocks alone would not fill the GPU, of one block and one slice of the
// block's positions.  Positions go in batches of four (eight 16-byte loads in flight,
// one running-max rescale per batch, weights by ex2.approx on log2-scaled gates); the slices of a
// block are merged through shared memory.
// Sequence position v is frontier row v (v < n_frontier) or new row v - n_frontier.  One extra CTA
// copies the new frontier (the positions after the last full block).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ds4x_internal.h"
#include "ds4x_ptx.cuh"

namespace ds4x {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 4;  // positions loaded before their running-max update

struct CompressParams {
  const uint16_t* x;   // [T, D]
  const uint16_t* g;   // [T, D]
  const float* bias;   // [ratio, D]
  const uint16_t* fx;  // [nf, D] frontier rows in
  const uint16_t* fg;
  uint16_t* rows;      // [n_out, D]
  uint16_t* fx_out;    // [rem, D] frontier rows out
  uint16_t* fg_out;
  int nf, T, D, ratio, n_out, rem;
  int cg;     // channel groups (of 4 or 8 channels) per CTA slab
  int slabs;  // slabs per block (D / channels a group / cg)
  int ns;     // position slices per block
  int bpc;    // blocks per CTA
  int main_ctas;  // CTAs of blocks (one more copies the frontier)
};

// CPT channels a thread: their 16-bit values move as one vector (16 bytes for 8, 8 for 4)
template <int CPT>
struct Vec;
template <>
struct Vec<8> {
  using T = uint4;
  static constexpr int kWords = 4;
};
template <>
struct Vec<4> {
  using T = uint2;
  static constexpr int kWords = 2;
};

template <int CPT>
__device__ __forceinline__ void words_of(const typename Vec<CPT>::T& u, uint32_t (&w)[CPT / 2]) {
  if constexpr (CPT == 8) {
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  } else {
    w[0] = u.x; w[1] = u.y;
  }
}

template <bool kBf16, int CPT>
__device__ __forceinline__ void unpack(const typename Vec<CPT>::T& u, float (&f)[CPT]) {
  uint32_t w[CPT / 2];
  words_of<CPT>(u, w);
#pragma unroll
  for (int k = 0; k < CPT / 2; ++k) {
    if constexpr (kBf16) {
      const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
      f[2 * k] = __low2float(h);
      f[2 * k + 1] = __high2float(h);
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      f[2 * k] = __low2float(h);
      f[2 * k + 1] = __high2float(h);
    }
  }
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (kBf16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

__device__ __forceinline__ const uint16_t* seq_row(const uint16_t* held, const uint16_t* fresh, int nf, int64_t v,
                                                   int D) {
  return v < nf ? held + v * D : fresh + (v - nf) * D;
}

__device__ __forceinline__ uint4 ldg_vec(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ldg_vec(const uint2* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// 2^x with the hardware approximation (MUFU.EX2; flushes subnormal results to zero); 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// z = (g + bias) log2(e) for the CPT channels of one position (the product rounded on its own,
// never fused with what uses it, so that both compressor paths round a gate alike)
template <bool kBf16, int CPT>
__device__ __forceinline__ void gate(const typename Vec<CPT>::T& ug, const float* bias_row, float (&z)[CPT]) {
  unpack<kBf16, CPT>(ug, z);
#pragma unroll
  for (int k4 = 0; k4 < CPT / 4; ++k4) {
    const float4 b = __ldg(reinterpret_cast<const float4*>(bias_row) + k4);
    z[4 * k4] = __fmul_rn(z[4 * k4] + b.x, 1.4426950408889634f);
    z[4 * k4 + 1] = __fmul_rn(z[4 * k4 + 1] + b.y, 1.4426950408889634f);
    z[4 * k4 + 2] = __fmul_rn(z[4 * k4 + 2] + b.z, 1.4426950408889634f);
    z[4 * k4 + 3] = __fmul_rn(z[4 * k4 + 3] + b.w, 1.4426950408889634f);
  }
}

template <bool kBf16, int CPT>
__global__ void __launch_bounds__(kThreads, CPT == 4 ? 3 : 1) compress_kernel(const CompressParams p) {
  using V = typename Vec<CPT>::T;
  __shared__ float part[kThreads][3 * CPT];  // a slice's (m, l, acc) of its CPT channels
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  if ((int)blockIdx.x >= p.main_ctas) {
    // ------------------------------------------------ the new frontier: rem positions of x and g
    const int per_row = p.D / 8;
    for (int idx = tid; idx < p.rem * per_row; idx += blockDim.x) {
      const int i = idx / per_row, c = idx - i * per_row;
      const int64_t v = (int64_t)p.n_out * p.ratio + i;
      reinterpret_cast<uint4*>(p.fx_out + (int64_t)i * p.D)[c] =
          reinterpret_cast<const uint4*>(seq_row(p.fx, p.x, p.nf, v, p.D))[c];
      reinterpret_cast<uint4*>(p.fg_out + (int64_t)i * p.D)[c] =
          reinterpret_cast<const uint4*>(seq_row(p.fg, p.g, p.nf, v, p.D))[c];
    }
    return;
  }
  const int c = tid % p.cg;
  const int s = (tid / p.cg) % p.ns;
  const int b = tid / (p.cg * p.ns);
  const int slab = blockIdx.x % p.slabs;
  const int64_t j = (int64_t)(blockIdx.x / p.slabs) * p.bpc + b;
  const int grp = slab * p.cg + c;  // CPT-channel group within the row
  const bool active = b < p.bpc && j < p.n_out;
  // running max (log2 units), sum and weighted sum of the CPT channels
  float m[CPT], l[CPT], acc[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    m[k] = -INFINITY;
    l[k] = 0.f;
    acc[k] = 0.f;
  }
  if (active) {
    const int i0 = (int)((int64_t)s * p.ratio / p.ns), i1 = (int)((int64_t)(s + 1) * p.ratio / p.ns);
    for (int i = i0; i < i1; i += kBatch) {
      const int nb = min(kBatch, i1 - i);
      V ux[kBatch], ug[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        if (q < nb) {
          const int64_t v = j * p.ratio + i + q;
          ux[q] = ldg_vec(reinterpret_cast<const V*>(seq_row(p.fx, p.x, p.nf, v, p.D)) + grp);
          ug[q] = ldg_vec(reinterpret_cast<const V*>(seq_row(p.fg, p.g, p.nf, v, p.D)) + grp);
        }
      }
      // the batch's max raises the running max once; then its weights
      float bm[CPT];
#pragma unroll
      for (int k = 0; k < CPT; ++k) bm[k] = -INFINITY;
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        if (q < nb) {
          float z[CPT];
          gate<kBf16, CPT>(ug[q], p.bias + (int64_t)(i + q) * p.D + grp * CPT, z);
#pragma unroll
          for (int k = 0; k < CPT; ++k) bm[k] = fmaxf(bm[k], z[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        const float mn = fmaxf(m[k], bm[k]);
        const float sc = ex2_approx(m[k] - mn);  // 0 while m is still -inf
        l[k] *= sc;
        acc[k] *= sc;
        m[k] = mn;
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        if (q < nb) {
          float z[CPT], xv[CPT];
          gate<kBf16, CPT>(ug[q], p.bias + (int64_t)(i + q) * p.D + grp * CPT, z);
          unpack<kBf16, CPT>(ux[q], xv);
#pragma unroll
          for (int k = 0; k < CPT; ++k) {
            const float a = ex2_approx(z[k] - m[k]);
            l[k] += a;
            acc[k] = fmaf(a, xv[k], acc[k]);
          }
        }
      }
    }
  }
  if (p.ns > 1) {
    // merge the slices of each (block, channel group) as a tree in shared memory:
    // M = max m_s, L = sum l_s 2^(m_s - M), the same for acc
    for (int half = p.ns / 2; half >= 1; half /= 2) {
      if (s >= half && s < 2 * half) {
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
          part[tid][k] = m[k];
          part[tid][CPT + k] = l[k];
          part[tid][2 * CPT + k] = acc[k];
        }
      }
      __syncthreads();
      if (s < half) {
        const int o = tid + half * p.cg;  // slice s + half of the same (block, channel group)
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
          const float mo = part[o][k];
          const float mn = fmaxf(m[k], mo);
          if (mn == -INFINITY) continue;
          const float sa = ex2_approx(m[k] - mn), sb = ex2_approx(mo - mn);
          l[k] = l[k] * sa + part[o][CPT + k] * sb;
          acc[k] = acc[k] * sa + part[o][2 * CPT + k] * sb;
          m[k] = mn;
        }
      }
      __syncthreads();
    }
    if (s != 0) return;
  }
  if (!active) return;
  uint32_t w[CPT / 2];
#pragma unroll
  for (int k = 0; k < CPT / 2; ++k) w[k] = pack2<kBf16>(acc[2 * k] / l[2 * k], acc[2 * k + 1] / l[2 * k + 1]);
  V o;
  if constexpr (CPT == 8) {
    o = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    o = make_uint2(w[0], w[1]);
  }
  reinterpret_cast<V*>(p.rows + j * p.D)[grp] = o;
}

// ------------------------------------------------------------------ long batches, streamed
// A long batch (ratio <= 4, D a power of two <= 512) streams its x and g rows through a ring of
// shared-memory stages that bulk copies fill: one producer lane keeps up to kStages x 64 KB of a
// CTA's rows in flight without holding them in registers, and 512 threads reduce whole blocks
// from shared memory.  A stage holds kStageBytes of x and of g, srows = kStageBytes / (2 D)
// consecutive positions, i.e. srows / ratio blocks.  Consumer thread t always owns channel group
// t % (D / 8) (512 is a multiple of D / 8), so its 8 channels' bias stays in registers.  A block's
// arithmetic is the one-pass kernel's, step for step, so a row does not depend on the path.  The block that draws on held-over
// frontier rows (block 0 when n_frontier > 0) and the new frontier go to one extra CTA.
constexpr int kSConsumers = 512;
constexpr int kSThreads = kSConsumers + 32;  // + the producer warp
constexpr int kStages = 3;
constexpr int kStageBytes = 32768;
constexpr int kSSmem = kStages * 2 * kStageBytes + 2 * kStages * 8;

struct StreamParams {
  const uint16_t* x;
  const uint16_t* g;
  const float* bias;
  const uint16_t* fx;
  const uint16_t* fg;
  uint16_t* rows;
  uint16_t* fx_out;
  uint16_t* fg_out;
  int nf, D, n_out, rem;
  int j0;         // first block of the stream: 1 when block 0 draws on frontier rows
  int srows;      // positions a stage holds (a multiple of the ratio)
  int nstages;    // stages of the stream
  int main_ctas;  // CTAs of the stream; the next one takes block 0 and the frontier
  int lg;         // log2 of the channel groups a row (D / 8)
  int* status;
};

// count bytes from global memory into shared memory, completed on bar (addresses and size are
// multiples of 16 bytes)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

template <bool kBf16, int R>
__global__ void __launch_bounds__(kSThreads, 1) compress_stream_kernel(const StreamParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * 2 * kStageBytes);
  uint64_t* empty = full + kStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSConsumers / 32);
    }
    fence_mbarrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const float kLog2e = 1.4426950408889634f;
  if ((int)blockIdx.x >= p.main_ctas) {
    // ------------------------------------- block 0 over frontier rows, and the new frontier
    if (p.j0 == 1) {
      for (int d = tid; d < p.D; d += blockDim.x) {
        float m = -INFINITY, z[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const uint16_t gv = seq_row(p.fg, p.g, p.nf, i, p.D)[d];
          const float gf = kBf16 ? __bfloat162float(__ushort_as_bfloat16(gv)) : __half2float(__ushort_as_half(gv));
          z[i] = __fmul_rn(gf + p.bias[i * p.D + d], kLog2e);
          m = fmaxf(m, z[i]);
        }
        float l = 0.f, acc = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const uint16_t xv = seq_row(p.fx, p.x, p.nf, i, p.D)[d];
          const float xf = kBf16 ? __bfloat162float(__ushort_as_bfloat16(xv)) : __half2float(__ushort_as_half(xv));
          const float a = ex2_approx(z[i] - m);
          l += a;
          acc = fmaf(a, xf, acc);
        }
        const float r = acc / l;
        p.rows[d] = kBf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(r)) : __half_as_ushort(__float2half_rn(r));
      }
    }
    const int per_row = p.D / 8;
    for (int idx = tid; idx < p.rem * per_row; idx += blockDim.x) {
      const int i = idx / per_row, c = idx - i * per_row;
      const int64_t v = (int64_t)p.n_out * R + i;
      reinterpret_cast<uint4*>(p.fx_out + (int64_t)i * p.D)[c] =
          reinterpret_cast<const uint4*>(seq_row(p.fx, p.x, p.nf, v, p.D))[c];
      reinterpret_cast<uint4*>(p.fg_out + (int64_t)i * p.D)[c] =
          reinterpret_cast<const uint4*>(seq_row(p.fg, p.g, p.nf, v, p.D))[c];
    }
    return;
  }
  const int bps = p.srows / R;  // blocks a stage
  const int G = 1 << p.lg;      // channel groups of 8 a row
  const size_t row_bytes = (size_t)p.D * 2;
  const int my_stages = (p.nstages - (int)blockIdx.x + p.main_ctas - 1) / p.main_ctas;
  if (warp == kSConsumers / 32) {
    // ------------------------------------------------------------------------- producer
    if (lane == 0) {
      int k = 0;
      for (; k < my_stages; ++k) {
        const int slot = k % kStages;
        if (!mbar_wait(&empty[slot], ((k / kStages) & 1) ^ 1, p.status, 71)) break;
        const int64_t jb = p.j0 + (int64_t)((int)blockIdx.x + k * p.main_ctas) * bps;
        const int nb = (int)min((int64_t)bps, (int64_t)p.n_out - jb);
        const int64_t row0 = jb * R - p.nf;  // x row of the stage's first position (jb >= j0)
        const uint32_t bytes = (uint32_t)((size_t)nb * R * row_bytes);
        uint8_t* sx = smem + slot * 2 * kStageBytes;
        mbar_arrive_expect_tx(&full[slot], 2 * bytes);
        bulk_load(sx, p.x + row0 * p.D, bytes, &full[slot]);
        bulk_load(sx + kStageBytes, p.g + row0 * p.D, bytes, &full[slot]);
      }
      // the copies issued have landed before the CTA can exit (the consumers normally waited for
      // all of them; after a wait that gave up, wait here, bounded)
      for (int q = max(0, k - kStages); q < k; ++q) mbar_wait(&full[q % kStages], (q / kStages) & 1, p.status, 72);
    }
    return;
  }
  // ----------------------------------------------------------------------------- consumers
  const int c = tid & (G - 1);
  float bb[R][8];  // bias of this thread's 8 channels for the R positions of a block
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(p.bias + (int64_t)i * p.D + c * 8));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(p.bias + (int64_t)i * p.D + c * 8) + 1);
    bb[i][0] = b0.x;
    bb[i][1] = b0.y;
    bb[i][2] = b0.z;
    bb[i][3] = b0.w;
    bb[i][4] = b1.x;
    bb[i][5] = b1.y;
    bb[i][6] = b1.z;
    bb[i][7] = b1.w;
  }
  for (int k = 0; k < my_stages; ++k) {
    const int slot = k % kStages;
    if (!mbar_wait(&full[slot], (k / kStages) & 1, p.status, 70)) break;
    const uint8_t* sx = smem + slot * 2 * kStageBytes;
    const uint8_t* sg = sx + kStageBytes;
    const int64_t jb = p.j0 + (int64_t)((int)blockIdx.x + k * p.main_ctas) * bps;
    const int nb = (int)min((int64_t)bps, (int64_t)p.n_out - jb);
    for (int t = tid; t < (nb << p.lg); t += kSConsumers) {
      const int jj = t >> p.lg;  // block within the stage (and t & (G - 1) == c)
      const uint8_t* rx = sx + (size_t)jj * R * row_bytes + c * 16;
      const uint8_t* rg = sg + (size_t)jj * R * row_bytes + c * 16;
      float m[8], l[8], acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        m[q] = -INFINITY;
        l[q] = 0.f;
        acc[q] = 0.f;
      }
      // the block's max gate a channel, then the weights and sums (gates recomputed), in the
      // one-pass kernel's arithmetic and order: a block's row is the same whichever path made it
#pragma unroll
      for (int i = 0; i < R; ++i) {
        float gv[8];
        unpack<kBf16, 8>(*reinterpret_cast<const uint4*>(rg + i * row_bytes), gv);
#pragma unroll
        for (int q = 0; q < 8; ++q) m[q] = fmaxf(m[q], __fmul_rn(gv[q] + bb[i][q], kLog2e));
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
        float gv[8], xv[8];
        unpack<kBf16, 8>(*reinterpret_cast<const uint4*>(rg + i * row_bytes), gv);
        unpack<kBf16, 8>(*reinterpret_cast<const uint4*>(rx + i * row_bytes), xv);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float a = ex2_approx(__fmul_rn(gv[q] + bb[i][q], kLog2e) - m[q]);
          l[q] += a;
          acc[q] = fmaf(a, xv[q], acc[q]);
        }
      }
      uint4 o;
      o.x = pack2<kBf16>(acc[0] / l[0], acc[1] / l[1]);
      o.y = pack2<kBf16>(acc[2] / l[2], acc[3] / l[3]);
      o.z = pack2<kBf16>(acc[4] / l[4], acc[5] / l[5]);
      o.w = pack2<kBf16>(acc[6] / l[6], acc[7] / l[7]);
      reinterpret_cast<uint4*>(p.rows + (jb + jj) * p.D)[c] = o;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
}

template <bool kBf16, int R>
cudaError_t launch_stream(const StreamParams& sp, int grid, cudaStream_t stream) {
  const cudaError_t e = ensure_dynamic_smem(compress_stream_kernel<kBf16, R>, kSSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(compress_stream_kernel<kBf16, R>, dim3(grid), dim3(kSThreads), (size_t)kSSmem, stream, sp);
}

// The streamed path takes a batch of at least two stages a CTA on every SM; shorter calls (a
// 2048-token chunk) keep the one-pass kernel, whose launch shape spreads few blocks wide.
// Returns 1 when the call was not for it.
int try_stream(const CompressArgs& a, int n_out, int rem, cudaStream_t stream) {
  const int R = a.ratio, D = a.D;
  if (!(R == 1 || R == 2 || R == 4) || D < 8 || D > 512 || (D & (D - 1)) != 0) return 1;
  StreamParams sp;
  sp.j0 = a.n_frontier > 0 ? 1 : 0;
  sp.srows = kStageBytes / (2 * D);
  const int bps = sp.srows / R;
  const int64_t nblk = (int64_t)n_out - sp.j0;
  const int sms = device_sm_count();
  if (nblk < 2ll * sms * bps) return 1;
  sp.x = static_cast<const uint16_t*>(a.x);
  sp.g = static_cast<const uint16_t*>(a.g);
  sp.bias = a.bias;
  sp.fx = static_cast<const uint16_t*>(a.fx);
  sp.fg = static_cast<const uint16_t*>(a.fg);
  sp.rows = static_cast<uint16_t*>(a.rows);
  sp.fx_out = static_cast<uint16_t*>(a.fx_out);
  sp.fg_out = static_cast<uint16_t*>(a.fg_out);
  sp.nf = a.n_frontier;
  sp.D = D;
  sp.n_out = n_out;
  sp.rem = rem;
  sp.nstages = (int)((nblk + bps - 1) / bps);
  sp.main_ctas = sp.nstages < sms ? sp.nstages : sms;
  sp.lg = 0;
  while ((8 << sp.lg) < D) ++sp.lg;
  sp.status = device_status_ptr();
  const int grid = sp.main_ctas + ((sp.j0 == 1 || rem > 0) ? 1 : 0);
  cudaError_t e;
  switch (R) {
    case 1: e = a.bf16 ? launch_stream<true, 1>(sp, grid, stream) : launch_stream<false, 1>(sp, grid, stream); break;
    case 2: e = a.bf16 ? launch_stream<true, 2>(sp, grid, stream) : launch_stream<false, 2>(sp, grid, stream); break;
    default: e = a.bf16 ? launch_stream<true, 4>(sp, grid, stream) : launch_stream<false, 4>(sp, grid, stream); break;
  }
  if (e != cudaSuccess) return DS4X_ERR_CUDA;
  count_launch();
  return DS4X_OK;
}

}  // namespace

// Launch shape: channels a thread, ns position slices, a slab of cg channel groups (the largest
// divisor of the row's groups with cg * ns <= kThreads), bpc blocks per CTA filling kThreads.
int launch_compress(const CompressArgs& a, cudaStream_t stream) {
  CompressParams p;
  p.x = static_cast<const uint16_t*>(a.x);
  p.g = static_cast<const uint16_t*>(a.g);
  p.bias = a.bias;
  p.fx = static_cast<const uint16_t*>(a.fx);
  p.fg = static_cast<const uint16_t*>(a.fg);
  p.rows = static_cast<uint16_t*>(a.rows);
  p.fx_out = static_cast<uint16_t*>(a.fx_out);
  p.fg_out = static_cast<uint16_t*>(a.fg_out);
  p.nf = a.n_frontier;
  p.T = a.T;
  p.D = a.D;
  p.ratio = a.ratio;
  const int64_t n = (int64_t)a.n_frontier + a.T;
  p.n_out = (int)(n / a.ratio);
  p.rem = (int)(n % a.ratio);
  if (p.n_out == 0 && p.rem == 0) return DS4X_OK;
  const int rs = try_stream(a, p.n_out, p.rem, stream);
  if (rs != 1) return rs;
  // 8 channels a thread (16-byte loads) when the blocks alone give about four CTAs of work per SM,
  // else 4 (more threads, fewer registers: three CTAs per SM) and position slices as needed
  const int64_t want = 4ll * device_sm_count() * kThreads;
  const int CPT = (int64_t)p.n_out * (a.D / 8) >= want ? 8 : 4;
  const int groups = a.D / CPT;
  // position slices: as many as it takes for about four CTAs of work per SM (a power of two, at
  // most 32 and at most ratio / kBatch), so a ratio-128 block of a 2048-token chunk spreads out
  // while a long batch of blocks streams its positions in one thread
  int ns = 1;
  while (2 * ns <= a.ratio / kBatch && 2 * ns <= 32 && (int64_t)p.n_out * groups * ns < want) ns *= 2;
  int cg = groups < kThreads / ns ? groups : kThreads / ns;
  while (groups % cg) --cg;
  p.cg = cg;
  p.slabs = groups / cg;
  p.ns = ns;
  p.bpc = kThreads / (cg * ns);
  p.main_ctas = (int)((p.n_out + p.bpc - 1) / p.bpc) * p.slabs;
  const int grid = p.main_ctas + (p.rem > 0 ? 1 : 0);
  cudaError_t e;
  if (CPT == 8)
    e = a.bf16 ? launch_pdl(compress_kernel<true, 8>, dim3(grid), dim3(kThreads), 0, stream, p)
               : launch_pdl(compress_kernel<false, 8>, dim3(grid), dim3(kThreads), 0, stream, p);
  else
    e = a.bf16 ? launch_pdl(compress_kernel<true, 4>, dim3(grid), dim3(kThreads), 0, stream, p)
               : launch_pdl(compress_kernel<false, 4>, dim3(grid), dim3(kThreads), 0, stream, p);
  if (e != cudaSuccess) return DS4X_ERR_CUDA;
  count_launch();
  return DS4X_OK;
}

}  // namespace ds4x
