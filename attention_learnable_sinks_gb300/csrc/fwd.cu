// Forward of sink attention: O and LSE.
//
// Online softmax over key chunks, seeded with the sink: the running maximum
// starts at S_h and the running sum at exp(S_h - S_h) = 1, so the virtual
// token enters the denominator once and adds nothing to the output (page
// "GPT-OSS Agentic RL Training: A Practical Retrospective", section "The Role
// of Attention Sinks").
//
// Persistent CTAs take (query tile, head) work items from the device-built
// tile list, longest first; consecutive items are the heads of one tile, so
// the GQA group's K/V rows are reused from L2.
#include <algorithm>
#include <cmath>

#include "internal.h"

namespace sinkattn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;  // keys per staged chunk
constexpr int kPad = 65;    // padded smem row (floats) for per-lane dot products
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr size_t kSmemFloats = kTile * 64      // Qs
                               + kChunk * kPad  // Ks
                               + kChunk * 64    // Vs
                               + kTile * 64     // Os (accumulator)
                               + kWarps * 64    // Ps
                               + 2 * kTile;     // m, l
constexpr size_t kSmemBytes = kSmemFloats * sizeof(float);

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ bool visible(const Problem& p, int i, int j, int L) {
  if (j >= L) return false;
  if (p.causal && j > i) return false;
  if (p.window > 0 && i - j >= p.window) return false;
  return true;
}

__global__ void __launch_bounds__(kThreads)
fwd_kernel(Problem p, const int2* __restrict__ items, int32_t* __restrict__ meta) {
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Ks = Qs + kTile * 64;
  float* Vs = Ks + kChunk * kPad;
  float* Os = Vs + kChunk * 64;
  float* Ps = Os + kTile * 64;
  float* ms = Ps + kWarps * 64;
  float* ls = ms + kTile;
  __shared__ int s_w;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwork = meta[0] * p.Hq;

  for (;;) {
    __syncthreads();
    if (tid == 0) s_w = atomicAdd(&meta[1], 1);
    __syncthreads();
    const int w = s_w;
    if (w >= nwork) break;
    const int2 it = items[w / p.Hq];
    const int h = w % p.Hq, kvh = h / p.G;
    const int base = p.cu[it.x], L = p.cu[it.x + 1] - base;
    const int r0 = it.y * kTile, r1 = min(L, r0 + kTile), nrows = r1 - r0;
    const float sink2 = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;

    for (int e = tid; e < kTile * 64; e += kThreads) {
      const int r = e >> 6, d = e & 63;
      float x = 0.f;
      if (r < nrows)
        x = __bfloat162float(p.q[(int64_t)(base + r0 + r) * p.q_stride + h * 64 + d]) * p.scale_log2;
      Qs[e] = x;
      Os[e] = 0.f;
    }
    for (int r = tid; r < kTile; r += kThreads) {
      ms[r] = sink2;
      ls[r] = p.sinks ? 1.f : 0.f;
    }
    int klo, khi;
    visible_keys(p.causal, p.window, L, r0, r1, &klo, &khi);
    for (int c0 = klo & ~(kChunk - 1); c0 < khi; c0 += kChunk) {
      __syncthreads();
      for (int e = tid; e < kChunk * 64; e += kThreads) {
        const int j = e >> 6, d = e & 63;
        float kx = 0.f, vx = 0.f;
        if (c0 + j < L) {
          kx = __bfloat162float(p.k[(int64_t)(base + c0 + j) * p.k_stride + kvh * 64 + d]);
          vx = __bfloat162float(p.v[(int64_t)(base + c0 + j) * p.v_stride + kvh * 64 + d]);
        }
        Ks[j * kPad + d] = kx;
        Vs[j * 64 + d] = vx;
      }
      __syncthreads();
      for (int rr = warp; rr < nrows; rr += kWarps) {
        const int i = r0 + rr;
        const float* qrow = Qs + rr * 64;
        float s0 = 0.f, s1 = 0.f;
        for (int d = 0; d < 64; ++d) {
          const float qd = qrow[d];
          s0 += qd * Ks[lane * kPad + d];
          s1 += qd * Ks[(lane + 32) * kPad + d];
        }
        if (!visible(p, i, c0 + lane, L)) s0 = -INFINITY;
        if (!visible(p, i, c0 + lane + 32, L)) s1 = -INFINITY;
        const float m_old = ms[rr];
        const float m_new = fmaxf(m_old, warp_max(fmaxf(s0, s1)));
        float alpha = 1.f, p0 = 0.f, p1 = 0.f;
        if (m_new != -INFINITY) {
          alpha = exp2f(m_old - m_new);
          p0 = exp2f(s0 - m_new);
          p1 = exp2f(s1 - m_new);
        }
        const float rs = warp_sum(p0 + p1);
        Ps[warp * 64 + lane] = p0;
        Ps[warp * 64 + lane + 32] = p1;
        __syncwarp();
        float a0 = Os[rr * 64 + 2 * lane] * alpha, a1 = Os[rr * 64 + 2 * lane + 1] * alpha;
        for (int kk = 0; kk < kChunk; ++kk) {
          const float pk = Ps[warp * 64 + kk];
          a0 += pk * Vs[kk * 64 + 2 * lane];
          a1 += pk * Vs[kk * 64 + 2 * lane + 1];
        }
        Os[rr * 64 + 2 * lane] = a0;
        Os[rr * 64 + 2 * lane + 1] = a1;
        const float l_old = ls[rr];
        __syncwarp();
        if (lane == 0) {
          ms[rr] = m_new;
          ls[rr] = l_old * alpha + rs;
        }
        __syncwarp();
      }
    }
    __syncthreads();
    for (int e = tid; e < nrows * 64; e += kThreads) {
      const int r = e >> 6, d = e & 63;
      const float l = ls[r];
      p.o[(int64_t)(base + r0 + r) * p.Hq * 64 + h * 64 + d] =
          __float2bfloat16_rn(l > 0.f ? Os[e] / l : 0.f);
    }
    if (p.lse)
      for (int r = tid; r < nrows; r += kThreads) {
        const float l = ls[r];
        p.lse[(int64_t)h * p.total + base + r0 + r] =
            l > 0.f ? (ms[r] + log2f(l)) * kLn2 : -INFINITY;
      }
  }
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, const TileList& qtiles, int num_sms, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t work = (int64_t)qtiles.capacity * p.Hq;
  const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms * 2);
  if (grid <= 0) return cudaSuccess;
  fwd_kernel<<<grid, kThreads, kSmemBytes, s>>>(p, qtiles.items, qtiles.meta);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
