// Backward of sink attention: dq, dk, dv and dL/dS_h (page "GPT-OSS Agentic
// RL Training: A Practical Retrospective", section "Implementation in
// FlashAttention v3", step 2: the backward that also returns the sink
// gradient).
//
// With the sink carrying no value, D_i = rowsum(dO_i * O_i) equals
// sum_j P_ij dP_ij, so dS_ij = P_ij (dP_ij - D_i) as in plain attention, and the
// sink's own gradient is dS_h = -sum_i p_sink_i D_i, p_sink_i = exp(S_h - LSE_i).
//
// dS_h is a sum with heavy cancellation (its terms change sign with dO), so it
// is not formed from D, whose O is rounded to bf16: the key-stationary kernel
// accumulates p_sink_i * P_ij * dP_ij from its fp32 P and dP instead, per
// (key tile, head), and a final pass adds those partials in a fixed order.
//
// Kernels, in launch order:
//   preprocess  one pass over (token, head) rows: D = rowsum(dO * O)
//   dq          row-stationary: recompute P, dP, dS per key; dq = scale dS K
//   dkdv        key-stationary over the whole GQA group:
//               dv = sum P^T dO, dk = scale sum dS^T Q, and the per-head
//               partials of sum p_sink P dP
//   finish      dS_h = -(fixed-order fp64 sum of the partials)
#include <algorithm>
#include <cmath>

#include "internal.h"

namespace sinkattn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;
constexpr int kPad = 65;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPrepThreads = 128;  // tokens per preprocess block

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ bool visible(const Problem& p, int i, int j, int L) {
  if (i >= L || j >= L) return false;
  if (p.causal && j > i) return false;
  if (p.window > 0 && i - j >= p.window) return false;
  return true;
}

__device__ __forceinline__ int next_item(int32_t* meta, int* slot) {
  __syncthreads();
  if (threadIdx.x == 0) *slot = atomicAdd(&meta[1], 1);
  __syncthreads();
  return *slot;
}

// ---------------------------------------------------------------- preprocess
__global__ void __launch_bounds__(kPrepThreads)
preprocess_kernel(BwdProblem bp) {
  const Problem& p = bp.f;
  const int h = blockIdx.y;
  const int t = blockIdx.x * kPrepThreads + threadIdx.x;
  if (t < p.total) {
    const uint4* o4 = reinterpret_cast<const uint4*>(p.o + ((int64_t)t * p.Hq + h) * 64);
    const uint4* g4 = reinterpret_cast<const uint4*>(bp.dout + ((int64_t)t * p.Hq + h) * 64);
    float D = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 a = o4[c], b = g4[c];
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(b2[e]);
        D += x.x * y.x + x.y * y.y;
      }
    }
    bp.D[(int64_t)h * p.total + t] = D;
  }
}

// ---------------------------------------------------------------- dq
constexpr size_t kDqSmemBytes =
    (3 * kTile * 64 + 2 * kChunk * kPad + kWarps * 64 + 2 * kTile) * sizeof(float);

__global__ void __launch_bounds__(kThreads)
dq_kernel(BwdProblem bp, const int2* __restrict__ items, int32_t* __restrict__ meta) {
  const Problem& p = bp.f;
  extern __shared__ float sm[];
  float* Qs = sm;                    // q * scale * log2e
  float* dOs = Qs + kTile * 64;
  float* Acc = dOs + kTile * 64;     // sum_j dS_ij k_j
  float* Ks = Acc + kTile * 64;
  float* Vs = Ks + kChunk * kPad;
  float* Bs = Vs + kChunk * kPad;    // per-warp dS row
  float* lse2 = Bs + kWarps * 64;
  float* Ds = lse2 + kTile;
  __shared__ int s_w;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwork = meta[0] * p.Hq;
  for (;;) {
    const int w = next_item(meta, &s_w);
    if (w >= nwork) break;
    const int2 it = items[w / p.Hq];
    const int h = w % p.Hq, kvh = h / p.G;
    const int base = p.cu[it.x], L = p.cu[it.x + 1] - base;
    const int r0 = it.y * kTile, r1 = min(L, r0 + kTile), nrows = r1 - r0;
    for (int e = tid; e < kTile * 64; e += kThreads) {
      const int r = e >> 6, d = e & 63;
      float x = 0.f, g = 0.f;
      if (r < nrows) {
        x = __bfloat162float(p.q[(int64_t)(base + r0 + r) * p.q_stride + h * 64 + d]) * p.scale_log2;
        g = __bfloat162float(bp.dout[((int64_t)(base + r0 + r) * p.Hq + h) * 64 + d]);
      }
      Qs[e] = x;
      dOs[e] = g;
      Acc[e] = 0.f;
    }
    for (int r = tid; r < kTile; r += kThreads) {
      const bool in = r < nrows;
      lse2[r] = in ? p.lse[(int64_t)h * p.total + base + r0 + r] * kLog2e : 0.f;
      Ds[r] = in ? bp.D[(int64_t)h * p.total + base + r0 + r] : 0.f;
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
        Vs[j * kPad + d] = vx;
      }
      __syncthreads();
      for (int rr = warp; rr < nrows; rr += kWarps) {
        const int i = r0 + rr;
        float s0 = 0.f, s1 = 0.f, g0 = 0.f, g1 = 0.f;
        for (int d = 0; d < 64; ++d) {
          const float qd = Qs[rr * 64 + d], gd = dOs[rr * 64 + d];
          s0 += qd * Ks[lane * kPad + d];
          s1 += qd * Ks[(lane + 32) * kPad + d];
          g0 += gd * Vs[lane * kPad + d];
          g1 += gd * Vs[(lane + 32) * kPad + d];
        }
        const float P0 = visible(p, i, c0 + lane, L) ? exp2f(s0 - lse2[rr]) : 0.f;
        const float P1 = visible(p, i, c0 + lane + 32, L) ? exp2f(s1 - lse2[rr]) : 0.f;
        Bs[warp * 64 + lane] = P0 * (g0 - Ds[rr]);
        Bs[warp * 64 + lane + 32] = P1 * (g1 - Ds[rr]);
        __syncwarp();
        float a0 = Acc[rr * 64 + 2 * lane], a1 = Acc[rr * 64 + 2 * lane + 1];
        for (int kk = 0; kk < kChunk; ++kk) {
          const float ds = Bs[warp * 64 + kk];
          a0 += ds * Ks[kk * kPad + 2 * lane];
          a1 += ds * Ks[kk * kPad + 2 * lane + 1];
        }
        Acc[rr * 64 + 2 * lane] = a0;
        Acc[rr * 64 + 2 * lane + 1] = a1;
        __syncwarp();
      }
    }
    __syncthreads();
    for (int e = tid; e < nrows * 64; e += kThreads) {
      const int r = e >> 6, d = e & 63;
      bp.dq[((int64_t)(base + r0 + r) * p.Hq + h) * 64 + d] = __float2bfloat16_rn(Acc[e] * p.scale);
    }
  }
}

// ---------------------------------------------------------------- dk, dv
constexpr size_t kDkvSmemBytes =
    (4 * kTile * 64 + 2 * kChunk * kPad + 2 * kWarps * 64 + 3 * kChunk) * sizeof(float);

__global__ void __launch_bounds__(kThreads)
dkdv_kernel(BwdProblem bp, const int2* __restrict__ items, int32_t* __restrict__ meta) {
  const Problem& p = bp.f;
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = Ks + kTile * 64;
  float* dKs = Vs + kTile * 64;
  float* dVs = dKs + kTile * 64;
  float* Qs = dVs + kTile * 64;       // unscaled q rows of the chunk
  float* dOs = Qs + kChunk * kPad;
  float* Pb = dOs + kChunk * kPad;
  float* Sb = Pb + kWarps * 64;
  float* lse2 = Sb + kWarps * 64;
  float* Ds = lse2 + kChunk;
  float* Ps = Ds + kChunk;            // p_sink of the chunk's rows
  __shared__ int s_w;
  __shared__ float red[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwork = meta[0] * p.Hkv;
  for (;;) {
    const int w = next_item(meta, &s_w);
    if (w >= nwork) break;
    const int2 it = items[w / p.Hkv];
    const int kvh = w % p.Hkv;
    const int base = p.cu[it.x], L = p.cu[it.x + 1] - base;
    const int c0 = it.y * kTile, c1 = min(L, c0 + kTile), nkeys = c1 - c0;
    for (int e = tid; e < kTile * 64; e += kThreads) {
      const int j = e >> 6, d = e & 63;
      float kx = 0.f, vx = 0.f;
      if (j < nkeys) {
        kx = __bfloat162float(p.k[(int64_t)(base + c0 + j) * p.k_stride + kvh * 64 + d]);
        vx = __bfloat162float(p.v[(int64_t)(base + c0 + j) * p.v_stride + kvh * 64 + d]);
      }
      Ks[e] = kx;
      Vs[e] = vx;
      dKs[e] = 0.f;
      dVs[e] = 0.f;
    }
    int rlo, rhi;
    seeing_rows(p.causal, p.window, L, c0, c1, &rlo, &rhi);
    for (int hh = 0; hh < p.G; ++hh) {
      const int h = kvh * p.G + hh;
      const float sink2 = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
      float sacc = 0.f;  // this thread's share of sum p_sink P dP for head h
      for (int q0 = rlo & ~(kChunk - 1); q0 < rhi; q0 += kChunk) {
        __syncthreads();
        for (int e = tid; e < kChunk * 64; e += kThreads) {
          const int r = e >> 6, d = e & 63;
          float x = 0.f, g = 0.f;
          if (q0 + r < L) {
            x = __bfloat162float(p.q[(int64_t)(base + q0 + r) * p.q_stride + h * 64 + d]);
            g = __bfloat162float(bp.dout[((int64_t)(base + q0 + r) * p.Hq + h) * 64 + d]);
          }
          Qs[r * kPad + d] = x;
          dOs[r * kPad + d] = g;
        }
        for (int r = tid; r < kChunk; r += kThreads) {
          const bool in = q0 + r < L;
          lse2[r] = in ? p.lse[(int64_t)h * p.total + base + q0 + r] * kLog2e : 0.f;
          Ds[r] = in ? bp.D[(int64_t)h * p.total + base + q0 + r] : 0.f;
          Ps[r] = in && p.sinks ? exp2f(sink2 - lse2[r]) : 0.f;
        }
        __syncthreads();
        for (int kk = warp; kk < nkeys; kk += kWarps) {
          const int j = c0 + kk;
          float s0 = 0.f, s1 = 0.f, g0 = 0.f, g1 = 0.f;
          for (int d = 0; d < 64; ++d) {
            const float kd = Ks[kk * 64 + d], vd = Vs[kk * 64 + d];
            s0 += Qs[lane * kPad + d] * kd;
            s1 += Qs[(lane + 32) * kPad + d] * kd;
            g0 += dOs[lane * kPad + d] * vd;
            g1 += dOs[(lane + 32) * kPad + d] * vd;
          }
          const float P0 = visible(p, q0 + lane, j, L) ? exp2f(s0 * p.scale_log2 - lse2[lane]) : 0.f;
          const float P1 =
              visible(p, q0 + lane + 32, j, L) ? exp2f(s1 * p.scale_log2 - lse2[lane + 32]) : 0.f;
          Pb[warp * 64 + lane] = P0;
          Pb[warp * 64 + lane + 32] = P1;
          Sb[warp * 64 + lane] = P0 * (g0 - Ds[lane]);
          Sb[warp * 64 + lane + 32] = P1 * (g1 - Ds[lane + 32]);
          sacc += Ps[lane] * (P0 * g0) + Ps[lane + 32] * (P1 * g1);
          __syncwarp();
          float v0 = dVs[kk * 64 + 2 * lane], v1 = dVs[kk * 64 + 2 * lane + 1];
          float k0 = dKs[kk * 64 + 2 * lane], k1 = dKs[kk * 64 + 2 * lane + 1];
          for (int r = 0; r < kChunk; ++r) {
            const float pr = Pb[warp * 64 + r], sr = Sb[warp * 64 + r];
            v0 += pr * dOs[r * kPad + 2 * lane];
            v1 += pr * dOs[r * kPad + 2 * lane + 1];
            k0 += sr * Qs[r * kPad + 2 * lane];
            k1 += sr * Qs[r * kPad + 2 * lane + 1];
          }
          dVs[kk * 64 + 2 * lane] = v0;
          dVs[kk * 64 + 2 * lane + 1] = v1;
          dKs[kk * 64 + 2 * lane] = k0;
          dKs[kk * 64 + 2 * lane + 1] = k1;
          __syncwarp();
        }
      }
      // fixed-order reduction of the head's partial over the CTA
      sacc = warp_sum(sacc);
      __syncthreads();
      if (lane == 0) red[warp] = sacc;
      __syncthreads();
      if (tid == 0) {
        float s = 0.f;
        for (int i = 0; i < kWarps; ++i) s += red[i];
        bp.sink_part[(int64_t)h * bp.part_stride + w / p.Hkv] = s;
      }
    }
    __syncthreads();
    for (int e = tid; e < nkeys * 64; e += kThreads) {
      const int j = e >> 6, d = e & 63;
      const int64_t off = ((int64_t)(base + c0 + j) * p.Hkv + kvh) * 64 + d;
      bp.dk[off] = __float2bfloat16_rn(dKs[e] * p.scale);
      bp.dv[off] = __float2bfloat16_rn(dVs[e]);
    }
  }
}

// ---------------------------------------------------------------- finish
__global__ void finish_kernel(BwdProblem bp, const int32_t* __restrict__ kmeta) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= bp.f.Hq || !bp.dsinks) return;
  double acc = 0.0;
  if (bp.f.sinks) {
    const int n = kmeta[0];
    for (int c = 0; c < n; ++c) acc += (double)bp.sink_part[(int64_t)h * bp.part_stride + c];
  }
  bp.dsinks[h] = (float)(-acc);
}

template <class K>
cudaError_t allow_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdProblem& p, cudaStream_t s) {
  if (p.nchunks == 0) return cudaSuccess;
  preprocess_kernel<<<dim3(p.nchunks, p.f.Hq), kPrepThreads, 0, s>>>(p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdProblem& p, const TileList& qtiles, int num_sms,
                          cudaStream_t s) {
  cudaError_t e = allow_smem(dq_kernel, kDqSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t work = (int64_t)qtiles.capacity * p.f.Hq;
  const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms);
  if (grid <= 0) return cudaSuccess;
  dq_kernel<<<grid, kThreads, kDqSmemBytes, s>>>(p, qtiles.items, qtiles.meta);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdProblem& p, const TileList& ktiles, int num_sms,
                            cudaStream_t s) {
  cudaError_t e = allow_smem(dkdv_kernel, kDkvSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t work = (int64_t)ktiles.capacity * p.f.Hkv;
  const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms);
  if (grid <= 0) return cudaSuccess;
  dkdv_kernel<<<grid, kThreads, kDkvSmemBytes, s>>>(p, ktiles.items, ktiles.meta);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_finish(const BwdProblem& p, const TileList& ktiles, cudaStream_t s) {
  finish_kernel<<<(p.f.Hq + 127) / 128, 128, 0, s>>>(p, ktiles.meta);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
