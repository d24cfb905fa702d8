// Decode with sinks over a paged KV cache: one new query row per sequence
// (page "GPT-OSS Agentic RL Training: A Practical Retrospective", section
// "Implementation in FlashAttention v3", step 1, the forward with sinks, here
// on the inference side the pages took it from).
//
// The query of sequence b is the row at its last position, L - 1; it sees
// keys j in [max(0, L - W), L) (all of them without a window) and the sink of
// its head. The keys are split into ranges handled by separate CTAs:
//
//   split kernel    one CTA per (split, kv head, sequence): the G query heads
//                   of the kv head together, 128-key chunks of K and V brought
//                   in by TMA (one copy per cache block, double-buffered),
//                   scores on the CUDA cores (G x 64 x 128 per chunk is far
//                   below a tensor-core tile and the kernel is bound by HBM),
//                   an online softmax per head, and a partial
//                   (max, sum, unnormalised O) per split and head
//   combine kernel  per (sequence, head): max over the partials and the sink
//                   logit, then O = sum_s o_s 2^(m_s - M) / Z with
//                   Z = 2^(S_h - M) + sum_s l_s 2^(m_s - M), LSE = M + log Z
//
// Scores are kept in log2 units (q is pre-scaled by scale * log2 e), so every
// exponential is an exp2.
#include <algorithm>
#include <cmath>

#include "internal.h"
#include "sm100.cuh"

namespace sinkattn {
namespace {

using namespace sm100;

constexpr int kDecThreads = 128;
constexpr int kChunk = 128;                                // keys per chunk, one per thread
constexpr uint32_t kChunkBytes = kChunk * kHeadDim * 2;    // 16 KB of K (or V)
constexpr int kMaxGroup = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kErrInvalidArg = 1;  // SINKATTN_ERR_INVALID_ARG

struct __align__(1024) DecSmem {
  uint8_t k[2][kChunkBytes];      // chunk stages, rows of 128 bytes, 128-byte swizzled
  uint8_t v[2][kChunkBytes];
  float qs[kMaxGroup][kHeadDim];  // the group's queries, times scale * log2 e
  float pr[kMaxGroup][kChunk];    // the chunk's scores, then its probabilities
  uint64_t full[2];
  int abort;
  int bad;
};
constexpr size_t kDecSmemBytes = sizeof(DecSmem) + 1024;

__device__ __forceinline__ float2 bf2_to_f2(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// Key range of a sequence, in 128-key chunks aligned to the sequence start
// (the cache block size divides 128), and this split's share of the chunks.
struct Range {
  int L, k0, base_al, c_begin, c_end;
};

__device__ __forceinline__ Range split_range(const DecodeProblem& p, int b, int split) {
  Range r;
  r.L = p.seqlens[b];
  r.k0 = p.window > 0 ? max(0, r.L - p.window) : 0;
  r.base_al = (r.k0 / kChunk) * kChunk;
  const int nch = r.L > r.base_al ? (r.L - r.base_al + kChunk - 1) / kChunk : 0;
  const int per = (nch + p.nsplit - 1) / p.nsplit;
  r.c_begin = min(nch, split * per);
  r.c_end = min(nch, r.c_begin + per);
  return r;
}

template <int G>
__global__ void __launch_bounds__(kDecThreads)
decode_split_kernel(const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
                    DecodeProblem p) {
  constexpr int kTph = (kDecThreads / G) < 32 ? (kDecThreads / G) : 32;  // threads per head
  constexpr int kActive = G * kTph;                                       // softmax / PV threads
  constexpr int kDims = kHeadDim / kTph;                                  // output dims per thread
  constexpr int kKpt = kChunk / kTph;                                     // keys per thread (softmax)
  extern __shared__ uint8_t smem_raw[];
  DecSmem& sm = *reinterpret_cast<DecSmem*>(smem_raw + align1024_pad(smem_raw));
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x;
  const Guard g{&sm.abort, p.err};
  if (t == 0) {
    sm.abort = 0;
    sm.bad = 0;
    mbar_init(&sm.full[0], 1);
    mbar_init(&sm.full[1], 1);
    fence_barrier_init();
  }
  if (t == 32) tma_prefetch(&tm_kc);
  if (t == 33) tma_prefetch(&tm_vc);
  const Range r = split_range(p, b, split);
  const int bs = p.block_size;
  const int nlocal = r.c_end - r.c_begin;
  // the sequence length and this split's block indices must be in range
  __syncthreads();
  if (r.L < 0 || r.L > p.max_blocks * bs) {
    if (t == 0) sm.bad = 1;
  } else if (nlocal > 0) {
    const int lb0 = max((r.base_al + r.c_begin * kChunk) / bs, r.k0 / bs);
    const int lb1 = min((r.base_al + r.c_end * kChunk + bs - 1) / bs, (r.L + bs - 1) / bs);
    for (int lb = lb0 + t; lb < lb1; lb += kDecThreads) {
      const int pb = p.block_table[(int64_t)b * p.max_blocks + lb];
      if (pb < 0 || pb >= p.num_blocks) sm.bad = 1;
    }
  }
  // q of the group, scaled
  for (int i = t; i < G * kHeadDim; i += kDecThreads) {
    const int gg = i / kHeadDim, d = i % kHeadDim;
    const __nv_bfloat16 x = p.q[((int64_t)b * p.Hq + kvh * G + gg) * kHeadDim + d];
    sm.qs[gg][d] = __bfloat162float(x) * p.scale_log2;
  }
  __syncthreads();
  if (sm.bad) {
    if (t == 0) atomicCAS(p.err, 0, kErrInvalidArg);
    return;
  }

  // TMA of chunk c into stage c & 1: one box of `bs` rows per cache block
  // that holds visible keys (blocks wholly before the window are not read)
  auto issue = [&](int c) {
    const int st = c & 1;
    const int j0 = r.base_al + (r.c_begin + c) * kChunk;
    uint32_t bytes = 0;
    for (int i = 0; i < kChunk / bs; ++i) {
      const int j = j0 + i * bs;
      if (j < r.L && j + bs > r.k0) bytes += 2u * (uint32_t)bs * kHeadDim * 2u;
    }
    mbar_expect_tx(&sm.full[st], bytes);
    for (int i = 0; i < kChunk / bs; ++i) {
      const int j = j0 + i * bs;
      if (j >= r.L) break;
      if (j + bs <= r.k0) continue;
      const int pb = p.block_table[(int64_t)b * p.max_blocks + j / bs];
      tma_load_3d(sm.k[st] + i * bs * 128, &tm_kc, &sm.full[st], 0, kvh, pb * bs);
      tma_load_3d(sm.v[st] + i * bs * 128, &tm_vc, &sm.full[st], 0, kvh, pb * bs);
    }
  };
  if (t == 0) {
    if (nlocal > 0) issue(0);
    if (nlocal > 1) issue(1);
  }

  const int gh = t / kTph, sub = t % kTph;  // softmax / PV role: head gh, share sub
  float m_run = -INFINITY, l_run = 0.f;
  float o[kDims];
#pragma unroll
  for (int i = 0; i < kDims; ++i) o[i] = 0.f;
  bool ok = true;
  int c = 0;
  for (; c < nlocal; ++c) {
    const int st = c & 1;
    if (!mbar_wait(&sm.full[st], (c >> 1) & 1, g)) ok = false;
    ok = __syncthreads_and(ok);
    if (!ok) break;
    // scores: thread t takes key row t of the chunk
    {
      const int j = r.base_al + (r.c_begin + c) * kChunk + t;
      const bool valid = j >= r.k0 && j < r.L;
      uint64_t kv[32];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 x = *reinterpret_cast<const uint4*>(sm.k[st] + sw128_offset(t, cc));
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = bf2_to_f2(w4[e]);
          kv[cc * 4 + e] = f2pack(f.x, f.y);
        }
      }
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        uint64_t acc0 = f2pack(0.f, 0.f), acc1 = f2pack(0.f, 0.f);
#pragma unroll
        for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
          const float4 qq = *reinterpret_cast<const float4*>(&sm.qs[gg][4 * d4]);
          acc0 = ffma2(f2pack(qq.x, qq.y), kv[2 * d4], acc0);
          acc1 = ffma2(f2pack(qq.z, qq.w), kv[2 * d4 + 1], acc1);
        }
        const float2 a = f2unpack(acc0), bb = f2unpack(acc1);
        sm.pr[gg][t] = valid ? (a.x + a.y) + (bb.x + bb.y) : -INFINITY;
      }
    }
    __syncthreads();
    // online softmax per head over the chunk
    float alpha = 1.f;
    if (t < kActive) {
      float s[kKpt];
      float mloc = -INFINITY;
#pragma unroll
      for (int i = 0; i < kKpt; ++i) {
        s[i] = sm.pr[gh][sub * kKpt + i];
        mloc = fmaxf(mloc, s[i]);
      }
#pragma unroll
      for (int off = kTph / 2; off > 0; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
      const float m_new = fmaxf(m_run, mloc);
      const float msub = m_new == -INFINITY ? 0.f : m_new;
      alpha = ex2(m_run - msub);  // 0 while nothing was seen
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < kKpt; ++i) {
        const float pv = ex2(s[i] - msub);
        sm.pr[gh][sub * kKpt + i] = pv;
        lsum += pv;
      }
#pragma unroll
      for (int off = kTph / 2; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      l_run = l_run * alpha + lsum;
      m_run = m_new;
    }
    __syncthreads();
    // O += P V: thread (gh, sub) owns dims sub * kDims .. + kDims - 1. Rows
    // outside the sequence's keys are skipped rather than weighted by zero:
    // they may hold stale or never-written values.
    if (t < kActive) {
      const int d0 = sub * kDims;
#pragma unroll
      for (int i = 0; i < kDims; ++i) o[i] *= alpha;
      const uint32_t cc = d0 >> 3, within = (d0 & 7) * 2;
      const int j0 = r.base_al + (r.c_begin + c) * kChunk;
      const int jlo = max(r.k0 - j0, 0), jhi = min(r.L - j0, kChunk);
#pragma unroll 8
      for (int j = jlo; j < jhi; ++j) {
        const float pj = sm.pr[gh][j];
        const uint8_t* row = sm.v[st] + sw128_offset(j, cc) + within;
        if (kDims == 8) {
          const uint4 x = *reinterpret_cast<const uint4*>(row);
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = bf2_to_f2(w4[e]);
            o[2 * e] = fmaf(pj, f.x, o[2 * e]);
            o[2 * e + 1] = fmaf(pj, f.y, o[2 * e + 1]);
          }
        } else if (kDims == 4) {
          const uint2 x = *reinterpret_cast<const uint2*>(row);
          const float2 f0 = bf2_to_f2(x.x), f1 = bf2_to_f2(x.y);
          o[0] = fmaf(pj, f0.x, o[0]);
          o[1] = fmaf(pj, f0.y, o[1]);
          o[2] = fmaf(pj, f1.x, o[2]);
          o[3] = fmaf(pj, f1.y, o[3]);
        } else {  // kDims == 2
          const float2 f = bf2_to_f2(*reinterpret_cast<const uint32_t*>(row));
          o[0] = fmaf(pj, f.x, o[0]);
          o[1] = fmaf(pj, f.y, o[1]);
        }
      }
    }
    __syncthreads();  // stage st has been read by everyone
    if (t == 0 && c + 2 < nlocal) issue(c + 2);
  }
  if (!ok) {  // chunks c and c + 1 may still be in flight: let them land (bounded)
    if (t == 0)
      for (int cf = c; cf < nlocal && cf < c + 2; ++cf) {
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(&sm.full[cf & 1], (cf >> 1) & 1) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    return;
  }
  // partial result of this split
  if (t < kActive) {
    const int h = kvh * G + gh;
    const int64_t idx = ((int64_t)b * p.Hq + h) * p.nsplit + split;
    if (sub == 0) {
      p.part_ml[2 * idx] = m_run;
      p.part_ml[2 * idx + 1] = l_run;
    }
#pragma unroll
    for (int i = 0; i < kDims; ++i) p.part_o[idx * kHeadDim + sub * kDims + i] = o[i];
  }
}

// One warp per (sequence, head): two output dims per lane.
__global__ void __launch_bounds__(32) decode_combine_kernel(DecodeProblem p) {
  const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const int L = p.seqlens[b];
  if (L < 0 || L > p.max_blocks * p.block_size) return;  // reported by the split kernel
  const int64_t base = ((int64_t)b * p.Hq + h) * p.nsplit;
  const float sink2 = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
  float M = sink2;
  for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, p.part_ml[2 * (base + s)]);
  const float msub = M == -INFINITY ? 0.f : M;
  float Z = p.sinks ? ex2(sink2 - msub) : 0.f;
  float o0 = 0.f, o1 = 0.f;
  for (int s = 0; s < p.nsplit; ++s) {
    const float w = ex2(p.part_ml[2 * (base + s)] - msub);
    Z = fmaf(p.part_ml[2 * (base + s) + 1], w, Z);
    const float2 x = *reinterpret_cast<const float2*>(&p.part_o[(base + s) * kHeadDim + 2 * lane]);
    o0 = fmaf(x.x, w, o0);
    o1 = fmaf(x.y, w, o1);
  }
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  reinterpret_cast<uint32_t*>(p.o + ((int64_t)b * p.Hq + h) * kHeadDim)[lane] = pack_bf16(o0 * inv, o1 * inv);
  if (p.lse && lane == 0) p.lse[(int64_t)h * p.nseq + b] = Z > 0.f ? (msub + __log2f(Z)) * kLn2 : -INFINITY;
}

template <int G>
cudaError_t launch_split(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeProblem& p,
                         cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kDecSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.nsplit, p.Hkv, p.nseq);
  decode_split_kernel<G><<<grid, kDecThreads, kDecSmemBytes, s>>>(mk, mv, p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

size_t decode_workspace_bytes(int32_t nseq, int32_t Hq, int32_t nsplit) {
  const size_t n = (size_t)nseq * Hq * nsplit;
  return ((n * 2 * sizeof(float) + 255) & ~size_t(255)) + n * kHeadDim * sizeof(float);
}

cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t s) {
  if (p.nseq == 0) return cudaSuccess;
  CUtensorMap mk, mv;
  const int64_t rows = (int64_t)p.num_blocks * p.block_size;
  cudaError_t e = make_tmap_bf16_rows(&mk, p.k_cache, p.Hkv, (int)rows, (int64_t)p.Hkv * kHeadDim,
                                      p.block_size);
  if (e == cudaSuccess)
    e = make_tmap_bf16_rows(&mv, p.v_cache, p.Hkv, (int)rows, (int64_t)p.Hkv * kHeadDim, p.block_size);
  if (e != cudaSuccess) return e;
  switch (p.Hq / p.Hkv) {
    case 1: e = launch_split<1>(mk, mv, p, s); break;
    case 2: e = launch_split<2>(mk, mv, p, s); break;
    case 4: e = launch_split<4>(mk, mv, p, s); break;
    case 8: e = launch_split<8>(mk, mv, p, s); break;
    case 16: e = launch_split<16>(mk, mv, p, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<dim3(p.Hq, p.nseq), 32, 0, s>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
