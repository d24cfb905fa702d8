// Decode with sinks over a paged KV cache: one new query row per sequence
// (page "GPT-OSS Agentic RL Training: A Practical Retrospective", section
// "Implementation in FlashAttention v3", step 1, the forward with sinks, here
// on the inference side the pages took it from).
//
// The query of sequence b is the row at its last position, L - 1; it sees
// keys j in [max(0, L - W), L) (all of them without a window) and the sink of
// its head. The keys are split into ranges handled by separate CTAs:
//
//   split kernel    one CTA per (split, kv head, sequence) takes the G query
//                   heads of its kv head together. 128-key chunks of K and V
//                   come in by TMA (one copy per cache block), S = 3 chunks
//                   deep, or S = 1 when every split has at most two chunks
//                   (a short window): 44 KB of shared memory then lets four
//                   CTAs share an SM, so the whole grid runs in one wave.
//                   Both contractions run on the tensor cores with the keys
//                   on the long side, so the G heads (padded to N = 16) cost
//                   little: S^T = K Q^T (M = 128 keys) lands in tensor memory
//                   one key per thread, and O^T += V^T P^T (M = the 64 output
//                   dims) accumulates there across chunks. In between, each
//                   thread turns its key's scores into probabilities against a
//                   per-head reference maximum that moves only when a score
//                   exceeds it by 2^8 (then O^T and the sums are rescaled), so
//                   a chunk needs no reduction across threads.
//   combine kernel  per (sequence, head), when a sequence has several
//                   splits: max over the partials and the sink logit, then
//                   O = sum_s o_s 2^(m_s - M) / Z with
//                   Z = 2^(S_h - M) + sum_s l_s 2^(m_s - M), LSE = M + log Z.
//                   With one split the split kernel finishes the row itself.
//
// Scores are kept in log2 units (scale * log2 e is applied to the fp32
// scores), so every exponential is an exp2. The tensor cores are used because
// CUDA cores cannot keep up with HBM here: each K or V element costs 2G
// multiply-adds, and a CUDA-core version of this kernel (G = 8) needed about
// 5800 warp instructions per 32 KB chunk, as many as an SM can issue in the
// time HBM delivers the chunk.
#include <algorithm>
#include <cmath>

#include "internal.h"
#include "sm100.cuh"

namespace sinkattn {
namespace {

using namespace sm100;

constexpr int kDecThreads = 128;
constexpr int kChunk = 128;                                // keys per chunk, one per thread
constexpr uint32_t kPanelBytes = kChunk * 64 * 2;          // 128 keys x 64 features: 16 KB
constexpr int kN = 16;                                     // heads padded to the product's N
constexpr uint32_t kQPanelBytes = kN * 128;                // 16 heads x 64 features
constexpr float kLazy = 8.f;                               // log2 headroom of the reference max
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kErrInvalidArg = 1;  // SINKATTN_ERR_INVALID_ARG

// tensor memory columns
constexpr uint32_t kColO = 0;    // O^T: lanes = output dims (0..d-1), columns = heads
constexpr uint32_t kColS = 16;   // S^T, two buffers of 16: lanes = keys, columns = heads
constexpr uint32_t kTmemCols = 64;

// Head_dim 128: a chunk of K (or V) is two 64-feature panels of 128-byte
// rows, and so is Q; S^T walks both panels, and A = V^T of the second product
// spans them (M = 128 output dims, the panel distance its leading offset).
template <int S, int kD>
struct __align__(1024) DecSmem {
  static constexpr uint32_t kChunkBytes = kPanelBytes * (kD / 64);
  uint8_t k[S][kChunkBytes];        // chunk stages, panels of 128-byte rows, 128-byte swizzled
  uint8_t v[S][kChunkBytes];
  uint8_t q[kD / 64][kQPanelBytes]; // [16 heads][64 dims] bf16 per panel, 128-byte swizzled (rows >= G zero)
  uint8_t pt[2][2][kN * 128];       // P^T per buffer: [64-key block][16 heads][64 keys] bf16, swizzled
  float red[4][kN];                 // cross-warp max / sum per head
  int blk[S * (kChunk / 16)];       // physical blocks of the split's first S chunks
  uint64_t full[S];                 // TMA of a chunk landed
  uint64_t s_full[2];               // S^T of a chunk ready
  uint64_t pv_done[2];              // O^T += V^T P^T of a chunk done (stage and P^T free)
  uint32_t tmem_base;
  int abort;
  int bad;
};
template <int S, int kD>
constexpr size_t dec_smem_bytes() { return sizeof(DecSmem<S, kD>) + 1024; }

// Key range of a sequence in 128-key chunks aligned to the sequence start
// (the cache block size divides 128), and this split's share: splits take
// `split_chunks` chunks each, so work items have the same size whatever the
// sequence length, and the splits past a sequence's last chunk are empty.
struct Range {
  int L, k0, base_al, nch, c_begin, c_end;
};

__device__ __forceinline__ Range split_range(const DecodeProblem& p, int b, int split) {
  Range r;
  r.L = p.seqlens[b];
  r.k0 = p.window > 0 ? max(0, r.L - p.window) : 0;
  r.base_al = (r.k0 / kChunk) * kChunk;
  r.nch = r.L > r.base_al ? (r.L - r.base_al + kChunk - 1) / kChunk : 0;
  r.c_begin = min(r.nch, split * p.split_chunks);
  r.c_end = min(r.nch, r.c_begin + p.split_chunks);
  return r;
}

__device__ __forceinline__ bool length_ok(const DecodeProblem& p, const Range& r) {
  return r.L >= 0 && r.L <= p.max_blocks * p.block_size && r.nch <= p.split_chunks * p.nsplit;
}

// 16 consecutive 32-bit columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

template <int G, int S, int kD>
__global__ void __launch_bounds__(kDecThreads, (S == 1 ? 4 : 2) * 64 / kD)
decode_split_kernel(const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
                    DecodeProblem p) {
  constexpr int kStages = S;
  constexpr int kPanels = kD / 64;
  constexpr int kOutWarps = kD / 32;  // warps whose TMEM lanes hold output dims
  extern __shared__ uint8_t smem_raw[];
  DecSmem<S, kD>& sm = *reinterpret_cast<DecSmem<S, kD>*>(smem_raw + align1024_pad(smem_raw));
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  const Range r = split_range(p, b, split);
  const bool len_ok = length_ok(p, r);
  const int nlocal = r.c_end - r.c_begin;
  if (len_ok && nlocal == 0) {
    // past the sequence's last chunk: nothing to merge. A sequence without
    // keys and a single split gets the sink-only row here: o = 0 and
    // lse = S_h (or -inf without sinks).
    if (p.nsplit == 1 && r.L == 0) {
      for (int i = t; i < G * kD; i += kDecThreads)
        p.o[((int64_t)b * p.Hq + kvh * G) * kD + i] = __float2bfloat16_rn(0.f);
      if (p.lse && t < G) p.lse[(int64_t)(kvh * G + t) * p.nseq + b] = p.sinks ? p.sinks[kvh * G + t] : -INFINITY;
    }
    return;
  }
  const Guard g{&sm.abort, p.err, p.wait_limit_ns};
  if (t == 0) {
    sm.abort = 0;
    sm.bad = len_ok ? 0 : 1;
    for (int i = 0; i < kStages; ++i) mbar_init(&sm.full[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.pv_done[i], 1);
    }
    fence_barrier_init();
  }
  if (t == 32) tma_prefetch(&tm_kc);
  if (t == 33) tma_prefetch(&tm_vc);
  const int bs = p.block_size, nbox = kChunk / bs;
  const int64_t row_tab = (int64_t)b * p.max_blocks;
  __syncthreads();
  // every block index this split reads must be in range; those of its first
  // kStages chunks are kept for the first copies
  if (len_ok) {
    const int lbc0 = (r.base_al + r.c_begin * kChunk) / bs;
    const int lb0 = max(lbc0, r.k0 / bs);
    const int lb1 = min((r.base_al + r.c_end * kChunk) / bs, (r.L + bs - 1) / bs);
    for (int lb = lb0 + t; lb < lb1; lb += kDecThreads) {
      const int pb = p.block_table[row_tab + lb];
      if (pb < 0 || pb >= p.num_blocks) sm.bad = 1;
      if (lb - lbc0 < kStages * nbox) sm.blk[lb - lbc0] = pb;
    }
  }
  // Q of the group (rows >= G zero) and P^T rows >= G (zero for good), both
  // in the 128-byte-swizzled K-major layout the products read
  for (int i = t; i < kN * 8 * kPanels; i += kDecThreads) {
    const int pi = i / (kN * 8), h = (i / 8) % kN, cc = i % 8;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (h < G)
      x = *reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + kvh * G + h) * kD + 64 * pi + cc * 8);
    *reinterpret_cast<uint4*>(sm.q[pi] + sw128_offset(h, cc)) = x;
  }
  if constexpr (G < kN) {
    for (int i = t; i < 4 * (kN - G) * 8; i += kDecThreads) {
      const int cc = i % 8, h = G + (i / 8) % (kN - G), blk = i / (8 * (kN - G));
      *reinterpret_cast<uint4*>(&sm.pt[blk / 2][blk % 2][0] + sw128_offset(h, cc)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (sm.bad) {
    if (t == 0) atomicCAS(p.err, 0, kErrInvalidArg);
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    return;
  }

  auto chunk_start = [&](int c) { return r.base_al + (r.c_begin + c) * kChunk; };
  auto box_needed = [&](int j) { return j < r.L && j + bs > r.k0; };  // blocks before the window are skipped
  // Warp 0: block index of box `lane` of chunk c (read early, used at issue)
  auto load_blk = [&](int c) {
    const int j = chunk_start(c) + lane * bs;
    return (lane < nbox && box_needed(j)) ? p.block_table[row_tab + j / bs] : 0;
  };
  // Warp 0: TMA of chunk c into stage c % kStages, one box of `bs` rows per
  // block; lane i holds the block index of box i
  auto issue_tma = [&](int c, int pb_lane) {
    const int st = c % kStages, j0 = chunk_start(c);
    if (lane == 0) {
      uint32_t bytes = 0;
      for (int i = 0; i < nbox; ++i)
        if (box_needed(j0 + i * bs)) bytes += 2u * (uint32_t)bs * kD * 2u;
      mbar_expect_tx(&sm.full[st], bytes);
    }
    for (int i = 0; i < nbox; ++i) {
      const int pb = __shfl_sync(0xffffffffu, pb_lane, i);
      if (lane == 0 && box_needed(j0 + i * bs)) {
#pragma unroll
        for (int pi = 0; pi < kPanels; ++pi) {
          tma_load_3d(sm.k[st] + pi * kPanelBytes + i * bs * 128, &tm_kc, &sm.full[st], 64 * pi, kvh, pb * bs);
          tma_load_3d(sm.v[st] + pi * kPanelBytes + i * bs * 128, &tm_vc, &sm.full[st], 64 * pi, kvh, pb * bs);
        }
      }
    }
  };
  // Warp 0: S^T(c) = K Q^T into buffer c & 1 (K-major operands, 4 x K = 16)
  const uint32_t idS = idesc_bf16(128, kN, false, false);
  const uint32_t idO = idesc_bf16(128, kN, true, false);
  const uint64_t dQ = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
  auto issue_s = [&](int c) {
    const int st = c % kStages;
    const uint64_t dK = sdesc_sw128(smem_u32(sm.k[st]), 16, 1024);
#pragma unroll
    for (int k = 0; k < kD / 16; ++k) {  // +32 bytes per 16 features, panel by panel
      const uint64_t ok_ = (uint64_t)(k / 4) * (kPanelBytes >> 4) + 2 * (k % 4);
      const uint64_t oq = (uint64_t)(k / 4) * (kQPanelBytes >> 4) + 2 * (k % 4);
      umma_ss_warp(tmem + kColS + 16 * (c & 1), dK + ok_, dQ + oq, idS, k > 0);
    }
    umma_commit_warp(&sm.s_full[c & 1]);
  };
  // Warp 0: O^T += V^T P^T(c). A = V^T is the V tile read MN-major (M = 128
  // output rows): at head_dim 128 its two 64-dim panels, at 64 the one panel
  // twice (leading offset 0), the second copy's lanes of O^T never read.
  // B = P^T, two 64-key blocks of 2 KB.
  auto issue_pv = [&](int c) {
    const int st = c % kStages, pbuf = c & 1;
    const uint64_t dV = sdesc_sw128(smem_u32(sm.v[st]), kD == 128 ? kPanelBytes : 0, 1024);
#pragma unroll
    for (int k = 0; k < kChunk / 16; ++k) {
      const uint64_t dP = sdesc_sw128(smem_u32(sm.pt[pbuf][k / 4]), 16, 1024) + 2 * (k % 4);
      umma_ss_warp(tmem + kColO, dV + 128 * k, dP, idO, (c > 0 || k > 0) ? 1u : 0u);
    }
    umma_commit_warp(&sm.pv_done[pbuf]);
  };

  int n_tma = 0;  // chunks whose copies were issued (warp 0)
  int n_s = 0;    // chunks whose S^T was issued (warp 0)
  if (warp == 0) {
    // (test hook: with copies withheld, every wait below runs out)
    for (; n_tma < kStages && n_tma < nlocal && !p.withhold_copies; ++n_tma)
      issue_tma(n_tma, lane < nbox ? sm.blk[n_tma * nbox + lane] : 0);
    if (mbar_wait_warp(&sm.full[0], 0, g)) {
      tc_fence_after();
      issue_s(0);
      n_s = 1;
    }
  }

  const float sl2 = p.scale_log2;
  float m_ref[G], l_t[G];
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    m_ref[gg] = -INFINITY;
    l_t[gg] = 0.f;
  }
  int c = 0;
  for (; c < nlocal; ++c) {
    const int st = c % kStages, buf = c & 1, j0 = chunk_start(c);
    // chunk whose copies this iteration issues: with several stages the one
    // that reuses chunk c - 1's stage, with one stage the next chunk
    const int nxt = S == 1 ? c + 1 : c - 1 + kStages;
    const int pb_next = (warp == 0 && (S == 1 || c >= 1) && nxt < nlocal) ? load_blk(nxt) : 0;
    // S^T of the next chunk as early as its K tile is in
    if (warp == 0 && n_s == c + 1 && c + 1 < nlocal) {
      const int s1 = (c + 1) % kStages;
      const int ready = __shfl_sync(
          0xffffffffu, lane == 0 ? (int)mbar_try_wait(&sm.full[s1], ((c + 1) / kStages) & 1) : 0, 0);
      if (ready) {
        tc_fence_after();
        issue_s(c + 1);
        ++n_s;
      }
    }
    // scores of key t for every head
    const int j = j0 + t;
    const bool valid = j >= r.k0 && j < r.L;
    mbar_wait(&sm.s_full[buf], (c >> 1) & 1, g);
    tc_fence_after();
    uint32_t sr[16];
    tmem_ld16_wait(tmem + ((uint32_t)(32 * warp) << 16) + kColS + 16 * buf, sr);
    float x[G];
    bool need = false;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      x[gg] = valid ? __uint_as_float(sr[gg]) * sl2 : -INFINITY;
      need |= x[gg] > m_ref[gg] + kLazy;
    }
    if (!valid) {  // stale or never-written V rows must not reach the product (0 * NaN)
      mbar_wait(&sm.full[st], (c / kStages) & 1, g);  // the chunk's copies have landed (done long ago)
#pragma unroll
      for (int pi = 0; pi < kPanels; ++pi)
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4*>(sm.v[st] + pi * kPanelBytes + t * 128 + cc * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    need = __syncthreads_or(need);
    if (sm.abort) break;
    if (need) {  // move the reference maxima up to this chunk's maxima
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float v = x[gg];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) sm.red[warp][gg] = v;
      }
      __syncthreads();
      float alpha[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const float cm = fmaxf(fmaxf(sm.red[0][gg], sm.red[1][gg]), fmaxf(sm.red[2][gg], sm.red[3][gg]));
        const float m_new = fmaxf(m_ref[gg], cm);
        alpha[gg] = ex2(m_ref[gg] - m_new);  // 0 before the first chunk
        l_t[gg] *= alpha[gg];
        m_ref[gg] = m_new;
      }
      if (c > 0 && warp < kOutWarps) {  // rescale O^T (lanes 0..d-1 = dims) once the last product is in
        mbar_wait_warp(&sm.pv_done[(c - 1) & 1], ((c - 1) >> 1) & 1, g);
        tc_fence_after();
        uint32_t o[16];
        const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16) + kColO;
        tmem_ld16_wait(ta, o);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) o[gg] = __float_as_uint(__uint_as_float(o[gg]) * alpha[gg]);
        tmem_st16(ta, o);
        tmem_st_wait();
      }
    }
    // probabilities, as bf16 P^T for the product and summed per thread
    if (c >= 2) mbar_wait(&sm.pv_done[buf], ((c - 2) >> 1) & 1, g);  // P^T buffer free
    {
      uint8_t* prow = &sm.pt[buf][t / 64][0];
      const uint32_t col = t % 64;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const float pv = ex2(x[gg] - m_ref[gg]);
        l_t[gg] += pv;
        *reinterpret_cast<__nv_bfloat16*>(prow + sw128_offset(gg, col / 8) + (col % 8) * 2) =
            __float2bfloat16_rn(pv);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (sm.abort) break;
    if (warp == 0) {
      tc_fence_after();
      issue_pv(c);
      if constexpr (S == 1) {  // the only stage is free once this chunk's product is done
        if (nxt < nlocal && mbar_wait_warp(&sm.pv_done[c & 1], (c >> 1) & 1, g)) {
          issue_tma(nxt, pb_next);
          ++n_tma;
        }
      }
      if (n_s == c + 1 && c + 1 < nlocal) {  // the next K tile was late
        if (mbar_wait_warp(&sm.full[(c + 1) % kStages], ((c + 1) / kStages) & 1, g)) {
          issue_s(c + 1);
          ++n_s;
        }
      }
      if constexpr (S > 1) {
        if (c >= 1 && nxt < nlocal) {  // chunk c - 1's stage is free once its product is done
          if (mbar_wait_warp(&sm.pv_done[(c - 1) & 1], ((c - 1) >> 1) & 1, g)) {
            issue_tma(nxt, pb_next);
            ++n_tma;
          }
        }
      }
    }
  }
  bool ok = c == nlocal && !sm.abort;
  if (ok) {  // all products done: O^T complete
    mbar_wait(&sm.pv_done[(nlocal - 1) & 1], ((nlocal - 1) >> 1) & 1, g);
    tc_fence_after();
  }
  // per-head sums over the CTA
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    float v = l_t[gg];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) sm.red[warp][gg] = v;
  }
  __syncthreads();
  ok = ok && !sm.abort;
  if (ok && warp < kOutWarps) {
    float lsum[G];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) lsum[gg] = (sm.red[0][gg] + sm.red[1][gg]) + (sm.red[2][gg] + sm.red[3][gg]);
    uint32_t o[16];
    tmem_ld16_wait(tmem + ((uint32_t)(32 * warp) << 16) + kColO, o);
    const int d = t;  // output dim
    if (p.nsplit == 1) {
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const int h = kvh * G + gg;
        const float sink2 = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
        const float M = fmaxf(m_ref[gg], sink2);
        const float w = ex2(m_ref[gg] - M);
        const float Z = fmaf(lsum[gg], w, ex2(sink2 - M));
        p.o[((int64_t)b * p.Hq + h) * kD + d] = __float2bfloat16_rn(__uint_as_float(o[gg]) * (w / Z));
        if (p.lse && d == 0) p.lse[(int64_t)h * p.nseq + b] = (M + __log2f(Z)) * kLn2;
      }
    } else {
      const int64_t idx0 = ((int64_t)b * p.Hq + kvh * G) * p.nsplit + split;  // head kvh * G
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const int64_t idx = idx0 + (int64_t)gg * p.nsplit;
        p.part_o[idx * kD + d] = __uint_as_float(o[gg]);
        if (d == 0) {
          p.part_ml[2 * idx] = m_ref[gg];
          p.part_ml[2 * idx + 1] = lsum[gg];
        }
      }
    }
  }
  if (!ok && t == 0) {
    // let issued copies and products finish (bounded) before the memory goes
    for (int cf = max(0, n_tma - kStages); cf < n_tma; ++cf) {
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(&sm.full[cf % kStages], (cf / kStages) & 1) && global_ns() - t0 < kWaitLimitNs) {
      }
    }
    const uint64_t t0 = global_ns();
    if (c >= 1)
      while (!mbar_try_wait(&sm.pv_done[(c - 1) & 1], ((c - 1) >> 1) & 1) && global_ns() - t0 < kWaitLimitNs) {
      }
    if (n_s >= 1)
      while (!mbar_try_wait(&sm.s_full[(n_s - 1) & 1], ((n_s - 1) >> 1) & 1) &&
             global_ns() - t0 < kWaitLimitNs) {
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One warp per (sequence, head): d / 32 output dims per lane. Only the splits
// that hold keys of the sequence wrote partials.
template <int kD>
__global__ void __launch_bounds__(32) decode_combine_kernel(DecodeProblem p) {
  constexpr int kPer = kD / 32;  // consecutive dims per lane
  const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const Range r = split_range(p, b, 0);
  if (!length_ok(p, r)) return;  // reported by the split kernel
  const int ns = (r.nch + p.split_chunks - 1) / p.split_chunks;
  const int64_t base = ((int64_t)b * p.Hq + h) * p.nsplit;
  const float sink2 = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
  float M = sink2;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, p.part_ml[2 * (base + s)]);
  const float msub = M == -INFINITY ? 0.f : M;
  float Z = p.sinks ? ex2(sink2 - msub) : 0.f;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float w = ex2(p.part_ml[2 * (base + s)] - msub);
    Z = fmaf(p.part_ml[2 * (base + s) + 1], w, Z);
    const float* x = &p.part_o[(base + s) * kD + kPer * lane];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = fmaf(x[e], w, acc[e]);
  }
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  uint32_t* out = reinterpret_cast<uint32_t*>(p.o + ((int64_t)b * p.Hq + h) * kD + kPer * lane);
#pragma unroll
  for (int e = 0; e < kPer; e += 2) out[e / 2] = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
  if (p.lse && lane == 0) p.lse[(int64_t)h * p.nseq + b] = Z > 0.f ? (msub + __log2f(Z)) * kLn2 : -INFINITY;
}

template <int G, int S, int kD>
cudaError_t launch_split_s(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeProblem& p,
                           cudaStream_t s) {
  constexpr size_t bytes = dec_smem_bytes<S, kD>();
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<G, S, kD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.nsplit, p.Hkv, p.nseq);
  decode_split_kernel<G, S, kD><<<grid, kDecThreads, bytes, s>>>(mk, mv, p);
  note_launch();
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_split(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeProblem& p,
                         cudaStream_t s) {
  if (p.head_dim == kHeadDimWide)
    return p.split_chunks <= 2 ? launch_split_s<G, 1, kHeadDimWide>(mk, mv, p, s)
                               : launch_split_s<G, 3, kHeadDimWide>(mk, mv, p, s);
  return p.split_chunks <= 2 ? launch_split_s<G, 1, kHeadDim>(mk, mv, p, s)
                             : launch_split_s<G, 3, kHeadDim>(mk, mv, p, s);
}

}  // namespace

size_t decode_workspace_bytes(int32_t nseq, int32_t Hq, int32_t nsplit, int32_t head_dim) {
  const size_t n = (size_t)nseq * Hq * nsplit;
  return ((n * 2 * sizeof(float) + 255) & ~size_t(255)) + n * head_dim * sizeof(float);
}

cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t s) {
  if (p.nseq == 0) return cudaSuccess;
  CUtensorMap mk, mv;
  const int64_t rows = (int64_t)p.num_blocks * p.block_size;
  const int d = p.head_dim;
  cudaError_t e = make_tmap_bf16_rows(&mk, p.k_cache, p.Hkv, (int)rows, (int64_t)p.Hkv * d, p.block_size, d);
  if (e == cudaSuccess)
    e = make_tmap_bf16_rows(&mv, p.v_cache, p.Hkv, (int)rows, (int64_t)p.Hkv * d, p.block_size, d);
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
  if (p.nsplit == 1) return cudaSuccess;  // the split kernel finished every row
  if (d == kHeadDimWide)
    decode_combine_kernel<kHeadDimWide><<<dim3(p.Hq, p.nseq), 32, 0, s>>>(p);
  else
    decode_combine_kernel<kHeadDim><<<dim3(p.Hq, p.nseq), 32, 0, s>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
