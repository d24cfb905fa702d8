// Backward main kernel at head_dim 128: dK and dV of sink attention (page
// "GPT-OSS Agentic RL Training: A Practical Retrospective", section
// "Implementation in FlashAttention v3", step 2). dq comes from the
// query-stationary pass and dL/dS_h from the partials this kernel leaves for
// the finish pass, as at head_dim 64.
//
// Key-stationary like the head_dim 64 kernel: one CTA per SM owns a 128-key
// tile of one kv head at a time (persistent; units from the device-built
// key-tile list) and loops over the G query heads of the group x the 128-row
// query tiles that see the key tile, each taken as two 64-row blocks:
//   S^T  = K Q^T      [128 keys x 64 q]   SS, both K-major        -> TMEM
//   dP^T = V dO^T     [128 keys x 64 q]   SS, both K-major        -> TMEM
//   P^T  = exp2(S^T * scale * log2e - LSE * log2e),  dS^T = P^T (dP^T - D)
//        (softmax warpgroup, P^T written as bf16 over its own S^T columns,
//        dS^T to 128-byte-swizzled shared memory)
//   dV  += P^T dO     A = P^T (tensor memory), B = dO (MN-major)   TMEM
//   dK  += dS^T Q     A = dS^T (K-major), B = Q (MN-major)         TMEM
// dK and dV take 128 columns each, so tensor memory (512 columns) holds them
// plus two S^T / dP^T buffers and nothing else: the blocks alternate between
// the buffers (block parity), and each buffer has its own softmax warpgroup,
// so one warpgroup's softmax overlaps the products of the other's block.
// S^T / dP^T of block i + 2 are issued after the dV / dK products of block i,
// which read its P^T and dS^T: tcgen05 products of one thread execute in
// issue order, so the softmax that sees block i + 2's S^T complete may reuse
// the block's columns and dS^T buffer without another wait.
//
// Q, dO, K and V tiles are stored as 64-feature panels of 128-byte rows (one
// TMA copy each); the S^T / dP^T products walk both panels, and the MN-major
// dO / Q operands of dV / dK span them through the descriptor's panel stride.
//
// Warp roles (384 threads): warp 0 TMA producer (all lanes stage LSE / D /
// p_sink), warp 1 UMMA issuer, warps 4-7 / 8-11 softmax of the even / odd
// blocks and the dV / dK epilogue (warps 2-3 idle, so that each softmax
// warp's index mod 4 is its TMEM lane quarter). Tensor memory: S^T [0,128)
// and dP^T [128,256) as two 64-column buffers each, dV [256,384), dK
// [384,512). Shared memory: K, V 32 KB each, Q / dO blocks (16 KB each) in a
// 3-stage ring, dS^T double-buffered (16 KB each): 192 KB.
#include <algorithm>
#include <cmath>
#include <type_traits>

#include "internal.h"
#include "sm100.cuh"

namespace sinkattn {
namespace {

using namespace sm100;

constexpr int kD = kHeadDimWide;                     // 128 features
constexpr int kBlk = 64;                             // query rows per block
constexpr int kThreads = 384;
constexpr uint32_t kKPanel = kTile * 64 * 2;         // 128 key rows x 64 features: 16 KB
constexpr uint32_t kKBytes = kKPanel * (kD / 64);    // 32 KB
constexpr uint32_t kQPanel = kBlk * 64 * 2;          // 64 query rows x 64 features: 8 KB
constexpr uint32_t kQBytes = kQPanel * (kD / 64);    // 16 KB
constexpr uint32_t kDsBytes = kTile * kBlk * 2;      // dS^T [128 keys x 64 q]: 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;  // S^T / dP^T: + 64 per buffer
constexpr int kQStages = 3;
constexpr int kSchedSlots = 4;
constexpr int kSchedConsumers = 1 + 8;  // the UMMA warp and 8 softmax warps
constexpr float kLog2e = 1.4426950408889634f;

struct __align__(1024) Smem {
  uint8_t k[kKBytes];
  uint8_t v[kKBytes];
  uint8_t q[kQStages][kQBytes];
  uint8_t dout[kQStages][kQBytes];
  uint8_t dst[2][kDsBytes];             // dS^T, by block parity
  float4 rowld[kQStages][kBlk / 2];     // per query-row pair: {-LSE*log2e (+inf
                                        // outside the sequence) x2, -D x2}
  float2 rowps[kQStages][kBlk / 2];     // per query-row pair: p_sink x2
  uint64_t kv_full, kv_empty, q_full[kQStages], q_empty[kQStages];
  uint64_t sdp_full[2], pds_full[2];
  uint64_t dkv_full, dkv_empty, drain;
  uint64_t sched_full[kSchedSlots], sched_empty[kSchedSlots];
  int32_t sched_unit[kSchedSlots];  // work unit handed out, -1 = no more work
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Unit {
  int tidx, base, L, c0, nkeys, kvh, qt0, nq;
};

// Key tile it.y of sequence it.x, kv head w % Hkv (as at head_dim 64: the
// partials of dL/dS_h are stored under the key-tile number tidx).
__device__ __forceinline__ Unit decode(const Problem& p, const int2* items, int w) {
  Unit u;
  const int2 it = items[w / p.Hkv];
  u.kvh = w % p.Hkv;
  u.base = p.cu[it.x];
  u.L = p.cu[it.x + 1] - u.base;
  u.c0 = it.y * kTile;
  u.tidx = it.x + (u.base + u.c0) / kTile;
  const int c1 = min(u.L, u.c0 + kTile);
  u.nkeys = c1 - u.c0;
  int lo, hi;
  seeing_rows(p.causal, p.window, u.L, u.c0, c1, &lo, &hi);
  u.qt0 = lo / kTile;
  u.nq = (hi + kTile - 1) / kTile - u.qt0;
  return u;
}

template <class SmemT>
__device__ __forceinline__ int next_unit(SmemT& sm, uint32_t& n, const Guard& g, bool arrive,
                                         unsigned lanes) {
  const int s = n % kSchedSlots;
  if (!__all_sync(lanes, mbar_wait(&sm.sched_full[s], (n / kSchedSlots) & 1, g))) return -1;
  const int w = __shfl_sync(lanes, sm.sched_unit[s], 0);  // warp-uniform
  __syncwarp(lanes);
  if (arrive) mbar_arrive(&sm.sched_empty[s]);
  ++n;
  return w;
}

// Wait that ignores the abort flag (still time-bounded): used only to drain
// copies / products this CTA issued before it exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) break;
}

__global__ void __launch_bounds__(kThreads, 1)
bwd_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                BwdProblem bp, const int2* __restrict__ items, int32_t* __restrict__ meta) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw + align1024_pad(smem_raw));
  const Problem& p = bp.f;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Guard g{&sm.abort, p.err, p.wait_limit_ns};

  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.sdp_full[s], 1);
      mbar_init(&sm.pds_full[s], 128);
    }
    mbar_init(&sm.dkv_full, 1);
    mbar_init(&sm.dkv_empty, 256);
    mbar_init(&sm.drain, 1);
    for (int s = 0; s < kSchedSlots; ++s) {
      mbar_init(&sm.sched_full[s], 1);
      mbar_init(&sm.sched_empty[s], kSchedConsumers);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tm_q);
    tma_prefetch(&tm_k);
    tma_prefetch(&tm_v);
    tma_prefetch(&tm_do);
  }
  __syncthreads();
  tc_fence_after();
  // broadcast so the compiler sees a warp-uniform value (UMMA operands)
  const uint32_t tmem = __shfl_sync(0xffffffffu, sm.tmem_base, 0);
  const int nwork = meta[0] * p.Hkv;
  const int G = p.G;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t nunit = 0, nblk = 0, nsched = 0;
    bool ok = true;
    for (;;) {
      // take the next unit and publish it (or -1 when the list is exhausted)
      int w = 0;
      if (lane == 0) w = atomicAdd(&meta[1], 1);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w >= nwork) w = -1;
      {
        const int s = nsched % kSchedSlots;
        if (!mbar_wait_warp(&sm.sched_empty[s], ((nsched / kSchedSlots) & 1) ^ 1, g)) break;
        if (lane == 0) {
          sm.sched_unit[s] = w;
          mbar_arrive(&sm.sched_full[s]);
        }
        ++nsched;
      }
      if (w < 0) break;
      if (p.withhold_copies) break;  // test hook: the consumers' waits run out
      const Unit u = decode(p, items, w);
      // the unit's K / V load goes out right after its first Q / dO block
      bool kv_loaded = false;
      for (int i = 0; i < 2 * G * u.nq; ++i, ++nblk) {
        const int ti = i >> 1;
        const int h = u.kvh * G + ti / u.nq;
        const int q0 = (u.qt0 + ti % u.nq) * kTile + kBlk * (i & 1);
        const int st = nblk % kQStages;
        // global loads first (all in flight together), then the stage wait
        float lv[2], dv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int q = q0 + lane * 2 + e;
          const int64_t off = (int64_t)h * p.total + u.base + q;
          lv[e] = q < u.L ? __ldg(p.lse + off) : 0.f;
          dv[e] = q < u.L ? __ldg(bp.D + off) : 0.f;
        }
        const float sink2 = p.sinks ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
        if (!mbar_wait_warp(&sm.q_empty[st], ((nblk / kQStages) & 1) ^ 1, g)) {
          ok = false;
          break;
        }
        float l2[2], dd[2], ps[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool in = q0 + lane * 2 + e < u.L;
          l2[e] = in ? lv[e] * kLog2e : INFINITY;
          dd[e] = in ? dv[e] : 0.f;
          ps[e] = in && p.sinks ? ex2(sink2 - l2[e]) : 0.f;
        }
        sm.rowld[st][lane] = make_float4(-l2[0], -l2[1], -dd[0], -dd[1]);
        sm.rowps[st][lane] = make_float2(ps[0], ps[1]);
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(&sm.q_full[st], 2 * kQBytes);
#pragma unroll
          for (int pi = 0; pi < kD / 64; ++pi) {
            tma_load_3d(sm.q[st] + pi * kQPanel, &tm_q, &sm.q_full[st], 64 * pi, h, u.base + q0);
            tma_load_3d(sm.dout[st] + pi * kQPanel, &tm_do, &sm.q_full[st], 64 * pi, h, u.base + q0);
          }
        }
        if (!kv_loaded) {
          if (!mbar_wait_warp(&sm.kv_empty, (nunit & 1) ^ 1, g)) {
            ++nblk;  // this block's copy is in flight: the abort drain must see it
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(&sm.kv_full, 2 * kKBytes);
#pragma unroll
            for (int pi = 0; pi < kD / 64; ++pi) {
              tma_load_3d(sm.k + pi * kKPanel, &tm_k, &sm.kv_full, 64 * pi, u.kvh, u.base + u.c0);
              tma_load_3d(sm.v + pi * kKPanel, &tm_v, &sm.kv_full, 64 * pi, u.kvh, u.base + u.c0);
            }
          }
          ++nunit;
          kv_loaded = true;
        }
      }
      if (!ok) break;
    }
    if (lane == 0 && g.aborted()) {
      if (nunit) drain_wait(&sm.kv_full, (nunit - 1) & 1);
      for (uint32_t c = nblk > kQStages ? nblk - kQStages : 0; c < nblk; ++c)
        drain_wait(&sm.q_full[c % kQStages], (c / kQStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    // The whole warp runs this loop (uniform control flow and operands); one
    // elected lane issues each product and commit.
    const uint32_t idS = idesc_bf16(kTile, kBlk, false, false);
    const uint32_t idKV = idesc_bf16(kTile, kD, false, true);
    // descriptors built once; a product adds its byte offset / 16
    const uint64_t dK = sdesc_sw128(smem_u32(sm.k), 16, 1024);  // K-major
    const uint64_t dV = sdesc_sw128(smem_u32(sm.v), 16, 1024);
    const uint64_t dQk0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
    const uint64_t dOk0 = sdesc_sw128(smem_u32(sm.dout[0]), 16, 1024);
    // MN-major: the 64-feature panels of a block are kQPanel apart
    const uint64_t dQmn0 = sdesc_sw128(smem_u32(sm.q[0]), kQPanel, 1024);
    const uint64_t dOmn0 = sdesc_sw128(smem_u32(sm.dout[0]), kQPanel, 1024);
    const uint64_t dSk0 = sdesc_sw128(smem_u32(sm.dst[0]), 16, 1024);
    constexpr uint64_t kStageStep = kQBytes >> 4;  // q[1] - q[0], dout[1] - dout[0]
    constexpr uint64_t kDsStep = kDsBytes >> 4;    // dst[1] - dst[0]
    uint32_t nunit = 0, nblk = 0, npds[2] = {0, 0};
    bool ok = true;
    // S^T and dP^T of block `blk` into buffer blk & 1 (its Q / dO stage must
    // be full; the buffer's previous block's dV / dK were issued before)
    auto issue_sdp = [&](uint32_t blk) -> bool {
      const int st = blk % kQStages, b = blk & 1;
      if (!mbar_wait_warp(&sm.q_full[st], (blk / kQStages) & 1, g)) return false;
      tc_fence_after();
      const uint64_t bq = dQk0 + st * kStageStep;
      const uint64_t bo = dOk0 + st * kStageStep;
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) {  // +32 bytes per 16 features, panel by panel
        const uint64_t ok_ = (uint64_t)(k / 4) * (kKPanel >> 4) + 2 * (k % 4);
        const uint64_t oq = (uint64_t)(k / 4) * (kQPanel >> 4) + 2 * (k % 4);
        umma_ss_warp(tmem + kColS + 64 * b, dK + ok_, bq + oq, idS, k > 0);
        umma_ss_warp(tmem + kColDP + 64 * b, dV + ok_, bo + oq, idS, k > 0);
      }
      umma_commit_warp(&sm.sdp_full[b]);
      return true;
    };
    uint32_t nsched = 0;
    for (;;) {
      const int w = next_unit(sm, nsched, g, lane == 0, 0xffffffffu);
      if (w < 0) break;
      const Unit u = decode(p, items, w);
      const int nb = __shfl_sync(0xffffffffu, 2 * G * u.nq, 0);  // warp-uniform trip count (even, >= 2)
      if (!mbar_wait_warp(&sm.kv_full, nunit & 1, g)) break;
      if (!mbar_wait_warp(&sm.dkv_empty, (nunit & 1) ^ 1, g)) break;
      ++nunit;
      const uint32_t blk0 = nblk;
      if (!issue_sdp(blk0) || !issue_sdp(blk0 + 1)) break;
      for (int i = 0; i < nb && ok; ++i) {
        const uint32_t blk = blk0 + i;
        const int st = blk % kQStages, b = blk & 1;
        if (!mbar_wait_warp(&sm.pds_full[b], npds[b] & 1, g)) {
          ok = false;
          break;
        }
        ++npds[b];
        tc_fence_after();
        const uint32_t ap = tmem + kColS + 64 * b;  // P^T of this block (bf16 pairs, over its S^T)
        const uint64_t as = dSk0 + b * kDsStep;
        const uint64_t bo = dOmn0 + st * kStageStep;
        const uint64_t bq = dQmn0 + st * kStageStep;
#pragma unroll
        for (int k = 0; k < kBlk / 16; ++k) {  // 64 q rows, 16 at a time (+2048 B per panel)
          const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
          umma_ts_warp(tmem + kColDV, ap + 8 * k, bo + 128 * k, idKV, acc);
          umma_ss_warp(tmem + kColDK, as + 2 * k, bq + 128 * k, idKV, acc);
        }
        umma_commit_warp(&sm.q_empty[st]);  // last reader of this block's Q / dO
        if (i + 2 < nb && !issue_sdp(blk + 2)) ok = false;
      }
      nblk = blk0 + nb;
      if (!ok) break;
      umma_commit_warp(&sm.dkv_full);
      umma_commit_warp(&sm.kv_empty);
    }
    umma_commit_warp(&sm.drain);
    if (lane == 0) drain_wait(&sm.drain, 0);
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    // Warpgroup hf handles the blocks of parity hf (query rows 64 hf .. 64 hf
    // + 63 of every 128-row tile), each warp its 32 key rows (TMEM lanes),
    // read as two 16-lane groups in the .16x256b layout: thread t holds key
    // rows t/4 and t/4 + 8 of a group and, in every 8-column block, the query
    // pair 2(t%4), 2(t%4) + 1.
    const int hf = (warp - 4) / 4;
    const int quarter = warp & 3;
    const int gq = lane >> 2, qq = lane & 3;
    const uint64_t sl2x2 = f2pack(p.scale_log2, p.scale_log2);
    uint32_t nunit = 0, nblk0 = 0, nsd = 0, nsched = 0;
    bool ok = true;
    while (ok) {
      const int w = next_unit(sm, nsched, g, lane == 0, 0xffffffffu);
      if (w < 0) break;
      const Unit u = decode(p, items, w);
      // this thread's key rows: 32 quarter + 16 grp + 8 rh + gq, grp, rh in {0, 1}
      const int row_lo = 32 * quarter + gq, row_hi = row_lo + 24;
      const bool rows_valid = row_hi < u.nkeys;
      const int qlo_max = p.causal ? u.c0 + row_hi : 0;
      const int qhi_min = p.window > 0 ? u.c0 + row_lo + p.window : 0x7fffffff;
      uint64_t sa0 = f2pack(0.f, 0.f), sa1 = f2pack(0.f, 0.f);
      for (int ti = 0; ti < G * u.nq && ok; ++ti) {
        const uint32_t blk = nblk0 + 2 * ti + hf;
        const int hh = ti / u.nq;
        const int qb = (u.qt0 + ti % u.nq) * kTile + kBlk * hf;
        const int st = blk % kQStages;
        // the producer's LSE / D / p_sink rows of this block (acquire); the
        // first half of this thread's per-query constants is read while
        // S^T / dP^T are still being computed
        if (!mbar_wait_warp(&sm.q_full[st], (blk / kQStages) & 1, g)) {
          ok = false;
          break;
        }
        const float4* ld = &sm.rowld[st][qq];  // + 4 k: {-LSE*log2e x2, -D x2}
        const float2* pp = &sm.rowps[st][qq];  // + 4 k: p_sink x2
        float4 a4[4];
        float2 b2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          a4[k] = ld[4 * k];
          b2[k] = pp[4 * k];
        }
        if (!mbar_wait_warp(&sm.sdp_full[hf], nsd & 1, g)) {
          ok = false;
          break;
        }
        ++nsd;
        tc_fence_after();
        // one verdict per warp: both instantiations below are full of
        // warp-collective instructions, so the warp must not split between them
        const bool full =
            __all_sync(0xffffffffu, rows_valid && qb >= qlo_max && qb + kBlk - 1 < qhi_min);
        const uint32_t srow = smem_u32(sm.dst[hf]);
        // chunk c: lane group c & 1, 8-column blocks kb .. kb + 3 (kb = 4 (c >> 1));
        // the TMEM loads of chunk c + 1 are in flight while chunk c is computed
        auto taddr = [&](int c, uint32_t col) {
          return tmem + ((uint32_t)(32 * quarter + 16 * (c & 1)) << 16) + col + 32 * (c >> 1);
        };
        // the masked variant is a separate instantiation, so the arithmetic of
        // blocks strictly inside the band carries no masking work
        auto chunks = [&](auto mask_tag) {
          constexpr bool kMask = decltype(mask_tag)::value;
          uint32_t sv[2][16], pv[2][16];
          tmem_ld16x256b_x4x2_async(taddr(0, kColS + 64 * hf), taddr(0, kColDP + 64 * hf), sv[0], pv[0]);
          tmem_ld_wait();
          reg_fence16(sv[0]);
          reg_fence16(pv[0]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cur = c & 1, grp = c & 1, kb = 4 * (c >> 1);
            // P^T of chunk c goes to columns 16 (c >> 1) .. + 15 of lane group
            // grp, which the loads of chunks c and below have read; chunk
            // c + 1 reads the other lane group or columns 32 .. 63
            if (c < 3)
              tmem_ld16x256b_x4x2_async(taddr(c + 1, kColS + 64 * hf), taddr(c + 1, kColDP + 64 * hf),
                                        sv[cur ^ 1], pv[cur ^ 1]);
            if (grp == 0 && kb > 0) {  // second half of the constants
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                a4[k] = ld[4 * (kb + k)];
                b2[k] = pp[4 * (kb + k)];
              }
            }
            uint32_t pP[8], pS[8];  // [2 k + rh]: block kb + k, key row rh
            auto compute = [&](auto elem_tag) {
              constexpr bool kSelect = decltype(elem_tag)::value;
              // allowed query columns [clo, clo + span) of this thread's two key
              // rows (an empty range for rows past the end of the sequence)
              int clo[2];
              unsigned span[2];
#pragma unroll
              for (int rh = 0; rh < 2; ++rh) {
                const int rr = 32 * quarter + 16 * grp + 8 * rh + gq;
                const int j = u.c0 + rr;
                clo[rh] = (p.causal ? j : 0) - qb;
                const int chi = p.window > 0 ? j + p.window - qb : 0x40000000;
                span[rh] = rr < u.nkeys ? (unsigned)max(chi - clo[rh], 0) : 0u;
              }
#pragma unroll
              for (int k = 0; k < 4; ++k) {
#pragma unroll
                for (int rh = 0; rh < 2; ++rh) {
                  const int e = 4 * k + 2 * rh;
                  const float2 x = f2unpack(ffma2(f2pack(__uint_as_float(sv[cur][e]), __uint_as_float(sv[cur][e + 1])),
                                                  sl2x2, f2pack(a4[k].x, a4[k].y)));
                  float P0 = ex2(x.x), P1 = ex2(x.y);
                  if (kSelect) {  // one unsigned compare and a select per element
                    const int col = 8 * (kb + k) + 2 * qq;
                    P0 = (unsigned)(col - clo[rh]) < span[rh] ? P0 : 0.f;
                    P1 = (unsigned)(col + 1 - clo[rh]) < span[rh] ? P1 : 0.f;
                  }
                  const uint64_t P = f2pack(P0, P1);
                  const uint64_t t = fmul2(P, f2pack(__uint_as_float(pv[cur][e]), __uint_as_float(pv[cur][e + 1])));
                  if (rh)
                    sa1 = ffma2(f2pack(b2[k].x, b2[k].y), t, sa1);
                  else
                    sa0 = ffma2(f2pack(b2[k].x, b2[k].y), t, sa0);
                  const float2 ds = f2unpack(ffma2(P, f2pack(a4[k].z, a4[k].w), t));  // P (dP - D)
                  pP[2 * k + rh] = pack_bf16(P0, P1);
                  pS[2 * k + rh] = pack_bf16(ds.x, ds.y);
                }
              }
            };
            if constexpr (!kMask) {
              compute(std::false_type{});
            } else {
              // The chunk is key rows [j0, j0 + 16) x query columns [q0, q0 + 32),
              // the same for the whole warp. Where the band covers all of it,
              // or none of it, no element needs its own test.
              const int r0 = 32 * quarter + 16 * grp;
              const int j0 = u.c0 + r0, q0 = qb + 8 * kb;
              const bool none = r0 >= u.nkeys || (p.causal && q0 + 31 < j0) ||
                                (p.window > 0 && q0 >= j0 + 15 + p.window);
              const bool whole = r0 + 15 < u.nkeys && (!p.causal || q0 >= j0 + 15) &&
                                 (p.window <= 0 || q0 + 31 < j0 + p.window);
              if (none) {
#pragma unroll
                for (int e = 0; e < 8; ++e) pP[e] = pS[e] = 0u;
              } else if (whole) {
                compute(std::false_type{});
              } else {
                compute(std::true_type{});
              }
            }
            // P^T (bf16 pairs) over S^T -- warp-wide: column 4 (kb + k) + qq of
            // lanes rh = 0 / 1
            tmem_st16x128b_x4(tmem + ((uint32_t)(32 * quarter + 16 * grp) << 16) + kColS + 64 * hf + 4 * kb, pP);
            // dS^T to shared memory, as 8x8 blocks: block kb + k, rows rh
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
              const int m = lane >> 3, rh = m & 1, k = 2 * s2 + (m >> 1);
              const uint32_t rj = 32 * quarter + 16 * grp + 8 * rh + (lane & 7);
              stmatrix_x4(srow + rj * 128u + ((uint32_t)((kb + k) ^ (lane & 7)) << 4), pS[4 * s2],
                          pS[4 * s2 + 1], pS[4 * s2 + 2], pS[4 * s2 + 3]);
            }
            if (c < 3) {
              tmem_ld_wait();
              reg_fence16(sv[cur ^ 1]);
              reg_fence16(pv[cur ^ 1]);
            }
          }
        };
        if (full)
          chunks(std::false_type{});
        else
          chunks(std::true_type{});
        tmem_st_wait();
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.pds_full[hf]);
        if (ti % u.nq == u.nq - 1) {
          // head hh done: this warp's share of its sink-gradient partial
          const float2 s0 = f2unpack(sa0), s1 = f2unpack(sa1);
          float v = (s0.x + s0.y) + (s1.x + s1.y);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0)
            bp.sink_part[((int64_t)(u.kvh * G + hh) * bp.part_stride + u.tidx) * 8 + hf * 4 +
                         quarter] = v;
          sa0 = sa1 = f2pack(0.f, 0.f);
        }
      }
      nblk0 += 2 * G * u.nq;
      if (!ok) break;
      // epilogue: warpgroup 0 writes the dV rows, warpgroup 1 the dK rows,
      // one key row (TMEM lane) per thread
      if (!mbar_wait_warp(&sm.dkv_full, nunit & 1, g)) break;
      ++nunit;
      tc_fence_after();
      const int r = 32 * quarter + lane;
      const int j = u.c0 + r;
      const float sc = hf == 0 ? 1.f : p.scale;
      const uint32_t tcol = tmem + ((uint32_t)(32 * quarter) << 16) + (hf == 0 ? kColDV : kColDK);
      uint32_t ob[kD / 2];
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 64) {
        uint32_t a[64];
        tmem_ld64(tcol + c0, a);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          ob[c0 / 2 + e] = pack_bf16(__uint_as_float(a[2 * e]) * sc, __uint_as_float(a[2 * e + 1]) * sc);
      }
      tc_fence_before();
      mbar_arrive(&sm.dkv_empty);
      if (r < u.nkeys) {
        const int64_t off = ((int64_t)(u.base + j) * p.Hkv + u.kvh) * kD;
        uint4* dst = reinterpret_cast<uint4*>((hf == 0 ? bp.dv : bp.dk) + off);
#pragma unroll
        for (int c = 0; c < kD / 8; ++c)
          dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t prepare_bwd_wide(const BwdProblem& p, BwdWideLaunch* l) {
  const Problem& f = p.f;
  cudaError_t e = make_tmap_bf16_rows(&l->q64, f.q, f.Hq, f.total, f.q_stride, kBlk, kD);
  if (e == cudaSuccess) e = make_tmap_bf16_rows(&l->k, f.k, f.Hkv, f.total, f.k_stride, kTile, kD);
  if (e == cudaSuccess) e = make_tmap_bf16_rows(&l->v, f.v, f.Hkv, f.total, f.v_stride, kTile, kD);
  if (e == cudaSuccess)
    e = make_tmap_bf16_rows(&l->dout64, p.dout, f.Hq, f.total, (int64_t)f.Hq * kD, kBlk, kD);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bwd_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

cudaError_t launch_bwd_wide(const BwdProblem& p, const BwdWideLaunch& l, const TileList& ktiles,
                            int num_sms, cudaStream_t s) {
  const int64_t work = (int64_t)ktiles.capacity * p.f.Hkv;
  const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms);
  if (grid <= 0) return cudaSuccess;
  bwd_wide_kernel<<<grid, kThreads, kSmemBytes, s>>>(l.q64, l.k, l.v, l.dout64, p, ktiles.items,
                                                     ktiles.meta);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
