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
// is not formed from D, whose O is rounded to bf16: the main kernel
// accumulates p_sink_i * P_ij * dP_ij from its fp32 P and dP instead, per
// (key tile, head), and the last pass adds those partials in a fixed order.
//
// Kernels, in launch order:
//   preprocess  one pass over (token, head) rows: D = rowsum(dO * O); clears
//               the fp32 dq accumulator
//   main        key-stationary, on tcgen05 tensor cores (below)
//   finish      dq = bf16(dq accumulator); dS_h = -(fixed-order fp64 sum of
//               the partials, one warp per head)
//
// Main kernel. One CTA per SM owns a 128-key tile of one kv head at a time
// (persistent; units are taken dynamically from the device-built key-tile
// list, longest first) and loops over the G query heads of the group x the
// 128-row query tiles that see the key tile, each split in two 64-row halves:
//   S^T  = K Q^T      [128 keys x 64 q]   SS, both K-major        -> TMEM
//   dP^T = V dO^T     [128 keys x 64 q]   SS, both K-major        -> TMEM
//   P^T  = exp2(S^T * scale * log2e - LSE * log2e),  dS^T = P^T (dP^T - D)
//        (softmax warpgroup, one key row per thread; P^T written as bf16 to
//        tensor memory, dS^T to 128-byte-swizzled shared memory)
//   dV  += P^T dO     A = P^T (tensor memory), B = dO (MN-major)   TMEM
//   dK  += dS^T Q     A = dS^T (K-major), B = Q (MN-major)         TMEM
//   dQ   = dS K       per 128-row tile: A = the same dS^T buffer read
//        M-major, B = K (MN-major); read out by a second warpgroup and added
//        to the fp32 accumulator with TMA bulk reduce-adds, each warp its own
//        32 rows through its own 4 KB staging buffer (no block-wide
//        handshake: a shared staging buffer with mbarrier hand-offs was 5%
//        slower on the dense workload).
// Each half has its own tensor-memory S^T / dP^T buffer and its own softmax
// warpgroup, so the two halves of a tile run side by side and the products
// of one half overlap the softmax of the other; dS^T is double-buffered by
// tile so the dQ product stays off the softmax's path. dK and dV stay in
// tensor memory across the whole GQA group (no atomics) and are written once.
//
// Warp roles (512 threads): warp 0 TMA producer (all lanes stage LSE / D /
// p_sink), warp 1 UMMA issuer, warps 4-7 / 8-11 softmax of half 0 / 1 and
// the dV / dK epilogue, warps 12-15 dQ read-out (warps 2-3 idle). Tensor
// memory (512 columns): S^T [0,128) as two 64-column buffers, dP^T [128,256),
// dV [256,320), dK [320,384), dQ [384,448), P^T [448,512) (bf16 pairs, two
// 32-column halves). Q / dO are triple-buffered.
#include <algorithm>
#include <cmath>
#include <type_traits>

#include "internal.h"
#include "sm100.cuh"

namespace sinkattn {
namespace {

using namespace sm100;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPrepThreads = 256;

// ---------------------------------------------------------------- preprocess
// One warp per four (token, head) rows at head_dim 64 (two at 128), 16 bytes
// per lane: D = rowsum(dO * O) reduced over the row's lanes, and (head_dim 64,
// atomic dq) the row's 256 bytes of the fp32 dq accumulator cleared with
// coalesced stores.
template <int kD>
__global__ void __launch_bounds__(kPrepThreads)
preprocess_kernel(BwdProblem bp) {
  constexpr int kLanes = kD / 8;  // lanes per row
  const Problem& p = bp.f;
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = ((int64_t)blockIdx.x * kPrepThreads + threadIdx.x) >> 5;
  const int64_t row = warp_id * (32 / kLanes) + lane / kLanes;  // token * Hq + head
  const int sub = lane % kLanes;                                // 16-byte chunk of the row
  const bool in = row < (int64_t)p.total * p.Hq;
  float D = 0.f;
  if (in) {
    const uint4 a = *reinterpret_cast<const uint4*>(p.o + row * kD + sub * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(bp.dout + row * kD + sub * 8);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(b2[e]);
      D = fmaf(x.x, y.x, fmaf(x.y, y.y, D));
    }
    if (kD == kHeadDim && !bp.deterministic && !bp.acc_cleared) {  // the atomic dq path sums into the accumulator
      float4* acc = reinterpret_cast<float4*>(bp.dq_acc + row * kHeadDim) + sub * 2;
      acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (p.sinks) {  // sink partials: key tiles that do not exist stay zero
    const int64_t np = (int64_t)p.Hq * bp.part_stride * 8;
    for (int64_t e = (int64_t)blockIdx.x * kPrepThreads + threadIdx.x; e < np;
         e += (int64_t)gridDim.x * kPrepThreads)
      bp.sink_part[e] = 0.f;
  }
#pragma unroll
  for (int o = 1; o < kLanes; o <<= 1) D += __shfl_xor_sync(0xffffffffu, D, o);
  if (in && sub == 0) bp.D[(row % p.Hq) * p.total + row / p.Hq] = D;
}

// ---------------------------------------------------------------- main
constexpr int kThreads = 512;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2;  // 16 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;        // 64 rows
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384,
                   kColPT = 448;
constexpr int kQStages = 3;
constexpr int kSchedSlots = 4;
// consumers of a scheduler slot: the UMMA thread, 8 softmax warps, 4 dQ warps
constexpr int kSchedConsumers = 1 + 8 + 4;

struct __align__(1024) Smem {
  uint8_t k[kTileBytes];
  uint8_t v[kTileBytes];
  uint8_t q[kQStages][kTileBytes];
  uint8_t dout[kQStages][kTileBytes];
  uint8_t dst[2][2 * kTileBytes];  // dS^T, double-buffered by tile parity
  uint8_t dq[4][4096];             // dQ staging: per read-out warp, one [32 q][32] fp32 box
  float4 rowld[kQStages][kTile / 2];  // per query-row pair: {-LSE*log2e (-inf
                                      // outside the sequence) x2, -D x2}
  float2 rowps[kQStages][kTile / 2];  // per query-row pair: p_sink x2
  uint64_t kv_full, kv_empty, q_full[kQStages], q_empty[kQStages];
  uint64_t sdp_full[2], sdp_empty[2], pds_full[2], p_free[2], ds_free[2];
  uint64_t dq_full, dq_empty, dkv_full, dkv_empty, drain;
  uint64_t sched_full[kSchedSlots], sched_empty[kSchedSlots];
  int32_t sched_unit[kSchedSlots];  // work unit handed out, -1 = no more work
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Unit {
  int tidx, base, L, c0, nkeys, kvh, qt0, nq;
};

__device__ __forceinline__ Unit decode(const Problem& p, const int2* items, int w) {
  Unit u;
  const int2 it = items[w / p.Hkv];
  u.kvh = w % p.Hkv;
  u.base = p.cu[it.x];
  u.L = p.cu[it.x + 1] - u.base;
  u.c0 = it.y * kTile;
  // a number for the key tile that does not depend on the list's order:
  // b + (cu[b] + c0) / 128 is unique over the packing and below its tile
  // capacity (the sink-gradient partials are stored under it)
  u.tidx = it.x + (u.base + u.c0) / kTile;
  const int c1 = min(u.L, u.c0 + kTile);
  u.nkeys = c1 - u.c0;
  int lo, hi;
  seeing_rows(p.causal, p.window, u.L, u.c0, c1, &lo, &hi);
  u.qt0 = lo / kTile;
  u.nq = (hi + kTile - 1) / kTile - u.qt0;
  return u;
}

// Work units are handed out dynamically (longest first, from the device-built
// list): the producer warp takes the next index with an atomic and publishes
// it in a small ring; every other role reads the ring in order.
// `lanes` = the calling lanes of the warp (all of them read the slot before
// the arriving lane releases it; all of them get the same verdict).
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

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) break;
}

__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int c0,
                                                  int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}


// kDQ = false: the deterministic mode's instantiation, without the dQ
// products and read-out (dq then comes from the query-stationary pass).
template <bool kDQ>
__global__ void __launch_bounds__(kThreads, 1)
bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
           const __grid_constant__ CUtensorMap tm_dq, BwdProblem bp,
           const int2* __restrict__ items, int32_t* __restrict__ meta) {
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
      mbar_init(&sm.sdp_empty[s], 128);
      mbar_init(&sm.pds_full[s], 128);
      mbar_init(&sm.p_free[s], 1);
      mbar_init(&sm.ds_free[s], 1);
    }
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_empty, 128);
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
    if (kDQ) tma_prefetch(&tm_dq);
  }
  __syncthreads();
  tc_fence_after();
  // broadcast so the compiler sees a warp-uniform value (UMMA operands)
  const uint32_t tmem = __shfl_sync(0xffffffffu, sm.tmem_base, 0);
  const int nwork = meta[0] * p.Hkv;
  const int G = p.G;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t nunit = 0, ntile = 0, nsched = 0;
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
      // the unit's K / V load goes out right after its first Q / dO tile: a
      // Q / dO stage frees up a few tiles before the previous unit's K / V
      // do, so the two latencies overlap at the unit boundary
      bool kv_loaded = false;
      for (int i = 0; i < G * u.nq; ++i, ++ntile) {
        const int h = u.kvh * G + i / u.nq;
        const int q0 = (u.qt0 + i % u.nq) * kTile;
        const int st = ntile % kQStages;
        // global loads first (all in flight together), then the stage wait
        float lv[4], dv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = q0 + lane * 4 + e;
          const int64_t off = (int64_t)h * p.total + u.base + q;
          lv[e] = q < u.L ? __ldg(p.lse + off) : 0.f;
          dv[e] = q < u.L ? __ldg(bp.D + off) : 0.f;
        }
        const float sink2 = p.sinks ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
        if (!mbar_wait_warp(&sm.q_empty[st], ((ntile / kQStages) & 1) ^ 1, g)) {
          ok = false;
          break;
        }
        float l2[4], dd[4], ps[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool in = q0 + lane * 4 + e < u.L;
          l2[e] = in ? lv[e] * kLog2e : INFINITY;
          dd[e] = in ? dv[e] : 0.f;
          ps[e] = in && p.sinks ? ex2(sink2 - l2[e]) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          sm.rowld[st][lane * 2 + e / 2] = make_float4(-l2[e], -l2[e + 1], -dd[e], -dd[e + 1]);
          sm.rowps[st][lane * 2 + e / 2] = make_float2(ps[e], ps[e + 1]);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(&sm.q_full[st], 2 * kTileBytes);
          tma_load_3d(sm.q[st], &tm_q, &sm.q_full[st], 0, h, u.base + q0);
          tma_load_3d(sm.dout[st], &tm_do, &sm.q_full[st], 0, h, u.base + q0);
        }
        if (!kv_loaded) {
          if (!mbar_wait_warp(&sm.kv_empty, (nunit & 1) ^ 1, g)) {
            ++ntile;  // this tile's copy is in flight: the abort drain must see it
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(&sm.kv_full, 2 * kTileBytes);
            tma_load_3d(sm.k, &tm_k, &sm.kv_full, 0, u.kvh, u.base + u.c0);
            tma_load_3d(sm.v, &tm_v, &sm.kv_full, 0, u.kvh, u.base + u.c0);
          }
          ++nunit;
          kv_loaded = true;
        }
      }
      if (!ok) break;
    }
    if (lane == 0 && g.aborted()) {
      if (nunit) drain_wait(&sm.kv_full, (nunit - 1) & 1);
      for (uint32_t c = ntile > kQStages ? ntile - kQStages : 0; c < ntile; ++c)
        drain_wait(&sm.q_full[c % kQStages], (c / kQStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    // The whole warp runs this loop (uniform control flow and operands); one
    // elected lane issues each product and commit.
    const uint32_t idS = idesc_bf16(kTile, kTile, false, false);
    const uint32_t idKV = idesc_bf16(kTile, kHeadDim, false, true);
    const uint32_t idQ = idesc_bf16(kTile, kHeadDim, true, true);
    // descriptors built once; a product adds its byte offset / 16
    const uint64_t dK = sdesc_sw128(smem_u32(sm.k), 16, 1024);        // K-major
    const uint64_t dKmn = sdesc_sw128(smem_u32(sm.k), 8192, 1024);    // MN-major
    const uint64_t dV = sdesc_sw128(smem_u32(sm.v), 16, 1024);
    // per-stage / per-buffer operands differ by a fixed byte distance
    const uint64_t dQk0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
    const uint64_t dQmn0 = sdesc_sw128(smem_u32(sm.q[0]), 8192, 1024);
    const uint64_t dOk0 = sdesc_sw128(smem_u32(sm.dout[0]), 16, 1024);
    const uint64_t dOmn0 = sdesc_sw128(smem_u32(sm.dout[0]), 8192, 1024);
    const uint64_t dSk0 = sdesc_sw128(smem_u32(sm.dst[0]), 16, 1024);
    const uint64_t dSm0 = sdesc_sw128(smem_u32(sm.dst[0]), kTileBytes, 1024);
    constexpr uint64_t kStageStep = kTileBytes >> 4;        // q[1] - q[0], dout[1] - dout[0]
    constexpr uint64_t kDsStep = (2 * kTileBytes) >> 4;     // dst[1] - dst[0]
    uint32_t nunit = 0, ntile = 0, nsdp = 0, npds[2] = {0, 0}, ndq = 0;
    bool ok = true;
    // S^T and dP^T of a whole query tile, N = 128 (its Q / dO stage must be
    // full, and both softmax warpgroups must have read the previous tile's)
    auto issue_sdp = [&](uint32_t tile) -> bool {
      const int st = tile % kQStages;
      if (!mbar_wait_warp(&sm.sdp_empty[0], (nsdp & 1) ^ 1, g) ||
          !mbar_wait_warp(&sm.sdp_empty[1], (nsdp & 1) ^ 1, g))
        return false;
      ++nsdp;
      tc_fence_after();
      const uint64_t bq = dQk0 + st * kStageStep;
      const uint64_t bo = dOk0 + st * kStageStep;
#pragma unroll
      for (int k = 0; k < kHeadDim / 16; ++k) {  // +32 bytes per 16 features
        umma_ss_warp(tmem + kColS, dK + 2 * k, bq + 2 * k, idS, k > 0);
        umma_ss_warp(tmem + kColDP, dV + 2 * k, bo + 2 * k, idS, k > 0);
      }
      umma_commit_warp(&sm.sdp_full[0]);
      umma_commit_warp(&sm.sdp_full[1]);
      return true;
    };
    uint32_t nsched = 0;
    for (;;) {
      const int w = next_unit(sm, nsched, g, lane == 0, 0xffffffffu);
      if (w < 0) break;
      const Unit u = decode(p, items, w);
      const int nt = __shfl_sync(0xffffffffu, G * u.nq, 0);  // warp-uniform trip count
      if (!mbar_wait_warp(&sm.kv_full, nunit & 1, g)) break;
      if (!mbar_wait_warp(&sm.dkv_empty, (nunit & 1) ^ 1, g)) break;
      ++nunit;
      const uint32_t tile0 = ntile;
      if (!mbar_wait_warp(&sm.q_full[tile0 % kQStages], (tile0 / kQStages) & 1, g) ||
          !issue_sdp(tile0))
        break;
      for (int i = 0; i < nt && ok; ++i) {
        const uint32_t tile = tile0 + i;
        const int st = tile % kQStages, db = tile & 1;
        const bool more = i + 1 < nt;
        // S^T / dP^T of the next tile go in as soon as both softmax
        // warpgroups have read this tile's and its Q / dO have landed, always
        // before this tile's dV / dK. (Putting them after this tile's dQ when
        // Q / dO were late measured 1-1.6% slower on every workload.)
        if (more) {
          if (!mbar_wait_warp(&sm.sdp_empty[0], (nsdp & 1) ^ 1, g) ||
              !mbar_wait_warp(&sm.sdp_empty[1], (nsdp & 1) ^ 1, g) ||
              !mbar_wait_warp(&sm.q_full[(tile + 1) % kQStages], ((tile + 1) / kQStages) & 1, g) ||
              !issue_sdp(tile + 1)) {
            ok = false;
            break;
          }
        }
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait_warp(&sm.pds_full[hf], npds[hf] & 1, g)) {
            ok = false;
            break;
          }
          ++npds[hf];
          tc_fence_after();
          const uint32_t ap = tmem + kColPT + 32 * hf;  // P^T of this half (TMEM)
          const uint64_t as = dSk0 + db * kDsStep + hf * (kTileBytes >> 4);
          const uint64_t bo = dOmn0 + st * kStageStep + hf * (kHalfBytes >> 4);
          const uint64_t bq = dQmn0 + st * kStageStep + hf * (kHalfBytes >> 4);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 64 q rows of this half, 16 at a time
            const uint32_t acc = (i > 0 || hf > 0 || k > 0) ? 1u : 0u;
            umma_ts_warp(tmem + kColDV, ap + 8 * k, bo + 128 * k, idKV, acc);  // +2048 B / 16 rows
            umma_ss_warp(tmem + kColDK, as + 2 * k, bq + 128 * k, idKV, acc);
          }
          umma_commit_warp(&sm.p_free[hf]);
          if (hf == 1) umma_commit_warp(&sm.q_empty[st]);  // last reader of Q / dO
        }
        if (!ok) break;
        if constexpr (kDQ) {
          if (!mbar_wait_warp(&sm.dq_empty, (ndq & 1) ^ 1, g)) {
            ok = false;
            break;
          }
          ++ndq;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)  // 128 keys, 16 at a time (+2048 B)
            umma_ss_warp(tmem + kColDQ, dSm0 + db * kDsStep + 128 * k, dKmn + 128 * k, idQ, k > 0);
          umma_commit_warp(&sm.ds_free[db]);
          umma_commit_warp(&sm.dq_full);
        } else {
          umma_commit_warp(&sm.ds_free[db]);  // dK of both halves has read dS^T
        }
      }
      ntile = tile0 + nt;
      if (!ok) break;
      umma_commit_warp(&sm.dkv_full);
      umma_commit_warp(&sm.kv_empty);
    }
    umma_commit_warp(&sm.drain);
    if (lane == 0) drain_wait(&sm.drain, 0);
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax
    // Warpgroup hf handles half hf (query columns 64 hf .. 64 hf + 63) of
    // every tile, each warp its 32 key rows (TMEM lanes), read as two 16-lane
    // groups in the .16x256b layout: thread t holds key rows t/4 and t/4 + 8 of
    // a group and, in every 8-column block, the query pair 2(t%4), 2(t%4) + 1.
    // A thread so needs the per-query constants of 16 columns, not 64.
    const int hf = (warp - 4) / 4;
    const int quarter = warp & 3;
    const int gq = lane >> 2, qq = lane & 3;
    const uint64_t sl2x2 = f2pack(p.scale_log2, p.scale_log2);
    uint32_t nunit = 0, ntile = 0, nsd = 0, nsched = 0;
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
      for (int i = 0; i < G * u.nq && ok; ++i, ++ntile) {
        const int hh = i / u.nq;
        const int qb = (u.qt0 + i % u.nq) * kTile + 64 * hf;
        const int st = ntile % kQStages, db = ntile & 1;
        // the producer's LSE / D / p_sink rows of this tile (acquire); the
        // first half of this thread's per-query constants is read while
        // S^T / dP^T are still being computed
        if (!mbar_wait_warp(&sm.q_full[st], (ntile / kQStages) & 1, g)) {
          ok = false;
          break;
        }
        const float4* ld = &sm.rowld[st][32 * hf + qq];  // + 4 k: {-LSE*log2e x2, -D x2}
        const float2* pp = &sm.rowps[st][32 * hf + qq];  // + 4 k: p_sink x2
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
            __all_sync(0xffffffffu, rows_valid && qb >= qlo_max && qb + 63 < qhi_min);
        const uint32_t srow = smem_u32(sm.dst[db] + hf * kTileBytes);
        // chunk c: lane group c & 1, 8-column blocks kb .. kb + 3 (kb = 4 (c >> 1));
        // the TMEM loads of chunk c + 1 are in flight while chunk c is computed
        auto taddr = [&](int c, uint32_t col) {
          return tmem + ((uint32_t)(32 * quarter + 16 * (c & 1)) << 16) + col + 32 * (c >> 1);
        };
        // the masked variant is a separate instantiation, so the arithmetic of
        // tiles strictly inside the band carries no masking work
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
                if (kMask) {  // one unsigned compare and a select per element
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
            if (c == 0) {
              // P^T half free (dV / dK of the previous tile done), and this
              // tile's dS^T buffer free (dQ of the tile before that done)
              if (!mbar_wait_warp(&sm.p_free[hf], (ntile & 1) ^ 1, g) ||
                  !mbar_wait_warp(&sm.ds_free[db], ((ntile >> 1) & 1) ^ 1, g))
                ok = false;
            }
            // P^T (bf16 pairs) to tensor memory -- warp-wide, so always issued:
            // column 4 (kb + k) + qq of lanes rh = 0 / 1
            tmem_st16x128b_x4(tmem + ((uint32_t)(32 * quarter + 16 * grp) << 16) + kColPT + 32 * hf + 4 * kb, pP);
            // dS^T to shared memory, as 8x8 blocks: block kb + k, rows rh
            if (ok) {
#pragma unroll
              for (int s2 = 0; s2 < 2; ++s2) {
                const int m = lane >> 3, rh = m & 1, k = 2 * s2 + (m >> 1);
                const uint32_t rj = 32 * quarter + 16 * grp + 8 * rh + (lane & 7);
                stmatrix_x4(srow + rj * 128u + ((uint32_t)((kb + k) ^ (lane & 7)) << 4), pS[4 * s2],
                            pS[4 * s2 + 1], pS[4 * s2 + 2], pS[4 * s2 + 3]);
              }
            }
            if (c < 3) {
              tmem_ld_wait();
              reg_fence16(sv[cur ^ 1]);
              reg_fence16(pv[cur ^ 1]);
              if (c == 2) {  // all of this half's S^T / dP^T is in registers
                tc_fence_before();
                mbar_arrive(&sm.sdp_empty[hf]);
              }
            }
          }
        };
        if (full)
          chunks(std::false_type{});
        else
          chunks(std::true_type{});
        tmem_st_wait();
        if (!ok) break;
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.pds_full[hf]);
        if (i % u.nq == u.nq - 1) {
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
      if (!ok) break;
      // epilogue: warpgroup 0 writes the dV rows, warpgroup 1 the dK rows,
      // one key row (TMEM lane) per thread
      if (!mbar_wait_warp(&sm.dkv_full, nunit & 1, g)) break;
      ++nunit;
      tc_fence_after();
      const int r = 32 * quarter + lane;
      const int j = u.c0 + r;
      uint32_t a[64];
      tmem_ld64(tmem + ((uint32_t)(32 * quarter) << 16) + (hf == 0 ? kColDV : kColDK), a);
      tc_fence_before();
      mbar_arrive(&sm.dkv_empty);
      if (r < u.nkeys) {
        const float sc = hf == 0 ? 1.f : p.scale;
        uint32_t ob[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          ob[e] = pack_bf16(__uint_as_float(a[2 * e]) * sc, __uint_as_float(a[2 * e + 1]) * sc);
        const int64_t off = ((int64_t)(u.base + j) * p.Hkv + u.kvh) * kHeadDim;
        uint4* dst = reinterpret_cast<uint4*>((hf == 0 ? bp.dv : bp.dk) + off);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
      }
    }
  } else if (warp >= 12 && !kDQ) {
    // no dQ: these warps only keep the scheduler ring moving
    uint32_t nsched = 0;
    while (next_unit(sm, nsched, g, lane == 0, 0xffffffffu) >= 0) {
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ read-out
    // Each warp adds its own 32 query rows: TMEM -> registers -> its 4 KB
    // staging buffer -> TMA bulk reduce-add, with warp-level sync only.
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint8_t* buf = sm.dq[quarter];
    uint32_t ndq = 0, nsched = 0;
    bool ok = true;
    while (ok) {
      const int w = next_unit(sm, nsched, g, lane == 0, 0xffffffffu);
      if (w < 0) break;
      const Unit u = decode(p, items, w);
      for (int i = 0; i < G * u.nq; ++i) {
        const int h = u.kvh * G + i / u.nq;
        const int q0 = (u.qt0 + i % u.nq) * kTile;
        if (!mbar_wait_warp(&sm.dq_full, ndq & 1, g)) {
          ok = false;
          break;
        }
        ++ndq;
        tc_fence_after();
        uint32_t a[2][32];
        tmem_ld32(tmem + lane_off + kColDQ, a[0]);
        tmem_ld32(tmem + lane_off + kColDQ + 32, a[1]);
        tc_fence_before();
        mbar_arrive(&sm.dq_empty);
        // rows past the sequence end add zeros: a box wholly past it is skipped
        if (q0 + 32 * quarter >= u.L) continue;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (lane == 0) bulk_wait_read0();  // this warp's previous reduce has read the buffer
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t* v = &a[half][4 * c];
            *reinterpret_cast<uint4*>(buf + sw128_offset(lane, c)) = make_uint4(v[0], v[1], v[2], v[3]);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tm_dq, buf, 32 * half, h, u.base + q0 + 32 * quarter);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- finish
constexpr int kFinishThreads = 256;

__global__ void __launch_bounds__(kFinishThreads)
finish_kernel(BwdProblem bp) {
  const Problem& p = bp.f;
  // dS_h: one warp per head, over the partials in key-tile order (not list
  // order). Lane-strided fp64 sums, then a fixed butterfly, so the result
  // depends neither on timing nor on the work list's order.
  const int hw = blockIdx.x * (kFinishThreads / 32) + threadIdx.x / 32;
  if (bp.dsinks && hw < p.Hq) {
    const int lane = threadIdx.x & 31;
    double acc = 0.0;
    if (p.sinks) {
      const int n = 8 * bp.part_stride;
      const float* part = bp.sink_part + (int64_t)hw * bp.part_stride * 8;
      for (int c = lane; c < n; c += 32) acc += (double)part[c];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) bp.dsinks[hw] = bp.accumulate_dsinks ? bp.dsinks[hw] + (float)(-acc) : (float)(-acc);
  }
  const int64_t n8 = (int64_t)p.total * p.Hq * kHeadDim / 8;
  const int64_t e = (int64_t)blockIdx.x * kFinishThreads + threadIdx.x;  // 8 elements each
  if (!bp.deterministic && e < n8) {
    const float sc = p.scale;  // dq = scale * sum_j dS_ij k_j
    const float4 a = reinterpret_cast<const float4*>(bp.dq_acc)[2 * e];
    const float4 b = reinterpret_cast<const float4*>(bp.dq_acc)[2 * e + 1];
    reinterpret_cast<uint4*>(bp.dq)[e] =
        make_uint4(pack_bf16(a.x * sc, a.y * sc), pack_bf16(a.z * sc, a.w * sc),
                   pack_bf16(b.x * sc, b.y * sc), pack_bf16(b.z * sc, b.w * sc));
  }
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdProblem& p, cudaStream_t s) {
  const int64_t rows = (int64_t)p.f.total * p.f.Hq;
  if (rows == 0) return cudaSuccess;
  const int64_t rows_per_block = kPrepThreads * 8 / p.f.head_dim;  // lanes per row: head_dim / 8
  const unsigned blocks = (unsigned)((rows + rows_per_block - 1) / rows_per_block);
  if (p.f.head_dim == kHeadDimWide)
    preprocess_kernel<kHeadDimWide><<<blocks, kPrepThreads, 0, s>>>(p);
  else
    preprocess_kernel<kHeadDim><<<blocks, kPrepThreads, 0, s>>>(p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t prepare_bwd_main(const BwdProblem& p, BwdLaunch* l) {
  // the Q / K / V / dO maps also serve the deterministic dq pass (any head dim)
  const int d = p.f.head_dim;
  cudaError_t e = make_tmap_bf16_rows(&l->q, p.f.q, p.f.Hq, p.f.total, p.f.q_stride, kTile, d);
  if (e == cudaSuccess) e = make_tmap_bf16_rows(&l->k, p.f.k, p.f.Hkv, p.f.total, p.f.k_stride, kTile, d);
  if (e == cudaSuccess) e = make_tmap_bf16_rows(&l->v, p.f.v, p.f.Hkv, p.f.total, p.f.v_stride, kTile, d);
  if (e == cudaSuccess)
    e = make_tmap_bf16_rows(&l->dout, p.dout, p.f.Hq, p.f.total, (int64_t)p.f.Hq * d, kTile, d);
  if (e == cudaSuccess)  // bf16 dq, written by the dq pass in 32-row boxes of half the features
    e = make_tmap_bf16_box(&l->dqo, p.dq, p.f.Hq, p.f.total, (int64_t)p.f.Hq * d, d, d / 2, 32);
  if (e != cudaSuccess || d != kHeadDim) return e;
  e = make_tmap_f32_rows(&l->dq, p.dq_acc, p.f.Hq, p.f.total);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(p.deterministic ? bwd_kernel<false> : bwd_kernel<true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

cudaError_t launch_bwd_main(const BwdProblem& p, const BwdLaunch& l, const TileList& ktiles,
                            int num_sms, cudaStream_t s) {
  const int64_t work = (int64_t)ktiles.capacity * p.f.Hkv;
  const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms);
  if (grid <= 0) return cudaSuccess;
  if (p.deterministic)
    bwd_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(l.q, l.k, l.v, l.dout, l.dq, p, ktiles.items,
                                                         ktiles.meta);
  else
    bwd_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(l.q, l.k, l.v, l.dout, l.dq, p, ktiles.items,
                                                        ktiles.meta);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_finish(const BwdProblem& p, const TileList& ktiles, int num_sms,
                              cudaStream_t s) {
  (void)num_sms;
  (void)ktiles;
  const int64_t n8 = (int64_t)p.f.total * p.f.Hq * kHeadDim / 8;
  const int64_t head_blocks = (p.f.Hq + kFinishThreads / 32 - 1) / (kFinishThreads / 32);
  const int64_t blocks =
      p.deterministic ? head_blocks : std::max<int64_t>(head_blocks, (n8 + kFinishThreads - 1) / kFinishThreads);
  finish_kernel<<<(unsigned)blocks, kFinishThreads, 0, s>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
