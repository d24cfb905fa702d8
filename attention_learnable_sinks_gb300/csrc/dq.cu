// Deterministic dq of sink attention: a query-stationary pass on tcgen05
// tensor cores. Each 128-row tile of dq is owned by one CTA, which sums the
// key tiles the rows see in increasing order, so dq is bit-identical from run
// to run whatever the schedule (page "GPT-OSS Agentic RL Training: A
// Practical Retrospective", section "Implementation in FlashAttention v3",
// step 2; the gradient is the one the key-stationary main kernel forms, with
// the order of its sum fixed instead of left to atomics).
//
// For a query tile of head h and every key tile j it sees, in order:
//   S    = Q K_j^T      [128 q x 128 keys]  SS, both K-major        -> TMEM
//   dP   = dO V_j^T     [128 q x 128 keys]  SS, both K-major        -> TMEM
//   P    = exp2(S * scale * log2e - LSE * log2e),  dS = P (dP - D)
//   dQ  += dS K_j       A = dS (tensor memory), B = K_j (MN-major)  -> TMEM
// and dq = bf16(scale * dQ) is written once per tile. D = rowsum(dO * O) is
// the backward preprocess's; the sink enters only through LSE.
//
// One CTA per SM (persistent; query tiles x heads are taken dynamically from
// the device-built query-tile list, longest first, the heads of a tile
// consecutive so that a GQA group's K / V tiles come from L2).
// Warp roles (320 threads): warp 0 TMA producer (Q / dO double-buffered by
// unit, K / V in a 3-stage ring), warp 1 UMMA issuer, warps 2-5 and 6-9 two
// softmax warpgroups, one query row (TMEM lane) per thread, keys 0-63 / 64-127
// of each tile, then dq columns 0-31 / 32-63 of the epilogue. Each thread
// loads its S / dP half at once and releases the buffer, so S / dP of the next
// key tile are computed while it forms dS.
// Tensor memory (512 columns): S [0,128), dP [128,256), dS [256,384) as two
// 64-column bf16-pair buffers (by key tile), dQ [384,512) as two 64-column
// buffers at head_dim 64 (by unit, so one unit's epilogue overlaps the next
// unit's products), one 128-column buffer at head_dim 128.
//
// Head_dim 128: the tiles are two 64-feature panels of 128-byte rows each (a
// product over the features walks both); Q / dO have one buffer and K / V two
// stages (192 KB of shared memory), so a unit's Q / dO load waits until the
// previous unit's last S / dP have completed.
#include <algorithm>
#include <cmath>

#include "internal.h"
#include "sm100.cuh"

namespace sinkattn {
namespace {

using namespace sm100;

constexpr int kThreads = 320;
constexpr uint32_t kPanelBytes = kTile * 64 * 2;  // 128 rows x 64 features of bf16
constexpr uint32_t kTmemCols = 512;
template <int kD>
struct Cfg {
  static constexpr int kPanels = kD / 64;
  static constexpr uint32_t kTileBytes = kPanelBytes * kPanels;
  static constexpr int kQBufs = kD == 64 ? 2 : 1;      // Q / dO buffers (by unit)
  static constexpr int kKVStages = kD == 64 ? 3 : 2;   // K / V ring
  static constexpr int kDQBufs = kD == 64 ? 2 : 1;     // dQ accumulators (by unit)
};
constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColDQ = 384;  // + 64 per buffer
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSchedSlots = 4;
constexpr int kSchedConsumers = 1 + 8;  // the UMMA warp and 8 softmax warps
constexpr int kSoftmaxThreads = 256;

struct Unit {
  int base, L, r0, nrows, h, kvh, kt0, kt1;
};

template <int kD>
struct __align__(1024) Smem {
  static constexpr uint32_t kTileBytes = Cfg<kD>::kTileBytes;
  static constexpr int kQBufs = Cfg<kD>::kQBufs, kKVStages = Cfg<kD>::kKVStages;
  uint8_t q[kQBufs][kTileBytes];
  uint8_t dout[kQBufs][kTileBytes];
  uint8_t k[kKVStages][kTileBytes];
  uint8_t v[kKVStages][kTileBytes];
  uint64_t q_full[kQBufs], q_empty[kQBufs];
  uint64_t kv_full[kKVStages], kv_empty[kKVStages];
  uint64_t sdp_full, sdp_empty, ds_full[2], ds_free[2];
  uint64_t dq_full[Cfg<kD>::kDQBufs], dq_empty[Cfg<kD>::kDQBufs], drain;
  // dq staging: per softmax warp, its 32 rows x kD/2 columns (bf16), in the
  // swizzle of the TMA store that writes them (64 or 128 bytes per row)
  alignas(1024) uint8_t dqst[8][32 * kD];
  uint64_t sched_full[kSchedSlots], sched_empty[kSchedSlots];
  int32_t sched_unit[kSchedSlots];  // work unit handed out, -1 = no more work
  Unit sched_u[kSchedSlots];         // ... decoded by the producer
  uint32_t tmem_base;
  int abort;
};
template <int kD>
constexpr size_t smem_bytes() {
  return sizeof(Smem<kD>) + 1024;
}

__device__ __forceinline__ Unit decode(const Problem& p, const int2* items, int w) {
  const int2 it = items[w / p.Hq];
  Unit u;
  u.h = w % p.Hq;
  u.kvh = u.h / p.G;
  u.base = p.cu[it.x];
  u.L = p.cu[it.x + 1] - u.base;
  u.r0 = it.y * kTile;
  const int r1 = min(u.L, u.r0 + kTile);
  u.nrows = r1 - u.r0;
  int lo, hi;
  visible_keys(p.causal, p.window, u.L, u.r0, r1, &lo, &hi);
  u.kt0 = lo / kTile;
  u.kt1 = hi > lo ? (hi + kTile - 1) / kTile : u.kt0;
  return u;
}

// Wait that ignores the abort flag (still time-bounded): used only to drain
// copies / products this CTA issued before it exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) break;
}

template <int kD>
__global__ void __launch_bounds__(kThreads, 1)
dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
          const __grid_constant__ CUtensorMap tm_dqo, BwdProblem bp, const int2* __restrict__ items,
          int32_t* __restrict__ meta) {
  using C = Cfg<kD>;
  constexpr uint32_t kTileBytes = C::kTileBytes;
  constexpr int kQBufs = C::kQBufs, kKVStages = C::kKVStages, kDQBufs = C::kDQBufs;
  extern __shared__ uint8_t smem_raw[];
  Smem<kD>& sm = *reinterpret_cast<Smem<kD>*>(smem_raw + align1024_pad(smem_raw));
  const Problem& p = bp.f;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Guard g{&sm.abort, p.err, p.wait_limit_ns};

  if (threadIdx.x == 0) {
    sm.abort = 0;
    for (int s = 0; s < kQBufs; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.ds_full[s], kSoftmaxThreads);
      mbar_init(&sm.ds_free[s], 1);
    }
    for (int s = 0; s < kDQBufs; ++s) {
      mbar_init(&sm.dq_full[s], 1);
      mbar_init(&sm.dq_empty[s], kSoftmaxThreads);
    }
    for (int s = 0; s < kKVStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(&sm.sdp_full, 1);
    mbar_init(&sm.sdp_empty, kSoftmaxThreads);
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
  const int nwork = meta[0] * p.Hq;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t nq = 0, nkv = 0, nsched = 0;
      for (;;) {
        // take the next unit and publish it (or -1 when the list is exhausted)
        int w = atomicAdd(&meta[1], 1);
        if (w >= nwork) w = -1;
        Unit u{};
        if (w >= 0) u = decode(p, items, w);
        const int s = nsched % kSchedSlots;
        if (!mbar_wait(&sm.sched_empty[s], ((nsched / kSchedSlots) & 1) ^ 1, g)) break;
        sm.sched_unit[s] = w;
        sm.sched_u[s] = u;
        mbar_arrive(&sm.sched_full[s]);
        ++nsched;
        if (w < 0) break;
        if (p.withhold_copies) break;  // test hook: the consumers' waits run out
        const int qb = nq % kQBufs;
        if (!mbar_wait(&sm.q_empty[qb], ((nq / kQBufs) & 1) ^ 1, g)) break;
        mbar_expect_tx(&sm.q_full[qb], 2 * kTileBytes);
#pragma unroll
        for (int pi = 0; pi < C::kPanels; ++pi) {
          tma_load_3d(sm.q[qb] + pi * kPanelBytes, &tm_q, &sm.q_full[qb], 64 * pi, u.h, u.base + u.r0);
          tma_load_3d(sm.dout[qb] + pi * kPanelBytes, &tm_do, &sm.q_full[qb], 64 * pi, u.h, u.base + u.r0);
        }
        ++nq;
        bool ok = true;
        for (int kt = u.kt0; kt < u.kt1 && ok; ++kt) {
          const int st = nkv % kKVStages;
          if (!mbar_wait(&sm.kv_empty[st], ((nkv / kKVStages) & 1) ^ 1, g)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.kv_full[st], 2 * kTileBytes);
#pragma unroll
          for (int pi = 0; pi < C::kPanels; ++pi) {
            tma_load_3d(sm.k[st] + pi * kPanelBytes, &tm_k, &sm.kv_full[st], 64 * pi, u.kvh, u.base + kt * kTile);
            tma_load_3d(sm.v[st] + pi * kPanelBytes, &tm_v, &sm.kv_full[st], 64 * pi, u.kvh, u.base + kt * kTile);
          }
          ++nkv;
        }
        if (!ok) break;
      }
      if (g.aborted()) {  // let issued copies land before the CTA exits
        for (uint32_t c = nq > (uint32_t)kQBufs ? nq - kQBufs : 0; c < nq; ++c)
          drain_wait(&sm.q_full[c % kQBufs], (c / kQBufs) & 1);
        for (uint32_t c = nkv > kKVStages ? nkv - kKVStages : 0; c < nkv; ++c)
          drain_wait(&sm.kv_full[c % kKVStages], (c / kKVStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    // The whole warp runs this loop (uniform control flow and operands); one
    // elected lane issues each product and commit.
    const uint32_t idS = idesc_bf16(kTile, kTile, false, false);
    const uint32_t idQ = idesc_bf16(kTile, kD, false, true);
    // descriptors built once; a product adds its byte offset / 16
    const uint64_t dQ0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
    const uint64_t dO0 = sdesc_sw128(smem_u32(sm.dout[0]), 16, 1024);
    const uint64_t dK0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);       // K-major
    // MN-major: the 64-feature panels are kPanelBytes apart
    const uint64_t dKmn0 = sdesc_sw128(smem_u32(sm.k[0]), kPanelBytes, 1024);
    const uint64_t dV0 = sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);
    constexpr uint64_t kStageStep = kTileBytes >> 4;  // between stages of one array
    uint32_t nq = 0, nsdp = 0, nds = 0, nsched = 0;
    bool ok = true;
    // S and dP of the key tile in K / V stage c % kKVStages (the softmax must
    // have read the previous tile's)
    auto issue_sdp = [&](uint32_t qb, uint32_t c) -> bool {
      const int st = c % kKVStages;
      if (!mbar_wait_warp(&sm.kv_full[st], (c / kKVStages) & 1, g) ||
          !mbar_wait_warp(&sm.sdp_empty, (nsdp & 1) ^ 1, g))
        return false;
      ++nsdp;
      tc_fence_after();
      const uint64_t aq = dQ0 + qb * kStageStep, ao = dO0 + qb * kStageStep;
      const uint64_t bk = dK0 + st * kStageStep, bv = dV0 + st * kStageStep;
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) {  // +32 bytes per 16 features, panel by panel
        const uint64_t off = (uint64_t)(k / 4) * (kPanelBytes >> 4) + 2 * (k % 4);
        umma_ss_warp(tmem + kColS, aq + off, bk + off, idS, k > 0);
        umma_ss_warp(tmem + kColDP, ao + off, bv + off, idS, k > 0);
      }
      umma_commit_warp(&sm.sdp_full);
      return true;
    };
    // The units are one stream of (unit, key tile) steps: S / dP of the next
    // step -- the next unit's first tile at the end of a unit -- are issued
    // before dQ of the current one, so that a unit boundary leaves no gap in
    // the tensor pipe. fetch() returns 1 with the index of the next unit that
    // has key tiles (its Q / dO stage and dQ buffer are index % 2), 0 at the
    // end of the work, -1 on abort.  (Buffers: Q / dO index % kQBufs, dQ
    // index % kDQBufs.)
    auto fetch = [&](int& n, uint32_t& u) -> int {
      for (;;) {
        const int slot = nsched % kSchedSlots;
        if (!mbar_wait_warp(&sm.sched_full[slot], (nsched / kSchedSlots) & 1, g)) return -1;
        ++nsched;
        const int w = __shfl_sync(0xffffffffu, sm.sched_unit[slot], 0);  // warp-uniform
        n = __shfl_sync(0xffffffffu, sm.sched_u[slot].kt1 - sm.sched_u[slot].kt0, 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sched_empty[slot]);
        if (w < 0) return 0;
        u = nq++;
        if (!mbar_wait_warp(&sm.q_full[u % kQBufs], (u / kQBufs) & 1, g)) return -1;
        if (n > 0) return 1;
        // no key tile: nothing reads Q / dO, and dq is written as zero
        if (!mbar_wait_warp(&sm.dq_empty[u % kDQBufs], ((u / kDQBufs) & 1) ^ 1, g)) return -1;
        umma_commit_warp(&sm.q_empty[u % kQBufs]);
        umma_commit_warp(&sm.dq_full[u % kDQBufs]);
      }
    };
    // dQ of step jj of unit u (K / V load c): waits for dS, then 8 products
    auto dq_step = [&](uint32_t u, int jj, uint32_t c) -> bool {
      const int st = c % kKVStages, db = nds & 1;
      if (!mbar_wait_warp(&sm.ds_full[db], (nds >> 1) & 1, g)) return false;
      ++nds;
      tc_fence_after();
      const uint64_t bk = dKmn0 + st * kStageStep;
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k)  // dS from tensor memory; +2048 B of K per 16 keys
        umma_ts_warp(tmem + kColDQ + kD * (u % kDQBufs), tmem + kColDS + 64 * db + 8 * k, bk + 128 * k, idQ,
                     (jj > 0 || k > 0) ? 1u : 0u);
      umma_commit_warp(&sm.ds_free[db]);
      umma_commit_warp(&sm.kv_empty[st]);
      return true;
    };
    int n = 0;
    uint32_t u = 0, c = 0;  // c: K / V load of the current step
    int got = fetch(n, u);
    if (got > 0) {
      ok = issue_sdp(u % kQBufs, c);
      if (ok && n == 1) umma_commit_warp(&sm.q_empty[u % kQBufs]);  // last reader of Q / dO issued
    }
    while (got > 0 && ok) {
      // the unit's first dQ waits until the read-out of the unit that used
      // this accumulator before
      if (!mbar_wait_warp(&sm.dq_empty[u % kDQBufs], ((u / kDQBufs) & 1) ^ 1, g)) break;
      // every step but the last: S / dP of the next tile, then dQ of this one
      for (int jj = 0; jj + 1 < n && ok; ++jj, ++c) {
        ok = issue_sdp(u % kQBufs, c + 1);
        if (ok && jj + 2 == n) umma_commit_warp(&sm.q_empty[u % kQBufs]);
        if (ok) ok = dq_step(u, jj, c);
      }
      if (!ok) break;
      // the last step: the next unit's first S / dP go in before its dQ
      int n2 = 0;
      uint32_t u2 = 0;
      got = fetch(n2, u2);
      if (got < 0) break;
      if (got > 0) {
        if (!issue_sdp(u2 % kQBufs, c + 1)) break;
        if (n2 == 1) umma_commit_warp(&sm.q_empty[u2 % kQBufs]);
      }
      if (!dq_step(u, n - 1, c)) break;
      umma_commit_warp(&sm.dq_full[u % kDQBufs]);
      ++c;
      n = n2;
      u = u2;
    }
    umma_commit_warp(&sm.drain);  // every product issued above has completed
    if (lane == 0) drain_wait(&sm.drain, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int wg = (warp - 2) >> 2;  // key half of each tile, dq column half
    const int quarter = warp & 3;    // TMEM lanes 32 quarter .. 32 quarter + 31
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS + 64 * wg;
    const uint32_t tP = tmem + lane_off + kColDP + 64 * wg;
    const uint64_t sl2x2 = f2pack(p.scale_log2, p.scale_log2);
    uint32_t nsdp = 0, nds = 0, nunit = 0, nsched = 0;
    bool ok = true;
    // A unit's epilogue is deferred until this thread has formed dS of the
    // next unit's first key tile: by then the unit's last dQ product has
    // completed, and S / dP of the next unit were not kept waiting for it.
    // The pending unit's ring slot stays held until its epilogue.
    struct Pending {
      int64_t orow;  // output row (token * Hq + head)
      int slot;
      bool valid, any;
      int row0, h;   // the warp's first row (token) and the head, for its TMA store
    } pend{0, 0, false, false, 0, 0};
    uint8_t* stage = sm.dqst[warp - 2];
    bool has_pend = false;
    auto epilogue = [&]() -> bool {  // dq = bf16(scale * dQ), columns kD/2 wg .. kD/2 (wg + 1)
      constexpr int kHalf = kD / 2;
      const int dqb = nunit % kDQBufs;
      if (!mbar_wait_warp(&sm.dq_full[dqb], (nunit / kDQBufs) & 1, g)) return false;
      ++nunit;
      tc_fence_after();
      uint32_t a[kHalf];
      if constexpr (kHalf == 32)
        tmem_ld32(tmem + lane_off + kColDQ + kD * dqb + kHalf * wg, a);
      else
        tmem_ld64(tmem + lane_off + kColDQ + kD * dqb + kHalf * wg, a);
      tc_fence_before();
      mbar_arrive(&sm.dq_empty[dqb]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sched_empty[pend.slot]);  // the slot is no longer read
      const float sc = p.scale;  // dq = scale * sum_j dS_ij k_j
      uint32_t ob[kHalf / 2];
#pragma unroll
      for (int e = 0; e < kHalf / 2; ++e)
        ob[e] = pend.any ? pack_bf16(__uint_as_float(a[2 * e]) * sc, __uint_as_float(a[2 * e + 1]) * sc) : 0u;
      // rows through shared memory: a warp whose 32 rows all exist hands them
      // to one TMA store and goes on; a tail warp stores its valid rows itself
      constexpr int kChunks = kHalf / 8;  // 16-byte chunks per row: 4 or 8
      auto swz = [&](int row, int c) {    // the TMA swizzle of a row of kChunks 16-byte chunks
        return (uint32_t)(row * kChunks * 16) +
               ((uint32_t)(kChunks == 8 ? (c ^ (row & 7)) : (c ^ ((row >> 1) & 3))) << 4);
      };
      if (__all_sync(0xffffffffu, pend.valid)) {
        if (lane == 0) bulk_wait_read0();  // the previous store has read the staging rows
        __syncwarp();
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          *reinterpret_cast<uint4*>(stage + swz(lane, c)) = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_dqo, stage, kHalf * wg, pend.h, pend.row0);
          bulk_commit();
        }
      } else if (pend.valid) {
        uint4* dst = reinterpret_cast<uint4*>(bp.dq + pend.orow * kD + kHalf * wg);
#pragma unroll
        for (int c = 0; c < kChunks; ++c) dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
      }
      has_pend = false;
      return true;
    };
    while (ok) {
      const int slot = nsched % kSchedSlots;
      if (!mbar_wait_warp(&sm.sched_full[slot], (nsched / kSchedSlots) & 1, g)) break;
      ++nsched;
      if (sm.sched_unit[slot] < 0) break;  // no more work
      const volatile Unit& uv = sm.sched_u[slot];
      const int kt0 = uv.kt0, n = uv.kt1 - uv.kt0, L = uv.L;
      const int i = uv.r0 + r;
      const bool valid = r < uv.nrows;
      const int64_t roff = (int64_t)uv.h * p.total + uv.base + i;  // [Hq, total] row constants
      // rows past the tile's end get P = 0 (and are not written)
      const float nl2 = valid ? -__ldg(p.lse + roff) * kLog2e : -INFINITY;
      const float nd = valid ? -__ldg(bp.D + roff) : 0.f;
      const uint64_t nl2x2 = f2pack(nl2, nl2), ndx2 = f2pack(nd, nd);
      const int khi = p.causal ? min(i + 1, L) : L;
      const int klo = p.window > 0 ? max(0, i - p.window + 1) : 0;
      // one key tile: S / dP in, dS out
      auto tile = [&](int jj) -> bool {
        const int kb = (kt0 + jj) * kTile + 64 * wg;  // first key of this thread's half
        if (!mbar_wait_warp(&sm.sdp_full, nsdp & 1, g)) return false;
        ++nsdp;
        tc_fence_after();
        uint32_t sv[64], pv[64];
        tmem_ld64(tS, sv);
        tmem_ld64(tP, pv);
        tc_fence_before();
        mbar_arrive(&sm.sdp_empty);  // S / dP of the next tile may go in
        if (kb < klo || kb + 64 > khi) {
          // keys outside [klo, khi) get S = -inf (P = 0); one unsigned
          // compare and a select per element
          const int cl = klo - kb;
          const unsigned span = (unsigned)max(khi - klo, 0);
#pragma unroll
          for (int c = 0; c < 64; ++c)
            sv[c] = (unsigned)(c - cl) < span ? sv[c] : __float_as_uint(-INFINITY);
        }
        uint32_t ds[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x = f2unpack(ffma2(f2pack(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])),
                                          sl2x2, nl2x2));
          const uint64_t P = f2pack(ex2(x.x), ex2(x.y));
          const uint64_t t = fmul2(P, f2pack(__uint_as_float(pv[2 * c]), __uint_as_float(pv[2 * c + 1])));
          const float2 d = f2unpack(ffma2(P, ndx2, t));  // P dP - P D
          ds[c] = pack_bf16(d.x, d.y);
        }
        const int db = nds & 1;
        if (!mbar_wait_warp(&sm.ds_free[db], ((nds >> 1) & 1) ^ 1, g))  // dQ of tile jj - 2 done
          return false;
        ++nds;
        tc_fence_after();
        tmem_st32(tmem + lane_off + kColDS + 64 * db + 32 * wg, ds);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.ds_full[db]);
        return true;
      };
      // the previous unit's epilogue goes after the first tile (or at once
      // for a unit without key tiles)
      if (n > 0) ok = tile(0);
      if (ok && has_pend) ok = epilogue();
      for (int jj = 1; jj < n && ok; ++jj) ok = tile(jj);
      if (!ok) break;
      pend = Pending{(int64_t)(uv.base + i) * p.Hq + uv.h, slot, valid, n > 0,
                     uv.base + uv.r0 + 32 * quarter, uv.h};
      has_pend = true;
    }
    if (ok && has_pend) epilogue();  // the last unit
    if (lane == 0) bulk_wait0();     // this warp's dq stores are complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t prepare_bwd_dq(int head_dim) {
  if (head_dim == kHeadDimWide)
    return cudaFuncSetAttribute(dq_kernel<kHeadDimWide>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<kHeadDimWide>());
  return cudaFuncSetAttribute(dq_kernel<kHeadDim>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes<kHeadDim>());
}

cudaError_t launch_bwd_dq(const BwdProblem& p, const BwdLaunch& l, const TileList& qtiles,
                          int num_sms, cudaStream_t s) {
  const int64_t work = (int64_t)qtiles.capacity * p.f.Hq;
  const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms);
  if (grid <= 0) return cudaSuccess;
  if (p.f.head_dim == kHeadDimWide)
    dq_kernel<kHeadDimWide><<<grid, kThreads, smem_bytes<kHeadDimWide>(), s>>>(l.q, l.k, l.v, l.dout, l.dqo, p,
                                                                             qtiles.items, qtiles.meta);
  else
    dq_kernel<kHeadDim><<<grid, kThreads, smem_bytes<kHeadDim>(), s>>>(l.q, l.k, l.v, l.dout, l.dqo, p,
                                                                     qtiles.items, qtiles.meta);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
