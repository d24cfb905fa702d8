// Forward of sink attention on tcgen05 tensor cores: O and LSE.
//
// Online softmax over 128-key tiles, seeded with the sink: the running maximum
// starts at S_h and the running sum at exp(S_h - S_h) = 1, so the virtual
// token enters the denominator once and adds nothing to the output (page
// "GPT-OSS Agentic RL Training: A Practical Retrospective", section "The Role
// of Attention Sinks").
//
// One CTA owns one 128-row query tile of one head at a time (persistent;
// units are taken dynamically from the device-built tile list, longest first;
// the heads of a tile are consecutive work units, so a GQA group's K/V tiles
// are reused from L2). Two CTAs share an SM, which interleaves one CTA's softmax
// with the other's matrix products.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q tile, then K tiles (2-stage ring, one tile
//               ahead) and V tiles (2-stage ring); a K stage is released as
//               soon as S = Q K^T completes, a V stage after O += P V
//   warp 1      UMMA issuer: S = Q K^T (SS, K-major both) and O += P V (P from
//               tensor memory, V MN-major); S(j+1) is issued as soon as the
//               softmax has read S(j), so it overlaps softmax(j)
//   warps 2-5   softmax: one thread per query row (its TMEM lane); rescales O
//               only when the row maximum grows by more than 2^8; writes P as
//               bf16 into tensor memory; final O / l and LSE
// Tensor memory at head_dim 64 (256 columns, two CTAs per SM): S [0,128)
// fp32, P [128,192) bf16 pairs, O [192,256) fp32. At head_dim 128 (512
// columns, one CTA per SM): S [0,128), P [128,192), O [256,384). Q, K and V
// tiles are stored as 64-feature panels of 128-byte rows (one TMA copy and
// one 128-byte swizzle atom width each); a product over 128 features walks
// both panels.
//
// Decode instantiation (kDecode): one new query row per sequence against a
// paged KV cache, computed exactly as the training forward computes the last
// row of that sequence, so o and LSE agree with it bit for bit. A work unit is
// (sequence, kv head); its G query heads' rows sit in rows 0 .. G-1 of the
// query tile and all stand at position L - 1. The key tiles are the training
// forward's: 128 keys from the sequence start, in order, each loaded block by
// block from the cache; a block past the sequence end or wholly before the
// window is read out of bounds instead, which fills it with zeros (those keys
// are masked; the training forward sees finite keys there, so both add
// exact zeros), and value rows past the last key in its final block are
// zeroed before the P V product. The softmax and the products run the very
// same instructions as for a training row; a row's arithmetic does not depend
// on the other rows of its tile, nor on the tile's first key tile (the
// training forward may start one tile earlier with a fully masked tile, which
// adds exact zeros to O, the row sum and nothing to the maximum).
#include <algorithm>
#include <cmath>

#include "internal.h"
#include "sm100.cuh"

namespace sinkattn {
namespace {

using namespace sm100;

constexpr int kThreads = 192;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr uint32_t kPanelBytes = kTile * 64 * 2;  // 128 rows x 64 features of bf16
constexpr uint32_t kOPanelBytes = 32 * 128;        // O staging: 32 rows x 64 features of bf16
constexpr uint32_t kColS = 0, kColP = 128;
// per head dim: tile bytes, tensor-memory columns, O's column, CTAs per SM
template <int kD>
struct Cfg {
  static constexpr int kPanels = kD / 64;
  static constexpr uint32_t kTileBytes = kPanelBytes * kPanels;
  static constexpr uint32_t kTmemCols = kD == 64 ? 256 : 512;
  static constexpr uint32_t kColO = kD == 64 ? 192 : 256;
  static constexpr int kCtasPerSm = kD == 64 ? 2 : 1;
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;  // log2 units
constexpr int kSchedSlots = 4;
constexpr int kSchedConsumers = 1 + 4;  // the UMMA warp and 4 softmax warps
constexpr uint32_t kClearChunk = 4096;  // bytes of the backward's dq accumulator per copy

// Training: base = the sequence's first token, r0 = the tile's first row,
// nrows = rows in the tile, h = the query head. Decode: base = the sequence,
// r0 = L - 1 (every row's position), nrows = G, h = the group's first head.
struct Unit {
  int base, L, r0, nrows, h, kvh, kt0, kt1;
};

template <int kD>
struct __align__(1024) Smem {
  static constexpr uint32_t kTileBytes = Cfg<kD>::kTileBytes;
  uint8_t q[kTileBytes];
  uint8_t k[kKStages][kTileBytes];
  uint8_t v[kVStages][kTileBytes];
  uint8_t ostage[4][32 * kD * 2];  // per softmax warp: its 32 rows of O (bf16), 64-feature panels, swizzled
  uint8_t zeros[kClearChunk];   // source of the bulk copies that clear the backward's dq accumulator
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t q_full, q_empty, s_full, s_empty, p_full, o_done, drain;
  uint64_t sched_full[kSchedSlots], sched_empty[kSchedSlots];
  int32_t sched_unit[kSchedSlots];  // work unit handed out, -1 = no more work
  Unit sched_u[kSchedSlots];         // ... decoded by the producer
  float sched_sink[kSchedSlots];     // ... and its head's sink * log2(e) (-inf: none)
  uint32_t tmem_base;
  int abort;
};
template <int kD>
constexpr size_t smem_bytes() {
  return sizeof(Smem<kD>) + 1024;
}

// Decode: sequence w / Hkv, kv head w % Hkv, its keys [0, L) and the 128-key
// tiles the training forward's last row of the sequence would take.
__device__ __forceinline__ Unit decode_paged(const Problem& p, const PagedKV& kv, int w) {
  Unit u;
  u.base = w / p.Hkv;
  u.kvh = w % p.Hkv;
  u.h = u.kvh * p.G;
  u.nrows = p.G;
  int L = kv.seqlens[u.base];
  if (L < 0 || L > kv.max_blocks * kv.block_size) {
    atomicCAS(p.err, 0, 1 /* SINKATTN_ERR_INVALID_ARG */);
    L = 0;
  }
  u.L = L;
  u.r0 = L - 1;
  const int klo = p.window > 0 ? max(0, L - p.window) : 0;
  u.kt0 = klo / kTile;
  u.kt1 = (L + kTile - 1) / kTile;
  return u;
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
  u.kt1 = (hi + kTile - 1) / kTile;
  return u;
}

// Work units are handed out dynamically (longest first, from the device-built
// list): the producer thread takes the next index with an atomic, decodes it
// (the global loads of the tile list, cu_seqlens and the sink happen there,
// ahead of time) and publishes it in a small ring; the UMMA warp and the
// softmax warps read the ring in order. `lanes` = the calling lanes of the
// warp (all of them get the same verdict).
template <bool kDecode>
__device__ __forceinline__ Unit decode_unit(const Problem& p, const PagedKV& kv, const int2* items, int w) {
  if constexpr (kDecode)
    return decode_paged(p, kv, w);
  else
    return decode(p, items, w);
}

template <class SmemT>
__device__ __forceinline__ int next_unit(SmemT& sm, uint32_t& n, const Guard& g, bool arrive,
                                         unsigned lanes, Unit& u, float& sink2) {
  const int s = n % kSchedSlots;
  if (!__all_sync(lanes, mbar_wait(&sm.sched_full[s], (n / kSchedSlots) & 1, g))) return -1;
  const int w = __shfl_sync(lanes, sm.sched_unit[s], 0);  // warp-uniform
  u = sm.sched_u[s];
  sink2 = sm.sched_sink[s];
  __syncwarp(lanes);
  if (arrive) mbar_arrive(&sm.sched_empty[s]);
  ++n;
  return w;
}

// Bulk copy of shared memory to global memory (16-byte aligned, a multiple of
// 16 bytes), in the thread's bulk group; commit_group / wait_group below.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(gdst)),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { bulk_wait0(); }

// Wait that ignores the abort flag (still time-bounded): used only to drain
// copies / products this thread issued before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) break;
}

template <bool kDecode, int kD>
__global__ void __launch_bounds__(kThreads, Cfg<kD>::kCtasPerSm)
fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, Problem p,
           PagedKV kv, const int2* __restrict__ items, int32_t* __restrict__ meta) {
  static_assert(kD == 64 || kD == 128, "head_dim 64 or 128");
  using C = Cfg<kD>;
  constexpr uint32_t kTileBytes = C::kTileBytes;
  constexpr uint32_t kTmemCols = C::kTmemCols, kColO = C::kColO;
  extern __shared__ uint8_t smem_raw[];
  Smem<kD>& sm = *reinterpret_cast<Smem<kD>*>(smem_raw + align1024_pad(smem_raw));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Guard g{&sm.abort, p.err, p.wait_limit_ns};

  if (threadIdx.x == 0) {
    sm.abort = 0;
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_empty, 128);
    mbar_init(&sm.p_full, 128);
    mbar_init(&sm.o_done, 1);
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
  }
  if (!kDecode && p.clear) {  // the zero source of the clearing copies
    for (int i = threadIdx.x; i < (int)(kClearChunk / 16); i += kThreads)
      reinterpret_cast<uint4*>(sm.zeros)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();
  }
  __syncthreads();
  tc_fence_after();
  // broadcast so the compiler sees a warp-uniform value (UMMA operands)
  const uint32_t tmem = __shfl_sync(0xffffffffu, sm.tmem_base, 0);
  const int nwork = kDecode ? p.nseq * p.Hkv : meta[0] * p.Hq;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t nq = 0, nk = 0, nv = 0;
      // This CTA's share of the backward's dq accumulator, cleared a few
      // chunks per key-tile load (the forward leaves memory bandwidth unused)
      // and the rest after its last unit. The chunks per load come from the
      // key-tile loads a CTA can expect (the list's total cost x heads / CTAs),
      // so that short units (a narrow window) still spread the clear over
      // the whole kernel instead of leaving it to the end.
      int64_t clr = 0, clr_end = 0;
      int per_load = 1;
      if (!kDecode && p.clear) {
        const int64_t n16 = p.clear_bytes / 16;
        clr = n16 * blockIdx.x / gridDim.x * 16;
        clr_end = n16 * (blockIdx.x + 1) / gridDim.x * 16;
        const int64_t loads = (int64_t)meta[2] * p.Hq / gridDim.x;  // expected, this CTA
        const int64_t chunks = (clr_end - clr + kClearChunk - 1) / kClearChunk;
        // done by the last expected load (what a CTA with fewer loads leaves
        // goes after its last unit); at most 8 chunks per load
        per_load = (int)std::min<int64_t>(8, std::max<int64_t>(1, (chunks + loads - 1) / std::max<int64_t>(loads, 1)));
      }
      auto clear_some = [&]() {
        for (int r = 0; r < per_load && clr < clr_end; ++r) {
          const int64_t left = clr_end - clr;
          const uint32_t n = left < (int64_t)kClearChunk ? (uint32_t)left : kClearChunk;
          bulk_store(p.clear + clr, sm.zeros, n);
          clr += n;
        }
      };
      // a key tile: one copy, or (decode) one per cache block; a block past
      // the sequence end or wholly before the window is read out of bounds,
      // which fills it with zeros
      auto load_tile = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* bar, const Unit& u, int kt) {
        if constexpr (kDecode) {
          const int bs = kv.block_size;
          const int klo = p.window > 0 ? max(0, u.L - p.window) : 0;
          for (int i = 0; i < kTile / bs; ++i) {
            const int j0 = kt * kTile + i * bs;
            int row = kv.num_blocks * bs;  // the first row past the cache
            if (j0 < u.L && j0 + bs > klo) {
              const int pb = kv.block_table[(int64_t)u.base * kv.max_blocks + j0 / bs];
              if (pb >= 0 && pb < kv.num_blocks)
                row = pb * bs;
              else
                atomicCAS(p.err, 0, 1 /* SINKATTN_ERR_INVALID_ARG */);
            }
#pragma unroll
            for (int pi = 0; pi < C::kPanels; ++pi)
              tma_load_3d(dst + pi * kPanelBytes + i * bs * 128, map, bar, 64 * pi, u.kvh, row);
          }
        } else {
#pragma unroll
          for (int pi = 0; pi < C::kPanels; ++pi)
            tma_load_3d(dst + pi * kPanelBytes, map, bar, 64 * pi, u.kvh, u.base + kt * kTile);
        }
      };
      auto load_k = [&](const Unit& u, int kt) -> bool {
        const int s = nk % kKStages;
        if (!mbar_wait(&sm.k_empty[s], ((nk / kKStages) & 1) ^ 1, g)) return false;
        mbar_expect_tx(&sm.k_full[s], kTileBytes);
        load_tile(sm.k[s], &tm_k, &sm.k_full[s], u, kt);
        ++nk;
        clear_some();
        return true;
      };
      auto load_v = [&](const Unit& u, int kt) -> bool {
        const int s = nv % kVStages;
        if (!mbar_wait(&sm.v_empty[s], ((nv / kVStages) & 1) ^ 1, g)) return false;
        mbar_expect_tx(&sm.v_full[s], kTileBytes);
        load_tile(sm.v[s], &tm_v, &sm.v_full[s], u, kt);
        ++nv;
        return true;
      };
      uint32_t nsched = 0;
      for (;;) {
        // take the next unit and publish it (or -1 when the list is exhausted)
        int w = atomicAdd(&meta[1], 1);
        if (w >= nwork) w = -1;
        Unit u{};
        float sink2 = -INFINITY;
        if (w >= 0) {
          u = decode_unit<kDecode>(p, kv, items, w);
          if (p.sinks && !kDecode) sink2 = p.sinks[u.h] * kLog2e;
          if (kDecode && u.kt1 <= u.kt0) {
            // a sequence without keys: the sink alone, o = 0 and lse = S_h
            for (int r = 0; r < u.nrows; ++r) {
              uint4* dst = reinterpret_cast<uint4*>(p.o + ((int64_t)u.base * p.Hq + u.h + r) * kD);
              for (int c = 0; c < kD / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
              if (p.lse) p.lse[(int64_t)(u.h + r) * p.total + u.base] = p.sinks ? p.sinks[u.h + r] : -INFINITY;
            }
            continue;
          }
        }
        const int s = nsched % kSchedSlots;
        if (!mbar_wait(&sm.sched_empty[s], ((nsched / kSchedSlots) & 1) ^ 1, g)) break;
        sm.sched_unit[s] = w;
        sm.sched_u[s] = u;
        sm.sched_sink[s] = sink2;
        mbar_arrive(&sm.sched_full[s]);
        ++nsched;
        if (w < 0) break;
        if (p.withhold_copies) break;  // test hook: the consumers' waits run out
        if (!mbar_wait(&sm.q_empty, (nq & 1) ^ 1, g)) break;
        if (kDecode) {  // the G heads' rows of this sequence into rows 0 .. G-1
          mbar_expect_tx(&sm.q_full, (uint32_t)u.nrows * 128u * C::kPanels);
#pragma unroll
          for (int pi = 0; pi < C::kPanels; ++pi)
            tma_load_3d(sm.q + pi * kPanelBytes, &tm_q, &sm.q_full, 64 * pi, u.h, u.base);
        } else {
          mbar_expect_tx(&sm.q_full, kTileBytes);
#pragma unroll
          for (int pi = 0; pi < C::kPanels; ++pi)
            tma_load_3d(sm.q + pi * kPanelBytes, &tm_q, &sm.q_full, 64 * pi, u.h, u.base + u.r0);
        }
        ++nq;
        // K runs one tile ahead of V (S(j+1) is issued before P V(j))
        bool ok = load_k(u, u.kt0);
        for (int kt = u.kt0; kt < u.kt1 && ok; ++kt) {
          if (kt + 1 < u.kt1) ok = load_k(u, kt + 1);
          if (ok) ok = load_v(u, kt);
        }
        if (!ok) break;
      }
      if (!g.aborted())
        while (clr < clr_end) clear_some();
      bulk_wait_all();  // the clearing copies (this thread's own) are done
      if (g.aborted()) {  // let issued copies land before the CTA exits
        if (nq) drain_wait(&sm.q_full, (nq - 1) & 1);
        for (uint32_t c = nk > kKStages ? nk - kKStages : 0; c < nk; ++c)
          drain_wait(&sm.k_full[c % kKStages], (c / kKStages) & 1);
        for (uint32_t c = nv > kVStages ? nv - kVStages : 0; c < nv; ++c)
          drain_wait(&sm.v_full[c % kVStages], (c / kVStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    // The whole warp runs this loop (uniform control flow and operands); one
    // elected lane issues each product and commit.
    const uint32_t idS = idesc_bf16(kTile, kTile, false, false);
    const uint32_t idO = idesc_bf16(kTile, kD, false, true);
    // descriptors built once; a product adds its byte offset / 16. V is read
    // MN-major: its 64-feature panels are kPanelBytes apart.
    const uint64_t dQ = sdesc_sw128(smem_u32(sm.q), 16, 1024);
    const uint64_t dK0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
    const uint64_t dV0 = sdesc_sw128(smem_u32(sm.v[0]), kPanelBytes, 1024);
    constexpr uint64_t kStageStep = kTileBytes >> 4;  // k[1] - k[0], v[1] - v[0]
    uint32_t nq = 0, nk = 0, ns = 0, np = 0;
    bool ok = true;
    // S of the next key tile (K stage released when it completes)
    auto next_s = [&]() -> bool {
      const int s = nk % kKStages;
      if (!mbar_wait_warp(&sm.k_full[s], (nk / kKStages) & 1, g) ||
          !mbar_wait_warp(&sm.s_empty, (ns & 1) ^ 1, g))
        return false;
      ++ns;
      tc_fence_after();
      const uint64_t bk = dK0 + s * kStageStep;
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) {  // +32 bytes per 16 features, panel by panel
        const uint64_t off = (uint64_t)(k / 4) * (kPanelBytes >> 4) + 2 * (k % 4);
        umma_ss_warp(tmem + kColS, dQ + off, bk + off, idS, k > 0);
      }
      umma_commit_warp(&sm.s_full);
      umma_commit_warp(&sm.k_empty[s]);
      ++nk;
      return true;
    };
    uint32_t nsched = 0;
    while (ok) {
      Unit u;
      float sink2;
      const int w = next_unit(sm, nsched, g, lane == 0, 0xffffffffu, u, sink2);
      if (w < 0) break;
      const int n = __shfl_sync(0xffffffffu, u.kt1 - u.kt0, 0);  // warp-uniform trip count
      if (!mbar_wait_warp(&sm.q_full, nq & 1, g)) break;
      ++nq;
      if (!next_s()) break;
      if (n == 1) umma_commit_warp(&sm.q_empty);
      for (int jj = 0; jj < n; ++jj) {
        if (jj + 1 < n) {
          if (!next_s()) {
            ok = false;
            break;
          }
          if (jj + 2 == n) umma_commit_warp(&sm.q_empty);
        }
        const int sv = np % kVStages;
        if (!mbar_wait_warp(&sm.p_full, np & 1, g) ||
            !mbar_wait_warp(&sm.v_full[sv], (np / kVStages) & 1, g)) {
          ok = false;
          break;
        }
        ++np;
        if constexpr (kDecode) {
          // value rows past the sequence's last key (cache slots never
          // written) are zeroed, as the training forward's are finite there
          const int rs = u.L - (u.kt0 + jj) * kTile;
          if (rs < kTile) {
            for (int e = lane; e < (kTile - rs) * 8 * C::kPanels; e += 32) {
              const int pi = e / ((kTile - rs) * 8), f = e % ((kTile - rs) * 8);
              *reinterpret_cast<uint4*>(sm.v[sv] + pi * kPanelBytes + (rs + f / 8) * 128 + (f % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_async_smem();
            __syncwarp();
          }
        }
        tc_fence_after();
        const uint64_t bv = dV0 + sv * kStageStep;
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)  // P from tensor memory; +2048 B of V per 16 keys
          umma_ts_warp(tmem + kColO, tmem + kColP + 8 * k, bv + 128 * k, idO, (jj > 0 || k > 0) ? 1u : 0u);
        umma_commit_warp(&sm.v_empty[sv]);
        umma_commit_warp(&sm.o_done);
      }
    }
    umma_commit_warp(&sm.drain);  // every product issued above has completed
    if (lane == 0) drain_wait(&sm.drain, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS, tP = tmem + lane_off + kColP,
                   tO = tmem + lane_off + kColO;
    const float sl2 = p.scale_log2;
    uint32_t nsf = 0, nod = 0, nsched = 0;
    bool ok = true;
    while (ok) {
      // the ring slot stays held until the epilogue, and the unit's fields
      // are read from it where they are used (no registers held across the
      // tile loop)
      const int slot = nsched % kSchedSlots;
      if (!mbar_wait_warp(&sm.sched_full[slot], (nsched / kSchedSlots) & 1, g)) break;
      ++nsched;
      if (sm.sched_unit[slot] < 0) break;  // no more work
      const volatile Unit& uv = sm.sched_u[slot];
      const int kt0 = uv.kt0;
      const int n = uv.kt1 - kt0;
      // decode: every row stands at L - 1, row r is head h + r with its own sink
      const float sink2 = kDecode ? (p.sinks && r < uv.nrows ? __ldg(p.sinks + uv.h + r) * kLog2e : -INFINITY)
                                  : sm.sched_sink[slot];
      const int i = kDecode ? uv.r0 : uv.r0 + r;
      const int L = uv.L;
      const int khi = p.causal ? min(i + 1, L) : L;
      const int klo = p.window > 0 ? max(0, i - p.window + 1) : 0;
      float m = sink2;  // -inf without sinks
      float l = p.sinks ? 1.f : 0.f;
      for (int jj = 0; jj < n; ++jj) {
        const int c0 = (kt0 + jj) * kTile;
        if (!mbar_wait_warp(&sm.s_full, nsf & 1, g)) {
          ok = false;
          break;
        }
        ++nsf;
        tc_fence_after();
        float s[kTile];
        {
          uint32_t v[kTile];
          tmem_ld128(tS, v);
#pragma unroll
          for (int e = 0; e < kTile; ++e) s[e] = __uint_as_float(v[e]);
        }
        tc_fence_before();
        mbar_arrive(&sm.s_empty);
        if (c0 < klo || c0 + kTile > khi) {
          // keys outside [cl, ch) get -inf; one unsigned compare and a select
          // per element, no branches
          const int cl = klo - c0;
          const unsigned span = (unsigned)max(khi - klo, 0);
#pragma unroll
          for (int c = 0; c < kTile; ++c) s[c] = (unsigned)(c - cl) < span ? s[c] : -INFINITY;
        }
        // row maximum with three-input max (two new values per instruction)
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < kTile; c += 8) {
          mx0 = fmax3(mx0, s[c], s[c + 1]);
          mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
          mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
          mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
        }
        const float m_new = fmaxf(m, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2);
        // lazy rescale: keep the stale maximum unless it grew by > 2^8
        const bool resc = m_new > m + kRescale;
        const float alpha = resc ? ex2(m - m_new) : 1.f;
        if (resc) {
          l *= alpha;
          m = m_new;
        }
        const float msub = m == -INFINITY ? 0.f : m;
        uint64_t sumv = f2pack(0.f, 0.f);  // (even, odd) columns, two lanes per instruction
        uint32_t pa[32], pb[32];
#pragma unroll
        for (int c = 0; c < kTile / 2; ++c) {
          const float2 x = f2unpack(ffma2(f2pack(s[2 * c], s[2 * c + 1]), f2pack(sl2, sl2), f2pack(-msub, -msub)));
          const float p0 = ex2(x.x);
          const float p1 = ex2(x.y);
          sumv = fadd2(sumv, f2pack(p0, p1));
          if (c < 32)
            pa[c] = pack_bf16(p0, p1);
          else
            pb[c - 32] = pack_bf16(p0, p1);
        }
        {
          const float2 sv2 = f2unpack(sumv);
          l += sv2.x + sv2.y;
        }
        if (jj > 0) {
          // PV(jj-1) must be complete: it reads P and accumulates into O
          if (!mbar_wait_warp(&sm.o_done, nod & 1, g)) {
            ok = false;
            break;
          }
          ++nod;
          tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {  // O holds this unit's partial sum
#pragma unroll
            for (int c0 = 0; c0 < kD; c0 += 64) {
              uint32_t v[64];
              tmem_ld64(tO + c0, v);
              uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
              uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
#pragma unroll
              for (int e = 0; e < 64; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
              tmem_st32(tO + c0, v0);
              tmem_st32(tO + c0 + 32, v1);
            }
          }
        }
        tmem_st32(tP, pa);
        tmem_st32(tP + 32, pb);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full);
      }
      if (!ok) break;
      // epilogue: O / l, LSE
      if (!mbar_wait_warp(&sm.o_done, nod & 1, g)) break;
      ++nod;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t ob[kD / 2];
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 64) {
        uint32_t v[64];
        tmem_ld64(tO + c0, v);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          ob[c0 / 2 + e] = pack_bf16(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
      }
      const int nrows = uv.nrows, row0 = uv.base + uv.r0, h = uv.h;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sched_empty[slot]);  // the slot is no longer read
      if constexpr (kDecode) {  // row r: sequence base, head h + r
        const int b = row0 - uv.r0;
        if (r < nrows) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + ((int64_t)b * p.Hq + h + r) * kD);
#pragma unroll
          for (int c = 0; c < kD / 8; ++c) dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
          if (p.lse) p.lse[(int64_t)(h + r) * p.total + b] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
        }
        continue;
      }
      // O rows through shared memory, as 64-feature panels of 32 rows x 128
      // bytes in the 128-byte swizzle TMA uses. A warp whose 32 rows all
      // belong to the sequence hands them to one asynchronous TMA store per
      // panel and goes on to its next unit; a warp with rows past the
      // sequence end (they are the next sequence's) stores its valid rows
      // itself, four whole rows per instruction.
      constexpr int kChunks = kD / 8;
      uint8_t* ost = sm.ostage[quarter];
      if (lane == 0) bulk_wait_read0();  // this warp's previous store has read the staging rows
      __syncwarp();
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
        *reinterpret_cast<uint4*>(ost + (c / 8) * kOPanelBytes + lane * 128 + (((c % 8) ^ (lane & 7)) << 4)) =
            make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
      if (32 * quarter + 31 < nrows) {
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int pi = 0; pi < C::kPanels; ++pi)
            tma_store_3d(&tm_o, ost + pi * kOPanelBytes, 64 * pi, h, row0 + 32 * quarter);
          bulk_commit();
        }
      } else {
        __syncwarp();
#pragma unroll
        for (int pi = 0; pi < C::kPanels; ++pi) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + (lane >> 3), c = lane & 7;  // row of this warp, 16-byte chunk
            const uint4 x = *reinterpret_cast<const uint4*>(ost + pi * kOPanelBytes + rr * 128 + ((c ^ (rr & 7)) << 4));
            if (32 * quarter + rr < nrows)
              reinterpret_cast<uint4*>(p.o + ((int64_t)(row0 + 32 * quarter + rr) * p.Hq + h) * kD)[8 * pi + c] = x;
          }
        }
        __syncwarp();
      }
      if (p.lse && r < nrows)
        p.lse[(int64_t)h * p.total + row0 + r] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
    if (lane == 0) bulk_wait_all();  // this warp's O stores are complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t prepare_fwd(const Problem& p, FwdLaunch* l) {
  const int d = p.head_dim;
  cudaError_t e = make_tmap_bf16_rows(&l->q, p.q, p.Hq, p.total, p.q_stride, kTile, d);
  if (e == cudaSuccess) e = make_tmap_bf16_rows(&l->k, p.k, p.Hkv, p.total, p.k_stride, kTile, d);
  if (e == cudaSuccess) e = make_tmap_bf16_rows(&l->v, p.v, p.Hkv, p.total, p.v_stride, kTile, d);
  if (e == cudaSuccess) e = make_tmap_bf16_rows(&l->o, p.o, p.Hq, p.total, (int64_t)p.Hq * d, 32, d);
  if (e != cudaSuccess) return e;
  if (d == 128)
    return cudaFuncSetAttribute(fwd_kernel<false, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<128>());
  return cudaFuncSetAttribute(fwd_kernel<false, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes<64>());
}

cudaError_t launch_fwd(const Problem& p, const FwdLaunch& l, const TileList& qtiles, int num_sms,
                       cudaStream_t s) {
  const int64_t work = (int64_t)qtiles.capacity * p.Hq;
  const int per_sm = p.head_dim == 128 ? Cfg<128>::kCtasPerSm : Cfg<64>::kCtasPerSm;
  const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms * per_sm);
  if (grid <= 0) return cudaSuccess;
  if (p.head_dim == 128)
    fwd_kernel<false, 128><<<grid, kThreads, smem_bytes<128>(), s>>>(l.q, l.k, l.v, l.o, p, PagedKV{},
                                                                     qtiles.items, qtiles.meta);
  else
    fwd_kernel<false, 64><<<grid, kThreads, smem_bytes<64>(), s>>>(l.q, l.k, l.v, l.o, p, PagedKV{},
                                                                   qtiles.items, qtiles.meta);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_decode_exact(const Problem& p, const PagedKV& kv, const void* k_cache,
                                const void* v_cache, int32_t* counter, int num_sms, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  const int rows = kv.num_blocks * kv.block_size;
  const int d = p.head_dim;
  cudaError_t e = make_tmap_bf16_heads(&mq, p.q, p.Hq, p.nseq, p.G, d);
  if (e == cudaSuccess)
    e = make_tmap_bf16_rows(&mk, k_cache, p.Hkv, rows, (int64_t)p.Hkv * d, kv.block_size, d);
  if (e == cudaSuccess)
    e = make_tmap_bf16_rows(&mv, v_cache, p.Hkv, rows, (int64_t)p.Hkv * d, kv.block_size, d);
  if (e == cudaSuccess)
    e = d == 128 ? cudaFuncSetAttribute(fwd_kernel<true, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem_bytes<128>())
                 : cudaFuncSetAttribute(fwd_kernel<true, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem_bytes<64>());
  if (e == cudaSuccess) e = cudaMemsetAsync(counter, 0, 2 * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  const int64_t work = (int64_t)p.nseq * p.Hkv;
  const int per_sm = d == 128 ? Cfg<128>::kCtasPerSm : Cfg<64>::kCtasPerSm;
  const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms * per_sm);
  if (grid <= 0) return cudaSuccess;
  // (the decode form writes its rows itself: the O map argument is unused)
  if (d == 128)
    fwd_kernel<true, 128><<<grid, kThreads, smem_bytes<128>(), s>>>(mq, mk, mv, mq, p, kv, nullptr, counter);
  else
    fwd_kernel<true, 64><<<grid, kThreads, smem_bytes<64>(), s>>>(mq, mk, mv, mq, p, kv, nullptr, counter);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
