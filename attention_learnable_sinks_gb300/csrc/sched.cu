// Varlen tile scheduler: builds, on the device, the list of 128-row query
// tiles (forward) or 128-key key tiles (backward) of a packed batch, so that
// persistent CTAs taking items in order approximate a longest-processing-time-
// first schedule. Building on the device keeps the whole call asynchronous (no
// host copy of cu_seqlens, no stream sync).
//
// Cost of a query tile = number of key tiles it sees; cost of a key tile =
// number of query tiles that see it. Both follow from the causal / window
// mask and the sequence length.
//
// Two orders:
//   by cost           decreasing cost over the whole batch (the default)
//   sequence-major    sequence 0's tiles, then sequence 1's, ..., each
//                     sequence's by decreasing cost. Used for the backward
//                     when its fp32 dq accumulator is far larger than L2: the
//                     running units then cover one or two sequences, whose
//                     accumulator rows and Q / dO tiles stay in L2, instead of
//                     every sequence at once (on the 32-sequence varlen batch
//                     the backward main kernel took 17.5 ms instead of 24.6).
//                     When the batch has more sequences than the bucket table
//                     separates, the later ones share the last bucket.
#include "internal.h"

namespace sinkattn {
namespace {

constexpr int kBuckets = 4096;   // cost buckets; larger costs share the last
constexpr int kThreads = 1024;

__device__ inline int tile_cost(int by_keys, int causal, int window, int L, int t) {
  const int a = t * kTile;
  const int b = min(L, a + kTile);
  int lo, hi;
  if (by_keys)
    seeing_rows(causal, window, L, a, b, &lo, &hi);
  else
    visible_keys(causal, window, L, a, b, &lo, &hi);
  if (hi <= lo) return 0;
  return (hi + kTile - 1) / kTile - lo / kTile;
}

// Bucket of a tile: buckets are handed out from the highest index down.
__device__ inline int bucket_of(int seq_major, int levels, int b, int cost) {
  if (!seq_major) return min(cost, kBuckets - 1);
  const int key = b * levels + (levels - 1 - min(cost, levels - 1));
  return kBuckets - 1 - min(key, kBuckets - 1);
}

// One list to build: which tiles, in which order, where.
struct ListJob {
  int by_keys, seq_major, capacity;
  int2* items;
  int32_t* meta;
};

// One CTA per list (a forward can build the backward's key-tile list with its
// own query-tile list, in the same launch).
__global__ void __launch_bounds__(kThreads)
build_tile_list_kernel(const int32_t* __restrict__ cu, int nseq, int total, int max_seqlen,
                       int causal, int window, ListJob job0, ListJob job1,
                       int32_t* __restrict__ err) {
  const ListJob& job = blockIdx.x == 0 ? job0 : job1;
  const int by_keys = job.by_keys, seq_major = job.seq_major, capacity = job.capacity;
  int2* __restrict__ items = job.items;
  int32_t* __restrict__ meta = job.meta;
  // cost levels per sequence in sequence-major order
  const int levels = seq_major ? max(1, kBuckets / max(nseq, 1)) : 1;
  __shared__ int hist[kBuckets];
  __shared__ int warp_sums[kThreads / 32];
  __shared__ int bad;
  __shared__ unsigned long long total_cost;
  const int tid = threadIdx.x;
  for (int i = tid; i < kBuckets; i += kThreads) hist[i] = 0;
  if (tid == 0) {
    bad = (nseq >= 0 && (cu[0] != 0 || cu[nseq] != total)) ? 1 : 0;
    total_cost = 0ull;
  }
  __syncthreads();

  // pass 1: validate lengths, histogram of costs; a warp per sequence, its
  // lanes over the sequence's tiles
  const int lane = tid & 31, warp = tid >> 5;
  for (int b = warp; b < nseq; b += kThreads / 32) {
    const int L = cu[b + 1] - cu[b];
    if (L < 0 || L > max_seqlen) {
      if (lane == 0) atomicOr(&bad, 1);
      continue;
    }
    const int nt = (L + kTile - 1) / kTile;
    unsigned long long cost_sum = 0ull;
    for (int t = lane; t < nt; t += 32) {
      const int cost = tile_cost(by_keys, causal, window, L, t);
      atomicAdd(&hist[bucket_of(seq_major, levels, b, cost)], 1);
      cost_sum += (unsigned long long)cost;
    }
    // one shared-memory add per warp (every lane adding its own costs a
    // measurable few microseconds of contention)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cost_sum += __shfl_xor_sync(0xffffffffu, cost_sum, o);
    if (lane == 0 && cost_sum) atomicAdd(&total_cost, cost_sum);
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      meta[0] = 0;
      meta[1] = 0;
      meta[2] = 0;
      atomicCAS(err, 0, 1 /* SINKATTN_ERR_INVALID_ARG */);
    }
    return;
  }

  // exclusive scan in order of decreasing bucket: thread t owns the four
  // buckets kBuckets-1-4t ... kBuckets-4-4t
  constexpr int kPer = kBuckets / kThreads;
  int local[kPer];
  int sum = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    local[e] = hist[kBuckets - 1 - (tid * kPer + e)];
    sum += local[e];
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    warp_sums[lane] = wi - w;  // exclusive prefix of the warps
  }
  __syncthreads();
  int run = warp_sums[warp] + incl - sum;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    hist[kBuckets - 1 - (tid * kPer + e)] = run;  // start offset of the bucket
    run += local[e];
  }
  __shared__ int n_items;
  if (tid == kThreads - 1) n_items = run;
  __syncthreads();
  if (n_items > capacity) {
    if (tid == 0) {
      meta[0] = 0;
      meta[1] = 0;
      meta[2] = 0;
      atomicCAS(err, 0, 4 /* SINKATTN_ERR_WORKSPACE */);
    }
    return;
  }

  // pass 2: scatter items into their buckets (order inside a bucket is free)
  for (int b = warp; b < nseq; b += kThreads / 32) {
    const int L = cu[b + 1] - cu[b];
    const int nt = (L + kTile - 1) / kTile;
    for (int t = lane; t < nt; t += 32) {
      const int c = bucket_of(seq_major, levels, b, tile_cost(by_keys, causal, window, L, t));
      const int pos = atomicAdd(&hist[c], 1);
      items[pos] = make_int2(b, t);
    }
  }
  if (tid == 0) {
    meta[0] = n_items;
    meta[1] = 0;
    // total cost (key tiles seen by the query tiles, or query tiles seeing
    // the key tiles): the forward paces its clearing copies by it
    meta[2] = (int32_t)min(total_cost, 0x7fffffffull);
  }
}

}  // namespace

cudaError_t launch_build_tile_list(const Problem& p, int by_keys, int seq_major,
                                   const TileList& list, cudaStream_t s, const TileList* keys,
                                   int keys_seq_major) {
  const ListJob a{by_keys, seq_major, list.capacity, list.items, list.meta};
  const ListJob b = keys ? ListJob{1, keys_seq_major, keys->capacity, keys->items, keys->meta} : a;
  build_tile_list_kernel<<<keys ? 2 : 1, kThreads, 0, s>>>(p.cu, p.nseq, p.total, p.max_seqlen,
                                                           p.causal, p.window, a, b, p.err);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sinkattn
