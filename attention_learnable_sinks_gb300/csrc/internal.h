// Internal declarations shared by the translation units of libsinkattn.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>
#include <string>

namespace sinkattn {

constexpr int kHeadDim = 64;      // the head dim of decode and of the fp32 dq accumulator path
constexpr int kHeadDimWide = 128; // the other head dim of the forward and backward
constexpr int kTile = 128;  // rows per query tile and keys per key tile

// One problem as the kernels see it. Strides are in elements per token row.
struct Problem {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* sinks;          // null: no sink
  const int32_t* cu;           // device cu_seqlens
  __nv_bfloat16* o;
  float* lse;                  // [Hq, total]
  int64_t q_stride, k_stride, v_stride;
  int32_t nseq, total, max_seqlen, Hq, Hkv, G, causal, window;
  int32_t head_dim;            // 64 or 128
  float scale;                 // softmax scale
  float scale_log2;            // scale * log2(e)
  int32_t* err;                // device error word
  uint64_t wait_limit_ns;      // time limit of every wait inside the kernels
  int32_t withhold_copies;     // test hook: producers issue no copies (the
                               // consumers' waits run out)
  uint8_t* clear;              // forward: bytes to clear for the backward (or null)
  int64_t clear_bytes;         // a multiple of 16
};

struct BwdProblem {
  Problem f;
  const __nv_bfloat16* dout;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dsinks;
  float* D;                    // [Hq, total] workspace: rowsum(dO * O)
  float* sink_part;            // [Hq, part_stride, 8] workspace: per key tile
                               // (numbered b + (cu[b] + c0) / 128) and softmax
                               // warp, sum of p_sink * P * dP
  float* dq_acc;               // [total, Hq, 64] fp32 workspace (head_dim 64, atomic mode)
  int32_t nchunks;             // token chunks of the preprocess pass
  int32_t part_stride;         // key-tile capacity
  int32_t accumulate_dsinks;   // add to dsinks instead of overwriting it
  int32_t deterministic;       // dq from the query-stationary pass (no dq_acc);
                               // always set at head_dim 128
  int32_t acc_cleared;         // the forward cleared dq_acc: the preprocess skips it
};

// Decode over a paged KV cache, as the kernels see it.
struct DecodeProblem {
  const __nv_bfloat16* q;        // [nseq, Hq, head_dim]
  const __nv_bfloat16* k_cache;  // [num_blocks, block_size, Hkv, head_dim]
  const __nv_bfloat16* v_cache;
  const int32_t* block_table;    // [nseq, max_blocks]
  const int32_t* seqlens;        // [nseq]
  const float* sinks;            // null: no sink
  __nv_bfloat16* o;              // [nseq, Hq, head_dim]
  float* lse;                    // [Hq, nseq] or null
  float* part_ml;                // [nseq, Hq, nsplit, 2] workspace: running max (log2 units), sum
  float* part_o;                 // [nseq, Hq, nsplit, head_dim] workspace: unnormalised output
  int32_t nseq, num_blocks, block_size, max_blocks, Hq, Hkv, window;
  int32_t head_dim;              // 64 or 128
  int32_t nsplit;                // splits per sequence (grid x)
  int32_t split_chunks;          // 128-key chunks per split
  float scale_log2;              // softmax scale * log2(e)
  int32_t* err;                  // device error word
  uint64_t wait_limit_ns;        // time limit of every wait inside the kernels
  int32_t withhold_copies;       // test hook: the split kernel issues no copies
};

// The paged KV cache of the exact decode (the forward kernel's decode
// instantiation): keys of sequence b, logical block i are physical block
// block_table[b * max_blocks + i] of [num_blocks, block_size, Hkv, 64].
struct PagedKV {
  const int32_t* block_table;
  const int32_t* seqlens;
  int32_t num_blocks, block_size, max_blocks;
};

// Tile work list in the workspace: meta[0] = number of items, meta[1] = the
// next item to hand out (work stealing), meta[2] = the items' total cost,
// items[] = {sequence, tile} sorted by decreasing cost.
struct TileList {
  int32_t* meta;
  int2* items;
  int32_t capacity;
};

// Upper bound on the number of 128-row (or 128-key) tiles of a packing.
inline int32_t tile_capacity(int32_t nseq, int32_t total) {
  return (total + kTile - 1) / kTile + nseq;
}

// Keys visible from any row in [r0, r1) of a sequence of length L.
__host__ __device__ inline void visible_keys(int causal, int window, int L, int r0, int r1,
                                             int* lo, int* hi) {
  *hi = causal ? (r1 < L ? r1 : L) : L;
  int l = window > 0 ? r0 - window + 1 : 0;
  *lo = l > 0 ? l : 0;
}

// Rows that see any key in [c0, c1) of a sequence of length L.
__host__ __device__ inline void seeing_rows(int causal, int window, int L, int c0, int c1,
                                            int* lo, int* hi) {
  *lo = causal ? c0 : 0;
  int h = window > 0 ? c1 - 1 + window : L;
  *hi = h < L ? h : L;
}

// TMA descriptor for a bf16 [total, heads, head_dim] token-major tensor (row
// stride in elements): 3-D {head_dim, heads, total}, 128-byte swizzle, box
// {64, 1, box_rows}: one 64-feature panel (128-byte rows) per copy, so a
// head_dim 128 tile takes two copies, at feature 0 and 64.
cudaError_t make_tmap_bf16_rows(CUtensorMap* map, const void* base, int heads, int total,
                                int64_t row_stride, int box_rows = kTile, int head_dim = kHeadDim);

// TMA descriptor for a contiguous bf16 [rows, heads, head_dim] tensor read as
// boxes of 64 features of box_heads consecutive heads of one row: 3-D
// {head_dim, heads, rows}, 128-byte swizzle, box {64, box_heads, 1}.
cudaError_t make_tmap_bf16_heads(CUtensorMap* map, const void* base, int heads, int rows,
                                 int box_heads, int head_dim = kHeadDim);

// TMA descriptor for a bf16 [total, heads, head_dim] tensor with a box of
// box_rows tokens x box_inner features of one head and a swizzle of
// box_inner * 2 bytes (64 or 128).
cudaError_t make_tmap_bf16_box(CUtensorMap* map, const void* base, int heads, int total, int64_t row_stride,
                               int head_dim, int box_inner, int box_rows);

// TMA descriptor for the fp32 [total, heads, 64] dq accumulator (contiguous):
// 3-D {64, heads, total}, 128-byte swizzle, box {32, 1, 32}.
cudaError_t make_tmap_f32_rows(CUtensorMap* map, void* base, int heads, int total);

// Launchers (each returns the cudaGetLastError() of its launch).
// seq_major: sequence by sequence, each by decreasing cost (else by decreasing
// cost over the whole batch). keys (optional): a key-tile list to build in
// the same launch, in order keys_seq_major (the backward's, built by the
// forward).
cudaError_t launch_build_tile_list(const Problem& p, int by_keys, int seq_major,
                                   const TileList& list, cudaStream_t s,
                                   const TileList* keys = nullptr, int keys_seq_major = 0);
// Tensor maps and kernel attributes are prepared before a call's first
// launch, so that its kernels go out back to back (host-side preparation
// between two launches would leave the GPU idle).
struct FwdLaunch {
  CUtensorMap q, k, v, o;  // o: boxes of 32 rows x 64 features (the epilogue's TMA stores)
};
struct BwdLaunch {
  CUtensorMap q, k, v, dout, dq;
  CUtensorMap dqo;  // bf16 dq, boxes of 32 rows x head_dim / 2 (the dq pass's TMA stores)
};
cudaError_t prepare_fwd(const Problem& p, FwdLaunch* l);
cudaError_t prepare_bwd_main(const BwdProblem& p, BwdLaunch* l);
cudaError_t launch_fwd(const Problem& p, const FwdLaunch& l, const TileList& qtiles, int num_sms,
                       cudaStream_t s);
// Exact decode: p describes nseq query rows [nseq, Hq, head_dim] (q, o, lse [Hq, nseq],
// sinks, window, scale); the keys come from kv. counter: one int of device
// memory, zeroed here before the launch (work stealing).
cudaError_t launch_decode_exact(const Problem& p, const PagedKV& kv, const void* k_cache,
                                const void* v_cache, int32_t* counter, int num_sms, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const BwdProblem& p, cudaStream_t s);
cudaError_t launch_bwd_main(const BwdProblem& p, const BwdLaunch& l, const TileList& ktiles,
                            int num_sms, cudaStream_t s);
cudaError_t launch_bwd_finish(const BwdProblem& p, const TileList& ktiles, int num_sms,
                              cudaStream_t s);
// Deterministic dq: query-stationary pass over the query-tile list, on the
// main kernel's Q / K / V / dO tensor maps.
cudaError_t prepare_bwd_dq(int head_dim);
cudaError_t launch_bwd_dq(const BwdProblem& p, const BwdLaunch& l, const TileList& qtiles,
                          int num_sms, cudaStream_t s);
// head_dim 128: dK / dV by the key-stationary kernel over 64-row query blocks
// (dq from the query-stationary pass). Its Q / dO maps copy 64-row boxes.
struct BwdWideLaunch {
  CUtensorMap q64, k, v, dout64;
};
cudaError_t prepare_bwd_wide(const BwdProblem& p, BwdWideLaunch* l);
cudaError_t launch_bwd_wide(const BwdProblem& p, const BwdWideLaunch& l, const TileList& ktiles,
                            int num_sms, cudaStream_t s);

size_t decode_workspace_bytes(int32_t nseq, int32_t Hq, int32_t nsplit, int32_t head_dim);
cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t s);

// The limit of the waits inside kernels and the copy-withholding test hook,
// as set by sinkattn_set_wait_limit_ns / sinkattn_test_withhold_copies.
uint64_t wait_limit_ns();
int32_t withhold_copies();

// Counts kernel launches (sinkattn_launch_count).
void note_launch(int n = 1);

// Sets the calling thread's detail message (sinkattn_last_error_message).
void note_error_message(const std::string& msg);

}  // namespace sinkattn
