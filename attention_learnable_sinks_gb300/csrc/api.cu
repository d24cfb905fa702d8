// C ABI of libsinkattn.so (declared in include/sinkattn.h): argument checks,
// workspace layout and the order of kernel launches. No device memory is
// allocated here; every buffer, workspace included, belongs to the caller.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/sinkattn.h"
#include "internal.h"

namespace sinkattn {

namespace {

constexpr uint64_t sm100_default_wait_ns() { return 2000000000ull; }  // 2 s, as in sm100.cuh

__device__ int32_t g_error_word;  // first error recorded by any kernel

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit_ns{sm100_default_wait_ns()};
std::atomic<int32_t> g_withhold{0};
thread_local std::string g_message;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int32_t* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

sinkattn_status fail(sinkattn_status st, const std::string& msg) {
  g_message = msg;
  return st;
}

// Per-device constants: address of the error word, SM count.
sinkattn_status device_info(int32_t** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SINKATTN_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(SINKATTN_ERR_UNSUPPORTED, "device index out of range");
  // make the device's context current on this host thread before anything
  // else (tensor maps are encoded through the driver before the first launch,
  // e.g. on a thread that has made no CUDA call yet)
  static thread_local int bound_dev = -1;
  if (bound_dev != dev) {
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return fail(SINKATTN_ERR_CUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(e));
    bound_dev = dev;
  }
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_err_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_error_word);
    if (e != cudaSuccess)
      return fail(SINKATTN_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
      return fail(SINKATTN_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(SINKATTN_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300) only");
    g_err_ptr[dev] = static_cast<int32_t*>(ptr);
    g_num_sms[dev] = n;
  }
  *err = g_err_ptr[dev];
  *sms = g_num_sms[dev];
  return SINKATTN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The backward hands out key tiles sequence by sequence above this fp32 dq
// accumulator size (1.5x the 126 MB L2). Measured on GB300: the 2.2 GB
// accumulator of the 32-sequence varlen batch, 24.6 -> 17.5 ms for the main
// kernel; the 128 MB one of four 2048-token sequences, 5% slower, so it keeps
// the order by cost.
constexpr size_t kSeqMajorAccBytes = size_t(192) << 20;

// Key tiles sequence by sequence when the fp32 dq accumulator is well beyond
// L2 (the running units then share their sequences' rows of it).
bool keys_seq_major(const Problem& p, bool deterministic) {
  return !deterministic && p.head_dim == kHeadDim && p.nseq > 1 &&
         (size_t)p.total * p.Hq * kHeadDim * sizeof(float) > kSeqMajorAccBytes;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Workspace layout. Forward: [meta | q-tile items]. Backward:
// [meta | k-tile items | D | sink partials | meta | q-tile items | dq_acc]
// (the query-tile list serves the deterministic dq pass, which has no use for
// the fp32 dq accumulator: that mode needs only the bytes before it).
struct Layout {
  size_t q_meta, q_items, k_meta, k_items, D, part, dq_acc, bytes;
  int32_t capacity, nchunks;
  size_t bytes_for(bool deterministic) const { return deterministic ? dq_acc : bytes; }
};

Layout layout(int32_t nseq, int32_t total, int32_t Hq, bool bwd) {
  Layout l{};
  l.capacity = tile_capacity(nseq, total);
  l.nchunks = (total + kTile - 1) / kTile;
  size_t off = 0;
  if (!bwd) {
    l.q_meta = off;
    off += 256;
    l.q_items = off;
    off += align256(sizeof(int2) * (size_t)l.capacity);
  } else {
    l.k_meta = off;
    off += 256;
    l.k_items = off;
    off += align256(sizeof(int2) * (size_t)l.capacity);
    l.D = off;
    off += align256(sizeof(float) * (size_t)Hq * total);
    l.part = off;
    off += align256(sizeof(float) * 8 * (size_t)Hq * l.capacity);
    l.q_meta = off;
    off += 256;
    l.q_items = off;
    off += align256(sizeof(int2) * (size_t)l.capacity);
    l.dq_acc = off;
    off += align256(sizeof(float) * (size_t)total * Hq * kHeadDim);
  }
  l.bytes = off;
  return l;
}

bool shape_ok(int32_t nseq, int32_t total, int32_t Hq, int32_t Hkv) {
  return nseq >= 0 && total >= 0 && Hq > 0 && Hkv > 0 && Hq % Hkv == 0 && Hq <= 65535;
}

bool head_dim_ok(int32_t d) { return d == kHeadDim || d == kHeadDimWide; }

// The backward at head_dim 128 always takes dq from the query-stationary pass:
// tensor memory holds dK and dV (256 columns) and the S^T / dP^T buffers, with
// no room left for a dQ accumulator.
bool bwd_deterministic(int32_t head_dim, int32_t deterministic) {
  return deterministic != 0 || head_dim != kHeadDim;
}

// Checks shared by forward and backward; fills the kernels' view.
sinkattn_status check_fwd(const sinkattn_fwd_params* a, Problem* p) {
  if (!a) return fail(SINKATTN_ERR_INVALID_ARG, "params is NULL");
  if (!head_dim_ok(a->head_dim))
    return fail(SINKATTN_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (!shape_ok(a->nseq, a->total, a->Hq, a->Hkv))
    return fail(SINKATTN_ERR_INVALID_ARG, "need nseq >= 0, total >= 0, 0 < Hkv, Hq % Hkv == 0, Hq <= 65535");
  if (a->causal != 0 && a->causal != 1) return fail(SINKATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (a->window > 0 && !a->causal)
    return fail(SINKATTN_ERR_UNSUPPORTED, "a sliding window needs causal = 1");
  if (a->max_seqlen < 0 || (a->total > 0 && a->max_seqlen < 1))
    return fail(SINKATTN_ERR_INVALID_ARG, "max_seqlen must be >= 1 (>= 0 when total is 0)");
  if (!a->cu_seqlens) return fail(SINKATTN_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (std::isnan(a->softmax_scale) || std::isinf(a->softmax_scale))
    return fail(SINKATTN_ERR_INVALID_ARG, "softmax_scale is not finite");
  const int64_t d = a->head_dim;
  const int64_t qs = a->q_row_stride ? a->q_row_stride : (int64_t)a->Hq * d;
  const int64_t ks = a->k_row_stride ? a->k_row_stride : (int64_t)a->Hkv * d;
  const int64_t vs = a->v_row_stride ? a->v_row_stride : (int64_t)a->Hkv * d;
  if (qs < (int64_t)a->Hq * d || ks < (int64_t)a->Hkv * d || vs < (int64_t)a->Hkv * d ||
      qs % 8 || ks % 8 || vs % 8)
    return fail(SINKATTN_ERR_INVALID_ARG, "row strides must cover all heads and be multiples of 8 elements");
  if (a->total > 0) {
    if (!a->q || !a->k || !a->v || !a->o) return fail(SINKATTN_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->o) ||
        (a->lse && !aligned16(a->lse)))
      return fail(SINKATTN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  }
  p->q = static_cast<const __nv_bfloat16*>(a->q);
  p->k = static_cast<const __nv_bfloat16*>(a->k);
  p->v = static_cast<const __nv_bfloat16*>(a->v);
  p->sinks = a->sinks;
  p->cu = a->cu_seqlens;
  p->o = static_cast<__nv_bfloat16*>(a->o);
  p->lse = a->lse;
  p->q_stride = qs;
  p->k_stride = ks;
  p->v_stride = vs;
  p->nseq = a->nseq;
  p->total = a->total;
  p->max_seqlen = a->max_seqlen;
  p->Hq = a->Hq;
  p->Hkv = a->Hkv;
  p->G = a->Hq / a->Hkv;
  p->causal = a->causal;
  p->head_dim = a->head_dim;
  // a window at least as long as every sequence restricts nothing
  p->window = (a->window > 0 && a->window < a->max_seqlen) ? a->window : 0;
  p->scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / std::sqrt((float)a->head_dim);
  p->scale_log2 = p->scale * 1.4426950408889634f;
  p->wait_limit_ns = wait_limit_ns();
  p->withhold_copies = withhold_copies();
  return SINKATTN_OK;
}

sinkattn_status cuda_fail(cudaError_t e, const char* where) {
  return fail(SINKATTN_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

void record(void* ev, cudaStream_t s) {
  if (ev) cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library links no driver import.
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
int32_t withhold_copies() { return g_withhold.load(std::memory_order_relaxed); }

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

void note_error_message(const std::string& msg) { g_message = msg; }

cudaError_t make_tmap_bf16_rows(CUtensorMap* map, const void* base, int heads, int total,
                                int64_t row_stride, int box_rows, int head_dim) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)total};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)row_stride * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  const cuuint32_t elem[3] = {1, 1, 1};
  // a box row is 128 bytes, one head of one token; promoting the L2 fill to
  // 256 bytes would also fetch the neighbouring head's row (measured 12%
  // slower on the 32-sequence varlen backward, no faster elsewhere)
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_bf16_heads(CUtensorMap* map, const void* base, int heads, int rows,
                                 int box_heads, int head_dim) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)heads * head_dim * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_heads, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_bf16_box(CUtensorMap* map, const void* base, int heads, int total, int64_t row_stride,
                               int head_dim, int box_inner, int box_rows) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  if (box_inner != 32 && box_inner != 64) return cudaErrorInvalidValue;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)total};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)row_stride * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_inner, 1, (cuuint32_t)box_rows};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                         box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         box_inner == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_f32_rows(CUtensorMap* map, void* base, int heads, int total) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)heads, (cuuint64_t)total};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 4, (cuuint64_t)heads * kHeadDim * 4};
  const cuuint32_t box[3] = {32, 1, 32};  // 32 rows: one read-out warp's share of a tile
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace sinkattn

using namespace sinkattn;

extern "C" {

size_t sinkattn_fwd_workspace_size(int32_t nseq, int32_t total, int32_t Hq, int32_t Hkv,
                                   int32_t head_dim) {
  if (!shape_ok(nseq, total, Hq, Hkv) || !head_dim_ok(head_dim)) return 0;
  return layout(nseq, total, Hq, false).bytes;
}

size_t sinkattn_bwd_workspace_size(int32_t nseq, int32_t total, int32_t Hq, int32_t Hkv,
                                   int32_t head_dim) {
  return sinkattn_bwd_workspace_size_mode(nseq, total, Hq, Hkv, head_dim, 0);
}

size_t sinkattn_bwd_workspace_size_mode(int32_t nseq, int32_t total, int32_t Hq, int32_t Hkv,
                                        int32_t head_dim, int32_t deterministic) {
  if (!shape_ok(nseq, total, Hq, Hkv) || !head_dim_ok(head_dim)) return 0;
  return layout(nseq, total, Hq, true).bytes_for(bwd_deterministic(head_dim, deterministic));
}

sinkattn_status sinkattn_fwd(const sinkattn_fwd_params* a, void* stream) {
  g_message.clear();
  Problem p{};
  sinkattn_status st = check_fwd(a, &p);
  if (st != SINKATTN_OK) return st;
  const Layout l = layout(a->nseq, a->total, a->Hq, false);
  if (!a->workspace || a->workspace_bytes < l.bytes)
    return fail(SINKATTN_ERR_WORKSPACE, "workspace missing or smaller than sinkattn_fwd_workspace_size()");
  if (a->total == 0) return SINKATTN_OK;
  int sms = 0;
  st = device_info(&p.err, &sms);
  if (st != SINKATTN_OK) return st;
  // head_dim 64: prepare the backward's workspace (at 128 the backward has no
  // dq accumulator and builds its own lists: bwd_workspace is not used)
  const bool prep = a->bwd_workspace && p.head_dim == kHeadDim;
  if (prep) {
    // clear the backward's dq accumulator during the forward
    const Layout lb = layout(a->nseq, a->total, a->Hq, true);
    if (a->bwd_workspace_bytes < lb.bytes || !aligned16(a->bwd_workspace))
      return fail(SINKATTN_ERR_WORKSPACE,
                  "bwd_workspace smaller than sinkattn_bwd_workspace_size() or not 16-byte aligned");
    p.clear = static_cast<uint8_t*>(a->bwd_workspace) + lb.dq_acc;
    p.clear_bytes = (int64_t)(lb.bytes - lb.dq_acc);
  }
  // ... and builds its key-tile list, in the same launch as its own list
  TileList bkt{};
  if (prep) {
    const Layout lb = layout(a->nseq, a->total, a->Hq, true);
    char* bws = static_cast<char*>(a->bwd_workspace);
    bkt = TileList{reinterpret_cast<int32_t*>(bws + lb.k_meta), reinterpret_cast<int2*>(bws + lb.k_items),
                   lb.capacity};
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(a->workspace);
  TileList qt{reinterpret_cast<int32_t*>(ws + l.q_meta), reinterpret_cast<int2*>(ws + l.q_items),
              l.capacity};
  FwdLaunch fl;
  cudaError_t e = prepare_fwd(p, &fl);
  if (e != cudaSuccess) return cuda_fail(e, "forward tensor maps");
  e = launch_build_tile_list(p, 0, 0, qt, s, prep ? &bkt : nullptr,
                             keys_seq_major(p, false) ? 1 : 0);
  if (e != cudaSuccess) return cuda_fail(e, "tile list");
  record(a->timing_events[0], s);
  e = launch_fwd(p, fl, qt, sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "forward kernel");
  record(a->timing_events[1], s);
  return SINKATTN_OK;
}

sinkattn_status sinkattn_bwd(const sinkattn_bwd_params* a, void* stream) {
  g_message.clear();
  if (!a) return fail(SINKATTN_ERR_INVALID_ARG, "params is NULL");
  BwdProblem bp{};
  sinkattn_status st = check_fwd(&a->fwd, &bp.f);
  if (st != SINKATTN_OK) return st;
  const sinkattn_fwd_params& f = a->fwd;
  if (f.total > 0) {
    if (!f.lse || !a->dout || !a->dq || !a->dk || !a->dv)
      return fail(SINKATTN_ERR_INVALID_ARG, "lse, dout, dq, dk and dv must be non-NULL");
    if (!aligned16(a->dout) || !aligned16(a->dq) || !aligned16(a->dk) || !aligned16(a->dv))
      return fail(SINKATTN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  }
  const Layout l = layout(f.nseq, f.total, f.Hq, true);
  const bool det = bwd_deterministic(f.head_dim, a->deterministic);
  if (!a->workspace || a->workspace_bytes < l.bytes_for(det))
    return fail(SINKATTN_ERR_WORKSPACE,
                "workspace missing or smaller than sinkattn_bwd_workspace_size_mode()");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (f.total == 0) {
    if (a->dsinks && !a->accumulate_dsinks) {
      cudaError_t e = cudaMemsetAsync(a->dsinks, 0, sizeof(float) * f.Hq, s);
      if (e != cudaSuccess) return cuda_fail(e, "dsinks clear");
    }
    return SINKATTN_OK;
  }
  int sms = 0;
  st = device_info(&bp.f.err, &sms);
  if (st != SINKATTN_OK) return st;
  char* ws = static_cast<char*>(a->workspace);
  bp.dout = static_cast<const __nv_bfloat16*>(a->dout);
  bp.dq = static_cast<__nv_bfloat16*>(a->dq);
  bp.dk = static_cast<__nv_bfloat16*>(a->dk);
  bp.dv = static_cast<__nv_bfloat16*>(a->dv);
  bp.dsinks = a->dsinks;
  bp.accumulate_dsinks = a->accumulate_dsinks != 0;
  bp.deterministic = det;
  bp.acc_cleared = a->workspace_cleared != 0 && !bp.deterministic;
  bp.D = reinterpret_cast<float*>(ws + l.D);
  bp.sink_part = reinterpret_cast<float*>(ws + l.part);
  bp.dq_acc = reinterpret_cast<float*>(ws + l.dq_acc);
  bp.nchunks = l.nchunks;
  bp.part_stride = l.capacity;
  TileList kt{reinterpret_cast<int32_t*>(ws + l.k_meta), reinterpret_cast<int2*>(ws + l.k_items),
              l.capacity};
  TileList qt{reinterpret_cast<int32_t*>(ws + l.q_meta), reinterpret_cast<int2*>(ws + l.q_items),
              l.capacity};
  const bool wide = f.head_dim == kHeadDimWide;
  BwdLaunch bl;
  BwdWideLaunch wl;
  cudaError_t e = prepare_bwd_main(bp, &bl);
  if (e == cudaSuccess && wide) e = prepare_bwd_wide(bp, &wl);
  if (e == cudaSuccess && bp.deterministic) e = prepare_bwd_dq(f.head_dim);
  if (e != cudaSuccess) return cuda_fail(e, "backward tensor maps");
  // The key-tile list (unless the forward built it with the clear)
  if (!bp.acc_cleared) {
    e = launch_build_tile_list(bp.f, 1, keys_seq_major(bp.f, bp.deterministic) ? 1 : 0, kt, s);
    if (e != cudaSuccess) return cuda_fail(e, "key-tile list");
  }
  if (bp.deterministic) {
    e = launch_build_tile_list(bp.f, 0, 0, qt, s);
    if (e != cudaSuccess) return cuda_fail(e, "query-tile list");
  }
  e = launch_bwd_preprocess(bp, s);
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess");
  record(a->timing_events[0], s);
  e = wide ? launch_bwd_wide(bp, wl, kt, sms, s) : launch_bwd_main(bp, bl, kt, sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "backward main");
  record(a->timing_events[1], s);
  if (bp.deterministic) {
    record(a->timing_events_dq[0], s);
    e = launch_bwd_dq(bp, bl, qt, sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "deterministic dq");
    record(a->timing_events_dq[1], s);
  }
  e = launch_bwd_finish(bp, kt, sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "dq conversion / sink gradient");
  return SINKATTN_OK;
}

size_t sinkattn_decode_workspace_size(int32_t nseq, int32_t Hq, int32_t num_splits) {
  return sinkattn_decode_workspace_size_d(nseq, Hq, num_splits, kHeadDim);
}

size_t sinkattn_decode_workspace_size_d(int32_t nseq, int32_t Hq, int32_t num_splits, int32_t head_dim) {
  if (nseq < 0 || Hq <= 0 || Hq > 65535 || num_splits < 1 || num_splits > 64 || !head_dim_ok(head_dim))
    return 0;
  return decode_workspace_bytes(nseq, Hq, num_splits, head_dim);
}

}  // extern "C"

namespace {

// Checks shared by both decode entry points (nothing to do: nseq == 0 gives
// SINKATTN_OK with *empty set).
sinkattn_status check_decode(const sinkattn_decode_params* a, bool* empty) {
  *empty = false;
  if (!a) return fail(SINKATTN_ERR_INVALID_ARG, "params is NULL");
  if (!head_dim_ok(a->head_dim)) return fail(SINKATTN_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (a->nseq < 0 || a->nseq > 65535 || a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv || a->Hq > 65535)
    return fail(SINKATTN_ERR_INVALID_ARG, "need 0 <= nseq <= 65535, 0 < Hkv, Hq % Hkv == 0, Hq <= 65535");
  const int G = a->Hq / a->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(SINKATTN_ERR_UNSUPPORTED, "Hq / Hkv must be 1, 2, 4, 8 or 16");
  if (a->block_size != 16 && a->block_size != 32 && a->block_size != 64 && a->block_size != 128)
    return fail(SINKATTN_ERR_UNSUPPORTED, "block_size must be 16, 32, 64 or 128");
  if (a->num_blocks <= 0 || a->max_blocks_per_seq <= 0 ||
      (int64_t)a->num_blocks * a->block_size > INT32_MAX ||
      (int64_t)a->max_blocks_per_seq * a->block_size > INT32_MAX)
    return fail(SINKATTN_ERR_INVALID_ARG, "num_blocks and max_blocks_per_seq must be > 0 and cover < 2^31 tokens");
  if (a->num_splits < 0 || a->num_splits > 64)
    return fail(SINKATTN_ERR_INVALID_ARG, "num_splits must be in [0, 64]");
  if (std::isnan(a->softmax_scale) || std::isinf(a->softmax_scale))
    return fail(SINKATTN_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (a->nseq == 0) {
    *empty = true;
    return SINKATTN_OK;
  }
  if (!a->q || !a->k_cache || !a->v_cache || !a->block_table || !a->seqlens || !a->o)
    return fail(SINKATTN_ERR_INVALID_ARG, "q, k_cache, v_cache, block_table, seqlens and o must be non-NULL");
  if (!aligned16(a->q) || !aligned16(a->k_cache) || !aligned16(a->v_cache) || !aligned16(a->o))
    return fail(SINKATTN_ERR_INVALID_ARG, "q, the caches and o must be 16-byte aligned");
  return SINKATTN_OK;
}

}  // namespace

extern "C" {

sinkattn_status sinkattn_decode(const sinkattn_decode_params* a, void* stream) {
  g_message.clear();
  bool empty = false;
  sinkattn_status st0 = check_decode(a, &empty);
  if (st0 != SINKATTN_OK || empty) return st0;
  const int32_t d = a->head_dim;
  if (!a->workspace ||
      a->workspace_bytes < decode_workspace_bytes(a->nseq, a->Hq, std::max(a->num_splits, 1), d))
    return fail(SINKATTN_ERR_WORKSPACE, "workspace missing or smaller than sinkattn_decode_workspace_size_d()");
  int sms = 0;
  DecodeProblem p{};
  sinkattn_status st = device_info(&p.err, &sms);
  if (st != SINKATTN_OK) return st;
  // Splits: each takes `per` 128-key chunks. A sequence has at most `maxch`
  // chunks (its keys from the 128-aligned chunk holding the window's first
  // key). Automatic choice, from measurements on GB300: one split when a
  // sequence spans at most 4 chunks (the split kernel then finishes the rows
  // itself, without the combine pass); otherwise at least 4 splits, and enough
  // CTAs for about 4 per SM, at most 64 splits and never less than 2 chunks
  // each; fewer if the workspace is smaller.
  const int64_t keys = (int64_t)a->max_blocks_per_seq * a->block_size;
  const int64_t span = a->window > 0 ? std::min<int64_t>(keys, (int64_t)a->window + 127) : keys;
  const int64_t maxch = std::max<int64_t>(1, (span + 127) / 128);
  int64_t per;
  if (a->num_splits > 0) {
    per = (maxch + a->num_splits - 1) / a->num_splits;
  } else if (maxch <= 4) {
    per = maxch;
  } else {
    const int64_t units = (int64_t)a->nseq * a->Hkv;
    int64_t want = std::max<int64_t>(4, (4 * (int64_t)sms + units - 1) / units);
    want = std::min<int64_t>({want, 64, std::max<int64_t>(1, maxch / 2)});
    per = (maxch + want - 1) / want;
    while ((maxch + per - 1) / per > 1 &&
           decode_workspace_bytes(a->nseq, a->Hq, (int)((maxch + per - 1) / per), d) > a->workspace_bytes)
      ++per;
  }
  const int nsplit = (int)((maxch + per - 1) / per);
  if (a->workspace_bytes < decode_workspace_bytes(a->nseq, a->Hq, nsplit, d))
    return fail(SINKATTN_ERR_WORKSPACE, "workspace smaller than sinkattn_decode_workspace_size_d()");
  char* ws = static_cast<char*>(a->workspace);
  const size_t n = (size_t)a->nseq * a->Hq * nsplit;
  p.q = static_cast<const __nv_bfloat16*>(a->q);
  p.k_cache = static_cast<const __nv_bfloat16*>(a->k_cache);
  p.v_cache = static_cast<const __nv_bfloat16*>(a->v_cache);
  p.block_table = a->block_table;
  p.seqlens = a->seqlens;
  p.sinks = a->sinks;
  p.o = static_cast<__nv_bfloat16*>(a->o);
  p.lse = a->lse;
  p.part_ml = reinterpret_cast<float*>(ws);
  p.part_o = reinterpret_cast<float*>(ws + align256(n * 2 * sizeof(float)));
  p.nseq = a->nseq;
  p.num_blocks = a->num_blocks;
  p.block_size = a->block_size;
  p.max_blocks = a->max_blocks_per_seq;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.head_dim = d;
  p.window = a->window > 0 ? a->window : 0;
  p.nsplit = nsplit;
  p.split_chunks = (int32_t)per;
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / std::sqrt((float)d);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_ns();
  p.withhold_copies = withhold_copies();
  const cudaError_t e = launch_decode(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode kernels");
  return SINKATTN_OK;
}

sinkattn_status sinkattn_decode_exact(const sinkattn_decode_params* a, void* stream) {
  g_message.clear();
  bool empty = false;
  sinkattn_status st = check_decode(a, &empty);
  if (st != SINKATTN_OK || empty) return st;
  if (!a->workspace || a->workspace_bytes < 256)
    return fail(SINKATTN_ERR_WORKSPACE, "the exact decode needs a workspace of at least 256 bytes");
  Problem p{};
  int sms = 0;
  st = device_info(&p.err, &sms);
  if (st != SINKATTN_OK) return st;
  p.q = static_cast<const __nv_bfloat16*>(a->q);
  p.sinks = a->sinks;
  p.o = static_cast<__nv_bfloat16*>(a->o);
  p.lse = a->lse;
  p.nseq = a->nseq;
  p.total = a->nseq;  // lse is [Hq, nseq]
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.G = a->Hq / a->Hkv;
  p.causal = 1;
  p.head_dim = a->head_dim;
  p.window = a->window > 0 ? a->window : 0;
  p.scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / std::sqrt((float)a->head_dim);
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_ns();
  p.withhold_copies = withhold_copies();
  PagedKV kv{a->block_table, a->seqlens, a->num_blocks, a->block_size, a->max_blocks_per_seq};
  const cudaError_t e = launch_decode_exact(p, kv, a->k_cache, a->v_cache,
                                            static_cast<int32_t*>(a->workspace), sms,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "exact decode");
  return SINKATTN_OK;
}

const char* sinkattn_status_string(int32_t status) {
  switch (status) {
    case SINKATTN_OK: return "ok";
    case SINKATTN_ERR_INVALID_ARG: return "invalid argument";
    case SINKATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case SINKATTN_ERR_CUDA: return "CUDA error";
    case SINKATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case SINKATTN_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    default: return "unknown status";
  }
}

const char* sinkattn_last_error_message(void) { return g_message.c_str(); }

int32_t sinkattn_device_error(int32_t reset) {
  int32_t* err = nullptr;
  int sms = 0;
  if (device_info(&err, &sms) != SINKATTN_OK) return SINKATTN_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return SINKATTN_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SINKATTN_ERR_CUDA;
  if (reset) {
    const int32_t zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return SINKATTN_ERR_CUDA;
  }
  return word;
}

uint64_t sinkattn_launch_count(void) { return g_launches.load(); }

void sinkattn_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns ? ns : sm100_default_wait_ns(), std::memory_order_relaxed);
}

void sinkattn_test_withhold_copies(int32_t on) {
  g_withhold.store(on ? 1 : 0, std::memory_order_relaxed);
}

size_t sinkattn_params_size(int32_t which) {
  if (which == 0) return sizeof(sinkattn_fwd_params);
  if (which == 1) return sizeof(sinkattn_bwd_params);
  if (which == 2) return sizeof(sinkattn_decode_params);
  return 0;
}

}  // extern "C"
