// sinkattn_bwd_static_workspace: the backward for callers that cannot
// allocate device memory when they call it. Examples are a host that has
// already handed the whole device to its own memory pool, or code that runs
// where an allocation's implicit synchronisation is not allowed (a real-time
// loop). Such callers cannot provide the scratch memory sinkattn_bwd needs, so
// this entry point uses one fixed array that lives in the library itself.
//
// The array is a file-scope __device__ variable of
// SINKATTN_STATIC_BWD_WORKSPACE_BYTES bytes: every GPU that loads the library
// holds it until the process exits. Its device address is looked up once per
// device (with that device current) on the first call made on that device.
// That first call should therefore come before any stream capture.
//
// All calls share the array and it keeps the last call's contents. Nothing in
// it has to start at zero: the backward kernels rewrite every byte they read
// (tile list, D, the sink-gradient partials, and the dq accumulator, which the
// preprocess clears). Calls that overlap on the GPU, on any stream, race on the
// array.
#include <mutex>
#include <string>

#include "../../include/sinkattn.h"
#include "internal.h"

namespace {

__device__ __align__(256) unsigned char g_static_bwd_workspace[SINKATTN_STATIC_BWD_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_address[kMaxDevices] = {};

}  // namespace

extern "C" SINKATTN_API sinkattn_status sinkattn_bwd_static_workspace(
    const sinkattn_bwd_params* params, void* stream) {
  if (!params) return sinkattn_bwd(nullptr, stream);  // reports the NULL argument
  const sinkattn_fwd_params& f = params->fwd;
  const size_t need =
      sinkattn_bwd_workspace_size_mode(f.nseq, f.total, f.Hq, f.Hkv, f.head_dim, params->deterministic);
  if (need > SINKATTN_STATIC_BWD_WORKSPACE_BYTES) {
    sinkattn::note_error_message(
        "problem needs " + std::to_string(need) + " bytes of workspace; the static workspace holds " +
        std::to_string((size_t)SINKATTN_STATIC_BWD_WORKSPACE_BYTES) +
        " (use sinkattn_bwd with a caller-provided workspace)");
    return SINKATTN_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    sinkattn::note_error_message(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return SINKATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    sinkattn::note_error_message("current device " + std::to_string(dev) +
                                 " is beyond the " + std::to_string(kMaxDevices) +
                                 " devices the static workspace keeps addresses for");
    return SINKATTN_ERR_UNSUPPORTED;
  }
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_address[dev]) {
      // A host-side reference to the array names a host stand-in, not device
      // memory: the kernels need the device address, looked up here.
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_static_bwd_workspace);
      if (e != cudaSuccess) {
        sinkattn::note_error_message(std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
        return SINKATTN_ERR_CUDA;
      }
      g_address[dev] = ptr;
    }
    ws = g_address[dev];
  }
  sinkattn_bwd_params p = *params;
  p.workspace = ws;
  p.workspace_bytes = SINKATTN_STATIC_BWD_WORKSPACE_BYTES;
  return sinkattn_bwd(&p, stream);
}
