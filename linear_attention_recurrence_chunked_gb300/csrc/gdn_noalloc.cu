// gdn_noalloc.cu -- the gated-delta-rule prefill for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand over a workspace: a plug-in running inside
// a host framework that owns all device memory and forbids its plug-ins to
// allocate, an inference engine that reserved its whole memory budget up front,
// or a latency-critical loop that must not pay the implicit device-wide
// synchronisation of cudaMalloc/cudaFree.  la_gdn_prefill_noalloc serves them:
// its scratch (the per-chunk records of the two-kernel schedule, or the
// segment maps and entry states of long sequences) lives in a fixed array in
// this library's device memory, so the call allocates nothing -- no
// cudaMalloc, no cudaFree, no allocating library routine.
//
// Cost: every GPU that loads the library holds kNoallocScratchBytes of device
// memory for the array until the process exits.
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "la.h"

namespace {

// Upper bound of the scratch this entry point can use: 16 MiB, i.e. 256 of the
// 64 KiB fp32 128x128 blocks the segment scan keeps per segment map or entry
// state, or the chunk records of 225 (b,h,64-token chunk) triples.
// Problems whose minimum scratch is larger (a 16-head, 1M-token prefill needs
// 25 MiB) are refused; they go through la_gdn_prefill with a caller
// workspace.
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;

// The scratch array.  In host code `g_noalloc_scratch` is only a host-side
// stand-in for the symbol, never a device address: the device address is
// obtained per device with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
std::map<int, void*> g_scratch_addr;  // device ordinal -> device address of the array

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached.
la_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  auto it = g_scratch_addr.find(dev);
  if (it == g_scratch_addr.end()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LA_ERR_CUDA;
    it = g_scratch_addr.emplace(dev, p).first;
  }
  *out = it->second;
  return LA_OK;
}

}  // namespace

extern "C" la_status la_gdn_prefill_noalloc(const la_gdn_prefill_args* args, void* stream) {
  if (!args) return LA_ERR_INVALID_ARGUMENT;
  // Problems whose minimum scratch would not fit the fixed array are refused
  // before anything else happens (la_gdn_prefill_workspace_size_min reports
  // it).  Problems whose fastest schedule fits the array run that schedule;
  // the others run the single-kernel scan, whose scratch fits.
  const size_t need_min = la_gdn_prefill_workspace_size_min(args);
  if (need_min > kNoallocScratchBytes) return LA_ERR_WORKSPACE;
  const size_t need = la_gdn_prefill_workspace_size(args);
  if (need == 0) return la_gdn_prefill(args, nullptr, 0, stream);
  void* scratch = nullptr;
  const la_status st = scratch_address(&scratch);
  if (st != LA_OK) return st;
  // Both schedules write every scratch byte they read within the call, so
  // nothing in the array has to start at zero.
  return la_gdn_prefill(args, scratch, kNoallocScratchBytes, stream);
}
