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
#include <cuda.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "kernels.h"
#include "la.h"

namespace {

// Upper bound of the scratch this entry point can use: 16 MiB, i.e. 256 of the
// 64 KiB fp32 128x128 blocks the segment scan keeps per segment map or entry
// state, or the per-chunk inverse records (8 KiB each) of 2048 (b,h,64-token
// chunk) triples.  Problems whose minimum scratch is larger (a 16-head,
// 1M-token prefill needs 25 MiB) are refused; they go through la_gdn_prefill
// with a caller workspace.
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;

// The scratch array.  In host code `g_noalloc_scratch` is only a host-side
// stand-in for the symbol, never a device address: the device address is
// obtained with cudaGetSymbolAddress below, with the device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Driver calls that identify the current context, reached through the
// runtime's driver entry point (the library does not link libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};
const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return f;
}

// Process-unique id of the current context (0 when none is current yet).
la_status current_context_id(unsigned long long* id) {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return LA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return LA_ERR_CUDA;
  *id = 0;
  if (ctx == nullptr) return LA_OK;
  return f.get_id(ctx, id) == CUDA_SUCCESS ? LA_OK : LA_ERR_CUDA;
}

std::mutex g_scratch_mu;
std::map<unsigned long long, void*> g_scratch_addr;  // context id -> device address of the array

// Device address of the array in the current context.  It is looked up once
// per context and cached under the context's id, so a context that is
// destroyed and recreated (cudaDeviceReset, for one) gets a fresh lookup
// instead of a stale address.
la_status scratch_address(void** out) {
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    la::note_cuda_error((int)e);
    return LA_ERR_CUDA;
  }
  unsigned long long id = 0;
  la_status st = current_context_id(&id);
  if (st != LA_OK) return st;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (id != 0) {
    auto it = g_scratch_addr.find(id);
    if (it != g_scratch_addr.end()) {
      *out = it->second;
      return LA_OK;
    }
  }
  void* p = nullptr;
  // with no current context yet this also makes the device's primary context current
  const cudaError_t es = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (es != cudaSuccess || p == nullptr) {
    la::note_cuda_error((int)(es != cudaSuccess ? es : cudaErrorUnknown));
    return LA_ERR_CUDA;
  }
  if (id == 0) {
    st = current_context_id(&id);
    if (st != LA_OK) return st;
    if (id == 0) return LA_ERR_CUDA;
  }
  g_scratch_addr[id] = p;
  *out = p;
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
