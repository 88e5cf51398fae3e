// state_ops.cu -- operations on recurrent states between calls.
//
//   rescale  S <- lambda S per state, lambda in [0, 1]: the readout-boundary
//            rescaling of NoteBank App. D.1 (lambda = 1 keeps the state,
//            lambda = 0 resets it; a reset writes zeros whatever was stored);
//   gather   dst_i <- src_{index_i}: copy and branch states, e.g. the copy of
//            the state the question is processed on in NoteBank App. B,
//            Alg. 1 (one source state to several destinations).
// Both stream the states once (HBM-bound): 16-byte vectors when the state
// size allows it, grid sized in whole waves of the SMs.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

constexpr int kThreads = 256;

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
state_rescale_kernel(float* __restrict__ states, int64_t n_states, int64_t per, const float* __restrict__ lambda,
                     float lambda_all) {
  const int64_t total = n_states * per;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  if (kVec) {  // per % 4 == 0 and 16-byte aligned: whole float4s never straddle two states
    const int64_t per4 = per >> 2;
    float4* s4 = reinterpret_cast<float4*>(states);
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < (total >> 2); e += stride) {
      const float l = lambda ? lambda[e / per4] : lambda_all;
      float4 x = l == 0.f ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldcs(s4 + e);
      x.x *= l; x.y *= l; x.z *= l; x.w *= l;
      __stcs(s4 + e, x);
    }
  } else {
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += stride) {
      const float l = lambda ? lambda[e / per] : lambda_all;
      states[e] = l == 0.f ? 0.f : l * states[e];
    }
  }
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
state_gather_kernel(float* __restrict__ dst, const float* __restrict__ src, const int64_t* __restrict__ index,
                    int64_t n_dst, int64_t n_src, int64_t per, unsigned* status) {
  for (int64_t i = blockIdx.y; i < n_dst; i += gridDim.y) {
    const int64_t j = index[i];
    if (j < 0 || j >= n_src) {  // nothing is read or written for this destination
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, kStatusBadIndex);
      continue;
    }
    if (kVec) {
      const float4* s4 = reinterpret_cast<const float4*>(src + j * per);
      float4* d4 = reinterpret_cast<float4*>(dst + i * per);
      for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < (per >> 2); e += (int64_t)gridDim.x * kThreads)
        __stcs(d4 + e, __ldcs(s4 + e));
    } else {
      for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < per; e += (int64_t)gridDim.x * kThreads)
        dst[i * per + e] = src[j * per + e];
    }
  }
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      n = v;
    else
      n = 148;
  }
  return n;
}

}  // namespace

cudaError_t launch_state_rescale(float* states, int64_t n_states, int64_t per, const float* lambda, float lambda_all,
                                 cudaStream_t stream) {
  const int64_t total = n_states * per;
  if (total == 0) return cudaSuccess;
  const bool vec = per % 4 == 0 && (reinterpret_cast<uintptr_t>(states) & 15u) == 0;
  const int64_t work = vec ? total / 4 : total;
  const int64_t waves = (work + (int64_t)sm_count() * 4 * kThreads - 1) / ((int64_t)sm_count() * 4 * kThreads);
  const unsigned grid = (unsigned)(sm_count() * 4 * (waves < 8 ? waves : 8));
  if (vec)
    state_rescale_kernel<true><<<grid, kThreads, 0, stream>>>(states, n_states, per, lambda, lambda_all);
  else
    state_rescale_kernel<false><<<grid, kThreads, 0, stream>>>(states, n_states, per, lambda, lambda_all);
  return cudaGetLastError();
}

cudaError_t launch_state_gather(float* dst, const float* src, const int64_t* index, int64_t n_dst, int64_t n_src,
                                int64_t per, unsigned* status, cudaStream_t stream) {
  if (n_dst == 0 || per == 0) return cudaSuccess;
  const bool vec = per % 4 == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const int64_t work = vec ? per / 4 : per;
  const unsigned gx = (unsigned)((work + kThreads - 1) / kThreads < 64 ? (work + kThreads - 1) / kThreads : 64);
  const unsigned gy = (unsigned)(n_dst < 65535 ? n_dst : 65535);
  const dim3 grid(gx, gy);
  if (vec)
    state_gather_kernel<true><<<grid, kThreads, 0, stream>>>(dst, src, index, n_dst, n_src, per, status);
  else
    state_gather_kernel<false><<<grid, kThreads, 0, stream>>>(dst, src, index, n_dst, n_src, per, status);
  return cudaGetLastError();
}

}  // namespace la
