// swa_decode.cu -- one decode step of sliding-window softmax attention, the
// window layers of BASED (BASED notes Sec. 2.4: standard softmax over the
// last w tokens, whose KV the layer keeps; Sec. 2.5: the decode step fuses
// the dot products, the softmax and the weighted sum for the small window).
//
// Per (sequence, head) the keys and values of the last w tokens sit in a ring
// buffer: token p in slot p % w.  A step at position pos (tokens already
// seen) writes the new k, v into slot pos % w and attends over the
// min(pos + 1, w) tokens pos - w + 1 .. pos, the new one included:
//   o = sum_j softmax_j(scale q . k_j) v_j.
// One warp per (sequence, head), four per CTA: lane l scores the slots
// l, l + 32, ... (key rows read as 16-byte vectors), a warp max and sum by
// shuffles give the softmax, then lane l accumulates its d/32 consecutive
// output columns over the slots, eight slots in flight (each value row read
// by the warp in one coalesced piece).  The new token is written into its
// slot first, so all slots are read alike.  For d of 64 or 128 a second
// kernel stages each warp's whole window in shared memory with one round of
// 16-byte copies instead (a step then waits on memory once, not once per
// group of rows); larger windows than fit take the first kernel.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace la {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxWindow = 256;
constexpr int kMaxD = 128;
constexpr int kSlotsPerLane = kMaxWindow / 32;

// CPL consecutive elements as floats (CPL = 1, 2 or 4; the address is aligned to CPL elements)
template <int CPL>
__device__ __forceinline__ void load_n(const float* p, float* o) {
  if (CPL == 4) { const float4 x = *reinterpret_cast<const float4*>(p); o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w; }
  if (CPL == 2) { const float2 x = *reinterpret_cast<const float2*>(p); o[0] = x.x; o[1] = x.y; }
  if (CPL == 1) o[0] = *p;
}
template <int CPL>
__device__ __forceinline__ void load_n(const __nv_bfloat16* p, float* o) {
  if (CPL == 4) { const float4 x = load4(p); o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w; }
  if (CPL == 2) {
    const uint32_t r = *reinterpret_cast<const uint32_t*>(p);
    o[0] = __uint_as_float(r << 16);
    o[1] = __uint_as_float(r & 0xffff0000u);
  }
  if (CPL == 1) o[0] = __bfloat162float(*p);
}

// o[c] for this lane's CPL columns: sum_j p_j v_j[c] over the n slots, eight slots in flight
template <int CPL, typename TIn>
__device__ __forceinline__ void weighted_sum(const TIn* vc, int d, int n, const float* p, int lane, float* o) {
  float acc[8][CPL];
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[u][e] = 0.f;
  const TIn* base = vc + lane * CPL;
  int j = 0;
  for (; j + 8 <= n; j += 8) {
    float x[8][CPL];
#pragma unroll
    for (int u = 0; u < 8; ++u) load_n<CPL>(base + (int64_t)(j + u) * d, x[u]);
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int e = 0; e < CPL; ++e) acc[u][e] = fmaf(p[j + u], x[u][e], acc[u][e]);
  }
  for (; j < n; ++j) {
    float x[CPL];
    load_n<CPL>(base + (int64_t)j * d, x);
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[0][e] = fmaf(p[j], x[e], acc[0][e]);
  }
#pragma unroll
  for (int e = 0; e < CPL; ++e) {
    float t = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) t += acc[u][e];
    o[e] = t;
  }
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(32 * kWarps)
swa_decode_kernel(SwaDecodeLaunch a) {
  __shared__ float qs[kWarps][kMaxD];
  __shared__ float ps[kWarps][kMaxWindow];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t sh = (int64_t)blockIdx.x * kWarps + warp;
  grid_dependents_trigger();
  if (sh >= a.S * a.H) return;
  grid_dependency_wait();  // the caches, positions and inputs of this step are in memory
  const int64_t s = sh / a.H;
  const int d = a.d, w = a.window;
  const int64_t pos = a.pos[s];
  if (pos < 0) {  // nothing is read or written for this (sequence, head)
    if (lane == 0) atomicOr(a.status, kStatusBadIndex);
    return;
  }
  const int slot_new = (int)(pos % w);
  const int n = pos + 1 < w ? (int)(pos + 1) : w;  // valid slots: 0..n-1 (the ring fills from slot 0)
  const TIn* q = reinterpret_cast<const TIn*>(a.q) + sh * d;
  const TIn* k = reinterpret_cast<const TIn*>(a.k) + sh * d;
  const TIn* v = reinterpret_cast<const TIn*>(a.v) + sh * d;
  TIn* kc = reinterpret_cast<TIn*>(a.k_cache) + sh * (int64_t)w * d;
  TIn* vc = reinterpret_cast<TIn*>(a.v_cache) + sh * (int64_t)w * d;
  // the new token goes into its slot first, so every slot is read alike below
  for (int c = lane; c < d; c += 32) {
    qs[warp][c] = to_f(q[c]) * a.scale;
    kc[(int64_t)slot_new * d + c] = k[c];
    vc[(int64_t)slot_new * d + c] = v[c];
  }
  __syncwarp();  // orders the slot writes and qs before the lanes' reads
  // scores of this lane's slots (four partial sums per dot product)
  float sc[kSlotsPerLane];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kSlotsPerLane; ++i) {
    const int j = lane + 32 * i;
    float acc = -INFINITY;
    if (j < n) {
      const TIn* kr = kc + (int64_t)j * d;
      float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
      for (int c = 0; c < d; c += 8) {
        const float4 x = load4(kr + c), y = load4(kr + c + 4);
        p0 = fmaf(qs[warp][c], x.x, fmaf(qs[warp][c + 4], y.x, p0));
        p1 = fmaf(qs[warp][c + 1], x.y, fmaf(qs[warp][c + 5], y.y, p1));
        p2 = fmaf(qs[warp][c + 2], x.z, fmaf(qs[warp][c + 6], y.z, p2));
        p3 = fmaf(qs[warp][c + 3], x.w, fmaf(qs[warp][c + 7], y.w, p3));
      }
      acc = (p0 + p1) + (p2 + p3);
    }
    sc[i] = acc;
    m = fmaxf(m, acc);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
  float l = 0.f;
#pragma unroll
  for (int i = 0; i < kSlotsPerLane; ++i) {
    const int j = lane + 32 * i;
    if (j < n) {
      const float e = __expf(sc[i] - m);
      ps[warp][j] = e;
      l += e;
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) l += __shfl_xor_sync(kFullMask, l, off);
  __syncwarp();
  const float inv = 1.f / l;
  TOut* out = reinterpret_cast<TOut*>(a.out) + sh * d;
  if (d % 32 == 0) {
    // lane l owns the d/32 consecutive columns starting at l * d/32
    const int cpl = d >> 5;
    float o[4];
    if (cpl == 4) weighted_sum<4>(vc, d, n, ps[warp], lane, o);
    else if (cpl == 2) weighted_sum<2>(vc, d, n, ps[warp], lane, o);
    else weighted_sum<1>(vc, d, n, ps[warp], lane, o);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < cpl) store1(out + lane * cpl + e, o[e] * inv);
  } else {
    for (int c = lane; c < d; c += 32) {
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(ps[warp][j], to_f(vc[(int64_t)j * d + c]), acc);
      store1(out + c, acc * inv);
    }
  }
}

// The same step with the key window staged in shared memory (d = D of 64 or 128, 16-byte aligned
// caches): each warp copies its whole key window in one round of 16-byte cp.async copies, rows padded
// by 16 bytes (a lane per row then reads without bank conflicts), and replaces the copy of the new
// token's slot with the new k.  The values are read straight from the cache (one coalesced row per
// warp load, eight rows in flight), so a warp's shared memory is half what staging both would take
// and twice as many warps fit on an SM.
template <typename TIn, typename TOut, int D>
__global__ void __launch_bounds__(32 * kWarps)
swa_decode_staged_kernel(SwaDecodeLaunch a) {
  extern __shared__ __align__(16) uint8_t sw_smem[];
  __shared__ float qs[kWarps][D];
  __shared__ float ps[kWarps][kMaxWindow];
  constexpr int kRowBytes = D * (int)sizeof(TIn), kPitch = kRowBytes + 16, kVec = kRowBytes / 16;
  constexpr int kPerVec = 16 / (int)sizeof(TIn);  // elements per 16-byte vector
  constexpr int kCpl = D / 32;                     // output columns per lane
  const int nwarps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t sh = (int64_t)blockIdx.x * nwarps + warp;
  grid_dependents_trigger();
  if (sh >= a.S * a.H) return;  // warp-uniform; the kernel has no block-wide barrier
  grid_dependency_wait();       // the caches, positions and inputs of this step are in memory
  const int64_t s = sh / a.H;
  const int w = a.window;
  const int64_t pos = a.pos[s];
  if (pos < 0) {
    if (lane == 0) atomicOr(a.status, kStatusBadIndex);
    return;
  }
  const int slot_new = (int)(pos % w);
  const int n = pos + 1 < w ? (int)(pos + 1) : w;
  uint8_t* ks = sw_smem + (size_t)warp * w * kPitch;
  const uint8_t* kc = reinterpret_cast<const uint8_t*>(a.k_cache) + sh * (int64_t)w * kRowBytes;
  const TIn* vcache = reinterpret_cast<const TIn*>(a.v_cache) + sh * (int64_t)w * D;
  for (int i = lane; i < n * kVec; i += 32) {
    const int r = i / kVec, c = i - r * kVec;
    tc::cp_async16(tc::smem_u32(ks + r * kPitch + c * 16), kc + (int64_t)r * kRowBytes + c * 16, 16u);
  }
  tc::cp_async_commit();
  // meanwhile: q (scaled) and the new token into the ring buffer
  const TIn* q = reinterpret_cast<const TIn*>(a.q) + sh * D;
  const TIn* k = reinterpret_cast<const TIn*>(a.k) + sh * D;
  const TIn* v = reinterpret_cast<const TIn*>(a.v) + sh * D;
  TIn knew[kCpl], vnew[kCpl];
#pragma unroll
  for (int e = 0; e < kCpl; ++e) {
    const int c = lane * kCpl + e;
    qs[warp][c] = to_f(q[c]) * a.scale;
    knew[e] = k[c];
    vnew[e] = v[c];
    reinterpret_cast<TIn*>(a.k_cache)[(sh * w + slot_new) * D + c] = knew[e];
    reinterpret_cast<TIn*>(a.v_cache)[(sh * w + slot_new) * D + c] = vnew[e];
  }
  tc::cp_async_wait_all();
  __syncwarp();
  // the staged copy of the new token's slot may hold the old token: overwrite it (the value cache
  // itself already holds the new v: this warp's own stores, ordered by the __syncwarp)
#pragma unroll
  for (int e = 0; e < kCpl; ++e) reinterpret_cast<TIn*>(ks + slot_new * kPitch)[lane * kCpl + e] = knew[e];
  __syncwarp();
  // scores of this lane's slots
  float sc[kSlotsPerLane];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kSlotsPerLane; ++i) {
    const int j = lane + 32 * i;
    float acc = -INFINITY;
    if (j < n) {
      const uint8_t* kr = ks + j * kPitch;
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int c = 0; c < kVec; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(kr + c * 16);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
        if constexpr (sizeof(TIn) == 2) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            p0 = fmaf(qs[warp][c * kPerVec + 2 * t], __uint_as_float(wd[t] << 16), p0);
            p1 = fmaf(qs[warp][c * kPerVec + 2 * t + 1], __uint_as_float(wd[t] & 0xffff0000u), p1);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (t & 1) p1 = fmaf(qs[warp][c * kPerVec + t], __uint_as_float(wd[t]), p1);
            else p0 = fmaf(qs[warp][c * kPerVec + t], __uint_as_float(wd[t]), p0);
          }
        }
      }
      acc = p0 + p1;
    }
    sc[i] = acc;
    m = fmaxf(m, acc);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
  float l = 0.f;
#pragma unroll
  for (int i = 0; i < kSlotsPerLane; ++i) {
    const int j = lane + 32 * i;
    if (j < n) {
      const float e = __expf(sc[i] - m);
      ps[warp][j] = e;
      l += e;
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) l += __shfl_xor_sync(kFullMask, l, off);
  __syncwarp();
  // o = sum_j p_j v_j / l from the value cache, lane l owning columns [kCpl l, kCpl l + kCpl)
  float o[4];
  weighted_sum<kCpl>(vcache, D, n, ps[warp], lane, o);
  const float inv = 1.f / l;
  TOut* out = reinterpret_cast<TOut*>(a.out) + sh * D;
#pragma unroll
  for (int e = 0; e < kCpl; ++e) store1(out + lane * kCpl + e, o[e] * inv);
}

// The staged kernel for d = D: warps per CTA so that their windows fit in shared memory, 0 if even one
// warp's does not (the caller then takes the kernel above).
template <typename TIn, typename TOut, int D>
cudaError_t launch_staged(const SwaDecodeLaunch& a, cudaStream_t stream, bool& done) {
  constexpr int64_t kMaxDynamic = 200 * 1024;
  const int64_t per_warp = (int64_t)a.window * (D * (int64_t)sizeof(TIn) + 16);
  const int wpc = (int)std::min<int64_t>(kWarps, kMaxDynamic / per_warp);
  done = false;
  if (wpc == 0) return cudaSuccess;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(swa_decode_staged_kernel<TIn, TOut, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kMaxDynamic);
  });
  if (attr != cudaSuccess) return attr;
  const int64_t grid = (a.S * a.H + wpc - 1) / wpc;
  done = true;
  return launch_dependent(swa_decode_staged_kernel<TIn, TOut, D>, dim3((unsigned)grid), dim3(32 * wpc),
                          (size_t)(wpc * per_warp), stream, a);
}

template <typename TIn, typename TOut>
cudaError_t launch_typed(const SwaDecodeLaunch& a, cudaStream_t stream) {
  const bool aligned = ((reinterpret_cast<uintptr_t>(a.k_cache) | reinterpret_cast<uintptr_t>(a.v_cache)) & 15u) == 0;
  if (aligned && (a.d == 64 || a.d == 128)) {
    bool done = false;
    const cudaError_t e = a.d == 64 ? launch_staged<TIn, TOut, 64>(a, stream, done)
                                    : launch_staged<TIn, TOut, 128>(a, stream, done);
    if (e != cudaSuccess || done) return e;
  }
  const int64_t grid = (a.S * a.H + kWarps - 1) / kWarps;
  return launch_dependent(swa_decode_kernel<TIn, TOut>, dim3((unsigned)grid), dim3(32 * kWarps), 0, stream, a);
}

}  // namespace

cudaError_t launch_swa_decode(const SwaDecodeLaunch& a, cudaStream_t stream) {
  if (a.S * a.H == 0) return cudaSuccess;
  if (a.in_bf16 && a.out_bf16) return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, stream);
  if (a.in_bf16) return launch_typed<__nv_bfloat16, float>(a, stream);
  if (a.out_bf16) return launch_typed<float, __nv_bfloat16>(a, stream);
  return launch_typed<float, float>(a, stream);
}

}  // namespace la
