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
// slot first, so all slots are read alike.
#include "common.cuh"
#include "kernels.h"

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
  if (sh >= a.S * a.H) return;
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

}  // namespace

cudaError_t launch_swa_decode(const SwaDecodeLaunch& a, cudaStream_t stream) {
  const int64_t grid = (a.S * a.H + kWarps - 1) / kWarps;
  if (grid == 0) return cudaSuccess;
#define LA_SWA(TI, TO) swa_decode_kernel<TI, TO><<<(unsigned)grid, 32 * kWarps, 0, stream>>>(a)
  if (a.in_bf16 && a.out_bf16) LA_SWA(__nv_bfloat16, __nv_bfloat16);
  else if (a.in_bf16) LA_SWA(__nv_bfloat16, float);
  else if (a.out_bf16) LA_SWA(float, __nv_bfloat16);
  else LA_SWA(float, float);
#undef LA_SWA
  return cudaGetLastError();
}

}  // namespace la
