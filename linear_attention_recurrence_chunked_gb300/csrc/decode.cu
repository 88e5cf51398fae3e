// decode.cu -- one-token recurrent decode steps, state updated in place.
//
// Both kernels are bound by HBM: every step reads and writes the whole fp32
// state once (BASED reading notes Sec. 2.5: the fused decode still reads and
// writes the persistent state).  State rows are moved as coalesced 16-byte
// vectors with streaming cache hints; all of a warp's state loads are issued
// before any arithmetic so each SM keeps many bytes in flight.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

// ---------------------------------------------------------------------------
// Gated DeltaNet decode (NoteBank Sec. 2 Eq. (1), A = alpha (I - beta k k^T)):
//   a_i = S_i . k,  u_i = beta (v_i - alpha a_i),  S_i <- alpha S_i + u_i k^T,
//   o_i = S_i(new) . q = alpha (S_i . q) + u_i (k . q).
// With delta = 0 the same kernel runs the scalar gate A = alpha I
// (u_i = beta v_i).
// One CTA per (sequence, head); 8 warps x 16 rows; a lane holds 4 of the 128
// columns of each of its warp's rows.
constexpr int kGdnD = 128;
constexpr int kGdnRowsPerWarp = 16;
constexpr int kGdnThreads = 32 * (kGdnD / kGdnRowsPerWarp);

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kGdnThreads)
gdn_decode_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                  const float* __restrict__ alpha, const float* __restrict__ beta,
                  TOut* __restrict__ out, float* __restrict__ state, float q_scale, float delta) {
  const int64_t sh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = warp * kGdnRowsPerWarp;
  float* S = state + sh * (kGdnD * kGdnD) + (int64_t)row0 * kGdnD;
  grid_dependents_trigger();
  grid_dependency_wait();  // the previous step's state and this step's inputs are in memory

  float4 s[kGdnRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kGdnRowsPerWarp; ++r)
    s[r] = __ldcs(reinterpret_cast<const float4*>(S + r * kGdnD) + lane);

  const float4 kk = load4(k + sh * kGdnD + lane * 4);
  float4 qq = load4(q + sh * kGdnD + lane * 4);
  qq.x *= q_scale; qq.y *= q_scale; qq.z *= q_scale; qq.w *= q_scale;
  const float vv = lane < kGdnRowsPerWarp ? to_f(v[sh * kGdnD + row0 + lane]) : 0.f;
  const float al = alpha[sh], be = beta[sh];
  const float kq = warp_sum(dot4(kk, qq));

  // lanes 0..15 end with a_r = S_r . k, lanes 16..31 with c_r = S_r . q
  float part[2 * kGdnRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kGdnRowsPerWarp; ++r) {
    part[r] = dot4(s[r], kk);
    part[kGdnRowsPerWarp + r] = dot4(s[r], qq);
  }
  const float red = warp_reduce_scatter<2 * kGdnRowsPerWarp>(part);
  const float u = be * (vv - delta * (al * red));              // valid on lanes 0..15
  const float u_mate = __shfl_xor_sync(kFullMask, u, 16);      // lanes 16..31 get u_{lane-16}
  if (lane >= kGdnRowsPerWarp)
    store1(out + sh * kGdnD + row0 + (lane - kGdnRowsPerWarp), al * red + u_mate * kq);

#pragma unroll
  for (int r = 0; r < kGdnRowsPerWarp; ++r) {
    const float ur = __shfl_sync(kFullMask, u, r);
    float4 x = s[r];
    x.x = fmaf(al, x.x, ur * kk.x);
    x.y = fmaf(al, x.y, ur * kk.y);
    x.z = fmaf(al, x.z, ur * kk.z);
    x.w = fmaf(al, x.w, ur * kk.w);
    __stcs(reinterpret_cast<float4*>(S + r * kGdnD) + lane, x);
  }
}

// ---------------------------------------------------------------------------
// Taylor / BASED decode (BASED notes Sec. 2.2):
//   s_j <- s_j + phi(k)_j v,  z_j <- z_j + phi(k)_j,
//   y = (sum_j phi(q)_j s_j) / (sum_j phi(q)_j z_j + eps)   (new state).
// One CTA per (sequence, head); thread (rg, cg) owns columns 4cg..4cg+3 of
// rows j = rg, rg+16, ...; phi entries are formed on the fly from the 16
// projected coordinates held in shared memory.
constexpr int kTayF = 16;
constexpr int kTayDv = 64;
constexpr int kTayD = 1 + kTayF + kTayF * kTayF;  // 273
constexpr int kTayThreads = 256;
constexpr int kTayRowGroups = kTayThreads / (kTayDv / 4);  // 16
constexpr int kTayRowsPerThread = (kTayD + kTayRowGroups - 1) / kTayRowGroups;  // 18

__device__ __forceinline__ float taylor_phi(const float* x, int j) {
  if (j == 0) return 1.f;
  if (j <= kTayF) return x[j - 1];
  const int t = j - 1 - kTayF;
  return x[t >> 4] * x[t & 15] * 0.70710678118654752f;
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kTayThreads)
taylor_decode_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                     TOut* __restrict__ out, float* __restrict__ s_state, float* __restrict__ z_state,
                     float eps, const float* __restrict__ decay, int64_t H) {
  __shared__ float xk[kTayF], xq[kTayF];
  __shared__ float4 red[kTayRowGroups][kTayDv / 4];
  __shared__ float dred[kTayThreads / 32];
  const int64_t sh = blockIdx.x;
  const int tid = threadIdx.x, cg = tid & 15, rg = tid >> 4;
  float* s = s_state + sh * (kTayD * kTayDv);
  float* z = z_state + sh * kTayD;
  grid_dependents_trigger();
  grid_dependency_wait();  // the previous step's state and this step's inputs are in memory
  const float lam = decay ? decay[sh % H] : 1.f;  // s <- lam s + phi(k) v^T, z <- lam z + phi(k)

  float4 sv[kTayRowsPerThread];
#pragma unroll
  for (int i = 0; i < kTayRowsPerThread; ++i) {
    const int j = rg + kTayRowGroups * i;
    if (j < kTayD) sv[i] = __ldcs(reinterpret_cast<const float4*>(s + j * kTayDv) + cg);
  }
  float zv0 = __ldcs(z + tid);
  float zv1 = tid + kTayThreads < kTayD ? __ldcs(z + tid + kTayThreads) : 0.f;
  if (tid < kTayF) xk[tid] = to_f(k[sh * kTayF + tid]);
  else if (tid < 2 * kTayF) xq[tid - kTayF] = to_f(q[sh * kTayF + tid - kTayF]);
  const float4 vv = load4(v + sh * kTayDv + cg * 4);
  __syncthreads();

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kTayRowsPerThread; ++i) {
    const int j = rg + kTayRowGroups * i;
    if (j < kTayD) {
      const float fk = taylor_phi(xk, j), fq = taylor_phi(xq, j);
      float4 x = sv[i];
      x.x = fmaf(fk, vv.x, lam * x.x);
      x.y = fmaf(fk, vv.y, lam * x.y);
      x.z = fmaf(fk, vv.z, lam * x.z);
      x.w = fmaf(fk, vv.w, lam * x.w);
      __stcs(reinterpret_cast<float4*>(s + j * kTayDv) + cg, x);
      acc.x = fmaf(fq, x.x, acc.x);
      acc.y = fmaf(fq, x.y, acc.y);
      acc.z = fmaf(fq, x.z, acc.z);
      acc.w = fmaf(fq, x.w, acc.w);
    }
  }
  // normaliser rows: thread t owns z_t and z_{t+256}
  float dpart;
  {
    zv0 = fmaf(lam, zv0, taylor_phi(xk, tid));
    __stcs(z + tid, zv0);
    dpart = taylor_phi(xq, tid) * zv0;
    if (tid + kTayThreads < kTayD) {
      zv1 = fmaf(lam, zv1, taylor_phi(xk, tid + kTayThreads));
      __stcs(z + tid + kTayThreads, zv1);
      dpart = fmaf(taylor_phi(xq, tid + kTayThreads), zv1, dpart);
    }
  }
  red[rg][cg] = acc;
  dpart = warp_sum(dpart);
  if ((tid & 31) == 0) dred[tid >> 5] = dpart;
  __syncthreads();
  if (tid < kTayDv) {
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kTayThreads / 32; ++w) den += dred[w];
    const float* redf = reinterpret_cast<const float*>(&red[0][0]);
    float num = 0.f;
#pragma unroll
    for (int g = 0; g < kTayRowGroups; ++g) num += redf[g * kTayDv + tid];
    store1(out + sh * kTayDv + tid, num / (den + eps));
  }
}

}  // namespace

cudaError_t launch_gdn_decode(const DecodeLaunch& a, cudaStream_t stream) {
  const unsigned grid = (unsigned)(a.S * a.H);
  if (grid == 0) return cudaSuccess;
  cudaError_t e;
#define LA_GDN_DECODE(TI, TO)                                                                    \
  e = launch_dependent(gdn_decode_kernel<TI, TO>, dim3(grid), dim3(kGdnThreads), 0, stream, (const TI*)a.q,   \
                       (const TI*)a.k, (const TI*)a.v, a.alpha, a.beta, (TO*)a.out, a.state, a.q_scale, a.delta)
  if (a.in_bf16 && a.out_bf16) LA_GDN_DECODE(__nv_bfloat16, __nv_bfloat16);
  else if (a.in_bf16) LA_GDN_DECODE(__nv_bfloat16, float);
  else if (a.out_bf16) LA_GDN_DECODE(float, __nv_bfloat16);
  else LA_GDN_DECODE(float, float);
#undef LA_GDN_DECODE
  return e;
}

cudaError_t launch_taylor_decode(const DecodeLaunch& a, cudaStream_t stream) {
  const unsigned grid = (unsigned)(a.S * a.H);
  if (grid == 0) return cudaSuccess;
  cudaError_t e;
#define LA_TAY_DECODE(TI, TO)                                                                    \
  e = launch_dependent(taylor_decode_kernel<TI, TO>, dim3(grid), dim3(kTayThreads), 0, stream, (const TI*)a.q, \
                       (const TI*)a.k, (const TI*)a.v, (TO*)a.out, a.state, a.z, a.eps, a.decay, a.H)
  if (a.in_bf16 && a.out_bf16) LA_TAY_DECODE(__nv_bfloat16, __nv_bfloat16);
  else if (a.in_bf16) LA_TAY_DECODE(__nv_bfloat16, float);
  else if (a.out_bf16) LA_TAY_DECODE(float, __nv_bfloat16);
  else LA_TAY_DECODE(float, float);
#undef LA_TAY_DECODE
  return e;
}

}  // namespace la
