// prefill_recurrent.cu -- token-serial prefill kernels (fp32 CUDA cores).
//
// Each CTA walks the sequence one token at a time with its slice of the
// state held in registers, exactly as the recurrence reads
// (NoteBank Sec. 2 Eq. (1); BASED reading notes Sec. 2.2).  These serve fp32
// inputs, whose 1e-4 accuracy contract the bf16 tensor-core chunk kernels
// cannot meet; bf16 inputs take the chunked kernels.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

template <typename T>
__device__ __forceinline__ const T* at(const View4& x, int64_t b, int64_t h, int64_t t) {
  return reinterpret_cast<const T*>(x.ptr) + b * x.sb + h * x.sh + t * x.st;
}

// ---------------------------------------------------------------------------
// Gated DeltaNet: CTA = (b, h, 32-row slab of S); 4 warps x 8 rows.
constexpr int kD = 128;
constexpr int kRowsPerWarp = 8;
constexpr int kWarps = 4;
constexpr int kSlab = kRowsPerWarp * kWarps;

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(32 * kWarps)
gdn_prefill_recurrent_kernel(GdnPrefillLaunch a) {
  const int slabs = kD / kSlab;
  const int64_t bh = blockIdx.x / slabs;
  const int slab = blockIdx.x % slabs;
  const int64_t b = bh / a.H, h = bh % a.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = slab * kSlab + warp * kRowsPerWarp;

  float4 s[kRowsPerWarp];
  const int64_t st_off = bh * kD * kD + (int64_t)row0 * kD;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
    s[r] = a.S_in ? *(reinterpret_cast<const float4*>(a.S_in + st_off + r * kD) + lane)
                  : make_float4(0.f, 0.f, 0.f, 0.f);

  const float* al_p = a.alpha + b * a.a_sb + h * a.a_sh;
  const float* be_p = a.beta + b * a.b_sb + h * a.b_sh;
  TOut* o_base = reinterpret_cast<TOut*>(a.o) + b * a.o_sb + h * a.o_sh;
  const int my_row = row0 + (lane >> 1);  // row whose v this lane needs (lanes 0..15)

  float4 kk, qq;
  float vv = 0.f, al = 0.f, be = 0.f;
  auto fetch = [&](int64_t t, float4& k4, float4& q4, float& v1, float& a1, float& b1) {
    k4 = load4(at<TIn>(a.k, b, h, t) + lane * 4);
    q4 = load4(at<TIn>(a.q, b, h, t) + lane * 4);
    v1 = lane < 16 ? to_f(at<TIn>(a.v, b, h, t)[my_row]) : 0.f;
    a1 = al_p[t];
    b1 = be_p[t];
  };
  if (a.N > 0) fetch(0, kk, qq, vv, al, be);
  for (int64_t t = 0; t < a.N; ++t) {
    float4 kn = kk, qn = qq;
    float vn = 0.f, aln = 0.f, ben = 0.f;
    if (t + 1 < a.N) fetch(t + 1, kn, qn, vn, aln, ben);
    float4 q4 = qq;
    q4.x *= a.q_scale; q4.y *= a.q_scale; q4.z *= a.q_scale; q4.w *= a.q_scale;
    const float kq = warp_sum(dot4(kk, q4));
    float part[2 * kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      part[r] = dot4(s[r], kk);
      part[kRowsPerWarp + r] = dot4(s[r], q4);
    }
    // lane l: index l>>1 -> lanes 0..15 hold a_{l>>1}, lanes 16..31 hold c_{(l-16)>>1}
    const float red = warp_reduce_scatter<2 * kRowsPerWarp>(part);
    const float u = be * (vv - a.delta * (al * red));  // delta = 0: the scalar gate writes beta v
    const float u_mate = __shfl_xor_sync(kFullMask, u, 16);
    if (lane >= 16 && (lane & 1) == 0)
      store1(o_base + t * a.o_st + row0 + ((lane - 16) >> 1), al * red + u_mate * kq);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const float ur = __shfl_sync(kFullMask, u, 2 * r);
      s[r].x = fmaf(al, s[r].x, ur * kk.x);
      s[r].y = fmaf(al, s[r].y, ur * kk.y);
      s[r].z = fmaf(al, s[r].z, ur * kk.z);
      s[r].w = fmaf(al, s[r].w, ur * kk.w);
    }
    kk = kn; qq = qn; vv = vn; al = aln; be = ben;
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
    *(reinterpret_cast<float4*>(a.S_out + st_off + r * kD) + lane) = s[r];
}

// ---------------------------------------------------------------------------
// Taylor / BASED: CTA = (b, h), 256 threads; thread (rg, cg) owns columns
// 4cg..4cg+3 of state rows rg, rg+16, ...; one barrier per token.
constexpr int kF = 16;
constexpr int kDv = 64;
constexpr int kDt = 1 + kF + kF * kF;  // 273
constexpr int kTThreads = 256;
constexpr int kRG = 16;
constexpr int kRowsPerThread = (kDt + kRG - 1) / kRG;  // 18

__device__ __forceinline__ float phi_at(const float* x, int j) {
  if (j == 0) return 1.f;
  if (j <= kF) return x[j - 1];
  const int t = j - 1 - kF;
  return x[t >> 4] * x[t & 15] * 0.70710678118654752f;
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kTThreads)
taylor_prefill_recurrent_kernel(TaylorPrefillLaunch a) {
  __shared__ float xk[2][kF], xq[2][kF];
  __shared__ float4 red[2][kRG][kDv / 4];
  __shared__ float dred[2][kTThreads / 32];
  const int64_t bh = blockIdx.x;
  const int64_t b = bh / a.H, h = bh % a.H;
  const int tid = threadIdx.x, cg = tid & 15, rg = tid >> 4;
  const float lam = a.decay ? a.decay[h] : 1.f;  // s <- lam s + phi(k) v^T, z <- lam z + phi(k)

  float4 sv[kRowsPerThread];
  const float* s_in = a.s_in ? a.s_in + bh * kDt * kDv : nullptr;
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i) {
    const int j = rg + kRG * i;
    sv[i] = (s_in && j < kDt) ? *(reinterpret_cast<const float4*>(s_in + j * kDv) + cg)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float* z_in = a.z_in ? a.z_in + bh * kDt : nullptr;
  float zv0 = z_in ? z_in[tid] : 0.f;
  float zv1 = (z_in && tid + kTThreads < kDt) ? z_in[tid + kTThreads] : 0.f;
  TOut* y_base = reinterpret_cast<TOut*>(a.y) + b * a.y_sb + h * a.y_sh;

  float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (a.N > 0) {
    if (tid < kF) xk[0][tid] = to_f(at<TIn>(a.k, b, h, 0)[tid]);
    else if (tid < 2 * kF) xq[0][tid - kF] = to_f(at<TIn>(a.q, b, h, 0)[tid - kF]);
    vv = load4(at<TIn>(a.v, b, h, 0) + cg * 4);
  }
  __syncthreads();
  for (int64_t t = 0; t < a.N; ++t) {
    const int buf = (int)(t & 1);
    float xn = 0.f;
    float4 vn = vv;
    if (t + 1 < a.N) {
      if (tid < kF) xn = to_f(at<TIn>(a.k, b, h, t + 1)[tid]);
      else if (tid < 2 * kF) xn = to_f(at<TIn>(a.q, b, h, t + 1)[tid - kF]);
      vn = load4(at<TIn>(a.v, b, h, t + 1) + cg * 4);
    }
    const float* xkb = xk[buf];
    const float* xqb = xq[buf];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int j = rg + kRG * i;
      if (j < kDt) {
        const float fk = phi_at(xkb, j), fq = phi_at(xqb, j);
        sv[i].x = fmaf(fk, vv.x, lam * sv[i].x);
        sv[i].y = fmaf(fk, vv.y, lam * sv[i].y);
        sv[i].z = fmaf(fk, vv.z, lam * sv[i].z);
        sv[i].w = fmaf(fk, vv.w, lam * sv[i].w);
        acc.x = fmaf(fq, sv[i].x, acc.x);
        acc.y = fmaf(fq, sv[i].y, acc.y);
        acc.z = fmaf(fq, sv[i].z, acc.z);
        acc.w = fmaf(fq, sv[i].w, acc.w);
      }
    }
    zv0 = fmaf(lam, zv0, phi_at(xkb, tid));
    float dpart = phi_at(xqb, tid) * zv0;
    if (tid + kTThreads < kDt) {
      zv1 = fmaf(lam, zv1, phi_at(xkb, tid + kTThreads));
      dpart = fmaf(phi_at(xqb, tid + kTThreads), zv1, dpart);
    }
    red[buf][rg][cg] = acc;
    dpart = warp_sum(dpart);
    if ((tid & 31) == 0) dred[buf][tid >> 5] = dpart;
    if (t + 1 < a.N) {
      if (tid < kF) xk[buf ^ 1][tid] = xn;
      else if (tid < 2 * kF) xq[buf ^ 1][tid - kF] = xn;
    }
    __syncthreads();
    if (tid < kDv) {
      float den = 0.f;
#pragma unroll
      for (int w = 0; w < kTThreads / 32; ++w) den += dred[buf][w];
      const float* redf = reinterpret_cast<const float*>(&red[buf][0][0]);
      float num = 0.f;
#pragma unroll
      for (int g = 0; g < kRG; ++g) num += redf[g * kDv + tid];
      store1(y_base + t * a.y_st + tid, num / (den + a.eps));
    }
    vv = vn;
  }
  float* s_out = a.s_out + bh * kDt * kDv;
#pragma unroll
  for (int i = 0; i < kRowsPerThread; ++i) {
    const int j = rg + kRG * i;
    if (j < kDt) *(reinterpret_cast<float4*>(s_out + j * kDv) + cg) = sv[i];
  }
  float* z_out = a.z_out + bh * kDt;
  z_out[tid] = zv0;
  if (tid + kTThreads < kDt) z_out[tid + kTThreads] = zv1;
}

}  // namespace

cudaError_t launch_gdn_prefill_recurrent(const GdnPrefillLaunch& a, cudaStream_t stream) {
  const int64_t grid = a.B * a.H * (kD / kSlab);
  if (grid == 0) return cudaSuccess;
#define LA_GDN_PF(TI, TO) gdn_prefill_recurrent_kernel<TI, TO><<<(unsigned)grid, 32 * kWarps, 0, stream>>>(a)
  if (a.in_bf16 && a.out_bf16) LA_GDN_PF(__nv_bfloat16, __nv_bfloat16);
  else if (a.in_bf16) LA_GDN_PF(__nv_bfloat16, float);
  else if (a.out_bf16) LA_GDN_PF(float, __nv_bfloat16);
  else LA_GDN_PF(float, float);
#undef LA_GDN_PF
  return cudaGetLastError();
}

cudaError_t launch_taylor_prefill_recurrent(const TaylorPrefillLaunch& a, cudaStream_t stream) {
  const int64_t grid = a.B * a.H;
  if (grid == 0) return cudaSuccess;
#define LA_TAY_PF(TI, TO) taylor_prefill_recurrent_kernel<TI, TO><<<(unsigned)grid, kTThreads, 0, stream>>>(a)
  if (a.in_bf16 && a.out_bf16) LA_TAY_PF(__nv_bfloat16, __nv_bfloat16);
  else if (a.in_bf16) LA_TAY_PF(__nv_bfloat16, float);
  else if (a.out_bf16) LA_TAY_PF(float, __nv_bfloat16);
  else LA_TAY_PF(float, float);
#undef LA_TAY_PF
  return cudaGetLastError();
}

}  // namespace la
