// notebank.cu -- NoteBank's data-parallel write side and routing.
//
// "History Replays Itself: Unleashing Long-Context Capability in Linear
// Attention" (NoteBank), Sec. 2 and App. B:
//   scores   (Eqs. (3), (8))  per write chunk C and channel (l,h):
//            mu_C = unit(mean_{t in C} unit(k_t)),  d_t^{l,h} = 1 - <unit(k_t), mu_C>,
//            d_t = mean over the J = L x H channels, and the sums of d over a
//            sliding window (48 tokens in App. B.2) that the span selection
//            maximises;
//   address  (Eqs. (4), (9))  per note span I_i and channel: t* = argmax_{t in I_i}
//            d_t^{l,h}, rho_i^{l,h} = P^{l,h} q_{t*}: 16 fixed coordinates of the
//            query at t*, stored as bf16;
//   route    (Eq. (5))  s_i^{l,h} = max_tau <unit(u_tau), unit(rho_i)> in fp32, one
//            vote per channel for its argmax note, the at most R notes with the
//            most votes (ties to the earlier note), returned in text order.
// Readings: a zero vector normalises to zero; argmaxes take the earliest
// index on ties; only notes with a vote are retrieved.
//
// All three read their inputs once and are HBM- or latency-bound: the scores
// take one CTA per (channel, chunk) with one warp per token (lanes over the
// key width), the address one warp per (note, channel), the routing one CTA
// per channel over all notes plus one CTA for the vote.
#include <math.h>

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace la {
namespace {
namespace cg = cooperative_groups;

constexpr int kScoreThreads = 256;
constexpr int kMaxD = 256;               // key / query width, multiple of 32
constexpr int kAddr = kNoteAddrDims;     // d_rho = 16
constexpr int kRouteThreads = 256;
constexpr int kMaxQ = 512;               // question tokens held in shared memory

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p) { return to_f(*p); }

// One token row of a channel: lane l holds elements l, l + 32, ... (d / 32 of them).
template <typename T, int PER>
__device__ __forceinline__ void load_row(const T* row, float (&x)[PER]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < PER; ++i) x[i] = ld_elem(row + lane + 32 * i);
}

// ---------------------------------------------------------------- scores
template <typename T, int PER>
__global__ void __launch_bounds__(kScoreThreads)
notebank_chunk_scores_kernel(NotebankScoresLaunch a) {
  grid_dependents_trigger();  // the channel-mean kernel may be scheduled once every CTA is resident
  __shared__ float part[kScoreThreads / 32][kMaxD];
  __shared__ float mu[kMaxD];
  __shared__ float inv_norm[1024];  // per token of the chunk (chunk <= 1024)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kScoreThreads / 32;
  const int64_t nchunks = (a.N + a.chunk - 1) / a.chunk;
  const int64_t ch = blockIdx.x / nchunks, c = blockIdx.x % nchunks;
  const int64_t l = ch / a.H, h = ch % a.H;
  const int64_t t0 = c * a.chunk;
  const int n = (int)min((int64_t)a.chunk, a.N - t0);
  const T* base = reinterpret_cast<const T*>(a.k.ptr) + l * a.k.sb + h * a.k.sh;

  // pass 1: unit keys, their sum (per warp), and each key's inverse norm
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int r = warp; r < n; r += kWarps) {
    float x[PER];
    load_row<T, PER>(base + (t0 + r) * a.k.st, x);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) ss = fmaf(x[i], x[i], ss);
    ss = warp_sum(ss);
    const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;  // a zero key normalises to zero
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = fmaf(x[i], inv, acc[i]);
    if (lane == 0) inv_norm[r] = inv;
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) part[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  // mean direction, normalised (the 1/|C| of the mean cancels)
  if (warp == 0) {
    float m[PER];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += part[w][lane + 32 * i];
      m[i] = s;
      ss = fmaf(s, s, ss);
    }
    ss = warp_sum(ss);
    const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) mu[lane + 32 * i] = m[i] * inv;
  }
  __syncthreads();
  float mv[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) mv[i] = mu[lane + 32 * i];
  // pass 2: d_t = 1 - <k_t, mu> / |k_t| (the chunk's rows come back from L2)
  float* out = a.d_ch + ch * a.N + t0;
  for (int r = warp; r < n; r += kWarps) {
    float x[PER];
    load_row<T, PER>(base + (t0 + r) * a.k.st, x);
    float dt = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) dt = fmaf(x[i], mv[i], dt);
    dt = warp_sum(dt);
    if (lane == 0) out[r] = 1.f - dt * inv_norm[r];
  }
}

// Elements [PER lane, PER lane + PER) of a 16-byte aligned shared-memory row, as floats: one vector
// load per 16 bytes (a warp reads the whole row in d * sizeof(T) / 128 wavefronts).
template <typename T, int PER>
__device__ __forceinline__ void load_lane_run(const T* row, int lane, float (&x)[PER]) {
  const T* p = row + PER * lane;
  constexpr int kBytes = PER * (int)sizeof(T);
  if constexpr (kBytes % 16 == 0) {
#pragma unroll
    for (int v = 0; v < kBytes / 16; ++v) {
      const uint4 u = reinterpret_cast<const uint4*>(p)[v];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x[8 * v + 2 * j] = __uint_as_float(w[j] << 16);
          x[8 * v + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) x[4 * v + j] = __uint_as_float(w[j]);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < PER; ++i) x[i] = to_f(p[i]);
  }
}

// The same scores with each chunk split over a cluster of kClusterCtas CTAs
// that keep their share of the chunk's keys in shared memory: the keys are
// read from HBM once.  Each CTA sums its unit keys; after a cluster barrier
// every warp adds the kClusterCtas partial sums (in rank order, so all get the
// same bits) through distributed shared memory; a second barrier at the end
// keeps every CTA's partial alive until all have read it.
constexpr int kClusterCtas = 4;

template <typename T, int PER>
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kScoreThreads)
notebank_chunk_scores_cluster_kernel(NotebankScoresLaunch a, int sub) {
  extern __shared__ __align__(16) uint8_t nb_smem[];
  T* rows = reinterpret_cast<T*>(nb_smem);                       // [sub][d]
  float* inv_norm = reinterpret_cast<float*>(rows + (int64_t)sub * a.d);  // [sub]
  __shared__ float part[kScoreThreads / 32][kMaxD];
  __shared__ float cpart[kMaxD];  // this CTA's sum of unit keys, read by the whole cluster
  __shared__ float mu[kMaxD];
  grid_dependents_trigger();  // the channel-mean kernel may be scheduled once every CTA is resident
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kScoreThreads / 32;
  const int d = (int)a.d;
  const int64_t nchunks = (a.N + a.chunk - 1) / a.chunk;
  const int64_t item = blockIdx.x / kClusterCtas;
  const int64_t ch = item / nchunks, c = item % nchunks;
  const int64_t l = ch / a.H, h = ch % a.H;
  const int64_t t0 = c * a.chunk;
  const int n = (int)min((int64_t)a.chunk, a.N - t0);
  const int r0 = rank * sub, r1 = min(n, r0 + sub);  // this CTA's rows of the chunk
  const T* base = reinterpret_cast<const T*>(a.k.ptr) + l * a.k.sb + h * a.k.sh;

  // this CTA's rows into shared memory, all requested at once (16-byte copies; the views are
  // 16-byte aligned with rows of d * sizeof(T), a multiple of 64 bytes)
  {
    const int vrow = d * (int)sizeof(T) / 16;
    const int nv = max(r1 - r0, 0) * vrow;
    const uint32_t sdst = tc::smem_u32(nb_smem);
    for (int v = threadIdx.x; v < nv; v += kScoreThreads) {
      const int rr = v / vrow, cv = v - rr * vrow;
      tc::cp_async16(sdst + (uint32_t)(rr * vrow + cv) * 16u,
                     reinterpret_cast<const uint8_t*>(base + (t0 + r0 + rr) * a.k.st) + cv * 16, 16u);
    }
    tc::cp_async_commit();
    tc::cp_async_wait_all();
    __syncthreads();
  }
  // pass 1: inverse norms and the sum of unit keys.  Lane l holds dims [PER l, PER l + PER) of a row;
  // the partial sums, their cluster-wide total and mu keep dim PER l + i at position 32 i + l, so that
  // a warp's accesses to them are free of bank conflicts
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  // kU rows per warp at a time (rows r, r + kWarps, ...): independent load / reduce chains overlap
  constexpr int kU = 4;
  for (int rb = r0 + warp; rb < r1; rb += kU * kWarps) {
    float x[kU][PER], ss[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = rb + u * kWarps;
      if (r < r1) load_lane_run<T, PER>(rows + (int64_t)(r - r0) * d, lane, x[u]);
      else
#pragma unroll
        for (int i = 0; i < PER; ++i) x[u][i] = 0.f;
      ss[u] = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) ss[u] = fmaf(x[u][i], x[u][i], ss[u]);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) ss[u] = warp_sum(ss[u]);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = rb + u * kWarps;
      const float inv = ss[u] > 0.f ? rsqrtf(ss[u]) : 0.f;  // a zero key (or a row past the end) adds nothing
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(x[u][i], inv, acc[i]);
      if (lane == 0 && r < r1) inv_norm[r - r0] = inv;
    }
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) part[warp][32 * i + lane] = acc[i];
  __syncthreads();
  for (int i = warp; i < PER; i += kWarps) {  // the warps' partial sums, warp by warp in a fixed order
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += part[w][32 * i + lane];
    cpart[32 * i + lane] = s;
  }
  cluster.sync();
  // mean direction of the whole chunk, normalised (the 1/|C| of the mean cancels), formed by warp 0 from
  // the kClusterCtas partial sums in rank order (so every CTA gets the same bits)
  if (warp == 0) {
    float m[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) m[i] = 0.f;
    for (int q = 0; q < kClusterCtas; ++q) {
      const float* rp = cluster.map_shared_rank(cpart, q);
#pragma unroll
      for (int i = 0; i < PER; ++i) m[i] += rp[32 * i + lane];
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) ss = fmaf(m[i], m[i], ss);
    ss = warp_sum(ss);
    const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) mu[32 * i + lane] = m[i] * inv;
  }
  __syncthreads();
  float mv[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) mv[i] = mu[32 * i + lane];
  // pass 2 from shared memory: d_t = 1 - <k_t, mu> / |k_t|
  float* out = a.d_ch + ch * a.N + t0;
  for (int rb = r0 + warp; rb < r1; rb += kU * kWarps) {
    float dt[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = rb + u * kWarps;
      float x[PER];
      if (r < r1) load_lane_run<T, PER>(rows + (int64_t)(r - r0) * d, lane, x);
      else
#pragma unroll
        for (int i = 0; i < PER; ++i) x[i] = 0.f;
      dt[u] = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) dt[u] = fmaf(x[i], mv[i], dt[u]);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) dt[u] = warp_sum(dt[u]);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int r = rb + u * kWarps;
      if (lane == 0 && r < r1) out[r] = 1.f - dt[u] * inv_norm[r - r0];
    }
  }
  cluster.sync();  // this CTA's partial sums stay alive until every CTA of the cluster has read them
}

// d_t = mean over the channels (fixed order), and the window sums of d.
// Block b covers tokens [b*256, b*256+256) and recomputes the window's halo.
__global__ void __launch_bounds__(kScoreThreads)
notebank_token_scores_kernel(NotebankScoresLaunch a) {
  extern __shared__ float dsm[];  // kScoreThreads + window - 1 token means
  grid_dependency_wait();  // the channel scores come from the kernel before (launched as its dependent)
  grid_dependents_trigger();
  const int64_t t0 = (int64_t)blockIdx.x * kScoreThreads;
  const int64_t J = a.L * a.H;
  const float invJ = 1.f / (float)J;
  const int span = kScoreThreads + (int)a.window - 1;
  for (int i = threadIdx.x; i < span; i += kScoreThreads) {
    const int64_t t = t0 + i;
    float s = 0.f;
    if (t < a.N)
      for (int64_t j = 0; j < J; ++j) s += a.d_ch[j * a.N + t];
    dsm[i] = s * invJ;
    if (i < kScoreThreads && t < a.N) a.d_mean[t] = dsm[i];
  }
  __syncthreads();
  const int64_t t = t0 + threadIdx.x;
  if (a.w && t + a.window <= a.N) {
    float s = 0.f;
    for (int u = 0; u < (int)a.window; ++u) s += dsm[threadIdx.x + u];
    a.w[t] = s;
  }
}

// ---------------------------------------------------------------- address
template <typename T>
__global__ void __launch_bounds__(256)
notebank_address_kernel(NotebankAddressLaunch a, unsigned* status) {
  grid_dependency_wait();  // the channel scores may come from the kernels just before
  const int64_t J = a.L * a.H;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // (note, channel)
  const int lane = threadIdx.x & 31;
  if (gw >= a.n_notes * J) return;
  const int64_t note = gw / J, ch = gw % J;
  const int64_t l = ch / a.H, h = ch % a.H;
  const int64_t s0 = a.spans[2 * note], len = a.spans[2 * note + 1];
  int32_t* ts = a.t_star + gw;
  __nv_bfloat16* rho = reinterpret_cast<__nv_bfloat16*>(a.rho) + gw * kAddr;
  const bool bad_span = s0 < 0 || len < 1 || s0 + len > a.N;
  const int coord = lane < kAddr ? a.coords[ch * kAddr + lane] : 0;
  const bool bad_coord = __any_sync(kFullMask, lane < kAddr && (coord < 0 || coord >= a.d));
  if (bad_span || bad_coord) {  // reported; the note's outputs are -1 / zeros
    if (lane == 0) {
      atomicOr(status, kStatusBadIndex);
      *ts = -1;
    }
    if (lane < kAddr) rho[lane] = __float2bfloat16_rn(0.f);
    return;
  }
  // argmax over the span, earliest token on ties
  const float* dr = a.d_ch + ch * a.N;
  float best = -INFINITY;
  int64_t bt = s0;
  for (int64_t t = s0 + lane; t < s0 + len; t += 32) {
    const float v = dr[t];
    if (v > best) { best = v; bt = t; }  // lanes see increasing t: the first maximum is kept
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float ov = __shfl_xor_sync(kFullMask, best, off);
    const int64_t ot = __shfl_xor_sync(kFullMask, bt, off);
    if (ov > best || (ov == best && ot < bt)) { best = ov; bt = ot; }
  }
  if (lane == 0) *ts = (int32_t)bt;
  if (lane < kAddr) {
    const T* qrow = reinterpret_cast<const T*>(a.q.ptr) + l * a.q.sb + h * a.q.sh + bt * a.q.st;
    rho[lane] = __float2bfloat16_rn(to_f(qrow[coord]));
  }
}

// ---------------------------------------------------------------- route
__device__ __forceinline__ void load_unit16(const __nv_bfloat16* p, float (&x)[kAddr]) {
  const uint4 a0 = reinterpret_cast<const uint4*>(p)[0];
  const uint4 a1 = reinterpret_cast<const uint4*>(p)[1];
  const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
#pragma unroll
  for (int i = 0; i < kAddr; ++i) ss = fmaf(x[i], x[i], ss);
  const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
  for (int i = 0; i < kAddr; ++i) x[i] *= inv;
}

// One CTA per channel: s_i = max_tau <unit(u_tau), unit(rho_i)> for every note; the channel's
// winner is the first note with the largest s.
__global__ void __launch_bounds__(kRouteThreads)
notebank_route_channel_kernel(NotebankRouteLaunch a) {
  __shared__ float un[kMaxQ][kAddr];
  __shared__ float rbest[kRouteThreads / 32];
  __shared__ int rarg[kRouteThreads / 32];
  const int64_t j = blockIdx.x;
  const __nv_bfloat16* u = reinterpret_cast<const __nv_bfloat16*>(a.u) + j * a.n_q * kAddr;
  for (int t = threadIdx.x; t < a.n_q; t += kRouteThreads) {
    float x[kAddr];
    load_unit16(u + (int64_t)t * kAddr, x);
#pragma unroll
    for (int i = 0; i < kAddr; ++i) un[t][i] = x[i];
  }
  __syncthreads();
  const __nv_bfloat16* rho = reinterpret_cast<const __nv_bfloat16*>(a.rho);
  float best = -INFINITY;
  int barg = 0x7fffffff;
  for (int64_t i = threadIdx.x; i < a.n_notes; i += kRouteThreads) {  // increasing i: first maximum kept
    float x[kAddr];
    load_unit16(rho + (i * a.J + j) * kAddr, x);
    float s = -INFINITY;
    for (int t = 0; t < a.n_q; ++t) {
      float dt = 0.f;
#pragma unroll
      for (int e = 0; e < kAddr; ++e) dt = fmaf(x[e], un[t][e], dt);
      s = fmaxf(s, dt);
    }
    if (a.s) a.s[i * a.J + j] = s;
    if (s > best) { best = s; barg = (int)i; }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float ob = __shfl_xor_sync(kFullMask, best, off);
    const int oa = __shfl_xor_sync(kFullMask, barg, off);
    if (ob > best || (ob == best && oa < barg)) { best = ob; barg = oa; }
  }
  if (lane == 0) { rbest[warp] = best; rarg[warp] = barg; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = rbest[0];
    int g = rarg[0];
    for (int w = 1; w < kRouteThreads / 32; ++w)
      if (rbest[w] > b || (rbest[w] == b && rarg[w] < g)) { b = rbest[w]; g = rarg[w]; }
    a.winner[j] = g;
  }
}

// Votes per note, then the at most R notes with the most votes (ties to the earlier note), in text order.
__global__ void __launch_bounds__(1024)
notebank_vote_kernel(NotebankRouteLaunch a) {
  __shared__ int64_t key_best[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.n_notes == 0) {  // nothing stored yet: no winners, nothing retrieved
    for (int64_t j = tid; j < a.J; j += blockDim.x) a.winner[j] = -1;
    for (int64_t r = tid; r < a.R; r += blockDim.x) a.top[r] = -1;
    return;
  }
  for (int64_t i = tid; i < a.n_notes; i += blockDim.x) a.votes[i] = 0;
  __syncthreads();
  for (int64_t j = tid; j < a.J; j += blockDim.x) atomicAdd(a.votes + a.winner[j], 1);
  __syncthreads();
  // selection key: larger is better; votes in the high bits, earlier note in the low bits
  auto key_of = [&](int64_t i) -> int64_t {
    const int v = a.votes[i];
    return v < 1 ? -1 : ((int64_t)v << 32) | (int64_t)(0x7fffffff - i);
  };
  int64_t chosen_prev = INT64_MAX;  // keys of earlier picks are strictly larger
  int picked = 0;
  for (int r = 0; r < a.R; ++r) {
    int64_t kbest = -1;
    for (int64_t i = tid; i < a.n_notes; i += blockDim.x) {
      const int64_t kk = key_of(i);
      if (kk < chosen_prev && kk > kbest) kbest = kk;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) kbest = max(kbest, (int64_t)__shfl_xor_sync(kFullMask, kbest, off));
    if (lane == 0) key_best[warp] = kbest;
    __syncthreads();
    if (tid == 0) {
      int64_t kb = -1;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) kb = max(kb, key_best[w]);
      key_best[0] = kb;
    }
    __syncthreads();
    const int64_t kb = key_best[0];
    __syncthreads();
    if (kb < 0) break;
    if (tid == 0) a.top[r] = (int32_t)(0x7fffffff - (kb & 0xffffffff));
    chosen_prev = kb;
    ++picked;
  }
  __syncthreads();
  if (tid == 0) {
    for (int r = picked; r < a.R; ++r) a.top[r] = -1;
    // text order: insertion sort of the picks by (position, index)
    for (int x = 1; x < picked; ++x) {
      const int32_t v = a.top[x];
      const int64_t pv = a.positions ? a.positions[v] : v;
      int y = x - 1;
      while (y >= 0) {
        const int32_t w = a.top[y];
        const int64_t pw = a.positions ? a.positions[w] : w;
        if (pw < pv || (pw == pv && w < v)) break;
        a.top[y + 1] = w;
        --y;
      }
      a.top[y + 1] = v;
    }
  }
}

constexpr size_t kClusterSmemMax = 160 * 1024;  // keys of a cluster's share of a chunk, plus norms

template <typename T, int PER>
cudaError_t launch_scores_pd(const NotebankScoresLaunch& a, cudaStream_t stream) {
  const int64_t nchunks = (a.N + a.chunk - 1) / a.chunk;
  const int64_t items = a.L * a.H * nchunks;
  const int sub = (int)((a.chunk + kClusterCtas - 1) / kClusterCtas);
  const size_t smem = (size_t)sub * (size_t)a.d * sizeof(T) + (size_t)sub * sizeof(float);
  if (smem <= kClusterSmemMax && items * kClusterCtas <= (int64_t)INT32_MAX) {
    static cudaError_t attr = cudaFuncSetAttribute(notebank_chunk_scores_cluster_kernel<T, PER>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kClusterSmemMax);
    if (attr != cudaSuccess) return attr;
    notebank_chunk_scores_cluster_kernel<T, PER>
        <<<(unsigned)(items * kClusterCtas), kScoreThreads, smem, stream>>>(a, sub);
  } else {  // the share of a chunk does not fit: two passes over global memory
    notebank_chunk_scores_kernel<T, PER><<<(unsigned)items, kScoreThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_scores_typed(const NotebankScoresLaunch& a, cudaStream_t stream) {
  switch (a.d / 32) {
    case 1: return launch_scores_pd<T, 1>(a, stream);
    case 2: return launch_scores_pd<T, 2>(a, stream);
    case 3: return launch_scores_pd<T, 3>(a, stream);
    case 4: return launch_scores_pd<T, 4>(a, stream);
    case 5: return launch_scores_pd<T, 5>(a, stream);
    case 6: return launch_scores_pd<T, 6>(a, stream);
    case 7: return launch_scores_pd<T, 7>(a, stream);
    default: return launch_scores_pd<T, 8>(a, stream);
  }
}

}  // namespace

cudaError_t launch_notebank_scores(const NotebankScoresLaunch& a, cudaStream_t stream) {
  if (a.L * a.H == 0 || a.N == 0) return cudaSuccess;
  const cudaError_t e = a.in_bf16 ? launch_scores_typed<__nv_bfloat16>(a, stream) : launch_scores_typed<float>(a, stream);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((a.N + kScoreThreads - 1) / kScoreThreads);
  const size_t smem = (size_t)(kScoreThreads + a.window - 1) * sizeof(float);
  return launch_dependent(notebank_token_scores_kernel, dim3(grid), dim3(kScoreThreads), smem, stream, a);
}

cudaError_t launch_notebank_address(const NotebankAddressLaunch& a, unsigned* status, cudaStream_t stream) {
  const int64_t warps = a.n_notes * a.L * a.H;
  if (warps == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  if (a.in_bf16) return launch_dependent(notebank_address_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream, a, status);
  return launch_dependent(notebank_address_kernel<float>, dim3(grid), dim3(256), 0, stream, a, status);
}

cudaError_t launch_notebank_route(const NotebankRouteLaunch& a, cudaStream_t stream) {
  if (a.J == 0) return cudaSuccess;
  if (a.n_notes > 0) {
    notebank_route_channel_kernel<<<(unsigned)a.J, kRouteThreads, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  notebank_vote_kernel<<<1, 1024, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace la
