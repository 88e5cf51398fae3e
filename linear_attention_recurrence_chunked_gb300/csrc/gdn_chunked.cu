// gdn_chunked.cu -- chunked gated-delta-rule prefill on the tcgen05 tensor cores.
//
// Recurrence (NoteBank Sec. 2 Eq. (1) with A_t = alpha_t (I - beta_t k_t k_t^T)):
//   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,  o_t = S_t q_t.
// Chunk form for a chunk of C tokens with incoming state S0 (an exact
// re-association of the recurrence; the state is carried across chunk
// boundaries as in NoteBank Sec. 3.2):
//   g_r = sum_{j<=r} log alpha_j,  gamma_r = e^{g_r},  Gamma_rj = e^{g_r - g_j}
//   L   = strict_lower(diag(beta) (Gamma . K K^T)),   T = (I + L)^{-1}
//   W   = T diag(beta gamma) K,   U~ = T diag(beta) V,   U = U~ - W S0^T
//   O   = diag(gamma) Q S0^T + (tril(Gamma) . Q K^T) U     (times q_scale: O is linear in Q)
//   S_C = gamma_C S0 + U^T diag(gamma_C / gamma) K
//
// One CTA per (batch, head) walks the chunks in order with the fp32 state S
// resident in tensor memory.  Every product is issued as a tcgen05 MMA with
// M = 128 by putting the 128-wide head dimension on M (the transposed
// products W^T, U~^T, (S0 W^T), (S0 Q^T), (P U)^T), except [K;Q] K^T where
// the K and Q tiles of the chunk are stacked into one 128-row operand.
// Tiles arrive by TMA into a two-stage ring; the next chunk's tiles load
// while the current one is processed.  T is inverted on the CUDA cores by
// doubling: 16x16 diagonal blocks by forward substitution, then 32x32 and
// 64x64 blocks from [[A,0],[C,B]]^-1 = [[A^-1,0],[-B^-1 C A^-1, B^-1]].
// Two threads share each tensor-memory lane and split its columns.
//
// Sequence segments (few (b,h) pairs, long N).  With d_v = d_k a segment
// acts on the incoming state as an affine map S_end = S_start M + B.  Pass 1
// runs the same chunk scan over every segment but the last twice, writing no
// outputs: from S = 0 (its final state is B_g) and from S = I with V taken
// as zero (the recurrence is then linear in S, so the final state is M_g).
// A small fp32 kernel chains E_{g+1} = E_g M_g + B_g into every segment's
// entry state; pass 2 reruns each segment from its entry state and writes
// the outputs, and the last segment the final state.
#include <mutex>

#include "gdn_common.cuh"

namespace la {
namespace {
using namespace tc;
using namespace gdn;

// shared memory map, offsets from a 1024-byte aligned base
constexpr uint32_t kStageBytes = 49152;   // [K;Q] tile [128][128] bf16 (32 KB) + V [64][128] (16 KB)
constexpr uint32_t kOffKQ = 0;            // within a stage
constexpr uint32_t kOffV = 32768;         // within a stage
constexpr uint32_t kOffS0 = 2 * kStageBytes;      // bf16 S0 [128 i][128 k], K-major
constexpr uint32_t kOffW = kOffS0 + 32768;        // bf16 W [64 r][128 k], K-major
constexpr uint32_t kOffT1 = kOffW + 16384;        // bf16 T diag(beta gamma) [64 r][64 j]
constexpr uint32_t kOffT2 = kOffT1 + 8192;        // bf16 T diag(beta)       [64 r][64 j]
constexpr uint32_t kOffPo = kOffT2 + 8192;        // 2 x bf16 tril(Gamma) . Q K^T [64 r][64 j]
constexpr uint32_t kOffU = kOffPo + 16384;        // bf16 U^T [128 i][64 j]
constexpr uint32_t kOffUD = kOffU + 16384;        // bf16 U^T diag(gamma_C/gamma) [128 i][64 j]
constexpr uint32_t kOffGate = kOffUD + 16384;     // 2 x fp32 {g, beta, gamma, 1/gamma}[64]
constexpr uint32_t kSmemUsed = kOffGate + 2048;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;
// Scratch of the inversion of the NEXT chunk, in tiles that are dead meanwhile:
// L and the block products live in the S0 tile (read by MMA 3 before, rewritten
// after), T in fp32 in the W tile (read by MMA 3 before, rewritten after).
constexpr uint32_t kOffL = kOffS0;                // fp32 L [64][65]
constexpr uint32_t kOffZ = kOffL + 64 * 65 * 4;   // fp32 block products (4 KB)
static_assert(64 * 65 * 4 + 1024 * 4 <= 32768, "L/Z scratch exceeds the S0 tile");
static_assert(64 * kTStride * 4 <= 16384, "T scratch exceeds the W tile");
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// tensor-memory columns (fp32, lane = row of the M = 128 accumulator)
constexpr uint32_t kColS = 0;     // S [i][k], 128 columns
constexpr uint32_t kColKQ = 128;  // lanes 0..63: K K^T, lanes 64..127: Q K^T (64 columns)
constexpr uint32_t kColW = 192;   // W^T [k][r]
constexpr uint32_t kColUt = 256;  // U~^T [i][r]
constexpr uint32_t kColX = 320;   // (W S0^T)^T [i][r]
constexpr uint32_t kColY = 384;   // (Q S0^T)^T [i][r]
constexpr uint32_t kColPU = 448;  // (P_o U)^T [i][r]
constexpr uint32_t kTmemCols = 512;

template <typename TOut>
__global__ void __launch_bounds__(kThreads, 1)
gdn_chunked_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const GdnPrefillLaunch a, const GdnTask task,
                   unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_tma[2];
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base_sh;
  __shared__ float warp0_total;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127;   // tensor-memory lane owned with the partner thread
  const int half = tid >> 7;   // which half of the lane's columns
  const CtaWork wk = cta_work(a, task, (int)blockIdx.x);
  const int b = wk.b, h = wk.h;
  const int64_t t_begin = wk.t_begin, t_end = wk.t_end;
  const int64_t N = t_end;
  const int nchunks = wk.nchunks;
  const bool zero_v = wk.zero_v, write_out = wk.write_out;
  const float* s_entry = wk.s_entry;
  float* s_exit = wk.s_exit;
  float* Lsm = reinterpret_cast<float*>(sm + kOffL);
  float* Tsm = reinterpret_cast<float*>(sm + kOffW);
  float* Zsm = reinterpret_cast<float*>(sm + kOffZ);
  const uint32_t sbase = smem_u32(sm);
  const float* al_p = a.alpha + b * a.a_sb + h * a.a_sh;
  const float* be_p = a.beta + b * a.b_sb + h * a.b_sh;
  // per-chunk gate tables, double-buffered by chunk parity
  auto gsm = [&](int c) { return reinterpret_cast<float*>(sm + kOffGate + (c & 1) * 1024); };  // g_r
  auto gam = [&](int c) { return gsm(c) + 2 * kC; };  // gamma_r = e^{g_r}
  auto gin = [&](int c) { return gsm(c) + 3 * kC; };  // 1 / gamma_r
  auto stage = [&](int c) { return sbase + (uint32_t)(c & 1) * kStageBytes; };
  auto po = [&](int c) { return (uint32_t)kOffPo + (uint32_t)(c & 1) * 8192u; };

  if (tid == 0) {
    mbar_init(smem_u32(&bar_tma[0]), 1);
    mbar_init(smem_u32(&bar_tma[1]), 1);
    mbar_init(smem_u32(&bar_mma), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lane quarter

  auto issue_tma = [&](int c) {
    const uint32_t st = stage(c);
    const uint32_t bar = smem_u32(&bar_tma[c & 1]);
    const int t0 = (int)(t_begin + (int64_t)c * kC);
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_4d(st + kOffKQ + 0, &tmap_k, 0, t0, h, b, bar);
    tma_load_4d(st + kOffKQ + 16384, &tmap_k, 64, t0, h, b, bar);
    tma_load_4d(st + kOffKQ + 8192, &tmap_q, 0, t0, h, b, bar);
    tma_load_4d(st + kOffKQ + 24576, &tmap_q, 64, t0, h, b, bar);
    tma_load_4d(st + kOffV + 0, &tmap_v, 0, t0, h, b, bar);
    tma_load_4d(st + kOffV + 8192, &tmap_v, 64, t0, h, b, bar);
  };
  int tma_issued = 0;   // chunks whose loads have been issued (meaningful in thread 0)
  int tma_waited = 0;   // chunks whose loads have been waited for
  if (tid == 0) {
    issue_tma(0);
    tma_issued = 1;
    if (nchunks > 1) {
      issue_tma(1);
      tma_issued = 2;
    }
  }

  // Initial state: lane i holds row i of S; this thread columns [64 half, 64 half + 64).
  {
    const float* src = s_entry ? s_entry + (int64_t)row * kD + 64 * half : nullptr;
    float v[64];
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      const float4 x = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[j] = x.x; v[j + 1] = x.y; v[j + 2] = x.z; v[j + 3] = x.w;
    }
    if (zero_v) {  // identity entry state: the run then yields the segment's linear map M_g
#pragma unroll
      for (int j = 0; j < 64; ++j) v[j] = (64 * half + j == row) ? 1.f : 0.f;
    }
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) tmem_st16(tlane + kColS + 64 * half + c0, *reinterpret_cast<float(*)[16]>(v + c0));
    tmem_st_wait();
  }

  auto load_gates = [&](int c, float& lg, float& bt) {
    const int64_t t = t_begin + (int64_t)c * kC + tid;
    if (tid < kC && c < nchunks && t < t_end) {
      lg = logf(al_p[t]);
      bt = be_p[t];
    } else {
      lg = 0.f;
      bt = 0.f;
    }
  };
  float lg_next = 0.f, bt_next = 0.f;
  load_gates(0, lg_next, bt_next);

  uint32_t mma_phase = 0;
  bool ok = true;
  bool mma_pending = false;

  // ---------------------------------------------------------------- phases
  // gates of chunk cc: inclusive scan of log alpha (threads 0..63); ends with a barrier
  auto phase_gates = [&](int cc) {
    const float lg = lg_next, bt = bt_next;
    load_gates(cc + 1, lg_next, bt_next);
    gate_tables(tid, lg, bt, gsm(cc), &warp0_total);
  };
  auto wait_tma = [&](int cc) {
    ok = ok && mbar_wait(smem_u32(&bar_tma[cc & 1]), (uint32_t)((cc >> 1) & 1), status);
    tma_waited = cc + 1;
  };
  auto wait_mma = [&]() {
    ok = ok && mbar_wait(smem_u32(&bar_mma), mma_phase, status);
    mma_phase ^= 1;
    mma_pending = !ok;
  };
  auto mma_kq_of = [&](int cc) { mma_kq(tmem + kColKQ, stage(cc) + kOffKQ); };  // [K;Q] K^T of chunk cc -> KQ
  // L (into the S0-tile scratch) and P_o of chunk cc from KQ
  auto phase_L_Po_of = [&](int cc) { phase_L_Po(tlane + kColKQ + 32 * half, row, half, gsm(cc), Lsm, sm + po(cc), 1.f, a.delta); };
  // T = (I + L)^{-1} of chunk cc, then the bf16 tiles T diag(beta gamma), T diag(beta)
  auto phase_T_of = [&](int cc) {
    phase_T(tid, Lsm, [&](int r) { return Tsm + r * kTStride; }, Zsm, gsm(cc), zero_v, a.delta, sm + kOffT1,
            sm + kOffT2);
  };
  // W^T = K^T (T diag(beta gamma))^T, U~^T = V^T (T diag(beta))^T of chunk cc
  auto mma_wu_of = [&](int cc) {
    mma_wu(tmem + kColW, tmem + kColUt, stage(cc) + kOffKQ, stage(cc) + kOffV, sbase + kOffT1, sbase + kOffT2);
  };
  auto phase_Wtile = [&]() {  // lane k, rows r in [32 half, 32 half + 32)
    float w[32];
    ld32(tlane + kColW + 32 * half, w);
#pragma unroll
    for (int r = 0; r < 32; ++r) st_bf16(sm + kOffW + sw128_off(32 * half + r, row, 64), w[r]);
  };
  auto sync_for_mma = [&]() {  // generic-proxy tile writes -> visible to the tensor cores
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };

  // ---------------------------------------------------------------- prologue: intra-chunk work of chunk 0
  phase_gates(0);
  if (tid == 0) wait_tma(0);
  if (__syncthreads_or(!ok)) goto done;
  if (tid == 0) {
    tc_fence_after();
    mma_kq_of(0);
    mma_commit(smem_u32(&bar_mma));
  }
  mma_pending = true;
  wait_mma();
  if (__syncthreads_or(!ok)) goto done;
  tc_fence_after();
  phase_L_Po_of(0);
  __syncthreads();
  phase_T_of(0);
  sync_for_mma();
  if (tid == 0) {
    mma_wu_of(0);
    mma_commit(smem_u32(&bar_mma));
  }
  mma_pending = true;
  // the S0 tile (its region held the inversion scratch) gets the initial state now
  {
    float v[64];
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) tmem_ld16(tlane + kColS + 64 * half + c0, *reinterpret_cast<float(*)[16]>(v + c0));
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<uint4*>(sm + kOffS0 + sw128_off(row, 64 * half + 8 * q, 128)) = pack8_bf16(v + 8 * q);
  }
  wait_mma();
  if (__syncthreads_or(!ok)) goto done;
  tc_fence_after();
  phase_Wtile();
  sync_for_mma();

  // ---------------------------------------------------------------- main loop: chain of chunk c, intra of c+1
  for (int c = 0; c < nchunks; ++c) {
    const bool has_next = c + 1 < nchunks;
    const int64_t t0 = t_begin + (int64_t)c * kC;
    const int nvalid = (N - t0 < kC) ? (int)(N - t0) : kC;  // tokens of this chunk inside [t_begin, t_end)
    if (has_next) phase_gates(c + 1);
    if (tid == 0 && has_next) wait_tma(c + 1);
    if (__syncthreads_or(!ok)) break;

    // ---- MMA 3: X = S0 W^T, Y = S0 Q^T of chunk c; [K;Q] K^T of chunk c+1
    if (tid == 0) {
      tc_fence_after();
      const uint32_t st = stage(c);
      const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
        const uint32_t woff = (uint32_t)(ks >> 2) * 8192u + (uint32_t)(ks & 3) * 32u;
        mma_bf16(tmem + kColX, kmaj(sbase + kOffS0 + koff), kmaj(sbase + kOffW + woff), id, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
        mma_bf16(tmem + kColY, kmaj(sbase + kOffS0 + koff), kmaj(st + kOffKQ + 8192 + koff), id, ks > 0);
      }
      if (has_next) mma_kq_of(c + 1);
      mma_commit(smem_u32(&bar_mma));
    }
    mma_pending = true;
    {
      // S <- gamma_C S while the MMAs run (S itself is not an operand of this round)
      const float gamC = gam(c)[kC - 1];
      float v[64];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) tmem_ld16(tlane + kColS + 64 * half + c0, *reinterpret_cast<float(*)[16]>(v + c0));
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 64; ++j) v[j] *= gamC;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) tmem_st16(tlane + kColS + 64 * half + c0, *reinterpret_cast<float(*)[16]>(v + c0));
      tmem_st_wait();
    }
    wait_mma();
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();

    // ---- U^T = U~^T - X of chunk c (lane i, columns j in [32 half, 32 half + 32)), U^T diag(gamma_C/gamma);
    //      L and P_o of chunk c+1
    {
      float u[32], x[32];
      tmem_ld16(tlane + kColUt + 32 * half, *reinterpret_cast<float(*)[16]>(u));
      tmem_ld16(tlane + kColUt + 32 * half + 16, *reinterpret_cast<float(*)[16]>(u + 16));
      tmem_ld16(tlane + kColX + 32 * half, *reinterpret_cast<float(*)[16]>(x));
      tmem_ld16(tlane + kColX + 32 * half + 16, *reinterpret_cast<float(*)[16]>(x + 16));
      tmem_ld_wait();
      const float gamC = gam(c)[kC - 1];
      const float* gi = gin(c);
      const int j0 = 32 * half;
      float ud[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        u[j] -= x[j];
        ud[j] = u[j] * (gamC * gi[j0 + j]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        *reinterpret_cast<uint4*>(sm + kOffU + sw128_off(row, j0 + 8 * q, 128)) = pack8_bf16(u + 8 * q);
        *reinterpret_cast<uint4*>(sm + kOffUD + sw128_off(row, j0 + 8 * q, 128)) = pack8_bf16(ud + 8 * q);
      }
    }
    if (has_next) phase_L_Po_of(c + 1);
    sync_for_mma();

    // ---- MMA 4: (P_o U)^T = U^T P_o^T ; S += U^T diag(gamma_C/gamma) K  (chunk c)
    if (tid == 0) {
      const uint32_t st = stage(c);
      const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kColPU, kmaj(sbase + kOffU + ks * 32), kmaj(sbase + po(c) + ks * 32), id, ks > 0);
      const uint32_t id2 = idesc_bf16(128, 128, 0, 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kColS, kmaj(sbase + kOffUD + ks * 32), sw128_desc(st + kOffKQ + ks * 2048, 16384, 1024),
                 id2, 1u);
      mma_commit(smem_u32(&bar_mma));
    }
    mma_pending = true;
    if (has_next) phase_T_of(c + 1);  // overlaps MMA 4; its tiles are not operands of MMA 4
    sync_for_mma();
    wait_mma();
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();

    // ---- MMA 2 of chunk c+1 (W^T, U~^T), overlapped with chunk c's outputs and the next S0 tile
    if (tid == 0 && has_next) {
      mma_wu_of(c + 1);
      mma_commit(smem_u32(&bar_mma));
    }
    if (has_next) mma_pending = true;
    {
      float y[32], p[32], v[64];
      tmem_ld16(tlane + kColY + 32 * half, *reinterpret_cast<float(*)[16]>(y));
      tmem_ld16(tlane + kColY + 32 * half + 16, *reinterpret_cast<float(*)[16]>(y + 16));
      tmem_ld16(tlane + kColPU + 32 * half, *reinterpret_cast<float(*)[16]>(p));
      tmem_ld16(tlane + kColPU + 32 * half + 16, *reinterpret_cast<float(*)[16]>(p + 16));
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) tmem_ld16(tlane + kColS + 64 * half + c0, *reinterpret_cast<float(*)[16]>(v + c0));
      tmem_ld_wait();
      const int r0 = 32 * half;
      const float* gm = gam(c);
      if (write_out) {
        TOut* optr = reinterpret_cast<TOut*>(a.o) + b * a.o_sb + h * a.o_sh + (t0 + r0) * a.o_st + row;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          if (r0 + r < nvalid) store1(optr, a.q_scale * fmaf(gm[r0 + r], y[r], p[r]));
          optr += a.o_st;
        }
      }
      if (has_next) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(sm + kOffS0 + sw128_off(row, 64 * half + 8 * q, 128)) = pack8_bf16(v + 8 * q);
      }
    }
    if (has_next) {
      wait_mma();
      if (__syncthreads_or(!ok)) break;
      tc_fence_after();
      phase_Wtile();
    }
    sync_for_mma();
    if (tid == 0 && c + 2 < nchunks) {
      issue_tma(c + 2);  // stage c is free: every MMA that read it has completed
      tma_issued = c + 3;
    }
  }

done:
  if (ok && s_exit) {
    // final state: lane i row i, this thread columns [64 half, 64 half + 64)
    float* dst = s_exit + (int64_t)row * kD + 64 * half;
    float v[64];
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) tmem_ld16(tlane + kColS + 64 * half + c0, *reinterpret_cast<float(*)[16]>(v + c0));
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 64; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  } else if (!ok && tid == 0) {
    // a wait expired: let this CTA's own copies and MMAs drain (bounded) before freeing TMEM
    for (int k = tma_waited; k < tma_issued; ++k) mbar_wait(smem_u32(&bar_tma[k & 1]), (uint32_t)((k >> 1) & 1), status);
    if (mma_pending) mbar_wait(smem_u32(&bar_mma), mma_phase, status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ----------------------------------------------------------------------------- segment combine
// Entry states of the segments of one (b,h): E_0 = S_in (or 0),
// E_{g+1} = E_g M_g + B_g, in fp32 on the CUDA cores.  M_g and E_g are staged
// in shared memory; thread t owns 64 columns of row t/2.
constexpr int kCombineThreads = 256;
constexpr int kEStride = kD + 1;  // padded rows: conflict-free column reads
constexpr size_t kCombineSmem = (size_t)kD * kEStride * 4 + (size_t)kD * kD * 4;

__global__ void __launch_bounds__(kCombineThreads)
gdn_segment_combine_kernel(const float* S_in, const float* maps, float* states, int G) {
  extern __shared__ float cs[];
  grid_dependency_wait();  // the maps come from the kernel before (launched as its dependent)
  grid_dependents_trigger();
  float* E = cs;                    // [128][129]
  float* M = cs + kD * kEStride;    // [128][128]
  const int64_t bh = blockIdx.x;
  const int tid = threadIdx.x, i = tid >> 1, k0 = (tid & 1) * 64;
  float* out0 = states + bh * G * kStateElems;
  for (int e = tid; e < kD * kD; e += kCombineThreads) {
    const float x = S_in ? S_in[bh * kStateElems + e] : 0.f;
    E[(e >> 7) * kEStride + (e & 127)] = x;
    out0[e] = x;
  }
  for (int g = 0; g + 1 < G; ++g) {
    const float* Bg = maps + ((bh * (G - 1) + g) * 2 + 0) * kStateElems;
    const float* Mg = maps + ((bh * (G - 1) + g) * 2 + 1) * kStateElems;
    __syncthreads();
    for (int e = tid * 4; e < kD * kD; e += kCombineThreads * 4)
      *reinterpret_cast<float4*>(M + e) = *reinterpret_cast<const float4*>(Mg + e);
    __syncthreads();
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      const float4 bb = *reinterpret_cast<const float4*>(Bg + i * kD + k0 + j);
      acc[j] = bb.x; acc[j + 1] = bb.y; acc[j + 2] = bb.z; acc[j + 3] = bb.w;
    }
#pragma unroll 2
    for (int m = 0; m < kD; ++m) {
      const float e = E[i * kEStride + m];
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 mm = *reinterpret_cast<const float4*>(M + m * kD + k0 + j);
        acc[j] = fmaf(e, mm.x, acc[j]);
        acc[j + 1] = fmaf(e, mm.y, acc[j + 1]);
        acc[j + 2] = fmaf(e, mm.z, acc[j + 2]);
        acc[j + 3] = fmaf(e, mm.w, acc[j + 3]);
      }
    }
    __syncthreads();
    float* outg = states + (bh * G + g + 1) * kStateElems + i * kD + k0;
#pragma unroll
    for (int j = 0; j < 64; ++j) E[i * kEStride + k0 + j] = acc[j];
#pragma unroll
    for (int j = 0; j < 64; j += 4) *reinterpret_cast<float4*>(outg + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
  }
}

// ----------------------------------------------------------------------------- host side

template <typename TOut>
cudaError_t launch_typed(const GdnPrefillLaunch& a, void* ws, unsigned* status, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  // strides of 0 (broadcast views) or not multiples of 16 bytes cannot be described
  if (!gdn_make_map(&mq, a.q, a.B, a.H, a.N) || !gdn_make_map(&mk, a.k, a.B, a.H, a.N) ||
      !gdn_make_map(&mv, a.v, a.B, a.H, a.N))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gdn_chunked_kernel<TOut>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemAlloc);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const GdnSegPlan plan = gdn_segment_plan(a.B, a.H, a.N);
  const int64_t BH = a.B * a.H;
  if (plan.G == 1) {
    const GdnTask task{kWhole, 1, a.N, nullptr, nullptr, 0, nullptr};
    gdn_chunked_kernel<TOut><<<(unsigned)BH, kThreads, kSmemAlloc, stream>>>(mq, mk, mv, a, task, status);
    return cudaGetLastError();
  }
  float* maps = static_cast<float*>(ws);
  float* states = maps + BH * (plan.G - 1) * 2 * kStateElems;
  const GdnTask t1{kSegmentMaps, plan.G, plan.seg_len, maps, nullptr, 0, nullptr};
  gdn_chunked_kernel<TOut><<<(unsigned)(BH * (plan.G - 1) * 2), kThreads, kSmemAlloc, stream>>>(mq, mk, mv, a, t1,
                                                                                               status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_gdn_segment_combine(a.S_in, maps, states, plan.G, BH, stream);
  if (e != cudaSuccess) return e;
  const GdnTask t2{kSegmentOutputs, plan.G, plan.seg_len, nullptr, states, 0, nullptr};
  gdn_chunked_kernel<TOut><<<(unsigned)(BH * plan.G), kThreads, kSmemAlloc, stream>>>(mq, mk, mv, a, t2, status);
  return cudaGetLastError();
}

}  // namespace

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// bf16 [B, H, N, 128] view -> 4-D tensor map with a (64 features x 64 tokens) box, 128-byte swizzle.
bool gdn_make_map(CUtensorMap* m, const View4& x, int64_t B, int64_t H, int64_t N) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)(x.st * 2), (cuuint64_t)(x.sh * 2), (cuuint64_t)(x.sb * 2)};
  const cuuint32_t box[4] = {64, (cuuint32_t)kC, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x.ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gdn_segment_combine(const float* S_in, const float* maps, float* states, int G, int64_t BH,
                                       cudaStream_t stream) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gdn_segment_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kCombineSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  return launch_dependent(gdn_segment_combine_kernel, dim3((unsigned)BH), dim3(kCombineThreads), kCombineSmem, stream,
                          S_in, maps, states, G);
}

// Number of sequence segments per (b,h).  With one CTA per SM, the three
// launches cost about ceil(2 (G-1) BH / P) + ceil(G BH / P) waves of a
// segment's length, against ceil(BH / P) waves of the whole sequence for
// G = 1; segments are used when they save at least 20 %, keep at least 32
// chunks each, and G stays <= 16 (the combine is sequential in G).  P is the
// GB300's 152 SMs, a constant rather than a device query so that the
// workspace queries answer from the problem's sizes alone (also on a host
// without a GPU); on a part with fewer SMs the plan stays correct and only
// its wave count is off.
GdnSegPlan gdn_segment_plan(int64_t B, int64_t H, int64_t N) {
  GdnSegPlan p{1, N, 0};
  const int64_t BH = B * H;
  const int64_t nchunks = (N + kC - 1) / kC;
  if (BH <= 0 || N <= 0) return p;
  constexpr int64_t P = 152, kMinSegChunks = 32, kMaxG = 16;
  auto waves = [&](int64_t ctas) { return (ctas + P - 1) / P; };
  const double whole = (double)waves(BH);
  double best = whole;
  int64_t bestG = 1;
  for (int64_t G = 2; G <= kMaxG && G * kMinSegChunks <= nchunks; ++G) {
    const double cost = (double)(waves(2 * (G - 1) * BH) + waves(G * BH)) / (double)G;
    if (cost < 0.8 * whole && cost < best) {
      best = cost;
      bestG = G;
    }
  }
  if (bestG == 1) return p;
  const int64_t seg_chunks = (nchunks + bestG - 1) / bestG;
  p.G = (int)((nchunks + seg_chunks - 1) / seg_chunks);
  p.seg_len = seg_chunks * kC;
  p.ws_bytes = (size_t)(BH * (p.G - 1) * 2 + BH * p.G) * kStateElems * sizeof(float);
  if (p.G == 1) p.ws_bytes = 0;
  return p;
}

cudaError_t launch_gdn_prefill_chunked(const GdnPrefillLaunch& a, void* ws, size_t ws_bytes, unsigned* status,
                                       cudaStream_t stream) {
  if (a.B * a.H == 0 || a.N == 0) return cudaSuccess;
  const GdnSegPlan plan = gdn_segment_plan(a.B, a.H, a.N);
  if (plan.G > 1 && (ws == nullptr || ws_bytes < plan.ws_bytes)) return cudaErrorInvalidValue;
  return a.out_bf16 ? launch_typed<__nv_bfloat16>(a, ws, status, stream) : launch_typed<float>(a, ws, status, stream);
}

}  // namespace la
