// gdn_scan.cu -- the chunked gated-delta-rule prefill: per-chunk records that
// hold what needs the triangular inverse, and a warp-specialized scan that
// reads q, k, v and the records once.
//
// Chunk form (gdn_common.cuh; NoteBank Sec. 2 Eq. (1), the state carried
// across chunk boundaries as in NoteBank Sec. 3.2), chunk of 64 tokens with
// incoming state S0:
//   T  = (I + L)^{-1},  L = strict_lower(diag(beta) (Gamma . K K^T))
//   W  = T diag(beta gamma) K,  U~ = T diag(beta) V,  U = U~ - W S0^T
//   O  = q_scale diag(gamma) (Q S0^T + P U),  P_rj = (q_r . k_j) / gamma_j  (j <= r)
//   S_C = gamma_C S0 + U^T diag(gamma_C / gamma) K
//
// Records: what needs the inversion or the chunk's queries against its keys,
// neither of which depends on the state: the bf16 tiles T2 = T diag(beta) and P
// of every chunk (16 KB, the images the scan's MMAs read), in the caller's
// workspace.  T by doubling, its 64-level block as tcgen05 tf32 MMAs
// (invert_T_tc).  They are formed either by kernel 1 (gdn_tinv_kernel, one CTA
// per chunk over the whole GPU) before the scan, or, when the (b,h) pairs leave
// SMs free and sequences are not split, by CTAs of the scan's own cooperative
// launch beside it (inversion_role), handed over through per-record flags.
//
// The scan (gdn_scan_kernel, one CTA per (b,h) or sequence segment) walks the
// chunks with the fp32 state in tensor memory and does everything else on
// the tcgen05 tensor cores, from tiles it loads once:
//   w:  W^T = K^T (T2 diag gamma)^T                            (chunk-local)
//   u:  U~^T = V^T T2^T                                        (chunk-local)
//   x:  X = S0 W^T                                             (the state path)
//   y:  Y = S0 Q^T                                             (outputs)
//   e:  S~ += (U diag(1 / (sigma gamma)))^T K                  (the state update)
//   d:  Y += U^T P^T  (the chunk's outputs, O^T = q_scale Y diag(gamma))
// The state is held as S~ = S / sigma, sigma the running product of the
// chunk decays gamma_C (folded back into S~ whenever it drops below 2^-32):
// the decay then enters only through a scale of U's columns, and the update
// S~ += (U diag(1 / (sigma gamma)))^T K takes the raw K tile.
//
// Roles (18 warps): warps 0-7 own the state rows (two threads per row) and
// run the passes on the sequential path, U = U~ - X and the bf16 copy S0 of
// the state after each update; warps 8-11 run the chunk-local passes a chunk
// ahead (gates, T2 diag gamma, W^T from tensor memory); warps 12-15 drain
// the outputs; warp 16 issues every MMA and warp 17 every copy, each as soon
// as its inputs are ready.  Hand-offs between them are mbarriers with one
// arrival per warp, and every wait is bounded.
#include <mutex>

#include "gdn_common.cuh"

namespace la {
namespace {
using namespace tc;
using namespace gdn;

// Per-chunk record written by kernel 1 (bf16 tile images, 128-byte swizzle, exactly as the scan's
// MMAs read them): T2 = T diag(beta) [64 r][64 j], then P [64 r][64 j], P_rj = (q_r . k_j) / gamma_j
// for j <= r (0 above the diagonal).
constexpr uint32_t kRecT2 = 0, kRecP = 8192, kRec = 16384;

// ============================================================================ kernel 1
// T = (I + L)^{-1} of a 64-token chunk by doubling, [[A, 0], [C, B]]^{-1} = [[A^{-1}, 0],
// [-B^{-1} C A^{-1}, B^{-1}]]: the four 16x16 diagonal blocks by forward substitution and the
// 32-level blocks on the CUDA cores, the two 64-level products (32x32x32) as tcgen05 MMAs (kind::tf32:
// fp32 operands at tf32 precision, fp32 accumulation).  Every MMA operand is an fp32 K-major tile
// with the 128-byte swizzle (panels of [64 rows][32 columns], 8 KB):
//   LT  L, strictly lower (16 KB);      TA  T, row-major (16 KB);      TB  T^T (16 KB);
//   SMt 4 KB: the 32-level's products, then Z^T ([32][32]).
// The MMAs run at M = 128 with the chunk's 64 rows in lanes 0..63 (the accumulator layout of every
// other MMA here); A rows 64..127 run over the 8 KB that follow each A tile, which must be shared
// memory of this CTA, and give accumulator rows that are never read.
//   Z               = L_[32:64][0:32] T_[0:32][0:32]      (rows 32-63)   N = 32, K = 32
//   T_[32:64][0:32] = -T_[32:64][32:64] Z                                  N = 32, K = 32
constexpr uint32_t kPanel = 8192;  // one [64][32] fp32 panel

__device__ __forceinline__ float* f32_at(uint8_t* tile, int row, int col) {
  return reinterpret_cast<float*>(tile + sw128_off_f32((uint32_t)row, (uint32_t)col, 64));
}

// L = strict_lower(diag(beta gamma) [K K^T] diag(1/gamma)) times delta into LT, and the bf16 image of
// P_rj = (q_r . k_j) / gamma_j (j <= r) into po_tile, from [K;Q] K^T in TMEM (lanes 0..63: K K^T,
// 64..127: Q K^T).  kq_taddr: this thread's lane at the first of its 32 columns (half = column half).
__device__ __forceinline__ void phase_LT_Po(uint32_t kq_taddr, int row, int half, const float* gate, uint8_t* LT,
                                            uint8_t* po_tile, float delta) {
  float v[32];
  ld32(kq_taddr, v);
  const int j0 = 32 * half;
  const float* bt = gate + kC;
  const float* gm = gate + 2 * kC;
  const float* gi = gate + 3 * kC;
  if (row < kC) {
    const int r = row;
    const float f = bt[r] * gm[r] * delta;
    uint8_t* rowp = LT + (uint32_t)half * kPanel + (uint32_t)r * 128u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 g4 = *reinterpret_cast<const float4*>(gi + j0 + 4 * c);
      const int j = j0 + 4 * c;
      float4 o;
      o.x = j < r ? f * g4.x * v[4 * c] : 0.f;
      o.y = j + 1 < r ? f * g4.y * v[4 * c + 1] : 0.f;
      o.z = j + 2 < r ? f * g4.z * v[4 * c + 2] : 0.f;
      o.w = j + 3 < r ? f * g4.w * v[4 * c + 3] : 0.f;
      *reinterpret_cast<float4*>(rowp + ((c ^ (r & 7)) << 4)) = o;
    }
  } else {
    const int r = row - kC;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = (j0 + j <= r) ? gi[j0 + j] * v[j] : 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(po_tile + sw128_off(r, j0 + 8 * q, 64)) = pack8_bf16(v + 8 * q);
  }
}

// T from L (both as above), then the bf16 image T2 = T diag(beta) into t2_tile (shared or global).
// lt: thread 0..255 of the 256 that call it (warp lt / 32 must sit at a multiple of four warps in
// the CTA, so that it reads TMEM lanes 32 (lt / 32 % 4)..); tm: 64 TMEM columns of this group, free;
// bar: an mbarrier that takes one arrival per commit, mph its next phase parity (the same in every
// thread).  Thread lt == 0 issues the MMAs.  `sync` is a barrier of the 256.  An expired wait is
// recorded in *status and makes it return false; the steps still run, so that every barrier is met.
//   1. the 16x16 diagonal blocks by forward substitution (threads 0..63, one column each, rows of L
//      read 16 bytes at a time); TA gets the column, TB the same values as a row;
//   2. the 32-level blocks T_10 = -T_11 (L_10 T_00) and T_32 = -T_33 (L_32 T_22) on the CUDA cores
//      (16x16 products, two outputs a thread, through SMt);
//   3. Z = L_[32:64][0:32] T_[0:32][0:32] as an MMA; meanwhile the T2 image of everything already
//      final (rows 0-31, and rows 32-63 columns 32-63);
//   4. T_[32:64][0:32] = -T_[32:64][32:64] Z as an MMA, its T2 image stored from the registers.
template <typename Sync>
__device__ __forceinline__ bool invert_T_tc(int lt, uint8_t* LT, uint8_t* TA, uint8_t* TB, uint8_t* SMt, uint32_t tm,
                                            uint32_t bar, uint32_t& mph, const float* bt, uint8_t* t2_tile,
                                            unsigned* status, Sync sync) {
  const int w = lt >> 5, lane = lt & 31;
  bool ok = true;
  auto mma_done = [&] {
    ok = mbar_wait(bar, mph, status) && ok;
    mph ^= 1u;
    tc_fence_after();
  };
  // 16 consecutive fp32 of row `row` of a [64][64] tile from column c0 (c0 % 16 == 0) as 4 float4
  auto row16 = [](const uint8_t* tile, int row, int c0, float4 (&o)[4]) {
    const uint8_t* rp = tile + (uint32_t)(c0 >> 5) * kPanel + (uint32_t)row * 128u;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = *reinterpret_cast<const float4*>(rp + ((((uint32_t)((c0 & 31) >> 2) + q) ^ (uint32_t)(row & 7)) << 4));
  };
  if (lt < kC) {
    // x[r] = delta_rc - sum_{j<r} L[base+r][base+j] x[j]: column c of the block's inverse
    const int base = (lt >> 4) * 16, c = lt & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = (r == c) ? 1.f : 0.f;
      if (r > 0) {
        float4 l4[4];
        row16(LT, base + r, base, l4);
        const float* l = reinterpret_cast<const float*>(l4);
        float acc2 = 0.f;
#pragma unroll
        for (int j = 0; j < r; ++j) {
          if (j & 1) acc2 = fmaf(-l[j], x[j], acc2);
          else acc = fmaf(-l[j], x[j], acc);
        }
        acc += acc2;
      }
      x[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) *f32_at(TA, base + r, base + c) = x[r];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<float4*>(f32_at(TB, base + c, base + 4 * q)) =
          make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
  } else if (lt < 2 * kC) {
    // the two upper blocks an MMA reads: TB rows 16-31 x columns 0-15 (T_01 transposed) and TA rows
    // 32-47 x columns 48-63 (T_23): zero
    const int e = lt - kC, r = e >> 2, c = 4 * (e & 3);
    *reinterpret_cast<float4*>(f32_at(TB, 16 + r, c)) = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(f32_at(TA, 32 + r, 48 + c)) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  sync();
  // 32-level, pair k (blocks (1,0) for k = 0, (3,2) for k = 1): this thread's row r and columns c, c+1
  const int k2 = lt >> 7, r16 = (lt >> 3) & 15, cp = (lt & 7) * 2;
  float* Zt = reinterpret_cast<float*>(SMt) + k2 * 16 * 20;  // Z_k^T [16][20]
  {
    float4 lr[4], t0[4], t1[4];
    row16(LT, 32 * k2 + 16 + r16, 32 * k2, lr);      // L_(2k+1)(2k) row r
    row16(TB, 32 * k2 + cp, 32 * k2, t0);            // column cp of T_(2k)(2k)
    row16(TB, 32 * k2 + cp + 1, 32 * k2, t1);        // column cp+1
    const float* l = reinterpret_cast<const float*>(lr);
    const float* a0 = reinterpret_cast<const float*>(t0);
    const float* a1 = reinterpret_cast<const float*>(t1);
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      z0 = fmaf(l[m], a0[m], z0);
      z1 = fmaf(l[m], a1[m], z1);
    }
    Zt[cp * 20 + r16] = z0;
    Zt[(cp + 1) * 20 + r16] = z1;
  }
  sync();
  {
    float4 tr[4], z0[4], z1[4];
    const int R = 32 * k2 + 16 + r16;
    row16(TA, R, 32 * k2 + 16, tr);                  // T_(2k+1)(2k+1) row r
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      z0[q] = *reinterpret_cast<const float4*>(Zt + cp * 20 + 4 * q);
      z1[q] = *reinterpret_cast<const float4*>(Zt + (cp + 1) * 20 + 4 * q);
    }
    const float* t = reinterpret_cast<const float*>(tr);
    const float* b0 = reinterpret_cast<const float*>(z0);
    const float* b1 = reinterpret_cast<const float*>(z1);
    float o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      o0 = fmaf(t[p], b0[p], o0);
      o1 = fmaf(t[p], b1[p], o1);
    }
    const int C = 32 * k2 + cp;
    *f32_at(TA, R, C) = -o0;
    *f32_at(TA, R, C + 1) = -o1;
    *f32_at(TB, C, R) = -o0;
    *f32_at(TB, C + 1, R) = -o1;
  }
  fence_proxy_async_smem();
  sync();
  const uint32_t la = smem_u32(LT), ta = smem_u32(TA), tb = smem_u32(TB), sa = smem_u32(SMt);
  const uint32_t id32 = idesc_tf32(128, 32);
  if (lt == 0) {
    tc_fence_after();
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_tf32(tm + 0, kmaj(la + 32 * s), kmaj(tb + 32 * s), id32, s > 0);
    mma_commit(bar);
  }
  // T2 = T diag(beta) of what is final: rows 0-31 (thread: row lt / 8, 8 columns), and rows 32-63
  // columns 32-63 (threads 0..127: row 32 + lt / 4, 8 columns from 32); 0 above the diagonal
  auto t2_chunk = [&](int r, int c0) {
    float4 a4[2];
    const uint8_t* rp = TA + (uint32_t)(c0 >> 5) * kPanel + (uint32_t)r * 128u;
#pragma unroll
    for (int q = 0; q < 2; ++q)
      a4[q] = *reinterpret_cast<const float4*>(rp + ((((uint32_t)((c0 & 31) >> 2) + q) ^ (uint32_t)(r & 7)) << 4));
    const float* tv = reinterpret_cast<const float*>(a4);
    float t2[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) t2[j] = c0 + j <= r ? tv[j] * bt[c0 + j] : 0.f;
    *reinterpret_cast<uint4*>(t2_tile + sw128_off(r, c0, 64)) = pack8_bf16(t2);
  };
  t2_chunk(lt >> 3, (lt & 7) * 8);
  if (lt < 128) t2_chunk(32 + (lt >> 2), 32 + (lt & 3) * 8);
  mma_done();
  // Z (rows 32-63: warps 1 and 5, 16 columns each), transposed into SMt
  if (w == 1 || w == 5) {
    const int c0 = w == 1 ? 0 : 16;
    float v[16];
    tmem_ld16(tm + (32u << 16) + (uint32_t)c0, v);
    tmem_ld_wait();
#pragma unroll
    for (int n = 0; n < 16; ++n) *reinterpret_cast<float*>(SMt + sw128_off_f32(c0 + n, lane, 32)) = v[n];
  }
  tc_fence_before();
  fence_proxy_async_smem();
  sync();
  if (lt == 0) {
    tc_fence_after();
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_tf32(tm + 32, kmaj(ta + kPanel + 32 * s), kmaj(sa + 32 * s), id32, s > 0);
    mma_commit(bar);
  }
  mma_done();
  // T_[32:64][0:32] = -(T_[32:64][32:64] Z): its T2 image straight from the registers (warps 1 and
  // 5: row 32 + lane, 16 columns each; all below the diagonal)
  if (w == 1 || w == 5) {
    const int c0 = w == 1 ? 0 : 16;
    float v[16];
    tmem_ld16(tm + (32u << 16) + 32u + (uint32_t)c0, v);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = -v[j] * bt[c0 + j];
#pragma unroll
    for (int q = 0; q < 2; ++q)
      *reinterpret_cast<uint4*>(t2_tile + sw128_off(32 + lane, c0 + 8 * q, 64)) = pack8_bf16(v + 8 * q);
  }
  tc_fence_before();
  return ok;
}

// T2 = diag(beta), the image for delta = 0 (L = 0, so T = I): thread r = tid / 4, 16 columns from c0.
__device__ __forceinline__ void t2_identity(int tid, const float* bt, uint8_t* t2_tile) {
  const int r = tid >> 2, c0 = (tid & 3) * 16;
  float t2[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) t2[j] = (c0 + j == r) ? bt[r] : 0.f;
#pragma unroll
  for (int q = 0; q < 2; ++q)
    *reinterpret_cast<uint4*>(t2_tile + sw128_off(r, c0 + 8 * q, 64)) = pack8_bf16(t2 + 8 * q);
}

// Kernel 1, one CTA per chunk (record): shared memory (offsets from a 1024-byte aligned base) LT,
// then the [K;Q] tile (K rows 0-63, Q rows 64-127) for one M=128 MMA giving K K^T and Q K^T, which
// TA and TB overlay once it is done, then SMt and the gate tables.  Each A operand of the inversion
// has 8 KB of this CTA's shared memory after it.  Both images go to the record straight from
// registers.
constexpr uint32_t kIOffLT = 0;
constexpr uint32_t kIOffKQ = 16384;
constexpr uint32_t kIOffTA = kIOffKQ, kIOffTB = kIOffKQ + 16384;
constexpr uint32_t kIOffSM = kIOffKQ + 32768;
constexpr uint32_t kIOffGate = kIOffSM + 4096;
constexpr uint32_t kISmemUsed = kIOffGate + 1024;
constexpr uint32_t kISmemAlloc = kISmemUsed + 1024;
static_assert(4 * (kISmemAlloc + 1024) <= 233472, "four inversion CTAs per SM");
static_assert(kIOffLT + 2 * kPanel + 8192 <= kISmemUsed && kIOffTA + 2 * kPanel + 8192 <= kISmemUsed,
              "every inversion A operand has 8 KB of shared memory after it");

__global__ void __launch_bounds__(kThreads, 4)
gdn_tinv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const GdnPrefillLaunch a, int nch, uint8_t* rec_out, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_tma;
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base_sh;
  __shared__ float carry;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127, half = tid >> 7;
  const int64_t rec = blockIdx.x;
  const int64_t bh = rec / nch;
  const int c = (int)(rec % nch);
  const int b = (int)(bh / a.H), h = (int)(bh % a.H);
  const int64_t t0 = (int64_t)c * kC;
  const uint32_t sbase = smem_u32(sm);
  float* gate = reinterpret_cast<float*>(sm + kIOffGate);
  uint8_t* rp = rec_out + rec * kRec;

  float al = 1.f, bt = 0.f;
  if (tid < kC && t0 + tid < a.N) {
    al = a.alpha[b * a.a_sb + h * a.a_sh + t0 + tid];
    bt = a.beta[b * a.b_sb + h * a.b_sh + t0 + tid];
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar_tma), 1);
    mbar_init(smem_u32(&bar_mma), 1);
    fence_mbar_init();
    const uint32_t bar = smem_u32(&bar_tma);
    mbar_arrive_expect_tx(bar, 32768);
    tma_load_4d(sbase + kIOffKQ + 0, &tmap_k, 0, (int)t0, h, b, bar);
    tma_load_4d(sbase + kIOffKQ + 16384, &tmap_k, 64, (int)t0, h, b, bar);
    tma_load_4d(sbase + kIOffKQ + 8192, &tmap_q, 0, (int)t0, h, b, bar);
    tma_load_4d(sbase + kIOffKQ + 24576, &tmap_q, 64, (int)t0, h, b, bar);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), 64);
    tmem_relinquish();
  }
  gate_tables(tid, logf(al), bt, gate, &carry);  // padded tokens: alpha = 1, beta = 0
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  // Every thread waits on the barriers itself (sleeping in hardware).
  bool ok = true, tma_waited = false, mma_pending = false;
  uint32_t mph = 0;
  do {
    ok = mbar_wait(smem_u32(&bar_tma), 0, status);
    tma_waited = ok;
    if (__syncthreads_or(!ok)) break;
    if (tid == 0) {
      tc_fence_after();
      mma_kq(tmem, sbase + kIOffKQ);
      mma_commit(smem_u32(&bar_mma));
    }
    mma_pending = true;
    ok = mbar_wait(smem_u32(&bar_mma), mph, status);
    mph ^= 1u;
    if (__syncthreads_or(!ok)) break;
    mma_pending = false;
    tc_fence_after();
    // L (rows of K K^T) into LT, P (rows of Q K^T) into its image in the record
    phase_LT_Po(tlane + 32 * half, row, half, gate, sm + kIOffLT, rp + kRecP, a.delta);
    tc_fence_before();
    __syncthreads();
    if (a.delta != 0.f) {
      ok = invert_T_tc(tid, sm + kIOffLT, sm + kIOffTA, sm + kIOffTB, sm + kIOffSM, tmem, smem_u32(&bar_mma), mph,
                       gate + kC, rp + kRecT2, status, [] { __syncthreads(); });
    } else {
      t2_identity(tid, gate + kC, rp + kRecT2);  // the scalar gate: no inverse to form
    }
  } while (false);

  if (!ok && tid == 0) {
    if (!tma_waited) mbar_wait(smem_u32(&bar_tma), 0, status);
    if (mma_pending) mbar_wait(smem_u32(&bar_mma), mph ^ 1u, status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

// ============================================================================ inversion role
// The CTAs of a scan launch past its scan CTAs (GdnTask::ready set) form the records themselves, so
// that the inversion runs on the SMs the scan leaves idle, beside it.  Each such CTA runs two
// independent pipelines of 8 worker warps (warps 0-7 and 8-15) over the records in chunk-major
// order (record i: chunk i / BH of pair i % BH), so that every (b,h) gets its early chunks first, as
// its scan CTA wants them.  Per record the steps of gdn_tinv_kernel, with the [K;Q] tile in two
// stages (the copy of the record after next goes in once T, formed over the current stage, is dead)
// and the two images stored straight from registers to the record.  Warp 16 + g serves pipeline g
// off its critical path: its lane 0 issues the pipeline's copies and, once the workers report a
// record written, releases the record's flag (the GPU-scope fence that release needs waits for the
// record's stores, so no worker waits on it); the whole warp forms the gate tables two records
// ahead, into the buffer of the record just written.  The scan's copy issuer acquires a flag before
// it copies the record.
// One pipeline's shared memory: the two [K;Q] stages (TA and TB of a record over its dead stage), LT,
// SMt and two gate-table buffers.  The A operands of the inversion (LT, TA) have 8 KB of shared memory of
// the CTA after them (pipeline 1's LT: its SMt, gate tables and the unused end of the allocation).
constexpr uint32_t kIGOffLT = 65536;
constexpr uint32_t kIGOffSM = kIGOffLT + 2 * kPanel;
constexpr uint32_t kIGOffGate = kIGOffSM + 4096;  // two gate-table buffers (records k, k+1 by parity)
constexpr uint32_t kIGrp = kIGOffGate + 2048;
static_assert(kIGrp % 1024 == 0, "one inversion pipeline's shared memory");

// Pacing: the scan re-reads the [K;Q] tiles the formers have just loaded and the records they have
// just written, from L2 while the formers are at most a few chunks ahead of it.  Measured at
// B=4 H=16 N=16384, formers alone 0.514 ms and the scan alone 0.568 ms gave 0.637 ms together
// without pacing, 0.599 ms with the formers held within 8 chunks of the scans (0.616 within 12).
// So the serving lane holds the copy of a record of chunk m while the scans together have issued the
// copies of fewer than (m - lead) BH chunks: one counter for all scans, since a wait on the scan of
// one pair would hold the other pairs' records behind it.  A pipeline's consecutive records lie
// stride / BH chunks apart and the lane paces the record two ahead of the one being formed, so a
// lead under about three such spacings waits on records that are not formed yet (a lead of 2 to 5
// at that shape took 9 ms); lead = ceil(3 stride / BH) (9 there).  The wait is a hint, which no
// result depends on, and gives up after kPaceLimitNs.
constexpr uint64_t kPaceLimitNs = 100000;

__device__ __forceinline__ void inversion_role(const CUtensorMap* tmap_q, const CUtensorMap* tmap_k,
                                               const GdnPrefillLaunch& a, int nch, int n_ctas, int cta,
                                               uint8_t* sm, uint8_t* rec_out, unsigned* ready, const unsigned* progress,
                                               unsigned* status) {
  // per pipeline: [K;Q] landed in stage 0, in stage 1; MMA done; record written (one arrival per
  // worker warp); record released (the serving lane); gate tables in buffer 0, in buffer 1 written
  __shared__ uint64_t ibar[2][7];
  __shared__ uint32_t itmem_sh;
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool worker = warp < 16;
  const int g = worker ? warp >> 3 : warp - 16;  // the pipeline this warp works in or serves
  const int lt = tid & 255, row = lt & 127, half = lt >> 7;
  const int64_t BH = a.B * a.H, nrec = BH * nch;
  const int64_t stride = 2 * (int64_t)n_ctas;
  const int64_t first = 2 * (int64_t)cta + g;
  uint8_t* gsm = sm + (uint32_t)g * kIGrp;
  const uint32_t gbase = smem_u32(gsm);
  uint8_t* LT = gsm + kIGOffLT;
  uint8_t* SMt = gsm + kIGOffSM;
  float* gates = reinterpret_cast<float*>(gsm + kIGOffGate);  // buffer p at gates + 256 p
  const uint32_t bar_done = smem_u32(&ibar[g][3]), bar_rel = smem_u32(&ibar[g][4]);

  if (tid == 0) {
    for (int p = 0; p < 2; ++p) {
      for (int j = 0; j < 3; ++j) mbar_init(smem_u32(&ibar[p][j]), 1);
      mbar_init(smem_u32(&ibar[p][3]), 8);
      mbar_init(smem_u32(&ibar[p][4]), 1);
      mbar_init(smem_u32(&ibar[p][5]), 1);
      mbar_init(smem_u32(&ibar[p][6]), 1);
    }
    fence_mbar_init();
    tma_prefetch_desc(tmap_k);
    tma_prefetch_desc(tmap_q);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&itmem_sh), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = itmem_sh + 64u * (uint32_t)g;
  const uint32_t tlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  if (worker) {
    auto sync = [g] { named_bar_sync(1 + g, 256); };
    const uint32_t bar_mma = smem_u32(&ibar[g][2]);
    // record i's (b,h) pair and chunk, advanced by stride without divisions; *_n: record i + stride
    const int64_t dbh = stride % BH, dch = stride / BH;
    int64_t bh_c = first % BH, ch_c = first / BH;
    int64_t bh_n = bh_c + dbh, ch_n = ch_c + dch;
    if (bh_n >= BH) bh_n -= BH, ++ch_n;
    bool ok = true, mma_pending = false;
    uint32_t mph = 0;  // next phase parity of bar_mma (three commits a record with the inversion)
    int k = 0;
    for (int64_t i = first; i < nrec; i += stride, ++k) {
      const int st = k & 1;
      const float* gate = gates + 256 * st;
      ok = mbar_wait(smem_u32(&ibar[g][st]), (uint32_t)((k >> 1) & 1), status);
      if (named_bar_or(1 + g, 256, !ok)) break;
      if (lt == 0) {
        tc_fence_after();
        mma_kq(tmem, gbase + (uint32_t)st * 32768u);
        mma_commit(bar_mma);
      }
      mma_pending = true;
      ok = mbar_wait(bar_mma, mph, status);
      mph ^= 1u;
      // the gate tables of this record, formed by the serving warp
      ok = mbar_wait(smem_u32(&ibar[g][5 + st]), (uint32_t)((k >> 1) & 1), status) && ok;
      if (named_bar_or(1 + g, 256, !ok)) break;
      mma_pending = false;
      tc_fence_after();
      uint8_t* rp = rec_out + (bh_c * nch + ch_c) * kRec;
      phase_LT_Po(tlane + 32 * half, row, half, gate, LT, rp + kRecP, a.delta);
      tc_fence_before();
      sync();
      uint8_t* stage = gsm + (uint32_t)st * 32768u;  // TA and TB over the dead [K;Q] tile
      if (a.delta != 0.f) {
        if (!invert_T_tc(lt, LT, stage, stage + 16384, SMt, tmem, bar_mma, mph, gate + kC, rp + kRecT2, status, sync))
          ok = false;
      } else {
        t2_identity(lt, gate + kC, rp + kRecT2);
      }
      fence_proxy_async_smem();  // T's writes before the copy that overwrites the stage
      // record written: one arrival per warp, once the serving lane has released the record before
      // (so that this arrival opens the next phase only after that one was seen)
      __syncwarp();
      if ((tid & 31) == 0) {
        if (k > 0 && !mbar_wait(bar_rel, (uint32_t)((k - 1) & 1), status)) ok = false;
        mbar_arrive(bar_done);
      }
      sync();  // T and the TMEM columns are rewritten by the next record
      bh_c = bh_n, ch_c = ch_n;
      bh_n += dbh, ch_n += dch;
      if (bh_n >= BH) bh_n -= BH, ++ch_n;
    }
    if (lt == 0 && !ok && mma_pending) mbar_wait(bar_mma, mph ^ 1u, status);
  } else {
    // the serving warp of pipeline g: copies and flag releases (lane 0), gate tables (the warp)
    const int lane = tid & 31;
    int issued[2] = {0, 0};
    auto load = [&](int64_t i, int st) {
      const int64_t bh = i % BH;
      const int t0 = (int)((i / BH) * kC), b = (int)(bh / a.H), h = (int)(bh % a.H);
      const uint32_t bar = smem_u32(&ibar[g][st]), dst = gbase + (uint32_t)st * 32768u;
      mbar_arrive_expect_tx(bar, 32768);
      tma_load_4d(dst + 0, tmap_k, 0, t0, h, b, bar);
      tma_load_4d(dst + 16384, tmap_k, 64, t0, h, b, bar);
      tma_load_4d(dst + 8192, tmap_q, 0, t0, h, b, bar);
      tma_load_4d(dst + 24576, tmap_q, 64, t0, h, b, bar);
      ++issued[st];
    };
    // gate tables of record i into buffer p, then its arrival: lane l takes tokens l and 32 + l and
    // runs the same two 32-lane scans, carry and exponentials as gate_tables (the same bits)
    auto gates_of = [&](int64_t i, int p) {
      const int64_t bh = i % BH, t0 = (i / BH) * kC;
      const int b = (int)(bh / a.H), h = (int)(bh % a.H);
      float lg[2], bt[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t t = t0 + lane + 32 * e;
        float al = 1.f;
        bt[e] = 0.f;
        if (t < a.N) {
          al = a.alpha[b * a.a_sb + h * a.a_sh + t];
          bt[e] = a.beta[b * a.b_sb + h * a.b_sh + t];
        }
        lg[e] = logf(al);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(kFullMask, lg[e], off);
          if (lane >= off) lg[e] += y;
        }
      }
      lg[1] += __shfl_sync(kFullMask, lg[0], 31);
      float* gt = gates + 256 * p;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = lane + 32 * e;
        gt[t] = lg[e];
        gt[kC + t] = bt[e];
        gt[2 * kC + t] = __expf(lg[e]);
        gt[3 * kC + t] = __expf(-lg[e]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ibar[g][5 + p]));
    };
    if (lane == 0) {
      if (first < nrec) load(first, 0);
      if (first + stride < nrec) load(first + stride, 1);
    }
    // lane 0: hold record i while the scans together are more than `lead` chunks behind it
    const int64_t lead = (3 * stride + BH - 1) / BH;
    auto pace = [&](int64_t i) {
      const int64_t m = i / BH;
      if (m <= lead) return;
      const uint64_t need = (uint64_t)(m - lead) * (uint64_t)BH;
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        unsigned v;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(progress) : "memory");
        if ((uint64_t)v >= need || globaltimer_ns() - t0 > kPaceLimitNs) return;
        __nanosleep(256);
      }
    };
    if (first < nrec) gates_of(first, 0);
    if (first + stride < nrec) gates_of(first + stride, 1);
    bool ok = true;
    int k = 0;
    for (int64_t i = first; i < nrec; i += stride, ++k) {
      ok = mbar_wait(bar_done, (uint32_t)(k & 1), status);
      if (!ok) break;
      if (lane == 0) {
        // release this record first: the scans may need it before the pacing lets the next copy go
        const int64_t bh = i % BH, r = bh * nch + i / BH;
        flag_release(ready + r, 1u);
        mbar_arrive(bar_rel);
        if (i + 2 * stride < nrec) {
          pace(i + 2 * stride);
          load(i + 2 * stride, k & 1);  // the workers are done with T there
        }
      }
      if (i + 2 * stride < nrec) gates_of(i + 2 * stride, k & 1);  // and with this buffer
    }
    if (!ok && lane == 0) {
      // let this pipeline's own copies finish (bounded) before the CTA exits
      for (int st = 0; st < 2; ++st)
        if (issued[st] > 0) mbar_wait(smem_u32(&ibar[g][st]), (uint32_t)((issued[st] - 1) & 1), status);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(itmem_sh, 128);
}

// ============================================================================ placement
// Where a launch's CTAs sit matters for the scan: measured on GB300, 64 scan CTAs on the lowest SM
// ids (as a 64-CTA launch is placed) take ~540 us at 16K tokens, while the same CTAs spread eight to
// each group of 16 SM ids (as the full-GPU launch places its first 64 CTAs) take 660-750 us, with the
// other SMs idle or not.  So a launch that forms its own records gives its roles by placement: every
// CTA marks its SM id, all meet at one grid barrier (the launch is cooperative, so all CTAs are
// resident), and a CTA's rank among the marked ids is its index: the lowest n_scan scan.  Every CTA
// falls back to blockIdx.x, consistently, if the SM ids are out of range or shared, or the barrier
// expires (the status then reports it).
constexpr unsigned kMaxSmIds = 1024;
constexpr size_t kPlaceBytes = ((2 + kMaxSmIds) * sizeof(unsigned) + 255) & ~size_t(255);  // + the pacing counter

__device__ __forceinline__ int placement_rank(unsigned* place, unsigned* status) {
  __shared__ int rank_sh;
  __shared__ int bad_sh;
  unsigned smid, nsmid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  asm volatile("mov.u32 %0, %%nsmid;" : "=r"(nsmid));
  if (nsmid > kMaxSmIds) return (int)blockIdx.x;  // the same for every CTA of the launch
  if (threadIdx.x == 0) {
    rank_sh = 0;
    bad_sh = 0;
    atomicAdd(place + 1 + smid, 1u);
    asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(place) : "memory");
    if (!flag_wait(place, gridDim.x, status)) bad_sh = 1;
  }
  __syncthreads();
  int below = 0, shared_id = 0;
  for (unsigned s = threadIdx.x; s < nsmid; s += blockDim.x) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(place + 1 + s) : "memory");
    if (s < smid) below += (int)v;
    shared_id |= v > 1u;
  }
  if (below) atomicAdd(&rank_sh, below);
  if (shared_id) bad_sh = 1;
  __syncthreads();
  return bad_sh ? (int)blockIdx.x : rank_sh;
}

// ============================================================================ kernel 2
// Shared memory (offsets from a 1024-byte aligned base), three rings of copy
// slots and the tiles the workers write:
//   K ring, three slots (free once the chunk's state update is done): K
//       [64 r][128 k], the T2 image.  Three deep so that the copies of chunk
//       c+1 are in flight a whole chunk before W^T of it is wanted.
//   V ring, two slots (free once U~ of the chunk is computed): V [64][128].
//   Q ring, two slots (free once the chunk's outputs are done): Q [64 r][128 k],
//       the P image.
//   W^T [128 k][64 r] (rows k, the r contiguous: an MN-major operand), one
//       tile: W^T of chunk c+1 is computed after x(c) is issued, and copied
//       into the tile only once it is done.
// The bf16 copy S0 of the state is the A operand of x and y straight from
// tensor memory.
constexpr int kKSlots = 3;
constexpr uint32_t kKSlot = 24576;                    // one K slot
constexpr uint32_t kKOffK = 0, kKOffT2 = 16384;
constexpr uint32_t kVSlot = 16384;
constexpr uint32_t kQSlot = 24576;                    // one Q slot
constexpr uint32_t kQOffQ = 0, kQOffP = 16384;
constexpr uint32_t kSOffK = 0;
constexpr uint32_t kSOffV = kSOffK + kKSlots * kKSlot;  // 73728
constexpr uint32_t kSOffQ = kSOffV + 2 * kVSlot;        // 106496
constexpr uint32_t kSOffWT = kSOffQ + 2 * kQSlot;       // 155648
constexpr uint32_t kSOffT1 = kSOffWT + 16384;           // T2 diag(gamma), one buffer
constexpr uint32_t kSOffGate = kSOffT1 + 8192;        // gate slots
constexpr int kGateSlots = 8;
constexpr uint32_t kGateSlot = 576;                   // gamma[64], 1/(sigma gamma)[64], scalars
constexpr uint32_t kSSmemUsed = kSOffGate + kGateSlots * kGateSlot;
constexpr uint32_t kSSmemAlloc = kSSmemUsed + 1024;
static_assert(kKSlot % 1024 == 0 && kQSlot % 1024 == 0 && kSOffV % 1024 == 0 && kSOffQ % 1024 == 0 &&
                  kSOffWT % 1024 == 0 && kSOffT1 % 1024 == 0,
              "MMA operand tiles sit on 1024-byte boundaries");
static_assert(kSSmemAlloc + 512 <= 232448, "shared memory budget");
static_assert(kIGrp + kIGOffLT + 2 * kPanel + 8192 <= kSSmemUsed && 2 * kIGrp <= kSSmemUsed,
              "the inversion role's two pipelines, and the 8 KB after pipeline 1's LT, fit the scan's shared memory");
// gate slot layout (floats)
constexpr int kGGam = 0, kGKds = 64, kGSig = 128, kGSigAfter = 129, kGFold = 130;

// tensor-memory columns
constexpr uint32_t kTS = 0;     // S~ [i][k], fp32
constexpr uint32_t kTS0 = 128;  // S0 = bf16(sigma S~) [i][k], two per column (64 columns)
constexpr uint32_t kTX = 192;   // X [i][r]
constexpr uint32_t kTY = 256;   // Y [i][r]
constexpr uint32_t kTU = 320;   // U~^T [i][r], two buffers (320..383, 384..447)
// The U pass writes U (bf16, two per column) over the X columns it has read and U diag(1/(sigma gamma))
// over the U~ columns it has read: tokens [32 h, +32) of row i go to columns [32 h, +16) of either
// tile, so an MMA step over tokens [16 s, +16) reads A at column offset ua_off(s).
__host__ __device__ constexpr uint32_t ua_off(int s) { return 32u * (uint32_t)(s >> 1) + 8u * (uint32_t)(s & 1); }
constexpr uint32_t kTW = 448;   // W^T [k][r]
constexpr uint32_t kTCols = 512;

constexpr int kStateWarps = 8, kLocalWarps = 4, kOutWarps = 4;
constexpr int kLocal0 = kStateWarps * 32;            // first local thread
constexpr int kOut0 = kLocal0 + kLocalWarps * 32;    // first output thread
constexpr int kIssuer0 = kOut0 + kOutWarps * 32;     // the MMA issuer warp
constexpr int kLoader0 = kIssuer0 + 32;              // the copy issuer warp
constexpr int kScanThreads = kLoader0 + 32;
constexpr int kLocalBar = 1;                         // named barrier of the local warps
constexpr float kFoldBelow = 2.3283064e-10f;         // 2^-32

// One CTA per SM (shared memory and all 512 tensor-memory columns).  Warps
// take registers in groups of four, so the 18 warps are budgeted as 20: at
// most 96 registers a thread; the wide passes work on 32 columns at a time.
// GATED: the scalar gate (delta = 0), where W = 0 and X = 0, so U = U~ needs nothing from the state:
// the sequential path shrinks to e(c) -> S0 pass -> e(c+1), with y and d off it, S0 double-buffered in
// tensor memory (the X columns, unused then, hold the copy of odd chunks) and U in the W^T columns.
template <typename TOut, bool GATED>
__global__ void __launch_bounds__(kScanThreads, 1)
gdn_scan_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const GdnPrefillLaunch a, const GdnTask task,
                int nch_total, uint8_t* rec, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int cta = task.ready != nullptr ? placement_rank(task.place, status) : (int)blockIdx.x;
  if (task.ready != nullptr && cta >= task.n_scan) {
    inversion_role(&tmap_q, &tmap_k, a, nch_total, (int)gridDim.x - task.n_scan, cta - task.n_scan, sm, rec,
                   task.ready, task.progress, status);
    return;
  }
  __shared__ uint64_t bar_k[kKSlots];  // K and the T2 image landed in their slot
  __shared__ uint64_t bar_v[2];        // V landed
  __shared__ uint64_t bar_q[2];        // Q and the P image landed
  __shared__ uint64_t bar_b;         // W^T, U~^T computed
  __shared__ uint64_t bar_x;         // X computed
  __shared__ uint64_t bar_e;         // state update done
  __shared__ uint64_t bar_o;         // Y += U^T P^T done: the chunk's outputs are complete
  __shared__ uint64_t bar_gate[kGateSlots];
  __shared__ uint64_t bar_fin;
  // Worker -> MMA issuer hand-offs, one arrival per warp, one phase per chunk: T1 written (bar_t1),
  // W^T written with Q and P landed (bar_wk), by the local warps; U written (bar_u) and S0 written
  // (bar_s0, phase 0 = the entry state), by the state warps; Y read (bar_of), by the output warps.
  // No group gets two phases ahead of the issuer's wait (each next hand-off needs an MMA issued after
  // that wait), so parities stay unambiguous.
  __shared__ uint64_t bar_t1, bar_wk, bar_u, bar_s0, bar_of;
  // Ring slots freed for the copy issuer, one arrival per warp, one phase per use of the slot: the
  // update (the last MMA to read K and T2) done (bar_kfree) and x issued after U~ done (bar_vfree),
  // by the state warps; Y read, so that the MMAs reading Q and P are done, by the output warps
  // (bar_qfree).  A slot's next phase needs the copy the issuer waits to make, so no phase is
  // passed unseen.
  __shared__ uint64_t bar_kfree[kKSlots], bar_vfree[2], bar_qfree[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ float lshare[2];        // local warps: scan carry, gamma_C

  const int tid = threadIdx.x, warp = tid >> 5;
  const CtaWork wk = cta_work(a, task, cta);
  const int b = wk.b, h = wk.h;
  const int n = wk.nchunks;
  const bool WOUT = wk.write_out, ZV = wk.zero_v;
  const int64_t rec0 = wk.bh * nch_total + wk.t_begin / kC;
  const uint32_t sb = smem_u32(sm);
  auto slot = [&](int c) { return reinterpret_cast<float*>(sm + kSOffGate + (uint32_t)(c % kGateSlots) * kGateSlot); };
  auto gate_par = [&](int c) { return (uint32_t)((c / kGateSlots) & 1); };
  auto kslot = [&](int c) { return kSOffK + (uint32_t)(c % kKSlots) * kKSlot; };
  auto kpar = [&](int c) { return (uint32_t)((c / kKSlots) & 1); };
  auto vslot = [&](int c) { return kSOffV + (uint32_t)(c & 1) * kVSlot; };
  auto qslot = [&](int c) { return kSOffQ + (uint32_t)(c & 1) * kQSlot; };
  auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait(smem_u32(bar), parity, status); };
  // tensor-memory columns of the bf16 state copy S0 of chunk c, and of U
  auto s0col = [&](int c) { return (GATED && (c & 1)) ? kTX : kTS0; };
  constexpr uint32_t kTUb = GATED ? kTW : kTX;

  if (tid == 0) {
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(smem_u32(&bar_k[i]), 1);
      mbar_init(smem_u32(&bar_kfree[i]), kStateWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_v[i]), 1);
      mbar_init(smem_u32(&bar_q[i]), 1);
      mbar_init(smem_u32(&bar_vfree[i]), kStateWarps);
      mbar_init(smem_u32(&bar_qfree[i]), kOutWarps);
    }
    mbar_init(smem_u32(&bar_b), 1);
    mbar_init(smem_u32(&bar_x), 1);
    mbar_init(smem_u32(&bar_e), 1);
    mbar_init(smem_u32(&bar_o), 1);
    for (int i = 0; i < kGateSlots; ++i) mbar_init(smem_u32(&bar_gate[i]), kLocalWarps);
    mbar_init(smem_u32(&bar_fin), 1);
    mbar_init(smem_u32(&bar_t1), kLocalWarps);
    mbar_init(smem_u32(&bar_wk), kLocalWarps);
    mbar_init(smem_u32(&bar_u), kStateWarps);
    mbar_init(smem_u32(&bar_s0), kStateWarps);
    mbar_init(smem_u32(&bar_of), kOutWarps);

    fence_mbar_init();
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), kTCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lane quarter
  // launched as a dependent of the kernel before it: everything above overlapped its end; what
  // follows reads the records, maps or entry states it wrote
  grid_dependency_wait();
  grid_dependents_trigger();
  // U pass of chunk c for this thread's row (its warp's lane quarter), tokens [32 h, +32):
  // U^T = U~^T - X and U^T diag(1 / (sigma gamma)), both bf16, into tensor memory over the X (the W^T
  // columns for the scalar gate) and U~ columns this thread has just read
  auto u_pass = [&](int c, int h) {
    const uint32_t par = (uint32_t)(c & 1);
#pragma unroll
    for (int part = 0; part < 2; ++part) {  // tokens [32 h + 16 part, +16)
      const int c0 = 32 * h + 16 * part;
      float x[16], u[16];
      if constexpr (!GATED) tmem_ld16(tlane + kTX + c0, x);  // the scalar gate has X = 0
      if (!ZV) tmem_ld16(tlane + kTU + 64 * par + c0, u);
      tmem_ld_wait();
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 16; ++j) u[j] = (ZV ? 0.f : u[j]) - (GATED ? 0.f : x[j]);
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = pack2_bf16(u[2 * j], u[2 * j + 1]);
      tmem_st8u(tlane + kTUb + 32 * h + 8 * part, w);
      const float4* kds = reinterpret_cast<const float4*>(slot(c) + kGKds + c0);  // 1/(sigma gamma_r)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 f = kds[q];
        u[4 * q] *= f.x; u[4 * q + 1] *= f.y; u[4 * q + 2] *= f.z; u[4 * q + 3] *= f.w;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = pack2_bf16(u[2 * j], u[2 * j + 1]);
      tmem_st8u(tlane + kTU + 64 * par + 32 * h + 8 * part, w);
    }
    tmem_st_wait();
    tc_fence_before();
  };

  if (warp == kIssuer0 / 32) {
    // ======================================================================= MMA issuer
    // Lane 0 issues every MMA in a fixed order, waiting before each for the hand-offs it needs.  The
    // tensor pipe runs MMAs in issue order, so the order decides the period: the state path
    // x(c) -> U pass -> e(c) -> S0 pass -> x(c+1) is sequential.  y(c) follows x(c) and runs during
    // the U pass; W^T of chunk c+1 goes in during the U pass too when its T1 is ready (else right
    // after e(c)), so that the local warps have copied it out by the time S0 of chunk c+1 is ready;
    // d(c) and U~^T of chunk c+1 follow e(c) and run during the S0 pass.  x(c+1) follows U~^T of
    // chunk c+1, so the U pass's wait on x also covers U~.
    if ((tid & 31) == 0) {
      const uint32_t id64 = idesc_bf16(128, 64, 0, 0);
      const uint32_t id64t = idesc_bf16(128, 64, 1, 0);    // A MN-major
      const uint32_t id64n = idesc_bf16(128, 64, 0, 1);    // B MN-major
      const uint32_t id128n = idesc_bf16(128, 128, 0, 1);  // B MN-major
      bool ok = true, mma_issued = false;
      auto ph = [](int m) { return (uint32_t)(m & 1); };
      // a hand-off that has already happened costs one non-suspending test
      auto wait_i = [&](uint64_t* bar, uint32_t parity) {
        return mbar_test_wait(smem_u32(bar), parity) || wait(bar, parity);
      };
      // w: W^T = K^T T1^T (chunk-local) into its tensor-memory tile, from the K slot and T1
      auto issue_w = [&](int m) {
        tc_fence_after();
        const uint32_t kt = sb + kslot(m) + kKOffK;
        const uint32_t t1 = sb + kSOffT1;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + kTW, sw128_desc(kt + ks * 2048, 8192, 1024), kmaj(t1 + ks * 32), id64t, ks > 0);
        mma_commit(smem_u32(&bar_b));
        mma_issued = true;
      };
      // u: U~^T = V^T T2^T (chunk-local) into the buffer of chunk m-2, whose U pass is done, once V
      // of the chunk has landed (T2 came with K, before T1)
      auto issue_u = [&](int m) -> bool {
        if (!wait_i(&bar_v[m & 1], (uint32_t)((m >> 1) & 1))) return false;
        tc_fence_after();
        const uint32_t vt = sb + vslot(m);
        const uint32_t t2 = sb + kslot(m) + kKOffT2;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + kTU + 64u * (uint32_t)(m & 1), sw128_desc(vt + ks * 2048, 8192, 1024),
                   kmaj(t2 + ks * 32), id64t, ks > 0);
        mma_issued = true;
        return true;
      };
      if constexpr (GATED) {
        // u of chunk m once K with T2 (its slot) and V have landed, then the commit the U pass waits on
        auto issue_ug = [&](int m) -> bool {
          if (!wait_i(&bar_k[m % kKSlots], kpar(m))) return false;
          if (!ZV && !issue_u(m)) return false;
          mma_commit(smem_u32(&bar_x));
          mma_issued = true;
          return true;
        };
        if (n > 0) ok = issue_ug(0);
        for (int c = 0; ok && c < n; ++c) {
          // ---- e: S~ += UD^T K, once U of the chunk is written and the S0 pass of the chunk before has
          // read the S~ this update changes
          ok = wait_i(&bar_u, ph(c)) && wait_i(&bar_s0, ph(c));
          if (!ok) break;
          tc_fence_after();
          {
            const uint32_t kt = sb + kslot(c) + kKOffK;
            const uint32_t ud = tmem + kTU + 64u * (uint32_t)(c & 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16_ts(tmem + kTS, ud + ua_off(ks), sw128_desc(kt + ks * 2048, 8192, 1024), id128n, 1u);
            mma_commit(smem_u32(&bar_e));
          }
          if (WOUT) {
            // ---- y: Y = S0 Q^T from the chunk's own S0 buffer, once Q and P have landed and the outputs
            // of the chunk before are drained; d: Y += U^T P^T
            ok = (c == 0 || wait_i(&bar_of, ph(c - 1))) && wait_i(&bar_q[c & 1], (uint32_t)((c >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            const uint32_t qt = sb + qslot(c) + kQOffQ;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off = (uint32_t)(ks >> 2) * 8192u + (uint32_t)(ks & 3) * 32u;
              mma_bf16_ts(tmem + kTY, tmem + s0col(c) + 8u * (uint32_t)ks, kmaj(qt + off), id64, ks > 0);
            }
            const uint32_t pp = sb + qslot(c) + kQOffP;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16_ts(tmem + kTY, tmem + kTUb + ua_off(ks), kmaj(pp + ks * 32), id64, 1u);
            mma_commit(smem_u32(&bar_o));
          }
          if (c + 1 < n) ok = issue_ug(c + 1);
        }
      } else {
      // prologue: the chunk-local products of chunk 0
      if (n > 0) {
        ok = wait_i(&bar_t1, 0);
        if (ok) {
          issue_w(0);
          if (!ZV) ok = issue_u(0);
        }
      }
      for (int c = 0; ok && c < n; ++c) {
        const bool next = c + 1 < n;
        // ---- x: X = S0 W^T, once S0 of the chunk is in tensor memory and W^T in its tile
        ok = wait_i(&bar_s0, ph(c)) && wait_i(&bar_wk, ph(c));
        if (!ok) break;
        tc_fence_after();
        {
          const uint32_t wt = sb + kSOffWT;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ts(tmem + kTX, tmem + kTS0 + 8u * (uint32_t)ks, sw128_desc(wt + ks * 2048, 0, 1024), id64n,
                        ks > 0);
          mma_commit(smem_u32(&bar_x));
        }
        // ---- y: Y = S0 Q^T, once the outputs of the chunk before are drained
        if (WOUT) {
          ok = c == 0 || wait_i(&bar_of, ph(c - 1));
          if (!ok) break;
          tc_fence_after();
          const uint32_t qt = sb + qslot(c) + kQOffQ;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (uint32_t)(ks >> 2) * 8192u + (uint32_t)(ks & 3) * 32u;
            mma_bf16_ts(tmem + kTY, tmem + kTS0 + 8u * (uint32_t)ks, kmaj(qt + off), id64, ks > 0);
          }
        }
        // ---- w of chunk c+1 now if T1 of it is ready (W^T of chunk c was copied out before x)
        bool w_done = false;
        if (next && mbar_test_wait(smem_u32(&bar_t1), ph(c + 1))) {
          issue_w(c + 1);
          w_done = true;
        }
        // ---- e: S~ += UD^T K, once the U pass is done (UD from tensor memory)
        ok = wait_i(&bar_u, ph(c));
        if (!ok) break;
        tc_fence_after();
        {
          const uint32_t kt = sb + kslot(c) + kKOffK;
          const uint32_t ud = tmem + kTU + 64u * (uint32_t)(c & 1);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ts(tmem + kTS, ud + ua_off(ks), sw128_desc(kt + ks * 2048, 8192, 1024), id128n, 1u);
          mma_commit(smem_u32(&bar_e));
        }
        if (next && !w_done && mbar_test_wait(smem_u32(&bar_t1), ph(c + 1))) {
          issue_w(c + 1);
          w_done = true;
        }
        // ---- d: Y += U^T P^T
        if (WOUT) {
          tc_fence_after();
          const uint32_t pp = sb + qslot(c) + kQOffP;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ts(tmem + kTY, tmem + kTX + ua_off(ks), kmaj(pp + ks * 32), id64, 1u);
          mma_commit(smem_u32(&bar_o));
        }
        if (next && !w_done) {
          ok = wait_i(&bar_t1, ph(c + 1));
          if (!ok) break;
          issue_w(c + 1);
        }
        if (next && !ZV) {
          ok = issue_u(c + 1);
          if (!ok) break;
        }
      }
      }
      if (!ok && mma_issued) {
        // let this CTA's own MMAs finish (bounded) before tensor memory is freed
        mma_commit(smem_u32(&bar_fin));
        mbar_wait(smem_u32(&bar_fin), 0, status);
      }
    }
    __syncwarp();
  } else if (warp == kLoader0 / 32) {
    // ======================================================================= copy issuer
    // Lane 0 issues the copies of every chunk in order, each into its ring slot once the slot's
    // earlier contents are no longer read: K and T2 of chunk m after the update of chunk m-3, V after
    // U~ of chunk m-2, Q and P after the outputs of chunk m-2.  When this launch forms the records
    // itself, the flag of chunk m+1's record is read early (relaxed, while the issuer waits for the
    // slots of chunk m) and, if already set, turned into an acquire with a fence where the copy is
    // issued; otherwise the issuer waits on it there.
    const bool leader = (tid & 31) == 0;
    int nk = 0, nv = 0, nq = 0;
    if (leader) {
      const unsigned* flags = task.ready != nullptr ? task.ready + rec0 : nullptr;
      unsigned seen = (flags != nullptr && n > 0) ? flag_peek(flags) : 0u;
      bool ok = true;
      for (int m = 0; ok && m < n; ++m) {
        const int t0 = (int)(wk.t_begin + (int64_t)m * kC);
        if (m >= kKSlots) ok = wait(&bar_kfree[m % kKSlots], kpar(m - kKSlots));
        if (ok && flags != nullptr) {
          if (seen == 1u) fence_acq_rel_gpu();  // the early read saw the flag: acquire
          else ok = flag_wait(flags + m, 1u, status);
          fence_proxy_async_global();
          seen = m + 1 < n ? flag_peek(flags + m + 1) : 0u;
        }
        if (!ok) break;
        {
          const uint32_t kt = sb + kslot(m);
          const uint32_t bar = smem_u32(&bar_k[m % kKSlots]);
          mbar_arrive_expect_tx(bar, 16384u + 8192u);
          tma_load_4d(kt + kKOffK + 0, &tmap_k, 0, t0, h, b, bar);
          tma_load_4d(kt + kKOffK + 8192, &tmap_k, 64, t0, h, b, bar);
          bulk_load(kt + kKOffT2, rec + (rec0 + m) * kRec + kRecT2, 8192, bar);
          ++nk;
          if (flags != nullptr)  // for the formers' pacing: one more chunk issued
            asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(task.progress) : "memory");
        }
        if (!ZV) {
          if (m >= 2) ok = wait(&bar_vfree[m & 1], (uint32_t)(((m - 2) >> 1) & 1));
          if (!ok) break;
          const uint32_t vt = sb + vslot(m);
          const uint32_t bar = smem_u32(&bar_v[m & 1]);
          mbar_arrive_expect_tx(bar, 16384u);
          tma_load_4d(vt + 0, &tmap_v, 0, t0, h, b, bar);
          tma_load_4d(vt + 8192, &tmap_v, 64, t0, h, b, bar);
          ++nv;
        }
        if (WOUT) {
          if (m >= 2) ok = wait(&bar_qfree[m & 1], (uint32_t)(((m - 2) >> 1) & 1));
          if (!ok) break;
          const uint32_t qt = sb + qslot(m);
          const uint32_t bar = smem_u32(&bar_q[m & 1]);
          mbar_arrive_expect_tx(bar, 16384u + 8192u);
          tma_load_4d(qt + kQOffQ + 0, &tmap_q, 0, t0, h, b, bar);
          tma_load_4d(qt + kQOffQ + 8192, &tmap_q, 64, t0, h, b, bar);
          bulk_load(qt + kQOffP, rec + (rec0 + m) * kRec + kRecP, 8192, bar);
          ++nq;
        }
      }
    }
    nk = __shfl_sync(kFullMask, nk, 0);
    nv = __shfl_sync(kFullMask, nv, 0);
    nq = __shfl_sync(kFullMask, nq, 0);
    // let this CTA's own copies land (bounded) before the CTA exits; a slot's phases complete in
    // order, so waiting for its last issued load covers the earlier ones
    for (int m = nk - kKSlots; m < nk; ++m)
      if (m >= 0) mbar_wait(smem_u32(&bar_k[m % kKSlots]), kpar(m), status);
    for (int m = nv - 2; m < nv; ++m)
      if (m >= 0) mbar_wait(smem_u32(&bar_v[m & 1]), (uint32_t)((m >> 1) & 1), status);
    for (int m = nq - 2; m < nq; ++m)
      if (m >= 0) mbar_wait(smem_u32(&bar_q[m & 1]), (uint32_t)((m >> 1) & 1), status);
  } else if (tid < kLocal0) {
    // ======================================================================= state warps
    // lane i = state row i; this thread: state columns [64 half, +64), U columns [32 half, +32)
    const int row = tid & 127, half = tid >> 7;
    bool ok = true;  // an expired wait skips this thread's later waits; every arrival is still made
    // S0 = bf16(v) for this thread's 64 state columns: packed columns [32 half, +32) of kTS0
    auto store_s0 = [&](const float* v) {
#pragma unroll
      for (int c0 = 0; c0 < 32; c0 += 16) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pack2_bf16(v[2 * (c0 + j)], v[2 * (c0 + j) + 1]);
        tmem_st16u(tlane + kTS0 + 32 * half + c0, w);
      }
    };
    {
      const float* src = wk.s_entry ? wk.s_entry + (int64_t)row * kD + 64 * half : nullptr;
      float v[64];
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 x = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[j] = x.x; v[j + 1] = x.y; v[j + 2] = x.z; v[j + 3] = x.w;
      }
      if (ZV) {  // identity entry state: the run then yields the segment's linear map
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = (64 * half + j == row) ? 1.f : 0.f;
      }
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16)
        tmem_st16(tlane + kTS + 64 * half + c0, *reinterpret_cast<float(*)[16]>(v + c0));
      store_s0(v);
      tmem_st_wait();
    }
    tc_fence_before();
    warp_arrive(smem_u32(&bar_s0));
    ok = wait(&bar_gate[0], 0);  // the gates of a chunk are waited for a chunk ahead, off the sequential path
    float sigma = 1.f;  // S = sigma S~ after the latest update
    for (int c = 0; c < n; ++c) {
      const uint32_t par = (uint32_t)(c & 1);
      // ---- U of chunk c, this row, tokens [32 half, +32)
      ok = ok && wait(&bar_x, par);
      tc_fence_after();
      warp_arrive(smem_u32(&bar_vfree[c & 1]));  // U~ of chunk c was done (before x): V may be refilled
      u_pass(c, half);
      warp_arrive(smem_u32(&bar_u));
      // ---- after the update: S0 of chunk c+1 = sigma' S~, folding sigma' into S~ when small
      ok = ok && wait(&bar_e, par);
      tc_fence_after();
      warp_arrive(smem_u32(&bar_kfree[c % kKSlots]));  // K and T2 of chunk c may be refilled
      const float* gs = slot(c);
      const float sig_after = gs[kGSigAfter];
      const bool fold = gs[kGFold] != 0.f;
      const bool has_next = c + 1 < n;
      if (!fold && has_next) {
        // this thread's 64 state columns, 32 at a time
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t col = 64 * half + 32 * part;
          float v[32];
          tmem_ld16(tlane + kTS + col, *reinterpret_cast<float(*)[16]>(v));
          tmem_ld16(tlane + kTS + col + 16, *reinterpret_cast<float(*)[16]>(v + 16));
          tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) w[j] = pack2_bf16(v[2 * j] * sig_after, v[2 * j + 1] * sig_after);
          tmem_st16u(tlane + s0col(c + 1) + col / 2, w);
        }
        tmem_st_wait();
      } else if (fold) {
        // sigma' folded into S~ (and S0 = S~ written if a chunk follows), 32 columns at a time
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t col = 64 * half + 32 * part;
          float v[32];
          tmem_ld16(tlane + kTS + col, *reinterpret_cast<float(*)[16]>(v));
          tmem_ld16(tlane + kTS + col + 16, *reinterpret_cast<float(*)[16]>(v + 16));
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= sig_after;
          if (has_next) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack2_bf16(v[2 * j], v[2 * j + 1]);
            tmem_st16u(tlane + s0col(c + 1) + col / 2, w);
          }
          tmem_st16(tlane + kTS + col, *reinterpret_cast<float(*)[16]>(v));
          tmem_st16(tlane + kTS + col + 16, *reinterpret_cast<float(*)[16]>(v + 16));
        }
        tmem_st_wait();
      }
      sigma = fold ? 1.f : sig_after;
      if (has_next) {
        tc_fence_before();
        warp_arrive(smem_u32(&bar_s0));
        ok = ok && wait(&bar_gate[(c + 1) % kGateSlots], gate_par(c + 1));
      }
    }
    ok = __all_sync(kFullMask, ok);  // warp-uniform: the loads below are warp-collective
    if (ok && wk.s_exit) {
      float* dst = wk.s_exit + (int64_t)row * kD + 64 * half;
      float v[64];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16)
        tmem_ld16(tlane + kTS + 64 * half + c0, *reinterpret_cast<float(*)[16]>(v + c0));
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 64; j += 4)
        *reinterpret_cast<float4*>(dst + j) =
            make_float4(sigma * v[j], sigma * v[j + 1], sigma * v[j + 2], sigma * v[j + 3]);
    }
  } else if (tid < kOut0) {
    // ======================================================================= local warps
    const int ltid = tid - kLocal0;  // 0..127 = this thread's tensor-memory lane
    bool ok = true;
    float sig_run = 1.f;  // sigma before the next chunk whose gates are formed
    const float* al_p = a.alpha + b * a.a_sb + h * a.a_sh;
    // alpha of chunk c for this thread's token (1 past the end), loaded a chunk before its gates are
    // formed so that the load's latency is not on the local warps' path
    auto load_alpha = [&](int c) {
      const int64_t t = wk.t_begin + (int64_t)c * kC + ltid;
      return (ltid < kC && c < n && t < wk.t_end) ? al_p[t] : 1.f;
    };
    // gates of chunk c from its alpha: g = cumsum log alpha, gamma = e^g, 1/(sigma gamma), sigma
    // bookkeeping
    auto gates = [&](int c, float al) {
      float* gs = slot(c);
      float g = ltid < kC ? logf(al) : 0.f;
      if (ltid < kC) {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(kFullMask, g, off);
          if ((ltid & 31) >= off) g += y;
        }
        if (ltid == 31) lshare[0] = g;
      }
      named_bar_sync(kLocalBar, kLocalWarps * 32);
      float gam = 0.f;
      if (ltid < kC) {
        if (ltid >= 32) g += lshare[0];
        gam = __expf(g);
        gs[kGGam + ltid] = gam;
        if (ltid == kC - 1) lshare[1] = gam;
      }
      named_bar_sync(kLocalBar, kLocalWarps * 32);
      const float gC = lshare[1];
      const float s_c = sig_run, s_after = s_c * gC;
      const bool fold = s_after < kFoldBelow;
      sig_run = fold ? 1.f : s_after;
      if (ltid < kC) gs[kGKds + ltid] = 1.f / (s_c * gam);
      if (ltid == 0) {
        gs[kGSig] = s_c;
        gs[kGSigAfter] = s_after;
        gs[kGFold] = fold ? 1.f : 0.f;
      }
      named_bar_sync(kLocalBar, kLocalWarps * 32);  // gates complete; lshare free again
      warp_arrive(smem_u32(&bar_gate[c % kGateSlots]));
    };
    // T1 = delta T2 diag(gamma) of chunk c (into the single T1 buffer; b of chunk c-1 has completed)
    auto t1_pass = [&](int c) {
      ok = ok && wait(&bar_k[c % kKSlots], kpar(c));
      const float* gam = slot(c) + kGGam;
      const uint8_t* t2 = sm + kslot(c) + kKOffT2;
      const int r = ltid >> 1, j0 = (ltid & 1) * 32;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t off = sw128_off(r, j0 + 8 * q, 64);
        const uint4 raw = *reinterpret_cast<const uint4*>(t2 + off);
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = __bfloat162float(x[e]) * gam[j0 + 8 * q + e] * a.delta;
        *reinterpret_cast<uint4*>(sm + kSOffT1 + off) = pack8_bf16(y);
      }
      fence_proxy_async_smem();
      warp_arrive(smem_u32(&bar_t1));
    };
    gates(0, load_alpha(0));
    if (n > 1) gates(1, load_alpha(1));
    if (n > 2) gates(2, load_alpha(2));
    float al_next = load_alpha(3);
    if constexpr (GATED) {
      // no T1 and no W^T: only the gates, three chunks ahead, paced by the updates (the gate slot of
      // chunk c+3 last served chunk c-5, whose S0 pass and outputs were done before the update of
      // chunk c)
      for (int c = 0; c + 3 < n; ++c) {
        ok = ok && wait(&bar_e, (uint32_t)(c & 1));
        const float al = al_next;
        al_next = load_alpha(c + 4);
        gates(c + 3, al);
      }
    } else {
    t1_pass(0);
    for (int c = 0; c < n; ++c) {
      const uint32_t par = (uint32_t)(c & 1);
      // ---- W^T (lane k of tensor memory holds row k) into its tile
      ok = ok && wait(&bar_b, par);
      tc_fence_after();
      {
        uint8_t* wt = sm + kSOffWT;
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // columns r, 32 at a time
          float w[32];
          tmem_ld16(tlane + kTW + 32 * part, *reinterpret_cast<float(*)[16]>(w));
          tmem_ld16(tlane + kTW + 32 * part + 16, *reinterpret_cast<float(*)[16]>(w + 16));
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(wt + sw128_off(ltid, 32 * part + 8 * q, 128)) = pack8_bf16(w + 8 * q);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (WOUT) ok = ok && wait(&bar_q[c & 1], (uint32_t)((c >> 1) & 1));  // Q and P of the chunk landed
      warp_arrive(smem_u32(&bar_wk));
      if (c + 1 < n) t1_pass(c + 1);
      if (c + 3 < n) {
        const float al = al_next;
        al_next = load_alpha(c + 4);
        gates(c + 3, al);
      }
    }
    }
  } else if (tid < kIssuer0) {
    // ======================================================================= output warps
    if (WOUT) {
      const int i = tid - kOut0;  // value index = tensor-memory lane
      bool ok = true;
      for (int c = 0; c < n; ++c) {
        ok = ok && wait(&bar_o, (uint32_t)(c & 1)) && wait(&bar_gate[c % kGateSlots], gate_par(c));
        tc_fence_after();
        float y[64];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) tmem_ld16(tlane + kTY + c0, *reinterpret_cast<float(*)[16]>(y + c0));
        tmem_ld_wait();
        const float* gam = slot(c) + kGGam;
#pragma unroll
        for (int r = 0; r < 64; ++r) y[r] *= a.q_scale * gam[r];
        tc_fence_before();
        warp_arrive(smem_u32(&bar_of));  // Y may be overwritten from here on
        warp_arrive(smem_u32(&bar_qfree[c & 1]));  // and Q, P of the chunk reloaded
        const int64_t t0 = wk.t_begin + (int64_t)c * kC;
        const int nvalid = (wk.t_end - t0 < kC) ? (int)(wk.t_end - t0) : kC;
        TOut* optr = reinterpret_cast<TOut*>(a.o) + b * a.o_sb + h * a.o_sh + t0 * a.o_st + i;
#pragma unroll
        for (int r = 0; r < 64; ++r) {
          if (r < nvalid) store1(optr, y[r]);
          optr += a.o_st;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTCols);
}

size_t records_bytes(int64_t BH, int64_t nch) { return (size_t)(BH * nch) * kRec; }
// one ready flag per record, for the launch that forms its records itself
// plus the placement scratch of that launch
// (whose first word counts the chunks all scans have issued, after the placement words), the flags
// rounded up to 256 bytes
size_t round256(size_t n) { return (n + 255) & ~size_t(255); }
size_t flags_bytes(int64_t BH, int64_t nch) { return round256((size_t)(BH * nch) * sizeof(unsigned)) + kPlaceBytes; }

// The fewest inversion CTAs worth a launch that forms its own records.
constexpr int kMinInversionCtas = 16;

// CTAs of the scan kernel that fit on the current device at once (0 if unknown).
template <typename K>
int coresident_ctas(K kernel) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kScanThreads, kSSmemAlloc) != cudaSuccess)
    return 0;
  return sms * per_sm;
}

template <typename TOut>
cudaError_t launch_scan_typed(const GdnPrefillLaunch& a, void* ws, unsigned* status, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!gdn_make_map(&mq, a.q, a.B, a.H, a.N) || !gdn_make_map(&mk, a.k, a.B, a.H, a.N) ||
      !gdn_make_map(&mv, a.v, a.B, a.H, a.N))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  static int coresident[2] = {0, 0};  // per scan instantiation, on the first device used
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gdn_tinv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kISmemAlloc);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gdn_scan_kernel<TOut, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kSSmemAlloc);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gdn_scan_kernel<TOut, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kSSmemAlloc);
    if (attr_err == cudaSuccess) {
      coresident[0] = coresident_ctas(gdn_scan_kernel<TOut, false>);
      coresident[1] = coresident_ctas(gdn_scan_kernel<TOut, true>);
    }
  });
  const bool gated = a.delta == 0.f;
  auto scan = gated ? gdn_scan_kernel<TOut, true> : gdn_scan_kernel<TOut, false>;
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t BH = a.B * a.H;
  const int64_t nch = (a.N + kC - 1) / kC;
  const GdnSegPlan plan = gdn_segment_plan(a.B, a.H, a.N);
  uint8_t* recT = static_cast<uint8_t*>(ws);
  float* seg = reinterpret_cast<float*>(recT + records_bytes(BH, nch));
  unsigned* ready = reinterpret_cast<unsigned*>(recT + records_bytes(BH, nch) + plan.ws_bytes);
  const int n_co = coresident[gated ? 1 : 0];
  if (plan.G == 1 && BH + kMinInversionCtas <= n_co) {
    // one launch: CTAs 0..BH-1 scan, the rest of the GPU forms the records beside them
    cudaError_t e = cudaMemsetAsync(ready, 0, flags_bytes(BH, nch), stream);
    if (e != cudaSuccess) return e;
    unsigned* place = ready + round256((size_t)(BH * nch) * sizeof(unsigned)) / sizeof(unsigned);
    unsigned* progress = place + 1 + kMaxSmIds;
    const GdnTask task{kWhole, 1, a.N, nullptr, nullptr, (int)BH, ready, place, progress};
    return launch_cooperative(scan, dim3((unsigned)n_co), dim3(kScanThreads), kSSmemAlloc, stream, mq, mk, mv, a,
                              task, (int)nch, recT, status);
  }
  gdn_tinv_kernel<<<(unsigned)(BH * nch), kThreads, kISmemAlloc, stream>>>(mq, mk, a, (int)nch, recT, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (plan.G == 1) {
    const GdnTask task{kWhole, 1, a.N, nullptr, nullptr, 0, nullptr};
    return launch_dependent(scan, dim3((unsigned)BH), dim3(kScanThreads), kSSmemAlloc, stream, mq,
                            mk, mv, a, task, (int)nch, recT, status);
  }
  float* maps = seg;
  float* states = maps + BH * (plan.G - 1) * 2 * kStateElems;
  const GdnTask t1{kSegmentMaps, plan.G, plan.seg_len, maps, nullptr, 0, nullptr};
  e = launch_dependent(scan, dim3((unsigned)(BH * (plan.G - 1) * 2)), dim3(kScanThreads), kSSmemAlloc,
                       stream, mq, mk, mv, a, t1, (int)nch, recT, status);
  if (e != cudaSuccess) return e;
  e = launch_gdn_segment_combine(a.S_in, maps, states, plan.G, BH, stream);
  if (e != cudaSuccess) return e;
  const GdnTask t2{kSegmentOutputs, plan.G, plan.seg_len, nullptr, states, 0, nullptr};
  return launch_dependent(scan, dim3((unsigned)(BH * plan.G)), dim3(kScanThreads), kSSmemAlloc, stream,
                          mq, mk, mv, a, t2, (int)nch, recT, status);
}

}  // namespace

size_t gdn_scan_workspace_bytes(int64_t B, int64_t H, int64_t N) {
  const int64_t BH = B * H;
  if (BH <= 0 || N <= 0) return 0;
  const int64_t nch = (N + kC - 1) / kC;
  return records_bytes(BH, nch) + gdn_segment_plan(B, H, N).ws_bytes + flags_bytes(BH, nch);
}

cudaError_t launch_gdn_prefill_scan(const GdnPrefillLaunch& a, void* ws, size_t ws_bytes, unsigned* status,
                                    cudaStream_t stream) {
  const int64_t BH = a.B * a.H;
  if (BH == 0 || a.N == 0) return cudaSuccess;
  const int64_t nch = (a.N + kC - 1) / kC;
  if (BH * nch > (int64_t)INT32_MAX) return cudaErrorInvalidValue;  // one inversion CTA per chunk
  if (ws == nullptr || ws_bytes < gdn_scan_workspace_bytes(a.B, a.H, a.N)) return cudaErrorInvalidValue;
  return a.out_bf16 ? launch_scan_typed<__nv_bfloat16>(a, ws, status, stream)
                    : launch_scan_typed<float>(a, ws, status, stream);
}

}  // namespace la
