// gdn_split.cu -- the chunked gated-delta-rule prefill as two kernels: a
// chunk-parallel kernel for everything that does not depend on the state,
// then a short sequential chain per (b,h) for what does.
//
// The chunk form (gdn_common.cuh; NoteBank Sec. 2 Eq. (1), the state carried
// across chunk boundaries as in NoteBank Sec. 3.2) splits into
//   chunk-local: gates, [K;Q] K^T, L, T = (I + L)^{-1}, W = T diag(beta gamma) K,
//                U~ = T diag(beta) V, P_o = tril(Gamma) . Q K^T
//   chain:       U = U~ - W S0^T,  O = (diag(gamma) Q) S0^T + P_o U,
//                S_C = gamma_C S0 + U^T diag(gamma_C / gamma) K.
// The single-kernel scan (gdn_chunked.cu) interleaves both in one CTA per
// (b,h): the chunk-local work, the inversion above all, sits on the
// sequential path and only B*H SMs work.  Here the first kernel runs one CTA
// per chunk over the whole GPU (two CTAs per SM) and leaves one record pair
// per chunk in the caller's workspace:
//   record A (41472 B): bf16 tile images exactly as the chain's MMAs read
//       them (128-byte swizzle): W [64 r][128 k], Q' = q_scale diag(gamma) Q
//       [64 r][128 k], P_o' = q_scale P_o [64][64]; then gamma_r and
//       1/gamma_r (fp32, 64 each);
//   record U (32768 B): U~^T in fp32, [128 i][64 r], the 16-byte chunks of
//       row i XOR-swizzled by i % 16 so that a warp reads 32 rows without
//       bank conflicts.
// The chain kernel has three roles.  One thread of warp 12 issues every copy
// (k by TMA, the records with the bulk-copy engine) and every MMA; warps 0-7
// run the CUDA-core passes of the critical path of each chunk,
//   X = S0 W^T -> U, U diag(1/(sigma gamma)) -> S update -> bf16 S0,
// two threads per state row, and hand over to the issuer through mbarriers;
// O^T = S0 Q'^T + U^T P_o'^T accumulates beside that path in one of two
// tensor-memory buffers, which warps 8-11 drain to global memory.  The
// decay gamma_C is never applied to the tensor-memory state: it holds
// S / sigma with sigma the running product of gamma_C, which enters through
// U diag(1 / (sigma gamma)) and the bf16 S0 copy, and is folded back into the
// state (one pass) whenever sigma drops below 2^-32.  The sequence-segment
// scheme (gdn_common.cuh) applies to the chain unchanged.
#include <mutex>

#include "gdn_common.cuh"

namespace la {
namespace {
using namespace tc;
using namespace gdn;

// ---------------------------------------------------------------- records
constexpr uint32_t kRecAW = 0;         // bf16 W [64 r][128 k], two [64][64] blocks
constexpr uint32_t kRecAQ = 16384;     // bf16 Q' = q_scale diag(gamma) Q [64 r][128 k], two blocks
constexpr uint32_t kRecAPo = 32768;    // bf16 P_o' = q_scale P_o [64 r][64 j]
constexpr uint32_t kRecAGate = 40960;  // fp32 gamma[64], then 1/gamma[64]
constexpr uint32_t kRecA = 41472;
constexpr uint32_t kRecU = 32768;      // fp32 U~^T [128 i][64 r], chunk-swizzled rows
static_assert(kRecA % 16 == 0 && kRecU % 16 == 0, "bulk copies move multiples of 16 bytes");

// ---------------------------------------------------------------- chunk-local kernel
// Shared memory (offsets from a 1024-byte aligned base), about 70 KB so that
// three CTAs share an SM: tiles die early and their space is reused.
constexpr uint32_t kLOffKQ = 0;                     // [K;Q] [128][128] bf16, two [128][64] blocks
constexpr uint32_t kLOffV = 32768;                  // V [64][128] bf16
constexpr uint32_t kLOffL = 49152;                  // fp32 L [64][65]
constexpr uint32_t kLOffZ = kLOffL + 64 * 65 * 4;   // fp32 block products (4 KB)
constexpr uint32_t kLOffGate = kLOffZ + 4096;       // fp32 gate tables [4][64]
constexpr uint32_t kLSmemUsed = kLOffGate + 1024;
constexpr uint32_t kLSmemAlloc = kLSmemUsed + 1024;
// T (fp32, 64 floats per row) in the Q rows of the [K;Q] tile once [K;Q] K^T
// and Q' are done: rows 0..31 in block 0, rows 32..63 in block 1
constexpr uint32_t kLOffT0 = kLOffKQ + 8192, kLOffT1Rows = kLOffKQ + 16384 + 8192;
// bf16 T diag(beta gamma) and T diag(beta) [64][64] over L once the inversion is done
constexpr uint32_t kLOffT1 = kLOffL, kLOffT2 = kLOffL + 8192;
// staging of the record parts written with one bulk copy each: Q' over L
// before L exists; W over the K rows of block 0 and U~^T over block 1 and V
// once the W/U~ MMAs are done
constexpr uint32_t kLOffQimg = kLOffL, kLOffWimg = kLOffKQ, kLOffUimg = kLOffKQ + 16384;
static_assert(kLOffL % 1024 == 0 && 16384 <= 64 * 65 * 4, "bf16 T tiles and the Q' image overlay L");
static_assert(kLOffUimg + kRecU <= kLOffV + 16384, "U~^T staging fits [K;Q] block 1 and V");
static_assert(3 * (kLSmemAlloc + 1024) <= 233472, "three chunk-local CTAs per SM");
// tensor memory: [K;Q] K^T in columns 0..63, then W^T over it and U~^T in 64..127
constexpr uint32_t kLColKQ = 0, kLColW = 0, kLColUt = 64, kLTmemCols = 128;

__global__ void __launch_bounds__(kThreads, 3)
gdn_local_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const GdnPrefillLaunch a, int nch, uint8_t* recA,
                 uint8_t* recU, unsigned* status) {
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
  float* gate = reinterpret_cast<float*>(sm + kLOffGate);
  float* Lsm = reinterpret_cast<float*>(sm + kLOffL);
  float* Zsm = reinterpret_cast<float*>(sm + kLOffZ);
  uint8_t* ra = recA + rec * kRecA;

  // this chunk's alpha and beta first: their latency overlaps the setup below
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
    mbar_arrive_expect_tx(bar, 49152);
    tma_load_4d(sbase + kLOffKQ + 0, &tmap_k, 0, (int)t0, h, b, bar);
    tma_load_4d(sbase + kLOffKQ + 16384, &tmap_k, 64, (int)t0, h, b, bar);
    tma_load_4d(sbase + kLOffKQ + 8192, &tmap_q, 0, (int)t0, h, b, bar);
    tma_load_4d(sbase + kLOffKQ + 24576, &tmap_q, 64, (int)t0, h, b, bar);
    tma_load_4d(sbase + kLOffV + 0, &tmap_v, 0, (int)t0, h, b, bar);
    tma_load_4d(sbase + kLOffV + 8192, &tmap_v, 64, (int)t0, h, b, bar);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), kLTmemCols);
    tmem_relinquish();
  }
  gate_tables(tid, logf(al), bt, gate, &carry);  // padded tokens: alpha = 1, beta = 0
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  bool ok = true, tma_waited = false, mma_pending = false;
  uint32_t mma_phase = 0;
  auto wait_mma = [&]() {
    ok = ok && mbar_wait(smem_u32(&bar_mma), mma_phase, status);
    mma_phase ^= 1;
    mma_pending = !ok;
  };
  do {
    if (tid == 0) {
      ok = mbar_wait(smem_u32(&bar_tma), 0, status);
      tma_waited = ok;
    }
    if (__syncthreads_or(!ok)) break;
    if (tid == 0) {
      tc_fence_after();
      mma_kq(tmem + kLColKQ, sbase + kLOffKQ);
      mma_commit(smem_u32(&bar_mma));
    }
    mma_pending = true;
    // Q' = q_scale diag(gamma) Q while [K;Q] K^T runs: the Q rows of the [K;Q] tile carry the same
    // 128-byte swizzle as rows of a [64][64] block, so each 16-byte chunk moves to the same place
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + i * kThreads, bk = e >> 9, r = (e >> 3) & 63, ch = e & 7;
      const uint4 raw = *reinterpret_cast<const uint4*>(sm + kLOffKQ + bk * 16384 + 8192 + r * 128 + ch * 16);
      const float f = a.q_scale * gate[2 * kC + r];
      const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
      float y[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) y[j] = f * __bfloat162float(x[j]);
      *reinterpret_cast<uint4*>(sm + kLOffQimg + bk * 8192 + r * 128 + ch * 16) = pack8_bf16(y);
    }
    if (tid < 32)  // gamma and 1/gamma
      reinterpret_cast<uint4*>(ra + kRecAGate)[tid] = reinterpret_cast<const uint4*>(gate + 2 * kC)[tid];
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(ra + kRecAQ, sbase + kLOffQimg, 16384);
      bulk_commit();
    }
    wait_mma();
    if (tid == 0) bulk_wait_read();  // the L region is written next
    if (__syncthreads_or(!ok)) break;  // also: every thread is done reading Q
    tc_fence_after();
    // L into shared memory, P_o' straight into record A
    phase_L_Po(tlane + kLColKQ + 32 * half, row, half, gate, Lsm, ra + kRecAPo, a.q_scale, a.delta);
    tc_fence_before();
    __syncthreads();
    phase_T(tid, Lsm,
            [&](int r) {
              return reinterpret_cast<float*>(sm + (r < 32 ? kLOffT0 + r * 256 : kLOffT1Rows + (r - 32) * 256));
            },
            Zsm, gate, false, a.delta, sm + kLOffT1, sm + kLOffT2);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      mma_wu(tmem + kLColW, tmem + kLColUt, sbase + kLOffKQ, sbase + kLOffV, sbase + kLOffT1, sbase + kLOffT2);
      mma_commit(smem_u32(&bar_mma));
    }
    mma_pending = true;
    wait_mma();
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    {
      // W image: lane k holds W^T[k][r] for r in [32 half, 32 half + 32)
      float w[32];
      ld32(tlane + kLColW + 32 * half, w);
#pragma unroll
      for (int r = 0; r < 32; ++r) st_bf16(sm + kLOffWimg + sw128_off(32 * half + r, row, 64), w[r]);
      // U~^T row `row`, columns [32 half, 32 half + 32): eight 16-byte chunks, swizzled by row % 16
      float u[32];
      ld32(tlane + kLColUt + 32 * half, u);
      uint8_t* ru = sm + kLOffUimg + row * 256;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int ch = 8 * half + q;
        *reinterpret_cast<float4*>(ru + ((ch ^ (row & 15)) << 4)) =
            make_float4(u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(ra + kRecAW, sbase + kLOffWimg, 16384);
      bulk_store(recU + rec * kRecU, sbase + kLOffUimg, kRecU);
      bulk_commit();
      bulk_wait_read();  // shared memory stays valid until the copies have read it
    }
  } while (false);

  if (!ok && tid == 0) {
    // a wait expired: let this CTA's own copies and MMAs drain (bounded) before freeing TMEM
    if (!tma_waited) mbar_wait(smem_u32(&bar_tma), 0, status);
    if (mma_pending) mbar_wait(smem_u32(&bar_mma), mma_phase, status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kLTmemCols);
}

// ---------------------------------------------------------------- chain kernel
// shared memory: two stages of {K tile, record A}, then U~^T, S0, U, UD
constexpr uint32_t kCStage = 58368;                // 16384 + 41472, rounded up to 1 KB
constexpr uint32_t kCOffK = 0;                     // within a stage: K [64][128] bf16, two [64][64] blocks
constexpr uint32_t kCOffRec = 16384;               // within a stage: record A
constexpr uint32_t kCOffUt = 2 * kCStage;          // fp32 U~^T [128][64] (one buffer)
constexpr uint32_t kCOffS0 = kCOffUt + kRecU;      // bf16 S0 [128 i][128 k], K-major
constexpr uint32_t kCOffU = kCOffS0 + 32768;       // bf16 U^T [128 i][64 j]
constexpr uint32_t kCOffUD = kCOffU + 16384;       // bf16 U^T diag(1/(sigma gamma)) [128 i][64 j]
constexpr uint32_t kCSmemUsed = kCOffUD + 16384;
constexpr uint32_t kCSmemAlloc = kCSmemUsed + 1024;
static_assert(kCOffRec + kRecA <= kCStage && kCStage % 1024 == 0, "stage layout");
static_assert(kCSmemAlloc <= 232448, "shared memory budget");
// tensor-memory columns
constexpr uint32_t kCColS = 0;     // S / sigma [i][k], 128 columns
constexpr uint32_t kCColX = 128;   // (W S0^T)^T [i][r]
constexpr uint32_t kCColO = 192;   // 2 x O^T [i][r], by chunk parity
constexpr uint32_t kCTmemCols = 512;
constexpr int kChainThreads = 256;   // warps 0-7: the chain's CUDA-core passes, two threads per state row
constexpr int kOutThreads = 128;     // warps 8-11: outputs
constexpr int kIssuerWarp = 12;      // warp 12: copies and MMAs
constexpr int kChainBlock = kChainThreads + kOutThreads + 32;
constexpr float kFoldBelow = 2.3283064e-10f;  // 2^-32: sigma is folded into the state below this

template <typename TOut>
__global__ void __launch_bounds__(kChainBlock, 1)
gdn_chain_kernel(const __grid_constant__ CUtensorMap tmap_k, const GdnPrefillLaunch a, const GdnTask task,
                 int nch_total, const uint8_t* recA, const uint8_t* recU, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_stage[2];  // k tile and record A landed, by stage
  __shared__ uint64_t bar_ut;        // record U landed
  __shared__ uint64_t bar_x;         // X of the chunk computed
  __shared__ uint64_t bar_s;         // state update of the chunk computed
  __shared__ uint64_t bar_o[2];      // O^T of the chunk computed, by parity
  __shared__ uint64_t bar_ofree[2];  // the output warps have read an O buffer, by parity
  __shared__ uint64_t bar_s0;        // the chain warps wrote the bf16 S0 tile of the chunk
  __shared__ uint64_t bar_u;         // the chain warps wrote the U tiles of the chunk
  __shared__ uint64_t bar_fin;       // drain after an expired wait
  __shared__ uint32_t tmem_base_sh;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127;   // state row / value index of this thread's TMEM lane
  const int half = (tid >> 7) & 1;  // chain warps: which half of the row's columns
  const CtaWork wk = cta_work(a, task);
  const int b = wk.b, h = wk.h;
  const int nchunks = wk.nchunks;
  const int64_t rec0 = wk.bh * nch_total + wk.t_begin / kC;  // record of this CTA's first chunk
  const uint32_t sbase = smem_u32(sm);
  auto stage = [&](int c) { return sbase + (uint32_t)(c & 1) * kCStage; };
  auto gate = [&](int c) {  // gamma_r of chunk c; 1/gamma_r follows
    return reinterpret_cast<const float*>(sm + (uint32_t)(c & 1) * kCStage + kCOffRec + kRecAGate);
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait(smem_u32(bar), parity, status); };

  if (tid == 0) {
    mbar_init(smem_u32(&bar_stage[0]), 1);
    mbar_init(smem_u32(&bar_stage[1]), 1);
    mbar_init(smem_u32(&bar_ut), 1);
    mbar_init(smem_u32(&bar_x), 1);
    mbar_init(smem_u32(&bar_s), 1);
    mbar_init(smem_u32(&bar_o[0]), 1);
    mbar_init(smem_u32(&bar_o[1]), 1);
    // one arrival per thread: measured slightly faster here than one per warp after __syncwarp
    mbar_init(smem_u32(&bar_ofree[0]), kOutThreads);
    mbar_init(smem_u32(&bar_ofree[1]), kOutThreads);
    mbar_init(smem_u32(&bar_s0), kChainThreads);
    mbar_init(smem_u32(&bar_u), kChainThreads);
    mbar_init(smem_u32(&bar_fin), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_k);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), kCTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  if (warp == kIssuerWarp) {
    // ================================================================ issuer (one thread)
    if ((tid & 31) == 0) {
      auto issue_stage = [&](int c) {  // k tile and record A of chunk c
        const uint32_t st = stage(c);
        const uint32_t bar = smem_u32(&bar_stage[c & 1]);
        const int t0 = (int)(wk.t_begin + (int64_t)c * kC);
        mbar_arrive_expect_tx(bar, 16384u + kRecA);
        tma_load_4d(st + kCOffK + 0, &tmap_k, 0, t0, h, b, bar);
        tma_load_4d(st + kCOffK + 8192, &tmap_k, 64, t0, h, b, bar);
        bulk_load(st + kCOffRec, recA + (rec0 + c) * kRecA, kRecA, bar);
      };
      auto issue_ut = [&](int c) {  // record U of chunk c
        const uint32_t bar = smem_u32(&bar_ut);
        mbar_arrive_expect_tx(bar, kRecU);
        bulk_load(sbase + kCOffUt, recU + (rec0 + c) * kRecU, kRecU, bar);
      };
      int st_issued = 0, st_done = 0;  // stage loads issued / known complete
      int ut_issued = 0, ut_done = 0;  // record-U loads issued / known complete
      bool ok = true, mma_issued = false;
      issue_stage(0);
      st_issued = 1;
      if (nchunks > 1) {
        issue_stage(1);
        st_issued = 2;
      }
      if (!wk.zero_v) {
        issue_ut(0);
        ut_issued = 1;
      }
      const uint32_t id = idesc_bf16(128, 64, 0, 0);
      const uint32_t id2 = idesc_bf16(128, 128, 0, 1);
      for (int c = 0; c < nchunks && ok; ++c) {
        const uint32_t par = (uint32_t)(c & 1);
        ok = wait(&bar_s0, par);  // the bf16 S0 tile of chunk c is written; chunk c-1 is done with its stage
        if (ok && c >= 1 && c + 1 < nchunks) {
          // stage of chunk c-1 -> chunk c+1, once the last MMAs reading it (O^T of chunk c-1) completed
          if (wk.write_out) ok = wait(&bar_o[par ^ 1u], (uint32_t)(((c - 1) >> 1) & 1));
          if (ok) {
            issue_stage(c + 1);
            st_issued = c + 2;
          }
        }
        ok = ok && wait(&bar_stage[c & 1], (uint32_t)((c >> 1) & 1));
        if (!ok) break;
        st_done = c + 1;
        tc_fence_after();
        const uint32_t st = stage(c);
        const uint32_t rec = st + kCOffRec;
        // X = S0 W^T
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t koff = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
          const uint32_t woff = (uint32_t)(ks >> 2) * 8192u + (uint32_t)(ks & 3) * 32u;
          mma_bf16(tmem + kCColX, kmaj(sbase + kCOffS0 + koff), kmaj(rec + kRecAW + woff), id, ks > 0);
        }
        mma_commit(smem_u32(&bar_x));
        mma_issued = true;
        // O^T = S0 Q'^T into the buffer of this parity, once the output warps drained it (chunk c-2)
        if (wk.write_out) {
          if (c >= 2) ok = wait(&bar_ofree[par], (uint32_t)(((c - 2) >> 1) & 1));
          if (!ok) break;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t koff = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
            const uint32_t qoff = (uint32_t)(ks >> 2) * 8192u + (uint32_t)(ks & 3) * 32u;
            mma_bf16(tmem + kCColO + 64 * par, kmaj(sbase + kCOffS0 + koff), kmaj(rec + kRecAQ + qoff), id, ks > 0);
          }
        }
        ok = wait(&bar_u, par);  // U tiles written; U~^T of chunk c read
        if (!ok) break;
        ut_done = wk.zero_v ? 0 : c + 1;
        tc_fence_after();
        if (c + 1 < nchunks && !wk.zero_v) {
          issue_ut(c + 1);
          ut_issued = c + 2;
        }
        // S/sigma += U^T diag(1/(sigma gamma)) K ; O^T += U^T P_o'^T
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + kCColS, kmaj(sbase + kCOffUD + ks * 32), sw128_desc(st + kCOffK + ks * 2048, 8192, 1024),
                   id2, 1u);
        mma_commit(smem_u32(&bar_s));
        if (wk.write_out) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + kCColO + 64 * par, kmaj(sbase + kCOffU + ks * 32), kmaj(rec + kRecAPo + ks * 32), id,
                     1u);
          mma_commit(smem_u32(&bar_o[par]));
        }
      }
      if (!ok) {
        // a wait expired: let this CTA's own copies and MMAs drain (bounded) before TMEM is freed
        for (int k = st_done; k < st_issued; ++k) wait(&bar_stage[k & 1], (uint32_t)((k >> 1) & 1));
        for (int k = ut_done; k < ut_issued; ++k) wait(&bar_ut, (uint32_t)(k & 1));
        if (mma_issued) {
          mma_commit(smem_u32(&bar_fin));  // arrives once every MMA issued so far has completed
          wait(&bar_fin, 0);
        }
      }
    }
  } else if (tid < kChainThreads) {
    // ================================================================ chain warps (lane i = row i of S;
    // this thread: columns [64 half, 64 half + 64) of the state, [32 half, 32 half + 32) of U)
    bool ok = true;
    // Initial state (sigma = 1) and its bf16 S0 copy.
    {
      const int hf = half;
      const float* src = wk.s_entry ? wk.s_entry + (int64_t)row * kD + 64 * hf : nullptr;
      float v[64];
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 x = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[j] = x.x; v[j + 1] = x.y; v[j + 2] = x.z; v[j + 3] = x.w;
      }
      if (wk.zero_v) {  // identity entry state: the run then yields the segment's linear map M_g
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = (64 * hf + j == row) ? 1.f : 0.f;
      }
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16)
        tmem_st16(tlane + kCColS + 64 * hf + c0, *reinterpret_cast<float(*)[16]>(v + c0));
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(sm + kCOffS0 + sw128_off(row, 64 * hf + 8 * q, 128)) = pack8_bf16(v + 8 * q);
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(smem_u32(&bar_s0));
    float sigma = 1.f;
    // An expired wait leaves this thread's `ok` false: it skips its later waits (so it meets at most one
    // expiry) but still makes every arrival, so no warp waits on it, and the final state is not written.

    for (int c = 0; c < nchunks; ++c) {
      const bool has_next = c + 1 < nchunks;
      const uint32_t par = (uint32_t)(c & 1);
      ok = ok && wait(&bar_stage[c & 1], (uint32_t)((c >> 1) & 1)) && wait(&bar_x, par) &&
           (wk.zero_v || wait(&bar_ut, par));
      tc_fence_after();
      // ---- U^T = U~^T - X and U^T diag(1 / (sigma gamma)), this row, columns [32 half, 32 half + 32)
      {
        const float* gi = gate(c) + kC;
        const float inv_sigma = 1.f / sigma;
        const uint8_t* ur = sm + kCOffUt + row * 256;
        {
          const int hf = half;
          float u[32], x[32];
          tmem_ld16(tlane + kCColX + 32 * hf, *reinterpret_cast<float(*)[16]>(x));
          tmem_ld16(tlane + kCColX + 32 * hf + 16, *reinterpret_cast<float(*)[16]>(x + 16));
          if (wk.zero_v) {
#pragma unroll
            for (int j = 0; j < 32; ++j) u[j] = 0.f;
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 f = *reinterpret_cast<const float4*>(ur + (((8 * hf + q) ^ (row & 15)) << 4));
              u[4 * q] = f.x; u[4 * q + 1] = f.y; u[4 * q + 2] = f.z; u[4 * q + 3] = f.w;
            }
          }
          tmem_ld_wait();
          float ud[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            u[j] -= x[j];
            ud[j] = u[j] * (gi[32 * hf + j] * inv_sigma);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            *reinterpret_cast<uint4*>(sm + kCOffU + sw128_off(row, 32 * hf + 8 * q, 128)) = pack8_bf16(u + 8 * q);
            *reinterpret_cast<uint4*>(sm + kCOffUD + sw128_off(row, 32 * hf + 8 * q, 128)) = pack8_bf16(ud + 8 * q);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_u));
      ok = ok && wait(&bar_s, par);
      tc_fence_after();

      // ---- sigma <- sigma gamma_C; bf16 S0 = sigma S~ for chunk c+1, folding sigma into S~ when small
      const float sigma_new = sigma * gate(c)[kC - 1];
      const bool fold = sigma_new < kFoldBelow;
      if (has_next || fold) {
        {
          const int hf = half;
          float v[64];
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 16)
            tmem_ld16(tlane + kCColS + 64 * hf + c0, *reinterpret_cast<float(*)[16]>(v + c0));
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 64; ++j) v[j] *= sigma_new;
          if (has_next) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(sm + kCOffS0 + sw128_off(row, 64 * hf + 8 * q, 128)) = pack8_bf16(v + 8 * q);
          }
          if (fold) {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16)
              tmem_st16(tlane + kCColS + 64 * hf + c0, *reinterpret_cast<float(*)[16]>(v + c0));
            tmem_st_wait();
          }
        }
      }
      sigma = fold ? 1.f : sigma_new;
      if (has_next) {
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_s0));
      }
    }

    ok = __all_sync(0xffffffffu, ok);  // warp-uniform: the final-state loads below are warp-collective
    if (ok && wk.s_exit) {
      // final state S = sigma S~: lane i row i, this thread's half of the columns
      float* dst = wk.s_exit + (int64_t)row * kD;
      {
        const int hf = half;
        float v[64];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16)
          tmem_ld16(tlane + kCColS + 64 * hf + c0, *reinterpret_cast<float(*)[16]>(v + c0));
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 64; j += 4)
          *reinterpret_cast<float4*>(dst + 64 * hf + j) =
              make_float4(sigma * v[j], sigma * v[j + 1], sigma * v[j + 2], sigma * v[j + 3]);
      }
    }
  } else if (wk.write_out) {
    // ================================================================ output warps
    // O^T of chunk c: lane i = value index, columns = the chunk's 64 tokens.
    bool ok = true;  // as in the chain warps: an expired wait skips the later waits, never an arrival
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t par = (uint32_t)(c & 1);
      ok = ok && wait(&bar_o[par], (uint32_t)((c >> 1) & 1));
      tc_fence_after();
      float o[64];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16)
        tmem_ld16(tlane + kCColO + 64 * par + c0, *reinterpret_cast<float(*)[16]>(o + c0));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_ofree[par]));  // the buffer may be overwritten from here on
      const int64_t t0 = wk.t_begin + (int64_t)c * kC;
      const int nvalid = (wk.t_end - t0 < kC) ? (int)(wk.t_end - t0) : kC;
      TOut* optr = reinterpret_cast<TOut*>(a.o) + b * a.o_sb + h * a.o_sh + t0 * a.o_st + row;
#pragma unroll
      for (int r = 0; r < 64; ++r) {
        if (r < nvalid) store1(optr, o[r]);
        optr += a.o_st;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kCTmemCols);
}

size_t records_bytes(int64_t BH, int64_t nch) { return (size_t)(BH * nch) * (size_t)(kRecA + kRecU); }

template <typename TOut>
cudaError_t launch_split_typed(const GdnPrefillLaunch& a, void* ws, unsigned* status, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!gdn_make_map(&mq, a.q, a.B, a.H, a.N) || !gdn_make_map(&mk, a.k, a.B, a.H, a.N) ||
      !gdn_make_map(&mv, a.v, a.B, a.H, a.N))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gdn_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLSmemAlloc);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gdn_chain_kernel<TOut>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kCSmemAlloc);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t BH = a.B * a.H;
  const int64_t nch = (a.N + kC - 1) / kC;
  uint8_t* recA = static_cast<uint8_t*>(ws);
  uint8_t* recU = recA + (size_t)(BH * nch) * kRecA;
  float* seg = reinterpret_cast<float*>(recA + records_bytes(BH, nch));
  gdn_local_kernel<<<(unsigned)(BH * nch), kThreads, kLSmemAlloc, stream>>>(mq, mk, mv, a, (int)nch, recA, recU,
                                                                           status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const GdnSegPlan plan = gdn_segment_plan(a.B, a.H, a.N);
  if (plan.G == 1) {
    const GdnTask task{kWhole, 1, a.N, nullptr, nullptr};
    gdn_chain_kernel<TOut><<<(unsigned)BH, kChainBlock, kCSmemAlloc, stream>>>(mk, a, task, (int)nch, recA, recU,
                                                                           status);
    return cudaGetLastError();
  }
  float* maps = seg;
  float* states = maps + BH * (plan.G - 1) * 2 * kStateElems;
  const GdnTask t1{kSegmentMaps, plan.G, plan.seg_len, maps, nullptr};
  gdn_chain_kernel<TOut><<<(unsigned)(BH * (plan.G - 1) * 2), kChainBlock, kCSmemAlloc, stream>>>(
      mk, a, t1, (int)nch, recA, recU, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_gdn_segment_combine(a.S_in, maps, states, plan.G, BH, stream);
  if (e != cudaSuccess) return e;
  const GdnTask t2{kSegmentOutputs, plan.G, plan.seg_len, nullptr, states};
  gdn_chain_kernel<TOut><<<(unsigned)(BH * plan.G), kChainBlock, kCSmemAlloc, stream>>>(mk, a, t2, (int)nch, recA,
                                                                                    recU, status);
  return cudaGetLastError();
}

}  // namespace

size_t gdn_split_workspace_bytes(int64_t B, int64_t H, int64_t N) {
  const int64_t BH = B * H;
  if (BH <= 0 || N <= 0) return 0;
  const int64_t nch = (N + kC - 1) / kC;
  return records_bytes(BH, nch) + gdn_segment_plan(B, H, N).ws_bytes;
}

cudaError_t launch_gdn_prefill_split(const GdnPrefillLaunch& a, void* ws, size_t ws_bytes, unsigned* status,
                                     cudaStream_t stream) {
  const int64_t BH = a.B * a.H;
  if (BH == 0 || a.N == 0) return cudaSuccess;
  const int64_t nch = (a.N + kC - 1) / kC;
  if (BH * nch > (int64_t)INT32_MAX) return cudaErrorInvalidValue;  // one chunk-local CTA per chunk
  if (ws == nullptr || ws_bytes < gdn_split_workspace_bytes(a.B, a.H, a.N)) return cudaErrorInvalidValue;
  return a.out_bf16 ? launch_split_typed<__nv_bfloat16>(a, ws, status, stream)
                    : launch_split_typed<float>(a, ws, status, stream);
}

}  // namespace la
