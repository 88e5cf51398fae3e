// gdn_common.cuh -- pieces shared by the two schedules of the chunked
// gated-delta-rule prefill: the single-kernel chunk scan (gdn_chunked.cu) and
// the two-kernel scan (gdn_scan.cu).  Sizes, the per-launch task of the
// sequence-segment scheme, and the chunk-local phases of the chunk form
// (NoteBank Sec. 2 Eq. (1), A_t = alpha_t (I - beta_t k_t k_t^T)):
//   g_r = sum_{j<=r} log alpha_j,  gamma_r = e^{g_r},  Gamma_rj = e^{g_r - g_j}
//   L   = strict_lower(diag(beta) (Gamma . K K^T)),   T = (I + L)^{-1}
//   W   = T diag(beta gamma) K,   U~ = T diag(beta) V,   P_o = tril(Gamma) . Q K^T
// None of these depends on the state; only U = U~ - W S0^T and what follows do.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace la {
namespace gdn {
using namespace tc;

// ---------------------------------------------------------------- helpers only these kernels use
// Orders this thread's generic-proxy view of global memory with its async-proxy (bulk copy)
// accesses: after acquiring a flag, before copying what the flag guards with cp.async.bulk.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------- flags between CTAs of one grid
// Release: every global write this thread has observed (its own, and those of the threads of its
// CTA ordered before it by a barrier) is visible GPU-wide before the flag reads `v`.
__device__ __forceinline__ void flag_release(unsigned* flag, unsigned v) {
  asm volatile("fence.acq_rel.gpu;\n\tst.relaxed.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(v) : "memory");
}
// Waits until *flag == v (acquire: what the releasing thread had observed is then visible to this
// thread); gives up after kWaitLimitNs, ORs kStatusTimeout into *status and returns false.  Only
// for flags set by CTAs of the same grid that are co-resident (a cooperative launch) and never
// wait on the waiting CTA.
__device__ __forceinline__ bool flag_wait(const unsigned* flag, unsigned v, unsigned* status) {
  uint64_t t0 = 0;
  for (int i = 0;; ++i) {
    unsigned x;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(x) : "l"(flag) : "memory");
    if (x == v) return true;
    if (i == 0) t0 = globaltimer_ns();
    else if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
    __nanosleep(128);
  }
}

// Cooperative launch: every CTA of the grid is resident at once (the launch fails otherwise), so
// CTAs may wait on flags other CTAs of the grid set.
template <typename... KArgs, typename... Args>
cudaError_t launch_cooperative(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// A relaxed GPU-scope read of a flag, issued early; if it already shows the value, fence_acq_rel_gpu
// where the guarded data is used makes the pair an acquire.
__device__ __forceinline__ unsigned flag_peek(const unsigned* flag) {
  unsigned x;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(x) : "l"(flag) : "memory");
  return x;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Instruction descriptor, kind::tf32: fp32 A/B read from shared memory at tf32 precision, both
// K-major, fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4)                       // D format: f32
         | (2u << 7)                     // A format: tf32
         | (2u << 10)                    // B format: tf32
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}
// D[tmem] (+)= A[smem] * B[smem]^T, fp32 operands at tf32 precision (one 8-deep K step: 32 bytes of
// each operand row), issued by one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Byte offset of fp32 element (row, col) in a K-major 128-byte-swizzled fp32 tile: panels of 32
// columns (128-byte rows), `rows` rows per panel; 16-byte chunks of a row permuted by row & 7.
__host__ __device__ __forceinline__ uint32_t sw128_off_f32(uint32_t row, uint32_t col, uint32_t rows) {
  return (col >> 5) * rows * 128u + row * 128u + ((((col & 31u) >> 2) ^ (row & 7u)) << 4) + ((col & 3u) << 2);
}

constexpr int kC = 64;         // tokens per chunk
constexpr int kD = 128;        // d_k = d_v
constexpr int kThreads = 256;  // two threads per tensor-memory lane, splitting its columns
constexpr int64_t kStateElems = (int64_t)kD * kD;
constexpr int kLStride = 65;  // fp32 L rows, padded
constexpr int kTStride = 64;  // fp32 T rows

// What one launch computes.  kWhole: every (b,h) from its entry state to the
// end.  Sequence segments (few (b,h) pairs, long N): with d_v = d_k a segment
// acts on its entry state as an affine map S_end = S_start M + B.
// kSegmentMaps runs the scan over every segment but the last twice without
// outputs, from S = 0 (final state B_g) and from S = I with V taken as zero
// (final state M_g); kSegmentOutputs reruns each segment from the entry state
// a combine kernel chained from the maps, writing outputs (and the last
// segment the final state).
constexpr int kWhole = 0, kSegmentMaps = 1, kSegmentOutputs = 2;
struct GdnTask {
  int mode;             // kWhole, kSegmentMaps or kSegmentOutputs
  int G;                // segments per (b,h)
  int64_t seg_len;      // tokens per segment (a multiple of the chunk)
  float* maps;          // kSegmentMaps: [BH][G-1][2][128][128]  (B_g, then M_g)
  const float* states;  // kSegmentOutputs: [BH][G][128][128] entry states
  // kWhole with the chunk records formed in the same launch: CTAs n_scan.. (by placement rank) run
  // the inversion and set ready[record] = 1 once a record is written (null: the records are complete
  // at launch); place: the launch's zeroed placement scratch (an arrival counter, then one word per
  // SM id); progress: zeroed, one word
  int n_scan;
  unsigned* ready;
  unsigned* place;
  unsigned* progress;  // chunks whose copies all scans together have issued (a pacing hint)
};

// The (b,h), segment, token range and entry/exit states of one CTA of `task`.
struct CtaWork {
  int64_t bh;
  int b, h, seg;
  int64_t t_begin, t_end;
  int nchunks;
  bool zero_v;     // identity entry state with V taken as zero (the map M_g)
  bool write_out;  // outputs are written
  const float* s_entry;
  float* s_exit;
};

// `cta`: this CTA's index in the task (its blockIdx.x unless the launch places its CTAs itself).
__device__ __forceinline__ CtaWork cta_work(const GdnPrefillLaunch& a, const GdnTask& task, int cta) {
  CtaWork w{};
  int which = 0;
  if (task.mode == kWhole) {
    w.bh = cta;
  } else if (task.mode == kSegmentMaps) {
    const int per = 2 * (task.G - 1);
    w.bh = cta / per;
    w.seg = (int)(cta % per) >> 1;
    which = (int)(cta % per) & 1;  // 0: B_g (zero entry state), 1: M_g (identity entry, V taken as 0)
  } else {
    w.bh = cta / task.G;
    w.seg = (int)(cta % task.G);
  }
  w.b = (int)(w.bh / a.H);
  w.h = (int)(w.bh % a.H);
  w.t_begin = task.mode == kWhole ? 0 : (int64_t)w.seg * task.seg_len;
  w.t_end = task.mode == kWhole ? a.N : min(a.N, w.t_begin + task.seg_len);
  w.nchunks = (int)((w.t_end - w.t_begin + kC - 1) / kC);
  w.zero_v = task.mode == kSegmentMaps && which == 1;
  w.write_out = task.mode != kSegmentMaps;
  w.s_entry = task.mode == kWhole            ? (a.S_in ? a.S_in + w.bh * kStateElems : nullptr)
              : task.mode == kSegmentOutputs ? task.states + (w.bh * task.G + w.seg) * kStateElems
                                             : nullptr;
  w.s_exit = task.mode == kWhole ? a.S_out + w.bh * kStateElems
             : task.mode == kSegmentMaps
                 ? task.maps + ((w.bh * (task.G - 1) + w.seg) * 2 + which) * kStateElems
                 : (w.seg == task.G - 1 ? a.S_out + w.bh * kStateElems : nullptr);
  return w;
}

__device__ __forceinline__ uint64_t kmaj(uint32_t addr) { return sw128_desc(addr, 0, 1024); }

// 32 consecutive TMEM columns of this thread's lane, one wait.
__device__ __forceinline__ void ld32(uint32_t taddr, float* v) {
  tmem_ld16(taddr, *reinterpret_cast<float(*)[16]>(v));
  tmem_ld16(taddr + 16, *reinterpret_cast<float(*)[16]>(v + 16));
  tmem_ld_wait();
}

__device__ __forceinline__ void st_bf16(uint8_t* p, float x) {
  *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(x);
}

// Gate tables of one chunk from this thread's log alpha and beta (threads
// 0..63 hold token tid of the chunk): inclusive scan of log alpha, then
// g, beta, gamma = e^g and 1/gamma into gate[0..63], [64..127], [128..191],
// [192..255].  Contains a block-wide barrier; `carry` is one shared float.
template <typename Sync>
__device__ __forceinline__ void gate_tables(int tid, float lg, float bt, float* gate, float* carry, Sync sync) {
  const int lane = tid & 31, warp = tid >> 5;
  float gx = lg;
  if (tid < kC) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(kFullMask, gx, off);
      if (lane >= off) gx += y;
    }
    if (tid == 31) *carry = gx;
  }
  sync();
  if (tid < kC) {
    if (warp == 1) gx += *carry;
    gate[tid] = gx;
    gate[kC + tid] = bt;
    gate[2 * kC + tid] = __expf(gx);
    gate[3 * kC + tid] = __expf(-gx);
  }
}
__device__ __forceinline__ void gate_tables(int tid, float lg, float bt, float* gate, float* carry) {
  gate_tables(tid, lg, bt, gate, carry, [] { __syncthreads(); });
}

// [K;Q] K^T of one chunk into 64 TMEM columns (lanes 0..63: K K^T, lanes
// 64..127: Q K^T).  kq_tile: the stacked [K;Q] tile, 128 rows in two
// 64-column blocks 16 KB apart (K rows first).  Issued by one thread.
__device__ __forceinline__ void mma_kq(uint32_t d_tmem, uint32_t kq_tile) {
  const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t koff = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
    mma_bf16(d_tmem, kmaj(kq_tile + koff), kmaj(kq_tile + koff), id, ks > 0);
  }
}

// W^T = K^T (T diag(beta gamma))^T and U~^T = V^T (T diag(beta))^T into 64
// TMEM columns each.  v_tile: [64][128] bf16 in two 64-column blocks 8 KB
// apart; t1, t2: bf16 [64][64] K-major tiles.  Issued by one thread.
__device__ __forceinline__ void mma_wu(uint32_t d_w, uint32_t d_ut, uint32_t kq_tile, uint32_t v_tile, uint32_t t1,
                                       uint32_t t2) {
  const uint32_t id = idesc_bf16(128, 64, 1, 0);
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
    mma_bf16(d_w, sw128_desc(kq_tile + ks * 2048, 16384, 1024), kmaj(t1 + ks * 32), id, ks > 0);
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
    mma_bf16(d_ut, sw128_desc(v_tile + ks * 2048, 8192, 1024), kmaj(t2 + ks * 32), id, ks > 0);
}

// delta * L (fp32 [64][kLStride]) and the bf16 tile po_scale * P_o [64][64]
// of one chunk from [K;Q] K^T in TMEM.  delta = 0 is the scalar gate
// (A_t = alpha_t I): nothing is erased, so L = 0 (T = I, U~ = diag(beta) V)
// here and W = 0 in phase_T.  kq_taddr: this thread's lane at the first of
// its 32 columns; gate: the chunk's gate tables.  A null po_tile skips P_o
// (the lanes of the Q rows then do nothing); po_row_gamma = false leaves out
// the row factor gamma_r (P_rj = po_scale (q_r . k_j) / gamma_j, j <= r).
__device__ __forceinline__ void phase_L_Po(uint32_t kq_taddr, int row, int half, const float* gate, float* Lsm,
                                           uint8_t* po_tile, float po_scale, float delta, bool po_row_gamma = true) {
  float v[32];
  ld32(kq_taddr, v);
  const int j0 = 32 * half;
  const float* bt = gate + kC;
  const float* gm = gate + 2 * kC;
  const float* gi = gate + 3 * kC;
  if (row < kC) {
    const int r = row;
    const float f = bt[r] * gm[r] * delta;
    float* Lrow = Lsm + r * kLStride + j0;
#pragma unroll
    for (int j = 0; j < 32; ++j) Lrow[j] = (j0 + j < r) ? f * gi[j0 + j] * v[j] : 0.f;
  } else if (po_tile != nullptr) {
    const int r = row - kC;
    const float f = (po_row_gamma ? gm[r] : 1.f) * po_scale;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = (j0 + j <= r) ? f * gi[j0 + j] * v[j] : 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(po_tile + sw128_off(r, j0 + 8 * q, 64)) = pack8_bf16(v + 8 * q);
  }
}

// T = (I + L)^{-1} by doubling (16x16 diagonal blocks by forward
// substitution, then 32x32 and 64x64 blocks from
// [[A,0],[C,B]]^-1 = [[A^-1,0],[-B^-1 C A^-1, B^-1]]), then the bf16 tiles
// delta T diag(beta gamma) (the erase of the incoming state; zero for the
// scalar gate) and T diag(beta) (zero when zero_v).  T is fp32 with 64
// floats per row; Trow(r) gives row r (16-byte aligned).  Zsm: 1024 fp32 of
// block products.  Every thread of the block calls it; it contains
// block-wide barriers, and L is no longer read once the last one has passed
// (the bf16 tiles may overlay it).
template <typename TRow>
__device__ __forceinline__ void phase_T(int tid, const float* Lsm, TRow Trow, float* Zsm, const float* gate,
                                        bool zero_v, float delta, uint8_t* t1_tile, uint8_t* t2_tile) {
  if (tid < kC) {
    // 16x16 diagonal blocks, right-looking substitution: one thread per block column
    const int base = (tid >> 4) * 16, col = tid & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) x[r] = (r == col) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      const float* Lc = Lsm + (base + j + 1) * kLStride + base + j;
#pragma unroll
      for (int r = j + 1; r < 16; ++r) x[r] = fmaf(-Lc[(r - j - 1) * kLStride], x[j], x[r]);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Trow(base + r)[base + col] = x[r];
  } else {
    // zero the six 16x16 blocks above the block diagonal
    for (int e = tid - kC; e < 6 * 256; e += kThreads - kC) {
      const int pr = e >> 8, w = e & 255;
      const int bi = pr < 3 ? 0 : (pr < 5 ? 1 : 2);
      const int bj = pr < 3 ? pr + 1 : (pr < 5 ? pr - 1 : 3);
      Trow(bi * 16 + (w >> 4))[bj * 16 + (w & 15)] = 0.f;
    }
  }
  __syncthreads();
  {
    // level 32: [[A,0],[C,B]]^-1 lower-left block = -B^-1 (C A^-1); blocks k = 0, 1
    const int k = tid >> 7, r = (tid >> 3) & 15, c0 = (tid & 7) * 2;
    const int R = 32 * k + 16, Cb = 32 * k;
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float l = Lsm[(R + r) * kLStride + Cb + m];
      const float* tm = Trow(Cb + m);
      z0 = fmaf(l, tm[Cb + c0], z0);
      z1 = fmaf(l, tm[Cb + c0 + 1], z1);
    }
    Zsm[k * 256 + r * 16 + c0] = z0;
    Zsm[k * 256 + r * 16 + c0 + 1] = z1;
    __syncthreads();
    float t0v = 0.f, t1v = 0.f;
    const float* tr = Trow(R + r);
#pragma unroll
    for (int p2 = 0; p2 < 16; ++p2) {
      const float tv = tr[R + p2];
      t0v = fmaf(tv, Zsm[k * 256 + p2 * 16 + c0], t0v);
      t1v = fmaf(tv, Zsm[k * 256 + p2 * 16 + c0 + 1], t1v);
    }
    Trow(R + r)[Cb + c0] = -t0v;
    Trow(R + r)[Cb + c0 + 1] = -t1v;
  }
  __syncthreads();
  {
    // level 64: rows 32.., columns 0..31; thread: 4 columns of one row
    const int r = tid >> 3, c0 = (tid & 7) * 4;
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const float l = Lsm[(32 + r) * kLStride + m];
      const float4 tv = *reinterpret_cast<const float4*>(Trow(m) + c0);
      z.x = fmaf(l, tv.x, z.x); z.y = fmaf(l, tv.y, z.y); z.z = fmaf(l, tv.z, z.z); z.w = fmaf(l, tv.w, z.w);
    }
    *reinterpret_cast<float4*>(Zsm + r * 32 + c0) = z;
    __syncthreads();
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* tr = Trow(32 + r);
#pragma unroll 8
    for (int p2 = 0; p2 < 32; ++p2) {
      const float tv = tr[32 + p2];
      const float4 zz = *reinterpret_cast<const float4*>(Zsm + p2 * 32 + c0);
      o.x = fmaf(tv, zz.x, o.x); o.y = fmaf(tv, zz.y, o.y); o.z = fmaf(tv, zz.z, o.z); o.w = fmaf(tv, zz.w, o.w);
    }
    *reinterpret_cast<float4*>(Trow(32 + r) + c0) = make_float4(-o.x, -o.y, -o.z, -o.w);
  }
  __syncthreads();
  {
    const int r = tid >> 2, c0 = (tid & 3) * 16;
    const float* bt = gate + kC;
    const float* gm = gate + 2 * kC;
    const float* tr = Trow(r);
    float t1[16], t2[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float tv = tr[c0 + j];
      t2[j] = tv * bt[c0 + j];
      t1[j] = t2[j] * gm[c0 + j] * delta;
    }
    if (zero_v) {  // V taken as zero: U~ = T diag(beta) V = 0
#pragma unroll
      for (int j = 0; j < 16; ++j) t2[j] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      *reinterpret_cast<uint4*>(t1_tile + sw128_off(r, c0 + 8 * q, 64)) = pack8_bf16(t1 + 8 * q);
      *reinterpret_cast<uint4*>(t2_tile + sw128_off(r, c0 + 8 * q, 64)) = pack8_bf16(t2 + 8 * q);
    }
  }
}

}  // namespace gdn

// Host side, defined in gdn_chunked.cu.
// Tensor map of a bf16 [B, H, N, 128] view: (64 features x 64 tokens) box,
// 128-byte swizzle; false when the view cannot be described (strides of 0 or
// not multiples of 16 bytes).
bool gdn_make_map(CUtensorMap* m, const View4& x, int64_t B, int64_t H, int64_t N);
// Entry states of the G segments of every (b,h) from their maps.
cudaError_t launch_gdn_segment_combine(const float* S_in, const float* maps, float* states, int G, int64_t BH,
                                       cudaStream_t stream);

}  // namespace la
