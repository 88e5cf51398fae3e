// api.cu -- the extern "C" entry points declared in include/la.h.
//
// Host side only: argument validation (before anything is launched), the
// N == 0 state pass-through, and dispatch to the kernel launchers.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "la.h"

namespace la {
namespace {
thread_local int t_last_cuda_error = 0;
}  // namespace
void note_cuda_error(int code) { t_last_cuda_error = code; }
int last_cuda_error() { return t_last_cuda_error; }
}  // namespace la

namespace {

// Device status word set by bounded waits that expire (LA_ERR_TIMEOUT).
__device__ unsigned g_la_device_status = 0;

unsigned* device_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_la_device_status) != cudaSuccess) return nullptr;
  return static_cast<unsigned*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(la_dtype t) { return t == LA_DTYPE_BF16 ? 2 : 4; }

bool valid_dtype(la_dtype t) { return t == LA_DTYPE_F32 || t == LA_DTYPE_BF16; }

// A [B,H,N,d] view: non-null (unless empty), 16-byte aligned base and token
// stride, non-negative strides, and rows that do not overlap along t.
bool valid_view(const la_tensor& x, int64_t B, int64_t H, int64_t N, int64_t d, la_dtype dt) {
  if (B * H * N == 0) return true;
  if (x.ptr == nullptr || !aligned16(x.ptr)) return false;
  if (x.stride_b < 0 || x.stride_h < 0 || x.stride_t < 0) return false;
  if (N > 1 && x.stride_t < d) return false;
  if ((x.stride_t * elem_bytes(dt)) % 16 != 0) return false;
  if ((x.stride_h * elem_bytes(dt)) % 16 != 0 || (x.stride_b * elem_bytes(dt)) % 16 != 0) return false;
  return true;
}

bool valid_gate(const la_tensor& x, int64_t B, int64_t H, int64_t N) {
  if (B * H * N == 0) return true;
  if (x.ptr == nullptr || (reinterpret_cast<uintptr_t>(x.ptr) & 3u) != 0) return false;
  if (x.stride_b < 0 || x.stride_h < 0) return false;
  return x.stride_t == 1;
}

la::View4 view(const la_tensor& x) { return la::View4{x.ptr, x.stride_b, x.stride_h, x.stride_t}; }

la_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return LA_OK;
  la::note_cuda_error((int)e);
  return LA_ERR_CUDA;
}

// N == 0: the final state is the initial state (or zero).
la_status pass_state(float* out, const float* in, size_t n_floats, cudaStream_t s) {
  if (n_floats == 0) return LA_OK;
  if (in == out) return LA_OK;
  const size_t bytes = n_floats * sizeof(float);
  if (in) return from_cuda(cudaMemcpyAsync(out, in, bytes, cudaMemcpyDeviceToDevice, s));
  return from_cuda(cudaMemsetAsync(out, 0, bytes, s));
}

constexpr int64_t kTaylorF = 16, kTaylorDv = 64, kTaylorD = 1 + 16 + 16 * 16;
constexpr int64_t kGdnD = 128;
constexpr int64_t kMaxDim = int64_t(1) << 40;
constexpr int64_t kMaxElems = int64_t(1) << 44;  // elements of one state array (64 TiB of fp32)

la_status check_based(const la_based_prefill_args* a) {
  if (!a) return LA_ERR_INVALID_ARGUMENT;
  if (a->B < 0 || a->H < 0 || a->N < 0 || a->B > kMaxDim || a->H > kMaxDim || a->N > kMaxDim)
    return LA_ERR_INVALID_ARGUMENT;
  if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return LA_ERR_INVALID_ARGUMENT;
  if (a->d_feat != kTaylorF || a->d_v != kTaylorDv) return LA_ERR_UNSUPPORTED;
  if (a->B * a->H > (int64_t(1) << 31) - 1) return LA_ERR_UNSUPPORTED;
  if (a->N > INT32_MAX - 128) return LA_ERR_UNSUPPORTED;  // tile coordinates are 32-bit
  const int64_t B = a->B, H = a->H, N = a->N;
  if (!valid_view(a->q, B, H, N, kTaylorF, a->in_dtype) || !valid_view(a->k, B, H, N, kTaylorF, a->in_dtype) ||
      !valid_view(a->v, B, H, N, kTaylorDv, a->in_dtype) || !valid_view(a->y, B, H, N, kTaylorDv, a->out_dtype))
    return LA_ERR_INVALID_ARGUMENT;
  if (B * H > 0) {
    if (!a->s_out || !a->z_out) return LA_ERR_INVALID_ARGUMENT;
    if (!aligned16(a->s_out) || !aligned16(a->s_in) || (reinterpret_cast<uintptr_t>(a->z_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(a->z_in) & 3u) || (reinterpret_cast<uintptr_t>(a->decay) & 3u))
      return LA_ERR_INVALID_ARGUMENT;
  }
  return LA_OK;
}

la_status check_gdn(const la_gdn_prefill_args* a) {
  if (!a) return LA_ERR_INVALID_ARGUMENT;
  if (a->B < 0 || a->H < 0 || a->N < 0 || a->B > kMaxDim || a->H > kMaxDim || a->N > kMaxDim)
    return LA_ERR_INVALID_ARGUMENT;
  if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return LA_ERR_INVALID_ARGUMENT;
  if (a->d_k != kGdnD || a->d_v != kGdnD) return LA_ERR_UNSUPPORTED;
  if (a->B * a->H > (int64_t(1) << 28)) return LA_ERR_UNSUPPORTED;
  if (a->N > INT32_MAX - 128) return LA_ERR_UNSUPPORTED;  // tile coordinates are 32-bit
  const int64_t B = a->B, H = a->H, N = a->N;
  if (!valid_view(a->q, B, H, N, kGdnD, a->in_dtype) || !valid_view(a->k, B, H, N, kGdnD, a->in_dtype) ||
      !valid_view(a->v, B, H, N, kGdnD, a->in_dtype) || !valid_view(a->o, B, H, N, kGdnD, a->out_dtype))
    return LA_ERR_INVALID_ARGUMENT;
  if (!valid_gate(a->alpha, B, H, N) || !valid_gate(a->beta, B, H, N)) return LA_ERR_INVALID_ARGUMENT;
  if (B * H > 0) {
    if (!a->S_out || !aligned16(a->S_out) || !aligned16(a->S_in)) return LA_ERR_INVALID_ARGUMENT;
  }
  return LA_OK;
}

}  // namespace

namespace {

// The GDN-family prefill: delta = 1 is the gated delta rule, delta = 0 the
// scalar gate A_t = alpha_t I; both share validation, workspace and kernels.
la_status gdn_family_prefill(const la_gdn_prefill_args* a, void* ws, size_t ws_bytes, void* stream, float delta) {
  const la_status st = check_gdn(a);
  if (st != LA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t BH = a->B * a->H;
  if (BH == 0) return LA_OK;
  if (a->N == 0) return pass_state(a->S_out, a->S_in, (size_t)(BH * kGdnD * kGdnD), s);
  // bf16: the two-kernel scan when the workspace holds its per-chunk inverse
  // records, else the single-kernel scan, which needs the segment scratch only
  bool split = false;
  if (a->in_dtype == LA_DTYPE_BF16) {
    if (ws != nullptr && !aligned16(ws)) return LA_ERR_WORKSPACE;
    const int64_t nch = (a->N + 63) / 64;
    split = ws != nullptr && ws_bytes >= la::gdn_scan_workspace_bytes(a->B, a->H, a->N) && BH * nch <= INT32_MAX;
    const size_t need_min = la::gdn_segment_plan(a->B, a->H, a->N).ws_bytes;
    if (!split && need_min > 0 && (ws == nullptr || ws_bytes < need_min)) return LA_ERR_WORKSPACE;
  }
  la::GdnPrefillLaunch L{};
  L.B = a->B; L.H = a->H; L.N = a->N;
  L.in_bf16 = a->in_dtype == LA_DTYPE_BF16;
  L.out_bf16 = a->out_dtype == LA_DTYPE_BF16;
  L.q = view(a->q); L.k = view(a->k); L.v = view(a->v);
  L.o = a->o.ptr; L.o_sb = a->o.stride_b; L.o_sh = a->o.stride_h; L.o_st = a->o.stride_t;
  L.alpha = static_cast<const float*>(a->alpha.ptr); L.a_sb = a->alpha.stride_b; L.a_sh = a->alpha.stride_h;
  L.beta = static_cast<const float*>(a->beta.ptr); L.b_sb = a->beta.stride_b; L.b_sh = a->beta.stride_h;
  L.q_scale = a->q_scale;
  L.S_in = a->S_in; L.S_out = a->S_out;
  L.delta = delta;
  if (!L.in_bf16) return from_cuda(la::launch_gdn_prefill_recurrent(L, s));
  unsigned* status = device_status_ptr();
  if (!status) return LA_ERR_CUDA;
  const cudaError_t e = split ? la::launch_gdn_prefill_scan(L, ws, ws_bytes, status, s)
                              : la::launch_gdn_prefill_chunked(L, ws, ws_bytes, status, s);
  if (e == cudaErrorInvalidValue) return LA_ERR_UNSUPPORTED;  // strides TMA cannot describe
  return from_cuda(e);
}

}  // namespace

extern "C" {

int la_abi_version(void) { return LA_ABI_VERSION; }

int la_last_cuda_error(void) { return la::last_cuda_error(); }

const char* la_cuda_error_name(int code) {
  const char* n = cudaGetErrorName(static_cast<cudaError_t>(code));
  return n ? n : "unknown CUDA error";
}

const char* la_status_string(la_status s) {
  switch (s) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID_ARGUMENT: return "invalid argument (null pointer, size, stride or alignment)";
    case LA_ERR_UNSUPPORTED: return "unsupported shape or dtype for the built kernels";
    case LA_ERR_WORKSPACE: return "workspace missing or too small";
    case LA_ERR_CUDA: return "CUDA call failed";
    case LA_ERR_TIMEOUT: return "a bounded device-side wait expired";
  }
  return "unknown status";
}

// The workspace queries depend on the problem's sizes and dtypes only (no
// pointer is inspected), so they may be asked before any buffer exists.
size_t la_based_prefill_workspace_size(const la_based_prefill_args* a) {
  (void)a;
  return 0;
}

// bf16 GDN problems the chunked kernels take (the fp32 path needs no scratch)
static bool gdn_chunked_shape(const la_gdn_prefill_args* a) {
  if (!a || a->B <= 0 || a->H <= 0 || a->N <= 0 || a->B > kMaxDim || a->H > kMaxDim || a->N > kMaxDim) return false;
  return a->d_k == kGdnD && a->d_v == kGdnD && a->in_dtype == LA_DTYPE_BF16;
}

size_t la_gdn_prefill_workspace_size(const la_gdn_prefill_args* a) {
  return gdn_chunked_shape(a) ? la::gdn_scan_workspace_bytes(a->B, a->H, a->N) : 0;
}

size_t la_gdn_prefill_workspace_size_min(const la_gdn_prefill_args* a) {
  return gdn_chunked_shape(a) ? la::gdn_segment_plan(a->B, a->H, a->N).ws_bytes : 0;
}

la_status la_based_prefill(const la_based_prefill_args* a, void* ws, size_t ws_bytes, void* stream) {
  const la_status st = check_based(a);
  if (st != LA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t BH = a->B * a->H;
  if (BH == 0) return LA_OK;
  if (a->N == 0) {
    la_status r = pass_state(a->s_out, a->s_in, (size_t)(BH * kTaylorD * kTaylorDv), s);
    if (r != LA_OK) return r;
    return pass_state(a->z_out, a->z_in, (size_t)(BH * kTaylorD), s);
  }
  (void)ws;
  (void)ws_bytes;
  la::TaylorPrefillLaunch L{};
  L.B = a->B; L.H = a->H; L.N = a->N;
  L.in_bf16 = a->in_dtype == LA_DTYPE_BF16;
  L.out_bf16 = a->out_dtype == LA_DTYPE_BF16;
  L.q = view(a->q); L.k = view(a->k); L.v = view(a->v);
  L.y = a->y.ptr; L.y_sb = a->y.stride_b; L.y_sh = a->y.stride_h; L.y_st = a->y.stride_t;
  L.s_in = a->s_in; L.z_in = a->z_in; L.s_out = a->s_out; L.z_out = a->z_out;
  L.eps = a->eps;
  L.decay = a->decay;
  if (!L.in_bf16) return from_cuda(la::launch_taylor_prefill_recurrent(L, s));
  unsigned* status = device_status_ptr();
  if (!status) return LA_ERR_CUDA;
  const cudaError_t e = la::launch_taylor_prefill_chunked(L, status, s);
  if (e == cudaErrorInvalidValue) return LA_ERR_UNSUPPORTED;  // strides TMA cannot describe
  return from_cuda(e);
}


la_status la_gdn_prefill(const la_gdn_prefill_args* a, void* ws, size_t ws_bytes, void* stream) {
  return gdn_family_prefill(a, ws, ws_bytes, stream, 1.f);
}

la_status la_gated_prefill(const la_gdn_prefill_args* a, void* ws, size_t ws_bytes, void* stream) {
  return gdn_family_prefill(a, ws, ws_bytes, stream, 0.f);
}

la_status la_decode_step(const la_decode_args* a, void* stream) {
  if (!a) return LA_ERR_INVALID_ARGUMENT;
  if (a->S < 0 || a->H < 0 || a->S > kMaxDim || a->H > kMaxDim) return LA_ERR_INVALID_ARGUMENT;
  if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return LA_ERR_INVALID_ARGUMENT;
  if (a->variant != LA_VARIANT_TAYLOR && a->variant != LA_VARIANT_GDN && a->variant != LA_VARIANT_GATED)
    return LA_ERR_INVALID_ARGUMENT;
  const bool gdn_family = a->variant != LA_VARIANT_TAYLOR;
  if (gdn_family && (a->d_k != kGdnD || a->d_v != kGdnD)) return LA_ERR_UNSUPPORTED;
  if (a->variant == LA_VARIANT_TAYLOR && (a->d_k != kTaylorF || a->d_v != kTaylorDv)) return LA_ERR_UNSUPPORTED;
  const int64_t SH = a->S * a->H;
  if (SH == 0) return LA_OK;
  if (SH > (int64_t(1) << 31) - 1) return LA_ERR_UNSUPPORTED;
  if (!a->q || !a->k || !a->v || !a->out || !a->state) return LA_ERR_INVALID_ARGUMENT;
  const int in_align = a->in_dtype == LA_DTYPE_BF16 ? 8 : 16;
  if ((reinterpret_cast<uintptr_t>(a->q) % in_align) || (reinterpret_cast<uintptr_t>(a->k) % in_align) ||
      (reinterpret_cast<uintptr_t>(a->v) % in_align) || !aligned16(a->state))
    return LA_ERR_INVALID_ARGUMENT;
  if (gdn_family && (!a->alpha || !a->beta)) return LA_ERR_INVALID_ARGUMENT;
  if (a->variant == LA_VARIANT_TAYLOR &&
      (!a->z || (reinterpret_cast<uintptr_t>(a->z) & 3u) || (reinterpret_cast<uintptr_t>(a->decay) & 3u)))
    return LA_ERR_INVALID_ARGUMENT;
  la::DecodeLaunch L{};
  L.S = a->S; L.H = a->H;
  L.in_bf16 = a->in_dtype == LA_DTYPE_BF16;
  L.out_bf16 = a->out_dtype == LA_DTYPE_BF16;
  L.q = a->q; L.k = a->k; L.v = a->v; L.alpha = a->alpha; L.beta = a->beta;
  L.out = a->out; L.state = a->state; L.z = a->z; L.eps = a->eps; L.q_scale = a->q_scale;
  L.delta = a->variant == LA_VARIANT_GDN ? 1.f : 0.f;
  L.decay = a->variant == LA_VARIANT_TAYLOR ? a->decay : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return from_cuda(gdn_family ? la::launch_gdn_decode(L, s) : la::launch_taylor_decode(L, s));
}

la_status la_state_rescale(float* states, int64_t n_states, int64_t elems_per_state, const float* lambda,
                           float lambda_all, void* stream) {
  if (n_states < 0 || elems_per_state < 0 || n_states > kMaxDim || elems_per_state > kMaxDim ||
      (elems_per_state > 0 && n_states > kMaxElems / elems_per_state))
    return LA_ERR_INVALID_ARGUMENT;
  if (n_states == 0 || elems_per_state == 0) return LA_OK;
  if (!states || (reinterpret_cast<uintptr_t>(states) & 3u)) return LA_ERR_INVALID_ARGUMENT;
  if (lambda && (reinterpret_cast<uintptr_t>(lambda) & 3u)) return LA_ERR_INVALID_ARGUMENT;
  return from_cuda(la::launch_state_rescale(states, n_states, elems_per_state, lambda, lambda_all,
                                            static_cast<cudaStream_t>(stream)));
}

la_status la_state_gather(float* dst, const float* src, const int64_t* index, int64_t n_dst, int64_t n_src,
                          int64_t elems_per_state, void* stream) {
  if (n_dst < 0 || n_src < 0 || elems_per_state < 0 || n_dst > kMaxDim || n_src > kMaxDim ||
      elems_per_state > kMaxDim ||
      (elems_per_state > 0 && (n_dst > kMaxElems / elems_per_state || n_src > kMaxElems / elems_per_state)))
    return LA_ERR_INVALID_ARGUMENT;
  if (n_dst == 0 || elems_per_state == 0) return LA_OK;
  if (!dst || !src || !index) return LA_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(dst) & 3u) || (reinterpret_cast<uintptr_t>(src) & 3u) ||
      (reinterpret_cast<uintptr_t>(index) & 7u))
    return LA_ERR_INVALID_ARGUMENT;
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst), d1 = d0 + (uintptr_t)(n_dst * elems_per_state) * 4u;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), s1 = s0 + (uintptr_t)(n_src * elems_per_state) * 4u;
  if (d0 < s1 && s0 < d1) return LA_ERR_INVALID_ARGUMENT;  // overlapping arrays
  unsigned* status = device_status_ptr();
  if (!status) return LA_ERR_CUDA;
  return from_cuda(la::launch_state_gather(dst, src, index, n_dst, n_src, elems_per_state, status,
                                           static_cast<cudaStream_t>(stream)));
}

la_status la_swa_decode_step(const la_swa_decode_args* a, void* stream) {
  if (!a) return LA_ERR_INVALID_ARGUMENT;
  if (a->S < 0 || a->H < 0 || a->S > kMaxDim || a->H > kMaxDim) return LA_ERR_INVALID_ARGUMENT;
  if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return LA_ERR_INVALID_ARGUMENT;
  if (a->d < 8 || a->d > 128 || a->d % 8 != 0 || a->window < 1 || a->window > 256) return LA_ERR_UNSUPPORTED;
  const int64_t SH = a->S * a->H;
  if (SH == 0) return LA_OK;
  if (SH > (int64_t(1) << 31) - 1) return LA_ERR_UNSUPPORTED;
  if (!a->q || !a->k || !a->v || !a->k_cache || !a->v_cache || !a->pos || !a->out) return LA_ERR_INVALID_ARGUMENT;
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->k_cache) ||
      !aligned16(a->v_cache) || !aligned16(a->out) || (reinterpret_cast<uintptr_t>(a->pos) & 7u))
    return LA_ERR_INVALID_ARGUMENT;
  unsigned* status = device_status_ptr();
  if (!status) return LA_ERR_CUDA;
  la::SwaDecodeLaunch L{};
  L.S = a->S; L.H = a->H; L.d = (int)a->d; L.window = (int)a->window;
  L.in_bf16 = a->in_dtype == LA_DTYPE_BF16;
  L.out_bf16 = a->out_dtype == LA_DTYPE_BF16;
  L.q = a->q; L.k = a->k; L.v = a->v; L.k_cache = a->k_cache; L.v_cache = a->v_cache;
  L.pos = a->pos; L.out = a->out; L.scale = a->scale; L.status = status;
  return from_cuda(la::launch_swa_decode(L, static_cast<cudaStream_t>(stream)));
}

la_status la_notebank_scores(const la_notebank_scores_args* a, void* stream) {
  if (!a) return LA_ERR_INVALID_ARGUMENT;
  if (a->L < 0 || a->H < 0 || a->N < 0 || a->L > kMaxDim || a->H > kMaxDim || a->N > kMaxDim)
    return LA_ERR_INVALID_ARGUMENT;
  if (!valid_dtype(a->in_dtype)) return LA_ERR_INVALID_ARGUMENT;
  if (a->d < 32 || a->d > 256 || a->d % 32 != 0) return LA_ERR_UNSUPPORTED;
  if (a->chunk < 1 || a->chunk > 1024 || a->window < 1 || a->window > 4096) return LA_ERR_INVALID_ARGUMENT;
  const int64_t J = a->L * a->H;
  if (J == 0 || a->N == 0) return LA_OK;
  if (J * ((a->N + a->chunk - 1) / a->chunk) > (int64_t(1) << 31) - 1) return LA_ERR_UNSUPPORTED;
  if (!valid_view(a->k, a->L, a->H, a->N, a->d, a->in_dtype)) return LA_ERR_INVALID_ARGUMENT;
  if (!a->d_ch || !a->d_mean || (reinterpret_cast<uintptr_t>(a->d_ch) & 3u) ||
      (reinterpret_cast<uintptr_t>(a->d_mean) & 3u) || (reinterpret_cast<uintptr_t>(a->w) & 3u))
    return LA_ERR_INVALID_ARGUMENT;
  la::NotebankScoresLaunch L{};
  L.L = a->L; L.H = a->H; L.N = a->N; L.d = a->d;
  L.in_bf16 = a->in_dtype == LA_DTYPE_BF16;
  L.k = view(a->k);
  L.chunk = a->chunk; L.window = a->window;
  L.d_ch = a->d_ch; L.d_mean = a->d_mean; L.w = a->N >= a->window ? a->w : nullptr;
  return from_cuda(la::launch_notebank_scores(L, static_cast<cudaStream_t>(stream)));
}

la_status la_notebank_address(const la_notebank_address_args* a, void* stream) {
  if (!a) return LA_ERR_INVALID_ARGUMENT;
  if (a->L < 0 || a->H < 0 || a->N < 0 || a->n_notes < 0 || a->L > kMaxDim || a->H > kMaxDim || a->N > kMaxDim ||
      a->n_notes > kMaxDim)
    return LA_ERR_INVALID_ARGUMENT;
  if (!valid_dtype(a->in_dtype)) return LA_ERR_INVALID_ARGUMENT;
  if (a->d < la::kNoteAddrDims || a->d > kMaxDim) return LA_ERR_UNSUPPORTED;
  const int64_t warps = a->n_notes * a->L * a->H;
  if (warps == 0) return LA_OK;
  if (warps > (int64_t(1) << 33)) return LA_ERR_UNSUPPORTED;  // grid of warps * 32 / 256 blocks
  if (a->N == 0) return LA_ERR_INVALID_ARGUMENT;  // no token to point at
  if (!valid_view(a->q, a->L, a->H, a->N, a->d, a->in_dtype)) return LA_ERR_INVALID_ARGUMENT;
  if (!a->d_ch || !a->coords || !a->spans || !a->t_star || !a->rho || (reinterpret_cast<uintptr_t>(a->d_ch) & 3u) ||
      (reinterpret_cast<uintptr_t>(a->coords) & 3u) || (reinterpret_cast<uintptr_t>(a->spans) & 7u) ||
      (reinterpret_cast<uintptr_t>(a->t_star) & 3u) || (reinterpret_cast<uintptr_t>(a->rho) & 1u))
    return LA_ERR_INVALID_ARGUMENT;
  unsigned* status = device_status_ptr();
  if (!status) return LA_ERR_CUDA;
  la::NotebankAddressLaunch L{};
  L.L = a->L; L.H = a->H; L.N = a->N; L.d = a->d; L.n_notes = a->n_notes;
  L.in_bf16 = a->in_dtype == LA_DTYPE_BF16;
  L.q = view(a->q);
  L.d_ch = a->d_ch; L.coords = a->coords; L.spans = a->spans; L.t_star = a->t_star; L.rho = a->rho;
  return from_cuda(la::launch_notebank_address(L, status, static_cast<cudaStream_t>(stream)));
}

la_status la_notebank_route(const la_notebank_route_args* a, void* stream) {
  if (!a) return LA_ERR_INVALID_ARGUMENT;
  if (a->n_notes < 0 || a->J < 0 || a->n_notes > (int64_t(1) << 31) - 2 || a->J > kMaxDim)
    return LA_ERR_INVALID_ARGUMENT;
  if (a->n_q < 1 || a->n_q > 512 || a->R < 1 || a->R > 64) return LA_ERR_UNSUPPORTED;
  if (a->J == 0) return LA_OK;
  if (!a->u || !a->winner || !a->top || !aligned16(a->u) || (reinterpret_cast<uintptr_t>(a->winner) & 3u) ||
      (reinterpret_cast<uintptr_t>(a->top) & 3u))
    return LA_ERR_INVALID_ARGUMENT;
  if (a->n_notes > 0 && (!a->rho || !a->votes || !aligned16(a->rho) || (reinterpret_cast<uintptr_t>(a->votes) & 3u) ||
                         (reinterpret_cast<uintptr_t>(a->s) & 3u) || (reinterpret_cast<uintptr_t>(a->positions) & 7u)))
    return LA_ERR_INVALID_ARGUMENT;
  la::NotebankRouteLaunch L{};
  L.n_notes = a->n_notes; L.J = a->J; L.n_q = a->n_q; L.R = a->R;
  L.rho = a->rho; L.u = a->u; L.positions = a->positions; L.s = a->s;
  L.winner = a->winner; L.votes = a->votes; L.top = a->top;
  return from_cuda(la::launch_notebank_route(L, static_cast<cudaStream_t>(stream)));
}

la_status la_selftest_bounded_wait(int arrive, int64_t limit_ns, void* stream) {
  if (limit_ns < 1000000 || limit_ns > 2000000000) return LA_ERR_INVALID_ARGUMENT;
  unsigned* status = device_status_ptr();
  if (!status) return LA_ERR_CUDA;
  return from_cuda(la::launch_bounded_wait_selftest(arrive, (uint64_t)limit_ns, status, static_cast<cudaStream_t>(stream)));
}

la_status la_device_status(void* stream, int clear) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_la_device_status, sizeof v) != cudaSuccess) return LA_ERR_CUDA;
  if (clear && v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_la_device_status, &zero, sizeof zero) != cudaSuccess) return LA_ERR_CUDA;
  }
  if (v & la::kStatusTimeout) return LA_ERR_TIMEOUT;
  return v ? LA_ERR_INVALID_ARGUMENT : LA_OK;  // kStatusBadIndex
}

}  // extern "C"
