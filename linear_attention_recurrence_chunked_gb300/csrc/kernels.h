// kernels.h -- internal launch descriptors shared by the C ABI layer and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace la {

// Bits of the device status word (read back by la_device_status).
constexpr unsigned kStatusTimeout = 1u;   // a bounded wait expired
constexpr unsigned kStatusBadIndex = 2u;  // a state index outside its array was skipped

// The cudaError_t behind the latest LA_ERR_CUDA returned to the calling
// thread (api.cu); noted by every path that maps a CUDA failure to it.
void note_cuda_error(int code);
int last_cuda_error();

struct View4 {        // strided [B, H, N, d] view, element strides
  const void* ptr;
  int64_t sb, sh, st;
};

struct DecodeLaunch {
  int64_t S, H;
  bool in_bf16, out_bf16;
  const void *q, *k, *v;
  const float *alpha, *beta;
  void* out;
  float* state;
  float* z;
  float eps, q_scale;
  float delta;  // GDN-family decode: 1 = gated delta rule, 0 = scalar gate (A_t = alpha_t I)
  const float* decay;  // Taylor decode: per-head retention [H] or null
};

struct TaylorPrefillLaunch {
  int64_t B, H, N;
  bool in_bf16, out_bf16;
  View4 q, k, v;
  void* y;
  int64_t y_sb, y_sh, y_st;
  const float* s_in;
  const float* z_in;
  float* s_out;
  float* z_out;
  float eps;
  const float* decay;  // per-head retention [H] or null (no decay)
};

struct GdnPrefillLaunch {
  int64_t B, H, N;
  bool in_bf16, out_bf16;
  View4 q, k, v;
  void* o;
  int64_t o_sb, o_sh, o_st;
  const float* alpha;
  int64_t a_sb, a_sh;
  const float* beta;
  int64_t b_sb, b_sh;
  float q_scale;
  const float* S_in;
  float* S_out;
  float delta;  // 1 = gated delta rule, A_t = alpha_t (I - beta_t k_t k_t^T); 0 = scalar gate, A_t = alpha_t I
};

// Sequence-segment plan of the gated-delta-rule prefill (see gdn_chunked.cu):
// G segments of seg_len tokens per (b,h); G == 1 runs the plain chunk scan.
struct GdnSegPlan {
  int G;
  int64_t seg_len;
  size_t ws_bytes;  // workspace: segment maps then segment entry states
};
GdnSegPlan gdn_segment_plan(int64_t B, int64_t H, int64_t N);

cudaError_t launch_gdn_decode(const DecodeLaunch& a, cudaStream_t stream);
cudaError_t launch_taylor_decode(const DecodeLaunch& a, cudaStream_t stream);
// fp32 inputs: token-serial CUDA-core kernels (fp32 arithmetic throughout).
cudaError_t launch_taylor_prefill_recurrent(const TaylorPrefillLaunch& a, cudaStream_t stream);
cudaError_t launch_gdn_prefill_recurrent(const GdnPrefillLaunch& a, cudaStream_t stream);
// bf16 inputs: chunked tcgen05 kernels.  The single-kernel scan needs the
// segment scratch of gdn_segment_plan only; the two-kernel scan (per-chunk
// inverse records, then the warp-specialized state scan) needs
// gdn_scan_workspace_bytes.
cudaError_t launch_gdn_prefill_chunked(const GdnPrefillLaunch& a, void* ws, size_t ws_bytes, unsigned* dev_status,
                                       cudaStream_t stream);
size_t gdn_scan_workspace_bytes(int64_t B, int64_t H, int64_t N);
cudaError_t launch_gdn_prefill_scan(const GdnPrefillLaunch& a, void* ws, size_t ws_bytes, unsigned* dev_status,
                                    cudaStream_t stream);
cudaError_t launch_taylor_prefill_chunked(const TaylorPrefillLaunch& a, unsigned* dev_status, cudaStream_t stream);
struct SwaDecodeLaunch {
  int64_t S, H;
  int d, window;
  bool in_bf16, out_bf16;
  const void *q, *k, *v;
  void *k_cache, *v_cache;
  const int64_t* pos;
  void* out;
  float scale;
  unsigned* status;  // device status word (a negative position sets kStatusBadIndex)
};
cudaError_t launch_swa_decode(const SwaDecodeLaunch& a, cudaStream_t stream);

// State operations between calls (state_ops.cu).  per = fp32 elements per state.
cudaError_t launch_state_rescale(float* states, int64_t n_states, int64_t per, const float* lambda, float lambda_all,
                                 cudaStream_t stream);
cudaError_t launch_state_gather(float* dst, const float* src, const int64_t* index, int64_t n_dst, int64_t n_src,
                                int64_t per, unsigned* dev_status, cudaStream_t stream);
cudaError_t launch_bounded_wait_selftest(int arrive, uint64_t limit_ns, unsigned* dev_status, cudaStream_t stream);

// NoteBank write side and routing (notebank.cu).
constexpr int kNoteAddrDims = 16;  // d_rho: query coordinates stored per channel and note
struct NotebankScoresLaunch {
  int64_t L, H, N, d;   // channels = L x H; key width d (multiple of 32, <= 256)
  bool in_bf16;
  View4 k;              // [L, H, N, d]
  int64_t chunk, window;
  float* d_ch;          // [L, H, N]
  float* d_mean;        // [N]
  float* w;             // [N - window + 1] or null
};
struct NotebankAddressLaunch {
  int64_t L, H, N, d, n_notes;
  bool in_bf16;
  View4 q;                // [L, H, N, d]
  const float* d_ch;      // [L, H, N]
  const int32_t* coords;  // [L, H, 16]
  const int64_t* spans;   // [n_notes, 2]: start, length
  int32_t* t_star;        // [n_notes, L, H]
  void* rho;              // [n_notes, L, H, 16] bf16
};
struct NotebankRouteLaunch {
  int64_t n_notes, J, n_q, R;
  const void* rho;           // [n_notes, J, 16] bf16
  const void* u;             // [J, n_q, 16] bf16
  const int64_t* positions;  // [n_notes] or null
  float* s;                  // [n_notes, J] or null
  int32_t* winner;           // [J]
  int32_t* votes;            // [n_notes]
  int32_t* top;              // [R]
};
cudaError_t launch_notebank_scores(const NotebankScoresLaunch& a, cudaStream_t stream);
cudaError_t launch_notebank_address(const NotebankAddressLaunch& a, unsigned* status, cudaStream_t stream);
cudaError_t launch_notebank_route(const NotebankRouteLaunch& a, cudaStream_t stream);

}  // namespace la
