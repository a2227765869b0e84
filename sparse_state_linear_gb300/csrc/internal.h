// internal.h -- host-side launchers shared between the translation units of
// the SDM library (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sdm.h"

namespace sdm {

// Resolved per-call parameters (validated by the API layer).
struct Dims {
  int B, H, T, s, dh, dv, W, R, kw, kr;
  int Ts;        // rows between chains in the [B, H, T, ...] layouts: T, or the
                 // full length when a call covers a window of steps
  int in_dtype;  // SDM_F32 / SDM_BF16
  int score;     // SDM_SCORE_DOT / SDM_SCORE_IDW
  float eps;
  int update;    // SDM_UPDATE_*
#ifdef __CUDACC__
  __host__ __device__
#endif
  long long N() const { return (long long)s * s; }
};

enum AddrMode { kAddrFused = 0, kAddrSelectOnly = 1, kAddrScoresOnly = 2 };

// Addressing kernels (address.cu).
//  kAddrFused:      q0 = q_w, q1 = q_r -> idx/wt of both branches.
//  kAddrSelectOnly: f0 = sub_w, f1 = sub_r (float32 sub-scores) -> idx/wt.
//  kAddrScoresOnly: q0 = the branch's half-queries -> S (float32).
// Whether the fused addressing of this shape runs on the tensor cores.
bool address_on_tensor_cores(const Dims& d);
cudaError_t launch_address(int mode, const Dims& d, const void* q0, const void* q1,
                           const void* K, const float* f0, const float* f1,
                           int32_t* idx_w, float* wt_w, int32_t* idx_r, float* wt_r,
                           float* S, unsigned* status, cudaStream_t stream);

// Plan codes per token: W + R rounded up to 8 (16-byte rows).
#ifdef __CUDACC__
__host__ __device__
#endif
inline int code_pitch(int W, int R) { return (W + R + 7) & ~7; }

// Hazard plan (plan.cu): per-row source codes of a segment into `codes`
// ([B*H*T, code_pitch(W, R)] int16) for a scan of ring depth `depth`.
cudaError_t launch_plan(const Dims& d, const int32_t* idx_w, const int32_t* idx_r,
                        int16_t* codes, int depth, unsigned* status, cudaStream_t stream);

// Scan (scan.cu): the plan kernel (writes per-row source codes into
// `workspace`) then the scan kernel.
size_t scan_workspace_bytes(const Dims& d);
// `undo` (may be null): log of each step's pre-write rows [B,H,T,W,d_v].
cudaError_t launch_scan(const Dims& d, const int32_t* idx_w, const float* wt_w,
                        const int32_t* idx_r, const float* wt_r, const void* alpha,
                        const void* beta, const void* v, float* M, float* y, float* undo,
                        void* workspace, int depth, int col_slice, unsigned* status,
                        cudaStream_t stream);
// The same in parts, for callers that run the plan on another stream (the
// overlapped forward): scan_setup picks the column slice and ring depth (it
// does not depend on T), launch_plan writes the codes for that depth, and
// launch_scan_kernel runs the scan kernel on them.
struct ScanSetup {
  int cw, depth;
  bool one_per_sm;   // every unit has an SM of its own (the MINB = 1 build)
  bool pair;         // exactly two units per SM: one CTA runs both
};
cudaError_t scan_setup(const Dims& d, int depth, int col_slice, bool logged, ScanSetup* out);
cudaError_t launch_scan_kernel(const Dims& d, const ScanSetup& c, const int32_t* idx_w,
                               const float* wt_w, const int32_t* idx_r, const float* wt_r,
                               const void* alpha, const void* beta, const void* v, float* M,
                               float* y, float* undo, const int16_t* codes, unsigned* status,
                               cudaStream_t stream);

// Undo of a logged segment (undo.cu): `workspace` holds B*H*N marks.
size_t undo_workspace_bytes(const Dims& d);
cudaError_t launch_undo(const Dims& d, const int32_t* idx_w, const float* undo, float* M,
                        void* workspace, unsigned* status, cudaStream_t stream);

// Per-head RMS-Norm and output gate on y (epilogue.cu).  g has d.in_dtype;
// out_dtype is SDM_F32 or SDM_BF16; gamma may be null.
cudaError_t launch_rmsnorm_gate(const Dims& d, const float* y, const void* g, const float* gamma,
                                float eps, void* out, int out_dtype, cudaStream_t stream);

// Fused decode (decode.cu): one CTA per (b,h) chain runs its T steps --
// addressing, write, read and, when out is non-null, the epilogue.
// sdm_api.cu: the overlapped forward (addressing of window k+1 beside the
// scan of window k).  forward_window_steps gives the window length (T = no
// windows), forward_segments the number of windows; run_segmented_forward
// returns a cudaError_t, or -1 if its streams could not be set up (nothing
// enqueued).
struct SegmentedForward {
  Dims d;
  const char* q_w;
  const char* q_r;
  const void* K;
  const char* alpha;
  const char* beta;
  const char* v;
  float* M;
  float* y;
  int32_t* idx_w;
  float* wt_w;
  int32_t* idx_r;
  float* wt_r;
  int16_t* codes;
  int in_bytes, depth, col_slice;
  unsigned* status;
};
int forward_window_steps(const Dims& d);
int forward_segments(const Dims& d);
int run_segmented_forward(const SegmentedForward& f, int window, cudaStream_t caller);

// rowtraffic.cu: random row pieces in the scan's unit layout, no arithmetic.
cudaError_t launch_row_traffic(const float* src, float* dst, long long chains, long long rows,
                               int dv, int col_slice, int T, int loads, int stores,
                               uint32_t seed, cudaStream_t stream);

cudaError_t launch_decode(const Dims& d, const void* q_w, const void* q_r, const void* K,
                          const void* alpha, const void* beta, const void* v, float* M, float* y,
                          int32_t* idx_w, float* wt_w, int32_t* idx_r, float* wt_r,
                          const void* g, const float* gamma, float eps, void* out,
                          int out_dtype, cudaStream_t stream);

// Limits of the current device, queried once per device (sdm_api.cu): SM
// count, shared memory per SM, and the opt-in maximum per CTA.
struct DeviceLimits {
  int sms;
  size_t smem_per_sm;
  size_t smem_per_cta;
};
DeviceLimits device_limits();

// Accessors of the API layer (sdm_api.cu) for other entry points.
sdm_status api_check_shape(const sdm_shape* shape, Dims* d);
sdm_status api_status_ptr(unsigned** out);
void api_scan_tuning(int* depth, int* col_slice);

}  // namespace sdm
