// sdm_api.cu -- the C ABI declared in include/sdm.h: argument checks, the
// per-device status word, and kernel dispatch.  No device memory is
// allocated here; every tensor belongs to the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sdm.h"

namespace sdm {
namespace {

// The status word of each device that loads this library (see sdm.h).
__device__ unsigned g_status = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_status_ptr[kMaxDevices] = {};
int g_depth = 0, g_colslice = 0;

sdm_status status_ptr(unsigned** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return SDM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return SDM_ERR_CUDA;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_status_ptr[dev];
  return SDM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sdm_status check_shape(const sdm_shape* sh, Dims* d) {
  if (!sh) return SDM_ERR_INVALID_ARG;
  if (sh->B < 0 || sh->H < 0 || sh->T < 0) return SDM_ERR_INVALID_ARG;
  if (sh->n_sub < 1 || sh->d_h < 1 || sh->d_v < 1 || sh->W < 1 || sh->R < 1)
    return SDM_ERR_INVALID_ARG;
  if (sh->k_w < 0 || sh->k_r < 0) return SDM_ERR_INVALID_ARG;
  if (sh->in_dtype != SDM_F32 && sh->in_dtype != SDM_BF16) return SDM_ERR_INVALID_ARG;
  if (sh->score != SDM_SCORE_DOT && sh->score != SDM_SCORE_IDW) return SDM_ERR_INVALID_ARG;
  if (sh->update != SDM_UPDATE_EQ4 && sh->update != SDM_UPDATE_SHARED_RESIDUAL)
    return SDM_ERR_INVALID_ARG;
  if (sh->score == SDM_SCORE_IDW && !(sh->idw_eps > 0.f)) return SDM_ERR_INVALID_ARG;
  const int s = sh->n_sub;
  const int kw = sh->k_w ? sh->k_w : (sh->W < s ? sh->W : s);
  const int kr = sh->k_r ? sh->k_r : (sh->R < s ? sh->R : s);
  if (kw > s || kr > s) return SDM_ERR_INVALID_ARG;
  if ((long long)kw * kw < sh->W || (long long)kr * kr < sh->R) return SDM_ERR_INVALID_ARG;
  // Supported envelope.
  if (s > 512) return SDM_ERR_UNSUPPORTED;
  if (sh->d_h != 16 && sh->d_h != 32 && sh->d_h != 64 && sh->d_h != 128 && sh->d_h != 256)
    return SDM_ERR_UNSUPPORTED;
  if (sh->d_v % 16 != 0 || sh->d_v > 2048) return SDM_ERR_UNSUPPORTED;
  if (sh->W > 64 || sh->R > 64 || kw > 64 || kr > 64) return SDM_ERR_UNSUPPORTED;
  const long long N = (long long)s * s;
  if ((long long)sh->B * sh->H * N * sh->d_v >= (1ll << 40)) return SDM_ERR_UNSUPPORTED;
  if ((long long)sh->B * sh->H * sh->T >= (1ll << 31)) return SDM_ERR_UNSUPPORTED;
  if ((long long)sh->B * sh->T >= (1ll << 31) / 16) return SDM_ERR_UNSUPPORTED;
  d->B = sh->B;
  d->H = sh->H;
  d->T = sh->T;
  d->Ts = sh->T;
  d->s = s;
  d->dh = sh->d_h;
  d->dv = sh->d_v;
  d->W = sh->W;
  d->R = sh->R;
  d->kw = kw;
  d->kr = kr;
  d->in_dtype = sh->in_dtype;
  d->score = sh->score;
  d->eps = sh->idw_eps;
  d->update = sh->update;
  return SDM_OK;
}

bool empty_work(const Dims& d) { return (long long)d.B * d.H * d.T == 0; }

sdm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SDM_OK : SDM_ERR_CUDA; }

#define SDM_CHECK_PTR(p) \
  do {                   \
    if (!(p) || !aligned16(p)) return SDM_ERR_INVALID_ARG; \
  } while (0)

__global__ void wait_timeout_selftest(unsigned* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) mbar_init(&bar, 1);
  __syncthreads();
  // Nothing arrives on `bar`: the bounded wait must give up and report.
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, timeout_ns))
    record_status(status, SDM_ERR_TIMEOUT);
}

}  // namespace

DeviceLimits device_limits() {
  static std::mutex mu;
  static DeviceLimits cache[64];
  static bool known[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!known[dev]) {
    int sms = 0, per_sm = 0, per_cta = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&per_cta, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cache[dev] = DeviceLimits{sms > 0 ? sms : 1, (size_t)(per_sm > 0 ? per_sm : 0),
                              (size_t)(per_cta > 0 ? per_cta : 0)};
    known[dev] = true;
  }
  return cache[dev];
}

// ----------------------------------------------------------- forward overlap
// sdm_forward cuts T into S windows of steps.  The addressing of window k+1
// (which reads only q and K) runs on a low-priority stream while the scan of
// window k (which carries M from window to window) runs on a high-priority
// one, so the addressing fills what the scan leaves of the GPU and the scan
// gets SMs first whenever they free up.  Each window's scan waits for its
// addressing; both streams are joined back into the caller's stream, so the
// call keeps one-stream semantics (and can be captured in a graph).  Results
// are bit-identical to sdm_address followed by sdm_scan: addressing is per
// token, and a scan of consecutive windows equals one scan.

// Windows: the tensor-core addressing of a window fits beside the scan in the
// SMs it leaves free, so short windows (512 steps, at most 32 of them) hide
// most of it; the FFMA addressing is too heavy to hide there, and only the
// scan's per-window ramps are worth overlapping (4 windows).
// Window length: T / windows rounded up to whole 64-step blocks (the
// addressing CTAs take 64 tokens of a chain, the plan kernel 64 steps), so no
// window leaves a partial block behind except the last.
int forward_window_steps(const Dims& d) {
  if (d.T < 2048) return d.T;
  int s = address_on_tensor_cores(d) ? d.T / 512 : 4;
  if (s > 32) s = 32;
  const int len = (d.T + s - 1) / s;
  return (len + 63) & ~63;
}

int forward_segments(const Dims& d) {
  const int len = forward_window_steps(d);
  return len <= 0 ? 1 : (d.T + len - 1) / len;
}

namespace {
struct ForwardStreams {
  bool ready = false;
  cudaStream_t hi = nullptr, lo = nullptr;
  cudaEvent_t start = nullptr, addr = nullptr, hi_end = nullptr, lo_end = nullptr;
};
std::mutex g_fwd_mu[64];
ForwardStreams g_fwd[64];
}  // namespace

int run_segmented_forward(const SegmentedForward& f, int window, cudaStream_t caller) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  // Enqueueing holds the device's lock: the side streams and events are shared.
  std::lock_guard<std::mutex> lk(g_fwd_mu[dev]);
  ForwardStreams& fs = g_fwd[dev];
  if (!fs.ready) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return -1;
    if (cudaStreamCreateWithPriority(&fs.hi, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&fs.lo, cudaStreamNonBlocking, least) != cudaSuccess ||
        cudaEventCreateWithFlags(&fs.start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&fs.addr, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&fs.hi_end, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&fs.lo_end, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    fs.ready = true;
  }
  const Dims& d = f.d;
  cudaError_t e = cudaEventRecord(fs.start, caller);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(fs.hi, fs.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(fs.lo, fs.start, 0);
  if (e != cudaSuccess) return (int)e;
  const int tseg = window;
  const size_t qrow = (size_t)2 * d.dh * f.in_bytes;       // bytes per token of q
  const size_t CP = (size_t)code_pitch(d.W, d.R);
  ScanSetup sc;
  e = scan_setup(d, f.depth, f.col_slice, false, &sc);
  // Window k's addressing on the low-priority stream; its hazard plan and
  // scan on the high-priority one (a plan queued behind the addressing
  // started late and held the scan back: slower on every workload).
  for (int t0 = 0; t0 < d.T && e == cudaSuccess; t0 += tseg) {
    Dims w = d;
    w.T = d.T - t0 < tseg ? d.T - t0 : tseg;
    w.Ts = d.T;
    int32_t* iw = f.idx_w + (size_t)t0 * d.W;
    int32_t* ir = f.idx_r + (size_t)t0 * d.R;
    float* ww = f.wt_w + (size_t)t0 * d.W;
    float* wr = f.wt_r + (size_t)t0 * d.R;
    int16_t* codes = f.codes + (size_t)t0 * CP;
    e = launch_address(kAddrFused, w, f.q_w + t0 * qrow, f.q_r + t0 * qrow, f.K, nullptr,
                       nullptr, iw, ww, ir, wr, nullptr, f.status, fs.lo);
    if (e == cudaSuccess) e = cudaEventRecord(fs.addr, fs.lo);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(fs.hi, fs.addr, 0);
    if (e == cudaSuccess) e = launch_plan(w, iw, ir, codes, sc.depth, f.status, fs.hi);
    if (e == cudaSuccess)
      e = launch_scan_kernel(w, sc, iw, ww, ir, wr, f.alpha + (size_t)t0 * f.in_bytes,
                             f.beta + (size_t)t0 * f.in_bytes,
                             f.v + (size_t)t0 * d.dv * f.in_bytes, f.M,
                             f.y + (size_t)t0 * d.dv, nullptr, codes, f.status, fs.hi);
  }
  // Join both streams back into the caller's, also after a failed launch, so
  // nothing of this call is left running behind the caller's back.
  cudaError_t j = cudaEventRecord(fs.hi_end, fs.hi);
  if (j == cudaSuccess) j = cudaEventRecord(fs.lo_end, fs.lo);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(caller, fs.hi_end, 0);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(caller, fs.lo_end, 0);
  return (int)(e != cudaSuccess ? e : j);
}

sdm_status api_check_shape(const sdm_shape* shape, Dims* d) { return check_shape(shape, d); }
sdm_status api_status_ptr(unsigned** out) { return status_ptr(out); }
void api_scan_tuning(int* depth, int* col_slice) {
  std::lock_guard<std::mutex> lk(g_mu);
  *depth = g_depth;
  *col_slice = g_colslice;
}

}  // namespace sdm

using namespace sdm;

extern "C" {

const char* sdm_status_string(sdm_status st) {
  switch (st) {
    case SDM_OK: return "ok";
    case SDM_ERR_INVALID_ARG: return "invalid argument";
    case SDM_ERR_UNSUPPORTED: return "unsupported shape or option";
    case SDM_ERR_CUDA: return "CUDA runtime error";
    case SDM_ERR_TIMEOUT: return "device wait timed out";
    case SDM_ERR_DEVICE_BOUNDS: return "slot index out of range";
    case SDM_ERR_DUPLICATE_SLOT: return "duplicate slot in a write set";
  }
  return "unknown status";
}

sdm_status sdm_subscores(const sdm_shape* shape, const void* q, const void* K, float* S,
                         void* stream) {
  Dims d;
  sdm_status st = check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if (empty_work(d)) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(q);
  SDM_CHECK_PTR(K);
  SDM_CHECK_PTR(S);
  unsigned* sp = nullptr;
  if ((st = status_ptr(&sp)) != SDM_OK) return st;
  return from_cuda(launch_address(kAddrScoresOnly, d, q, nullptr, K, nullptr, nullptr,
                                  nullptr, nullptr, nullptr, nullptr, S, sp,
                                  static_cast<cudaStream_t>(stream)));
}

sdm_status sdm_select(const sdm_shape* shape, const float* sub_w, const float* sub_r,
                      int32_t* idx_w, float* wt_w, int32_t* idx_r, float* wt_r,
                      void* stream) {
  Dims d;
  sdm_status st = check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if (empty_work(d)) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(sub_w);
  SDM_CHECK_PTR(sub_r);
  SDM_CHECK_PTR(idx_w);
  SDM_CHECK_PTR(wt_w);
  SDM_CHECK_PTR(idx_r);
  SDM_CHECK_PTR(wt_r);
  unsigned* sp = nullptr;
  if ((st = status_ptr(&sp)) != SDM_OK) return st;
  return from_cuda(launch_address(kAddrSelectOnly, d, nullptr, nullptr, nullptr, sub_w,
                                  sub_r, idx_w, wt_w, idx_r, wt_r, nullptr, sp,
                                  static_cast<cudaStream_t>(stream)));
}

sdm_status sdm_address(const sdm_shape* shape, const void* q_w, const void* q_r,
                       const void* K, int32_t* idx_w, float* wt_w, int32_t* idx_r,
                       float* wt_r, void* stream) {
  Dims d;
  sdm_status st = check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if (empty_work(d)) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(q_w);
  SDM_CHECK_PTR(q_r);
  SDM_CHECK_PTR(K);
  SDM_CHECK_PTR(idx_w);
  SDM_CHECK_PTR(wt_w);
  SDM_CHECK_PTR(idx_r);
  SDM_CHECK_PTR(wt_r);
  unsigned* sp = nullptr;
  if ((st = status_ptr(&sp)) != SDM_OK) return st;
  return from_cuda(launch_address(kAddrFused, d, q_w, q_r, K, nullptr, nullptr, idx_w, wt_w,
                                  idx_r, wt_r, nullptr, sp, static_cast<cudaStream_t>(stream)));
}

size_t sdm_workspace_size(const sdm_shape* shape) {
  Dims d;
  if (check_shape(shape, &d) != SDM_OK) return 0;
  return scan_workspace_bytes(d);
}

// sdm_scan and sdm_scan_logged: `undo` is null for the plain scan.
static sdm_status scan_entry(const sdm_shape* shape, const int32_t* idx_w, const float* wt_w,
                             const int32_t* idx_r, const float* wt_r, const void* alpha,
                             const void* beta, const void* v, float* M, float* y, float* undo,
                             bool logged, void* workspace, size_t ws_bytes, void* stream) {
  Dims d;
  sdm_status st = check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if (empty_work(d)) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(idx_w);
  SDM_CHECK_PTR(wt_w);
  SDM_CHECK_PTR(idx_r);
  SDM_CHECK_PTR(wt_r);
  SDM_CHECK_PTR(alpha);
  SDM_CHECK_PTR(beta);
  SDM_CHECK_PTR(v);
  SDM_CHECK_PTR(M);
  SDM_CHECK_PTR(y);
  if (logged) SDM_CHECK_PTR(undo);
  SDM_CHECK_PTR(workspace);
  if (ws_bytes < scan_workspace_bytes(d)) return SDM_ERR_INVALID_ARG;
  unsigned* sp = nullptr;
  if ((st = status_ptr(&sp)) != SDM_OK) return st;
  int depth, cs;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    depth = g_depth;
    cs = g_colslice;
  }
  if (cs && d.dv % cs != 0) return SDM_ERR_INVALID_ARG;
  return from_cuda(launch_scan(d, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y, undo,
                               workspace, depth, cs, sp, static_cast<cudaStream_t>(stream)));
}

sdm_status sdm_scan(const sdm_shape* shape, const int32_t* idx_w, const float* wt_w,
                    const int32_t* idx_r, const float* wt_r, const void* alpha,
                    const void* beta, const void* v, float* M, float* y, void* workspace,
                    size_t ws_bytes, void* stream) {
  return scan_entry(shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y, nullptr, false,
                    workspace, ws_bytes, stream);
}

sdm_status sdm_scan_logged(const sdm_shape* shape, const int32_t* idx_w, const float* wt_w,
                           const int32_t* idx_r, const float* wt_r, const void* alpha,
                           const void* beta, const void* v, float* M, float* y, float* undo,
                           void* workspace, size_t ws_bytes, void* stream) {
  return scan_entry(shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y, undo, true,
                    workspace, ws_bytes, stream);
}

size_t sdm_undo_workspace_size(const sdm_shape* shape) {
  Dims d;
  if (check_shape(shape, &d) != SDM_OK) return 0;
  return undo_workspace_bytes(d);
}

sdm_status sdm_scan_undo(const sdm_shape* shape, const int32_t* idx_w, const float* undo,
                         float* M, void* workspace, size_t ws_bytes, void* stream) {
  Dims d;
  sdm_status st = check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if (empty_work(d)) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(idx_w);
  SDM_CHECK_PTR(undo);
  SDM_CHECK_PTR(M);
  SDM_CHECK_PTR(workspace);
  if (ws_bytes < undo_workspace_bytes(d)) return SDM_ERR_INVALID_ARG;
  unsigned* sp = nullptr;
  if ((st = status_ptr(&sp)) != SDM_OK) return st;
  return from_cuda(launch_undo(d, idx_w, undo, M, workspace, sp,
                               static_cast<cudaStream_t>(stream)));
}

int sdm_forward_windows(const sdm_shape* shape) {
  Dims d;
  if (check_shape(shape, &d) != SDM_OK) return 0;
  return forward_segments(d);
}

sdm_status sdm_forward(const sdm_shape* shape, const void* q_w, const void* q_r,
                       const void* K, const void* alpha, const void* beta, const void* v,
                       float* M, float* y, int32_t* idx_w, float* wt_w, int32_t* idx_r,
                       float* wt_r, void* workspace, size_t ws_bytes, void* stream) {
  // Check the scan's arguments too before anything is enqueued.
  Dims d;
  sdm_status st = check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if (empty_work(d)) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(alpha);
  SDM_CHECK_PTR(beta);
  SDM_CHECK_PTR(v);
  SDM_CHECK_PTR(M);
  SDM_CHECK_PTR(y);
  SDM_CHECK_PTR(workspace);
  if (ws_bytes < scan_workspace_bytes(d)) return SDM_ERR_INVALID_ARG;
  const int S = forward_segments(d);
  if (S > 1) {
    SDM_CHECK_PTR(q_w);
    SDM_CHECK_PTR(q_r);
    SDM_CHECK_PTR(K);
    SDM_CHECK_PTR(idx_w);
    SDM_CHECK_PTR(wt_w);
    SDM_CHECK_PTR(idx_r);
    SDM_CHECK_PTR(wt_r);
    int depth, cs;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      depth = g_depth;
      cs = g_colslice;
    }
    if (cs && d.dv % cs != 0) return SDM_ERR_INVALID_ARG;
    unsigned* sp = nullptr;
    if ((st = status_ptr(&sp)) != SDM_OK) return st;
    const int ib = d.in_dtype == SDM_BF16 ? 2 : 4;
    SegmentedForward f{d,     static_cast<const char*>(q_w), static_cast<const char*>(q_r), K,
                       static_cast<const char*>(alpha), static_cast<const char*>(beta),
                       static_cast<const char*>(v), M, y, idx_w, wt_w, idx_r, wt_r,
                       static_cast<int16_t*>(workspace), ib, depth, cs, sp};
    const int rc = run_segmented_forward(f, forward_window_steps(d),
                                         static_cast<cudaStream_t>(stream));
    if (rc >= 0) return from_cuda(static_cast<cudaError_t>(rc));
    // The side streams could not be set up: one stream, unsegmented.
  }
  st = sdm_address(shape, q_w, q_r, K, idx_w, wt_w, idx_r, wt_r, stream);
  if (st != SDM_OK) return st;
  return sdm_scan(shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y, workspace, ws_bytes,
                  stream);
}

sdm_status sdm_rmsnorm_gate(const sdm_shape* shape, const float* y, const void* g,
                            const float* gamma, float eps, void* out, sdm_dtype out_dtype,
                            void* stream) {
  Dims d;
  sdm_status st = check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if (!(eps > 0.f) || !(eps < INFINITY)) return SDM_ERR_INVALID_ARG;
  if (out_dtype != SDM_F32 && out_dtype != SDM_BF16) return SDM_ERR_INVALID_ARG;
  if (empty_work(d)) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(y);
  SDM_CHECK_PTR(g);
  SDM_CHECK_PTR(out);
  if (gamma && !aligned16(gamma)) return SDM_ERR_INVALID_ARG;
  return from_cuda(launch_rmsnorm_gate(d, y, g, gamma, eps, out, out_dtype,
                                       static_cast<cudaStream_t>(stream)));
}

sdm_status sdm_decode(const sdm_shape* shape, const void* q_w, const void* q_r, const void* K,
                      const void* alpha, const void* beta, const void* v, float* M, float* y,
                      int32_t* idx_w, float* wt_w, int32_t* idx_r, float* wt_r,
                      const sdm_epilogue* epi, void* stream) {
  Dims d;
  sdm_status st = check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if (epi) {
    if (!(epi->eps > 0.f) || !(epi->eps < INFINITY)) return SDM_ERR_INVALID_ARG;
    if (epi->out_dtype != SDM_F32 && epi->out_dtype != SDM_BF16) return SDM_ERR_INVALID_ARG;
  }
  if (empty_work(d)) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(q_w);
  SDM_CHECK_PTR(q_r);
  SDM_CHECK_PTR(K);
  SDM_CHECK_PTR(alpha);
  SDM_CHECK_PTR(beta);
  SDM_CHECK_PTR(v);
  SDM_CHECK_PTR(M);
  SDM_CHECK_PTR(y);
  SDM_CHECK_PTR(idx_w);
  SDM_CHECK_PTR(wt_w);
  SDM_CHECK_PTR(idx_r);
  SDM_CHECK_PTR(wt_r);
  if (epi) {
    SDM_CHECK_PTR(epi->g);
    SDM_CHECK_PTR(epi->out);
    if (epi->gamma && !aligned16(epi->gamma)) return SDM_ERR_INVALID_ARG;
  }
  return from_cuda(launch_decode(d, q_w, q_r, K, alpha, beta, v, M, y, idx_w, wt_w, idx_r,
                                 wt_r, epi ? epi->g : nullptr, epi ? epi->gamma : nullptr,
                                 epi ? epi->eps : 0.f, epi ? epi->out : nullptr,
                                 epi ? (int)epi->out_dtype : 0,
                                 static_cast<cudaStream_t>(stream)));
}

sdm_status sdm_get_device_status(void* stream) {
  unsigned* sp = nullptr;
  sdm_status st = status_ptr(&sp);
  if (st != SDM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SDM_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, sp, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SDM_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpy(sp, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return SDM_ERR_CUDA;
  return static_cast<sdm_status>(v);
}

sdm_status sdm_set_scan_tuning(int depth, int col_slice) {
  if (depth < 0 || depth > 16) return SDM_ERR_INVALID_ARG;
  if (col_slice != 0 && col_slice != 16 && col_slice != 32 && col_slice != 64)
    return SDM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_depth = depth;
  g_colslice = col_slice;
  return SDM_OK;
}

sdm_status sdm_selftest_wait_timeout(long long timeout_ns, void* stream) {
  if (timeout_ns < 1000000ll || timeout_ns > 10000000000ll) return SDM_ERR_INVALID_ARG;
  unsigned* sp = nullptr;
  sdm_status st = status_ptr(&sp);
  if (st != SDM_OK) return st;
  wait_timeout_selftest<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      sp, (unsigned long long)timeout_ns);
  return from_cuda(cudaGetLastError());
}

sdm_status sdm_measure_row_traffic(const float* src, float* dst, long long chains,
                                   long long rows, int d_v, int col_slice, int T, int loads,
                                   int stores, unsigned seed, void* stream) {
  if (chains < 0 || rows < 1 || rows > 0xffffffffll || T < 0) return SDM_ERR_INVALID_ARG;
  if (col_slice != 16 && col_slice != 32 && col_slice != 64) return SDM_ERR_INVALID_ARG;
  if (d_v < col_slice || d_v % col_slice != 0) return SDM_ERR_INVALID_ARG;
  if (loads < 1 || loads > 128 || stores < 0 || stores > loads) return SDM_ERR_INVALID_ARG;
  if (chains * (d_v / col_slice) > 0x7fffffffll) return SDM_ERR_UNSUPPORTED;
  if (chains == 0 || T == 0) return SDM_OK;   // no work: pointers are not looked at
  SDM_CHECK_PTR(src);
  SDM_CHECK_PTR(dst);
  return from_cuda(launch_row_traffic(src, dst, chains, rows, d_v, col_slice, T, loads, stores,
                                      seed, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
