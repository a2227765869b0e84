/*
 * sdm.h -- C ABI of the GB300 (sm_103a) Sparse Delta Memory forward step.
 *
 * The method (web pages, cited by title and section):
 *   [SDM notes]   "Sparse Delta Memory：中文精读笔记" (reading notes on
 *                 arXiv 2607.07386v1): 2.2 symbols, 2.3 product-key addressing,
 *                 2.4 Eq. (3)-(5) write / untouched slots / read, 2.5 Fig. 2.
 *   [FwPKM notes] Fast-weight Product Key Memory reading notes, 2.2: half-query
 *                 against sub-key tables; inverse-distance sub-score.
 *
 * One forward step per token t of every (b, h) chain:
 *   addressing  S_p[j] = <q_p, K_p[j]> (or -ln(eps + |q_p - K_p[j]|^2)), p = 1, 2;
 *               top-k of each half; best W (R) of the k*k sums S_1[a] + S_2[b];
 *               slot = a*s + b; weights = softmax over the selected sums.
 *   write       for i in I^w:  M~[i] = alpha_t M[i];
 *                              M[i]  = M~[i] + beta_t w_i (v_t - M~[i])   (Eq. (4))
 *               rows not in I^w are left bit-identical.
 *   read        y_t = sum_{i in I^r} q_i M[i], after the write.        (Eq. (5))
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers to dense row-major arrays that
 *    the caller allocates and owns; the library keeps no pointer after return.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously; argument errors are returned before
 *    anything is enqueued.  Failures the device detects (an index out of
 *    range, a duplicate write slot, a wait that ran out) are recorded in a
 *    per-device status word that sdm_get_device_status() reads and clears.
 *  - Alignment: every tensor base must be 16-byte aligned.
 *  - A call with no work (B, H or T zero) enqueues nothing and returns
 *    SDM_OK after the shape check; its pointers are not looked at (empty
 *    tensors may pass NULL).
 *  - The library allocates no device memory (the status word is a static
 *    device variable; scratch is the caller's `workspace`).  There is no
 *    CPU fallback.
 *  - The device addresses of the library's static device arrays (the status
 *    word; the scratch of sdm_scan_noalloc) are looked up once per device and
 *    kept for the life of the process, and so are the two streams and the
 *    events sdm_forward uses for its overlapped windows (created on first
 *    use): do not go on using the library on a device after cudaDeviceReset
 *    (or any other teardown of its primary context), since those handles are
 *    then stale.
 */
#ifndef SDM_H
#define SDM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDM_OK = 0,
  SDM_ERR_INVALID_ARG = 1,     /* null pointer, bad size, misaligned base       */
  SDM_ERR_UNSUPPORTED = 2,     /* valid but outside the limits listed below     */
  SDM_ERR_CUDA = 3,            /* a CUDA runtime call failed                    */
  SDM_ERR_TIMEOUT = 4,         /* device: a bounded wait ran out                */
  SDM_ERR_DEVICE_BOUNDS = 5,   /* device: a slot index outside [0, N)           */
  SDM_ERR_DUPLICATE_SLOT = 6   /* device: a slot repeated within one write set  */
} sdm_status;

typedef enum { SDM_F32 = 0, SDM_BF16 = 1 } sdm_dtype;
typedef enum { SDM_SCORE_DOT = 0, SDM_SCORE_IDW = 1 } sdm_score_kind;
typedef enum { SDM_UPDATE_EQ4 = 0, SDM_UPDATE_SHARED_RESIDUAL = 1 } sdm_update_form;

typedef struct {
  int B, H, T;            /* batch, heads, tokens per chain                        */
  int n_sub;              /* s = sqrt(N) entries per sub-key table; N = s*s       */
  int d_h;                /* half-query / sub-key dimension                        */
  int d_v;                /* value width = row width of the table                 */
  int W, R;               /* write / read slots per token and head                */
  int k_w, k_r;           /* per-half top-k; 0 selects min(W, s) / min(R, s)      */
  sdm_dtype in_dtype;     /* dtype of q_w, q_r, K, v, alpha, beta                 */
  sdm_score_kind score;   /* sub-score kind                                        */
  float idw_eps;          /* eps of the inverse-distance score (1e-3 in [FwPKM])  */
  sdm_update_form update; /* SDM_UPDATE_EQ4: per-slot Eq. (4) [SDM notes 2.4].     */
                          /* SDM_UPDATE_SHARED_RESIDUAL: the residual shared by    */
                          /* the write set, read off Fig. 2 [SDM notes 2.5]:       */
                          /* M[i] = M~[i] + beta w_i (v - sum_j w_j M~[j]).        */
} sdm_shape;

/* Limits (anything else returns SDM_ERR_UNSUPPORTED):
 *   1 <= n_sub <= 512;  d_h in {16, 32, 64, 128, 256};  d_v a multiple of 16,
 *   16 <= d_v <= 2048;  1 <= W, R <= 64;  1 <= k <= min(64, n_sub) and
 *   W <= k_w^2, R <= k_r^2;  B*H*N*d_v < 2^40 elements;  B, H, T >= 0. */

/* Human-readable name of a status code (static string). */
const char* sdm_status_string(sdm_status st);

/* Sub-scores of one branch [SDM notes 2.3; FwPKM notes 2.2].
 *   q: [B,H,T,2,d_h] (in_dtype) half-queries of that branch;
 *   K: [H,2,s,d_h]   (in_dtype) the two sub-key tables of each head;
 *   S: [B,H,T,2,s]   float32 out: S[...,p,j] = <q_p, K_p[j]>, or
 *                    -ln(idw_eps + |q_p - K_p[j]|^2) when score = IDW.
 * Accumulation is fp32; used to compare addressing at the score level. */
sdm_status sdm_subscores(const sdm_shape* shape, const void* q, const void* K,
                         float* S, void* stream);

/* Product-key selection from given float32 sub-scores [SDM notes 2.3].
 *   sub_w, sub_r: [B,H,T,2,s] float32 sub-scores of the write / read branch;
 *   idx_w: [B,H,T,W] int32 out, wt_w: [B,H,T,W] float32 out;
 *   idx_r: [B,H,T,R] int32 out, wt_r: [B,H,T,R] float32 out.
 * Each half keeps its top k by (score desc, index asc); the k*k sums
 * fl32(S_1[a] + S_2[b]) are ranked by (sum desc, slot asc), slot = a*s + b;
 * the best W (R) are written in rank order, with the softmax of their sums.
 * Indices are exact: identical sub-scores give identical slots. */
sdm_status sdm_select(const sdm_shape* shape, const float* sub_w,
                      const float* sub_r, int32_t* idx_w, float* wt_w,
                      int32_t* idx_r, float* wt_r, void* stream);

/* Addressing: sdm_subscores + sdm_select for both branches, fused in one
 * kernel (the sub-scores never leave the chip).
 *   q_w, q_r: [B,H,T,2,d_h]; K: [H,2,s,d_h] (all in_dtype);
 *   outputs as in sdm_select. */
sdm_status sdm_address(const sdm_shape* shape, const void* q_w, const void* q_r,
                       const void* K, int32_t* idx_w, float* wt_w,
                       int32_t* idx_r, float* wt_r, void* stream);

/* Bytes of device workspace that sdm_scan / sdm_forward need for `shape`
 * (0 for an invalid shape).  The scan first resolves, for every row a step
 * touches, whether one of the few preceding steps still in flight wrote it
 * (a 16-bit code per token and row); the workspace holds those codes. */
size_t sdm_workspace_size(const sdm_shape* shape);

/* The write-then-read recurrence over t for every (b,h) chain
 * [SDM notes 2.4, Eq. (3)-(5)].
 *   idx_w/wt_w: [B,H,T,W] int32/float32; idx_r/wt_r: [B,H,T,R];
 *   alpha, beta: [B,H,T] (in_dtype); v: [B,H,T,d_v] (in_dtype);
 *   M: [B,H,N,d_v] float32, updated IN PLACE (the updated table is the result);
 *   y: [B,H,T,d_v] float32 out;
 *   workspace: device scratch of at least sdm_workspace_size(shape) bytes
 *   (ws_bytes), caller-owned, contents irrelevant on entry and on return.
 * shape->update selects the write: Eq. (4) per slot, or the shared residual
 * read off Fig. 2 (one prediction sum_j w_j M~[j] for the whole write set).
 * Write slots of one step must be distinct and all slots in [0, N); the
 * device checks both, skips the offending rows and records
 * SDM_ERR_DUPLICATE_SLOT / SDM_ERR_DEVICE_BOUNDS.  Calling this on
 * consecutive T-segments (the table carried in M) equals one call on the
 * concatenation.  M must not alias any other argument. */
sdm_status sdm_scan(const sdm_shape* shape, const int32_t* idx_w,
                    const float* wt_w, const int32_t* idx_r, const float* wt_r,
                    const void* alpha, const void* beta, const void* v,
                    float* M, float* y, void* workspace, size_t ws_bytes,
                    void* stream);

/* sdm_scan without a workspace, for callers that cannot allocate device
 * memory: e.g. a host framework that owns all device memory and only passes
 * in the tensors of a call, or a code path where a cudaMalloc (and the
 * device-wide synchronisation it may bring) is not allowed.  The paper has no
 * counterpart; this is an interface variant of sdm_scan, same arguments and
 * results minus `workspace`/`ws_bytes`.
 * Scratch: a fixed 8 MiB array of device memory in the library itself (every
 * GPU that loads the library holds it until the process exits).  Problems
 * needing more plan-code scratch than that, i.e.
 * B*H*T*round_up(W+R, 8)*2 bytes > 8 MiB (32768 token-heads at W = R = 64),
 * return SDM_ERR_UNSUPPORTED before anything is enqueued.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All calls
 * share the one array: calls whose work overlaps on the GPU (other streams,
 * other threads) race and must be serialised by the caller.  Nothing in the
 * array needs clearing: every value a call reads, that call wrote first.
 * Calls no cudaMalloc, cudaFree or allocating library routine. */
sdm_status sdm_scan_noalloc(const sdm_shape* shape, const int32_t* idx_w,
                            const float* wt_w, const int32_t* idx_r,
                            const float* wt_r, const void* alpha, const void* beta,
                            const void* v, float* M, float* y, void* stream);

/* sdm_scan that also keeps an undo log [SDM notes 2.9, appendix A.3: the
 * forward pass writes the table in place and the backward pass brings back
 * earlier states by undoing the sparse writes, for O(T*W*d_v) extra memory].
 *   undo: [B,H,T,W,d_v] float32 out, caller-owned: undo[b,h,t,j,:] is the
 *         value row idx_w[b,h,t,j] held just before step t's write (an
 *         exact copy of the fp32 table row).
 * All other arguments, the workspace and the results as in sdm_scan. */
sdm_status sdm_scan_logged(const sdm_shape* shape, const int32_t* idx_w,
                           const float* wt_w, const int32_t* idx_r,
                           const float* wt_r, const void* alpha, const void* beta,
                           const void* v, float* M, float* y, float* undo,
                           void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace sdm_scan_undo needs: B*H*N*4 (one mark per
 * table row; 0 for an invalid shape). */
size_t sdm_undo_workspace_size(const sdm_shape* shape);

/* Undo a logged segment: M [B,H,N,d_v] float32, in place, goes back to the
 * table it was before the sdm_scan_logged call that produced `undo` for the
 * same idx_w [B,H,T,W] (shape->T = that segment's length).  Every row the
 * segment wrote gets the copy logged at its earliest write; other rows are
 * untouched.  The result is bit-exact.  Undoing segments in reverse order
 * walks a long sequence back chunk by chunk.
 *   workspace: at least sdm_undo_workspace_size(shape) bytes, caller-owned,
 *   contents irrelevant on entry and on return.
 * Slots outside [0, N) are skipped and recorded as SDM_ERR_DEVICE_BOUNDS. */
sdm_status sdm_scan_undo(const sdm_shape* shape, const int32_t* idx_w,
                         const float* undo, float* M, void* workspace,
                         size_t ws_bytes, void* stream);

/* Per-head RMS-Norm and element-wise output gate on the read result
 * [SDM notes 2.4, after Eq. (5); the head-mixing projection that follows is
 * not part of this library]:
 *   out[b,h,t,:] = y[b,h,t,:] / sqrt(mean_c y[b,h,t,c]^2 + eps)
 *                  * gamma[h,:] * g[b,h,t,:]
 *   y:     [B,H,T,d_v] float32 (the scan's output);
 *   g:     [B,H,T,d_v] output gate, in shape->in_dtype, applied as given;
 *   gamma: [H,d_v] float32 per-head scale, or NULL for ones;
 *   eps:   > 0;  out: [B,H,T,d_v] in out_dtype (SDM_BF16 or SDM_F32).
 * One pass over y, bandwidth-bound.  Shape fields other than B, H, T, d_v
 * and in_dtype only need to be valid. */
sdm_status sdm_rmsnorm_gate(const sdm_shape* shape, const float* y, const void* g,
                            const float* gamma, float eps, void* out,
                            sdm_dtype out_dtype, void* stream);

/* Optional epilogue of sdm_decode: the arguments of sdm_rmsnorm_gate. */
typedef struct {
  const void* g;         /* [B,H,T,d_v] output gate, in shape->in_dtype      */
  const float* gamma;    /* [H,d_v] per-head scale, or NULL for ones         */
  float eps;             /* > 0                                              */
  void* out;             /* [B,H,T,d_v] in out_dtype                         */
  sdm_dtype out_dtype;   /* SDM_BF16 or SDM_F32                              */
} sdm_epilogue;

/* The forward step fused into one launch for short sequences -- decode,
 * T = 1 per call [SDM notes 2.3-2.5; section 3 reports decode speed at the
 * shapes of 2.8: sqrt N = 240 / 480, d_v = 960 / 1920].  Same arguments and
 * results as sdm_forward (y, M in place, selections in idx_w/wt_w/idx_r/wt_r)
 * plus, when `epi` is non-NULL, the sdm_rmsnorm_gate epilogue on y written
 * to epi->out.  Each (b,h) chain runs its T steps in order on one CTA, or,
 * when there are too few chains to fill the GPU, on up to 8 CTAs that each
 * own a range of its columns (with the epilogue they form one thread-block
 * cluster for the row norm); the latency of a step is one chain's dependent
 * path; use sdm_forward for long T.  Needs no workspace.  Sub-scores are fp32 FFMA for both
 * input dtypes, so a selection can differ from one made on sdm_forward's
 * tensor-core scores only where two candidate sums are within fp32 rounding
 * of each other. */
sdm_status sdm_decode(const sdm_shape* shape, const void* q_w, const void* q_r,
                      const void* K, const void* alpha, const void* beta,
                      const void* v, float* M, float* y, int32_t* idx_w,
                      float* wt_w, int32_t* idx_r, float* wt_r,
                      const sdm_epilogue* epi, void* stream);

/* One full forward step: sdm_address then sdm_scan on `stream`.
 * Inputs as above; M updated in place, y written, and the selected indices
 * and weights returned in the caller's idx_w/wt_w/idx_r/wt_r buffers. */
/* Number of step windows sdm_forward cuts T into (1 = none; 0 for an
 * invalid shape): from T = 2048 on, T/512 windows (at most 32) where the
 * addressing runs on the tensor cores, else 4; every window but the last is
 * a whole number of 64-step blocks.  With more than one, the addressing of
 * window k+1 runs on a low-priority internal stream while window k is
 * scanned on a high-priority one, both joined back into the caller's
 * stream; results are bit-identical to sdm_address followed by sdm_scan.
 * Each window launches the addressing, plan and scan kernels once.  The
 * internal streams and events are created by the first windowed call on a
 * device: make that call outside a CUDA graph capture; later calls can be
 * captured (the fork and join are recorded with the caller's stream).  If
 * the streams cannot be created, sdm_forward runs unwindowed on the
 * caller's stream. */
int sdm_forward_windows(const sdm_shape* shape);

sdm_status sdm_forward(const sdm_shape* shape, const void* q_w, const void* q_r,
                       const void* K, const void* alpha, const void* beta,
                       const void* v, float* M, float* y, int32_t* idx_w,
                       float* wt_w, int32_t* idx_r, float* wt_r, void* workspace,
                       size_t ws_bytes, void* stream);

/* Synchronizes `stream`, then returns and clears the device status word of
 * the current device (SDM_OK if no device-side failure was recorded). */
sdm_status sdm_get_device_status(void* stream);

/* Scan launch tuning for the calling process (0 = automatic):
 *   depth      steps whose rows are in flight per chain slice, 1..16;
 *   col_slice  columns of d_v per CTA, 16, 32 or 64 (must divide d_v).
 * Results do not depend on these; only speed does. */
sdm_status sdm_set_scan_tuning(int depth, int col_slice);

/* Self-test of the bounded device wait: launches one CTA that waits on a
 * barrier no thread ever completes, with a limit of `timeout_ns`
 * nanoseconds (1e6..1e10), then records SDM_ERR_TIMEOUT and returns.
 * Shows on a real device that a wait that runs out ends the kernel cleanly. */
sdm_status sdm_selftest_wait_timeout(long long timeout_ns, void* stream);

/* Measurement reference, not part of the method: the scan's row traffic
 * ([SDM notes] 2.4: per step of every (chain, column slice) unit, the W + R
 * rows it touches are fetched and the W written rows stored back) with no
 * arithmetic and no dependency between steps.  For each of chains x
 * (d_v / col_slice) units and each of T steps, `loads` row pieces of
 * col_slice floats are copied from rows drawn uniformly from the unit's chain
 * in `src` into shared memory, and the first `stores` of them are written to
 * other uniformly drawn rows of the same chain and columns in `dst`; draws
 * are a fixed hash of (seed, unit, step, position).  Bytes moved:
 * chains * d_v * T * (loads + stores) * 4.  A timed call gives the rate HBM
 * sustains for the scan's access pattern.
 *   src, dst   device [chains, rows, d_v] float32 (may be the same array; the
 *              contents of dst afterwards are unspecified); 16-byte aligned.
 *   col_slice  16, 32 or 64, dividing d_v;  1 <= loads <= 128;
 *   0 <= stores <= loads;  1 <= rows < 2^32.
 * Argument errors return SDM_ERR_INVALID_ARG before anything is enqueued. */
sdm_status sdm_measure_row_traffic(const float* src, float* dst, long long chains,
                                   long long rows, int d_v, int col_slice, int T, int loads,
                                   int stores, unsigned seed, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SDM_H */
