/*
 * sprint.h — C ABI of the GB300 (sm_103a) stale-weight SGD hot path.
 *
 * One process drives one GPU. The library computes the minibatch-SGD worker
 * step of a CNN/MLP (forward pass, dE/dW, dE/db, dE/dX by implicit-GEMM /
 * im2col convolution, FC GEMMs, 2x2 max-pooling, ReLU, softmax cross-entropy)
 * and the gradient-buffer / parameter-server update (GradBuf accumulation,
 * then plain SGD, momentum or per-parameter Adagrad), as set out in:
 *
 *   [S]  IPSJ SIG Technical Report Vol.2016-HPC-155 No.8, "SPRINT" ASGD CNN
 *        framework: Eq. (1) minibatch SGD; Eq. (2)-(3) network shapes;
 *        Sec. 3.3, Eq. (4)-(6) and the SGEMM role table that follows Eq. (6)
 *        (convolution, fc, dedw, dedb, dedx fc, dedx conv, im2col);
 *        Algorithm 1 (GPU thread: ComputeGradient, ComputeUpdateVal,
 *        UpdateGradient into GradBuf_t); Algorithm 2 (update thread:
 *        SumGradient, momentum via DeltaWeights, UpdateWeights).
 *   [PB] "Pipelined training of deep CNNs with stale weights", Sec. 4.1.
 *   [DB] "Google DistBelief Paper: Large Scale Distributed Deep Networks"
 *        (parameter-server update w' := w - eta*dw, Adagrad, n_push).
 *
 * Conventions for every entry point
 *  - Return value: a sprint_status (0 = SPRINT_OK). On error nothing is
 *    launched, and sprint_last_error() returns a message (thread-local).
 *  - Arguments are validated on the host before any launch.
 *  - Device pointers are caller-owned (the library never allocates, frees or
 *    keeps them past the call) and must be 16-byte aligned, else
 *    SPRINT_ERR_ALIGN. Host pointers are marked "host".
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream). Output buffers must not alias inputs unless the
 *    entry point says so.
 *  - All tensors are fp32. GEMM-shaped work runs on the tensor cores as TF32
 *    with FP32 accumulation; every other operation is exact fp32 arithmetic.
 *  - Layouts: activations NHWC [N][H][W][C]; conv weights [Cout][3][3][Cin]
 *    (GEMM K index = (kh*3 + kw)*Cin + ci); FC weights [out][in]; row-major.
 *  - Convolutions are 3x3, stride 1 ([S] Sec. 3.2, c = 3); `pad` is 0 or 1;
 *    the output is (H + 2*pad - 2) x (W + 2*pad - 2).
 *  - Kernels never trap. A bounded wait inside a kernel that gives up sets a
 *    device status word; sprint_device_status() reads it (SPRINT_ERR_DEVICE_FLAG).
 */
#ifndef SPRINT_H
#define SPRINT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* sprint_stream_t; /* a cudaStream_t */

typedef enum {
    SPRINT_OK = 0,
    SPRINT_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad flag    */
    SPRINT_ERR_SHAPE = 2,       /* inconsistent or out-of-range dimensions   */
    SPRINT_ERR_ALIGN = 3,       /* device pointer not 16-byte aligned        */
    SPRINT_ERR_UNSUPPORTED = 4, /* valid but not implemented (e.g. k > 16)   */
    SPRINT_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed         */
    SPRINT_ERR_DEVICE_FLAG = 6, /* a kernel reported a failed bounded wait   */
    SPRINT_ERR_WORKSPACE = 7    /* caller workspace missing or too small     */
} sprint_status;

/* Message of the last failed call on this thread ("" if none). Never NULL. */
const char* sprint_last_error(void);

/* ABI version (major*100 + minor). */
int sprint_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads). Host-side counter; no device call. */
uint64_t sprint_launch_count(void);

/* Reads (and with reset != 0 clears) the device status word that kernels set
 * when a bounded wait gives up. *flags_out = 0 means no kernel reported a
 * failure. Synchronises the device. Returns SPRINT_ERR_DEVICE_FLAG if a flag
 * was set, SPRINT_OK otherwise. */
int sprint_device_status(int* flags_out, int reset);

/* Plan queries (no page counterpart; for tests and tuning): how the library
 * would run a call, without running it. out[0 .. SPRINT_PLAN_FIELDS-1] (host):
 *   [0] path: SPRINT_PATH_TC (tcgen05 implicit GEMM / weight-gradient GEMM),
 *       SPRINT_PATH_SMALLC (direct CUDA-core kernel for <= 4 input channels),
 *       SPRINT_PATH_IM2COL (padded explicit im2col + tensor-core GEMM),
 *       SPRINT_PATH_SIMT (CUDA-core fallback)
 *   [1] tile width BN   [2] CTA pair (1) or single CTA (0)
 *   [3] split-K count of the weight gradient (1: none)
 *   [4] k-ranges of the last, partial round's tiles (1: no tail split; it is
 *       used only when the workspace holds its slabs)
 *   [5] taps per n-tile of the weight gradient (0: one tap per tile)
 *   [6] channel rows per packed tap   [7] k-tiles of 32 in the reduction
 *   [8..10] output-pixel box of the implicit GEMM (w, h, images)
 *   [11] layout of the weight gradient's transposed copies: 1 = blocked
 *       [H][W*N/32][C][32] (N % 32 == 0), 0 = [C][H][W][N]
 *   [12] 1 = weight gradient factored over kernel rows x columns on CTA pairs
 *       (Cin = Cout = 64, pad 1, N % 32 == 0)
 *   [13] 1 = forward / input gradient factored over the kernel columns on CTA
 *       pairs (64 output channels, input channels % 32 == 0, pad 1, rows of
 *       >= 96 pixels; uses the workspace for permuted weights)
 *   [14] 1 = forward / input gradient on halo-staged tiles (CTA pairs, pad
 *       1, input channels % 32 == 0; 64 outputs (forward or input gradient)
 *       with BN = 192, factored over the kernel columns, or 128 outputs of
 *       the forward pass with BN = 128): a tile is [9] rows of [8] output
 *       pixels, read once per 32-channel chunk with its one-pixel border;
 *       used where such tiles fill >= 80% of the 128 MMA rows
 *   [16] 1 = the halo-staged tiles of 128 outputs in their flipped form: the
 *       weights as the 128-row MMA operand and 256 tile positions ([9] rows
 *       of [8] pixels) as its N side, one CTA per tile ([1] = 128, [2] = 0)
 *   [15] 1 = forward of the RGB layer (3 input, 64 output channels, pad 1)
 *       on the tensor cores, its im2col rows written into shared memory (no
 *       workspace beyond the weights padded to 32 columns)
 * Returns SPRINT_ERR_SHAPE / SPRINT_ERR_INVALID_ARG like the calls they
 * describe. sprint_conv_plan: op, shape and have_wT as for the conv calls.
 * sprint_gemm_plan: the grouped tensor-core GEMM D[M][N] = A[M][K] B[N][K]^T
 * over `batch` problems (the batched FC calls), allow_tail as when the
 * workspace holds the tail slabs. */
#define SPRINT_PLAN_FIELDS 17
#define SPRINT_PATH_SIMT 0
#define SPRINT_PATH_TC 1
#define SPRINT_PATH_SMALLC 2
#define SPRINT_PATH_IM2COL 3
int sprint_conv_plan(int op, int N, int H, int W, int Cin, int Cout, int pad, int have_wT, int32_t* out, int n_out);
int sprint_gemm_plan(int M, int N, int K, int batch, int allow_tail, int32_t* out, int n_out);

/* Self-test of the failure path above (no page counterpart): launches one
 * block on `stream` whose thread waits, with the same bounded wait the
 * pipelined kernels use, on an mbarrier phase that nothing ever completes (no
 * copy or MMA is in flight). After limit_ns nanoseconds of wall time the wait
 * gives up, ORs 8 into the device status word and the kernel returns, so the
 * context stays usable; sprint_device_status then reports
 * SPRINT_ERR_DEVICE_FLAG with bit 8 set. limit_ns in [1e3, 1e10], else
 * SPRINT_ERR_INVALID_ARG. */
int sprint_selftest_bounded_wait(uint64_t limit_ns, sprint_stream_t stream);

/* ------------------------------------------------------------------------
 * im2col — the explicit unrolling of [S] Sec. 3.3, Eq. (5): rows x_l^2 * N,
 * columns c^2 * m_{l-1}.
 * x:   device [N][H][W][C]
 * col: device [N*Ho*Wo][9*C]; row (n,oh,ow), column (kh*3+kw)*C + ci holds
 *      x[n][oh+kh-pad][ow+kw-pad][ci], or 0 outside the image.
 * src_index: device [N*Ho*Wo][9*C] int32 or NULL; the flat NHWC index of the
 *      source element in x, or -1 for padding. Bit-exact by construction.
 * Errors: SHAPE if any size < 1, pad not in {0,1}, or N*Ho*Wo*9*C >= 2^31.
 */
int sprint_im2col(const float* x, int N, int H, int W, int C, int pad, float* col, int32_t* src_index,
                  sprint_stream_t stream);

/* ------------------------------------------------------------------------
 * Convolution forward — the "convolution" SGEMM role of [S] Sec. 3.3
 * (m = x_l^2 N, n = m_l, k = c^2 m_{l-1}), with the bias and ReLU of Sec. 3.2
 * fused into the epilogue:
 *   y[n,oh,ow,co] = act(b[co] + sum_{kh,kw,ci} x[n,oh+kh-pad,ow+kw-pad,ci] * w[co,kh,kw,ci])
 * act = ReLU if relu != 0, identity otherwise. b may be NULL (no bias).
 * x: device [N][H][W][Cin]; w: device [Cout][3][3][Cin]; b: device [Cout];
 * y: device [N][Ho][Wo][Cout] (written, must not alias x).
 * Implicit GEMM: no im2col buffer is formed. Layers whose channel counts the
 * tensor-core loader cannot tile (Cin or Cout not a multiple of 32, e.g. the
 * RGB input layer) run on a CUDA-core direct-convolution kernel instead.
 * ws: see sprint_conv_workspace_size(SPRINT_CONV_FWD, ...).
 */
int sprint_conv_fwd(const float* x, const float* w, const float* b, float* y, int N, int H, int W, int Cin,
                    int Cout, int pad, int relu, void* ws, size_t ws_bytes, sprint_stream_t stream);

/* Convolution input gradient — the "dedx conv" role of [S] Sec. 3.3:
 *   dx[n,i,j,ci] = mask(n,i,j,ci) * sum_{kh,kw,co} dy[n,i-kh+pad,j-kw+pad,co] * w[co,kh,kw,ci]
 * mask = (relu_src > 0) if relu_src != NULL (relu_src is this layer's input,
 * i.e. the previous layer's ReLU output, [N][H][W][Cin]), else 1.
 * dy: device [N][Ho][Wo][Cout]; dx: device [N][H][W][Cin] (fully written).
 * wT: device [3][3][Cin][Cout] = w transposed (sprint_transpose of w viewed as
 * [Cout][9*Cin]), or NULL: the tensor cores read both operands k-contiguous,
 * so without wT the call transposes w into its workspace first.
 * ws: see sprint_conv_workspace_size(SPRINT_CONV_DX, ...) (sized for wT == NULL). */
int sprint_conv_dX(const float* dy, const float* w, const float* wT, const float* relu_src, float* dx, int N, int H,
                   int W, int Cin, int Cout, int pad, void* ws, size_t ws_bytes, sprint_stream_t stream);

/* Convolution operations, for sprint_conv_workspace_size(). */
enum { SPRINT_CONV_FWD = 0, SPRINT_CONV_DX = 1, SPRINT_CONV_DW = 2 };

/* Workspace bytes the convolution `op` needs for this shape (split-K partial
 * sums, partial bias sums, transposed copies); 0 means none. Every conv entry
 * point takes a caller-owned device workspace `ws` of this many bytes (contents
 * on entry ignored, clobbered by the call; NULL allowed when the size is 0).
 * For SPRINT_CONV_FWD and SPRINT_CONV_DX the last part of the size may be room
 * for splitting the k range of the launch's last, partial round of tiles
 * (partial sums added afterwards in a fixed order: deterministic); a smaller
 * workspace that still holds the rest is accepted and that split is skipped.
 * Too small a workspace gives SPRINT_ERR_WORKSPACE. Calls that may overlap on
 * the GPU need separate workspaces. */
size_t sprint_conv_workspace_size(int op, int N, int H, int W, int Cin, int Cout, int pad);

/* Convolution weight and bias gradients — the "dedw" and "dedb" roles of
 * [S] Sec. 3.3 (dedw: m = c^2 m_{l-1}, n = m_l, k = x_l^2 N), fused with
 * UpdateGradient of Algorithm 1 (GradBuf_t <- Grad, or += Grad):
 *   dw[co,kh,kw,ci] = (accumulate ? dw : 0) + alpha * sum_{n,oh,ow} dy[n,oh,ow,co] x[n,oh+kh-pad,ow+kw-pad,ci]
 *   db[co]          = (accumulate ? db : 0) + alpha * sum_{n,oh,ow} dy[n,oh,ow,co]   (db may be NULL)
 * dy is the gradient w.r.t. the pre-activation (the ReLU mask already applied).
 * x: device [N][H][W][Cin]; dy: device [N][Ho][Wo][Cout]; dw: device
 * [Cout][3][3][Cin]; db: device [Cout]. With Cin <= 4 and Cout <= 64 (Cout even
 * when above 32; the RGB input layer) both sums run in FP32 on the CUDA cores
 * from x and dy as they are, and the workspace holds one partial per launched
 * block (Cout * (9 * Cin + 1) floats each), added in block order; otherwise the
 * workspace holds the transposed copies x^T, dy^T of the TF32 tensor-core
 * path ([C][H][W][N], or blocked [H][W*N/32][C][32] when N % 32 == 0) and its
 * partial sums.
 * ws: see sprint_conv_workspace_size(SPRINT_CONV_DW, ...). */
int sprint_conv_dW(const float* x, const float* dy, float* dw, float* db, float alpha, int accumulate, int N, int H,
                   int W, int Cin, int Cout, int pad, void* ws, size_t ws_bytes, sprint_stream_t stream);

/* The weight gradient's copy of its input made ahead of time (no page
 * counterpart: the re-layout the k-contiguous TF32 operands need, so a caller
 * can make it while the forward pass runs). When the tensor-core weight
 * gradient of this shape reads blocked copies (N % 32 == 0; plan field 11),
 * sprint_conv_xT_size returns the bytes of x^T = x as [H][W*N/32][C][32]
 * (pixels (h, w, n) with n fastest in blocks of 32 images, channel-major inside
 * a block), else 0. sprint_conv_xT writes that copy of x (device [N][H][W][C])
 * into xT (device, caller-owned; must not alias x); SPRINT_ERR_UNSUPPORTED when
 * the size is 0. sprint_conv_dW_xT is sprint_conv_dW reading x^T from xT
 * instead of forming it (xT must hold sprint_conv_xT's copy of this x; x is
 * still read by the paths that do not use copies); its workspace is the same
 * as sprint_conv_dW's (the x^T part is then left unused). */
size_t sprint_conv_xT_size(int N, int H, int W, int Cin, int Cout, int pad);
int sprint_conv_xT(const float* x, float* xT, int N, int H, int W, int Cin, int Cout, int pad,
                   sprint_stream_t stream);
int sprint_conv_dW_xT(const float* x, const float* xT, const float* dy, float* dw, float* db, float alpha,
                      int accumulate, int N, int H, int W, int Cin, int Cout, int pad, void* ws, size_t ws_bytes,
                      sprint_stream_t stream);

/* ------------------------------------------------------------------------
 * FC forward — the "fc" role of [S] Sec. 3.3 (m = N, n = m_l, k = m_{l-1}):
 *   y[n][o] = act(b[o] + sum_i x[n][i] * w[o][i]), act = ReLU if relu != 0.
 * x: device [N][in]; w: device [out][in]; b: device [out] or NULL;
 * y: device [N][out] (must not alias x). */
int sprint_fc_fwd(const float* x, const float* w, const float* b, float* y, int N, int in, int out, int relu,
                  sprint_stream_t stream);

/* FC backward — the "dedx fc", "dedw" and "dedb" roles of [S] Sec. 3.3,
 * with UpdateGradient of Algorithm 1 fused into the dW/db epilogue:
 *   dx[n][i] = mask[n][i] * sum_o dy[n][o] * w[o][i]       (skipped if dx == NULL)
 *   dw[o][i] = (accumulate ? dw : 0) + alpha * sum_n dy[n][o] * x[n][i]
 *   db[o]    = (accumulate ? db : 0) + alpha * sum_n dy[n][o]  (skipped if db == NULL)
 * mask = (relu_src > 0) when relu_src != NULL (this layer's input [N][in]),
 * else 1. dy is the gradient w.r.t. this layer's pre-activation output.
 * x [N][in], w [out][in], dy [N][out], relu_src: device inputs;
 * wT: device [in][out] = w transposed (sprint_transpose), or NULL (then
 * transposed into the workspace); dx [N][in], dw [out][in], db [out]: outputs.
 * The weight-gradient GEMM contracts over the batch; its operands are
 * transposed into the workspace (k contiguous for the tensor cores).
 * ws: device workspace of at least sprint_fc_workspace_size(N, in, out,
 * wT != NULL) bytes (caller-owned scratch, clobbered; NULL if that is 0). */
int sprint_fc_bwd(const float* x, const float* w, const float* wT, const float* dy, const float* relu_src, float* dx,
                  float* dw, float* db, float alpha, int accumulate, int N, int in, int out, void* ws, size_t ws_bytes,
                  sprint_stream_t stream);

/* Workspace bytes sprint_fc_bwd needs (have_wT: whether wT will be passed). */
size_t sprint_fc_workspace_size(int N, int in, int out, int have_wT);

/* FC backward without any allocation: the same computation and arguments as
 * sprint_fc_bwd, minus the workspace, which comes from a fixed scratch array
 * compiled into the library (the pages have no counterpart; this serves
 * callers that cannot allocate device memory: code under a memory manager
 * that owns all device memory, or paths that must not call cudaMalloc or
 * cudaFree because those may synchronise the device).
 *  - Limit: sprint_fc_bwd_static_scratch_bytes() bytes (24 MiB) per device. A
 *    shape whose sprint_fc_workspace_size(N, in, out, wT != NULL || dx == NULL)
 *    exceeds it is rejected with SPRINT_ERR_WORKSPACE before any launch.
 *  - The array is held by every GPU that loads the library until the process
 *    exits. The first call in a CUDA context looks up the array's device
 *    address there (cudaGetSymbolAddress) and caches it under the context's
 *    unique ID; make that first call before any stream capture. A context
 *    created later on the device (e.g. after cudaDeviceReset) gets its own
 *    lookup on its first call, which should also precede any capture.
 *  - No cudaMalloc, cudaFree or other allocating routine is called.
 *  - Every call shares the one array and it keeps the last call's contents;
 *    nothing in it needs to start at zero (each call writes what it reads).
 *    Calls that overlap on the GPU (e.g. on two streams) race on it. */
int sprint_fc_bwd_static_scratch(const float* x, const float* w, const float* wT, const float* dy,
                                 const float* relu_src, float* dx, float* dw, float* db, float alpha, int accumulate,
                                 int N, int in, int out, sprint_stream_t stream);

/* Size in bytes of the static scratch array sprint_fc_bwd_static_scratch uses. */
size_t sprint_fc_bwd_static_scratch_bytes(void);

/* ------------------------------------------------------------------------
 * Batched FC: `batch` independent problems of one shape in as few launches as
 * possible — the R logical replicas of one layer ([S] Algorithm 1 runs one
 * GPU thread per replica; here the replicas of a layer are one grouped
 * tensor-core launch, each problem with its own weight version).
 * Every array argument is a HOST array of `batch` device pointers (read during
 * the call only); problem g uses entry g of each. Each problem computes exactly
 * what sprint_fc_fwd / sprint_fc_bwd compute for it. Arrays the single-problem
 * call lets be NULL may be NULL arrays here (b, wT, relu_src, dx, db); entries
 * of b and relu_src may also be NULL individually. batch = 0 is a no-op.
 * Problems must not write the same memory. */
int sprint_fc_fwd_batched(const float* const* x, const float* const* w, const float* const* b, float* const* y,
                          float* const* yT, int batch, int N, int in, int out, int relu, void* ws, size_t ws_bytes,
                          sprint_stream_t stream);
/* yT (nullable array): also write each output transposed, yT[g] = device
 * [out][N] (row j = column j of y[g]), the k-contiguous operand a following
 * layer's weight-gradient GEMM reads (the TF32 tensor-core MMA takes only
 * k-contiguous operands). The tensor-core epilogue stores it next to y; other
 * paths transpose y afterwards. Must not overlap y or x. */

/* Optional workspace of sprint_fc_fwd_batched (device, 16-byte aligned): with
 * at least this many bytes the tensor-core launch may split the k range of its
 * last, partial round of tiles (partial sums parked in the workspace, then
 * added in a fixed order: deterministic); with less (or ws = NULL) it does not. */
size_t sprint_fc_fwd_batched_workspace_size(void);

/* Workspace bytes of sprint_fc_bwd_batched: `batch` slices of
 * sprint_fc_workspace_size(N, in, out, have_wT), each rounded up to 256, then
 * sprint_fc_fwd_batched_workspace_size() bytes for the last-round k split of
 * its GEMMs (optional: a workspace holding only the slices is accepted). */
size_t sprint_fc_batched_workspace_size(int batch, int N, int in, int out, int have_wT);

int sprint_fc_bwd_batched(const float* const* x, const float* const* xT1, const float* const* w,
                          const float* const* wT, const float* const* dy, const float* const* dyT,
                          const float* const* relu_src, float* const* dx, float* const* dxT, float* const* dw,
                          float* const* db, float alpha, int accumulate, int batch, int N, int in, int out, void* ws,
                          size_t ws_bytes, sprint_stream_t stream);
/* Optional transposed operands and outputs (nullable arrays; with all three
 * NULL the call is the plain batched backward):
 *  xT1[g]: device [in + 1][N], x[g] transposed (row i = column i of x[g])
 *    followed by one row of N ones. The weight-gradient GEMM reads it instead
 *    of transposing x, and the row of ones gives that GEMM one more output
 *    column, sum_n dy[g][n][o], which becomes db (alpha / accumulate as for
 *    db): dedb is computed inside the dedw GEMM ([S] Sec. 3.2, dedb = the
 *    column sums of dE/dy). x is still required (paths that do not take the
 *    tensor cores read it).
 *  dyT[g]: device [out][N], dy[g] transposed (read instead of transposing dy).
 *  dxT[g]: device [in][N], written with dx[g] transposed (needs dx); what the
 *    layer below passes as its dyT.
 * Results are those of the plain call up to the rounding of db (a TF32 GEMM
 * column instead of an fp32 sum when xT1 is given). */

/* Update rules of the parameter-server apply (see sprint_apply_update). */
typedef enum { SPRINT_OPT_SGD = 0, SPRINT_OPT_MOMENTUM = 1, SPRINT_OPT_ADAGRAD = 2, SPRINT_OPT_NESTEROV = 3 } sprint_opt;

/* The batched FC backward of the R replicas of one layer (arguments as
 * sprint_fc_bwd_batched; each dw[g] / db[g] is replica g's GradBuf, Algorithm 1)
 * followed by the parameter-server apply of that layer over those `batch`
 * GradBufs (SumGradient + UpdateWeights of Algorithm 2, [S] Sec. 3):
 *   S = dw[0] + dw[1] + ... + dw[batch-1]  (added in g order, per element)
 *   w_out = rule(w_in, S) with `opt`, eta, nu_or_eps and weight_decay exactly
 *   as sprint_apply_update computes it (bit for bit);
 *   b_out = rule(b_in, db[0] + ... + db[batch-1]) when db is given;
 *   wT_out (nullable): also w_out transposed, device [in][out].
 * w_in, w_out, w_state: device [out][in] (w_state: the momentum v or the
 * Adagrad G of w, updated in place; unused for SGD); b_in, b_out, b_state:
 * device [out] (required when db is given). w_out may equal w_in (in place)
 * but must not overlap any other argument. 1 <= batch <= 16.
 * The update runs after the backward pass in stream order: W' (and W'^T in
 * the same pass, as sprint_apply_update_t), then b'. */
int sprint_fc_bwd_update_batched(const float* const* x, const float* const* xT1, const float* const* w,
                                 const float* const* wT, const float* const* dy, const float* const* dyT,
                                 const float* const* relu_src, float* const* dx, float* const* dxT, float* const* dw,
                                 float* const* db, float alpha, int accumulate, int batch, int N, int in, int out,
                                 int opt, const float* w_in, const float* b_in, float* w_out, float* b_out,
                                 float* wT_out, float* w_state, float* b_state, float eta, float nu_or_eps,
                                 float weight_decay, void* ws, size_t ws_bytes, sprint_stream_t stream);

/* Transpose: dst[c][r] = src[r][c] for a row-major [rows][cols] matrix (the
 * w -> w^T copies the input-gradient GEMMs read). src and dst: device, must
 * not alias. */
int sprint_transpose(const float* src, float* dst, int rows, int cols, sprint_stream_t stream);

/* ------------------------------------------------------------------------
 * 2x2 stride-2 max-pool forward — the pooling p_l = 2 of [S] Sec. 3.2/Eq. (2).
 * x: device [N][H][W][C]; y: device [N][H/2][W/2][C] (floor; a trailing odd
 * row/column is ignored); argmax: device [N][H/2][W/2][C] uint8, code
 * 2*dy + dx of the first window element (row-major) that is strictly greater
 * than every element before it. Bit-exact on identical inputs. */
int sprint_pool_fwd(const float* x, float* y, uint8_t* argmax, int N, int H, int W, int C, sprint_stream_t stream);

/* Max-pool backward with the ReLU derivative of the pooled layer:
 *   dx[n, 2i+dy, 2j+dx, c] = dy[n,i,j,c] * (pooled[n,i,j,c] > 0)  at the argmax code, else 0.
 * pooled: the forward output y (device [N][H/2][W/2][C]) or NULL for no mask.
 * (The selected element of the ReLU output equals pooled, so this is the ReLU
 * derivative of the conv layer feeding the pool.)
 * dx: device [N][H][W][C], fully written (zeros off the argmax). */
int sprint_pool_bwd(const float* dy, const uint8_t* argmax, const float* pooled, float* dx, int N, int H, int W,
                    int C, sprint_stream_t stream);

/* ------------------------------------------------------------------------
 * Softmax cross-entropy — the softmax output layer of [S] Sec. 3.2:
 *   loss    = (1/N) sum_n [log sum_c exp(z[n][c]) - z[n][label[n]]]
 *   dlogits = (softmax(z) - onehot(label)) / N
 * With reduction_sum != 0 the 1/N factors are dropped (literal Eq. (1) sum).
 * logits: device [N][C]; labels: device int32 [N], each in [0, C) (a label
 * out of range is not read through: that row adds nothing to the loss, its
 * dlogits row is zero, and sprint_device_status reports flag 16);
 * loss: device fp32 scalar; dlogits: device [N][C] (may alias logits). */
int sprint_softmax_xent(const float* logits, const int32_t* labels, int N, int C, float* loss, float* dlogits,
                        int reduction_sum, sprint_stream_t stream);

/* The same for `batch` replicas of one shape in one launch (one block per
 * problem): logits, labels, loss, dlogits are HOST arrays of `batch` device
 * pointers; problem g writes *loss[g] and dlogits[g]. batch = 0 is a no-op. */
int sprint_softmax_xent_batched(const float* const* logits, const int32_t* const* labels, float* const* loss,
                                float* const* dlogits, int batch, int N, int C, int reduction_sum,
                                sprint_stream_t stream);

/* ------------------------------------------------------------------------
 * GradBuf accumulation — ComputeUpdateVal + UpdateGradient of Algorithm 1:
 *   buf[i] = (first ? 0 : buf[i]) + alpha * grad[i],  i < n.
 * alpha = 1 stores raw gradients (eta applied at the update); alpha = -eta is
 * the report's own form. buf and grad: device fp32 [n]. */
int sprint_gradbuf_accumulate(float* buf, const float* grad, size_t n, float alpha, int first, sprint_stream_t stream);

/* ------------------------------------------------------------------------
 * Parameter-server apply — SumGradient + UpdateWeights of Algorithm 2 and
 * the DistBelief rule w' := w - eta*dw, over k pending gradient buffers
 * (n_push accumulation). With S[i] = sum_{j<k} bufs[j][i] (summed in j order):
 *   sgd:      w_out = w_in - eta*S
 *   momentum: v = nu*v - eta*S;             w_out = w_in + v
 *   adagrad:  G = G + S*S;                  w_out = w_in - eta*S/(sqrt(G) + eps)
 * bufs: HOST array of k device pointers, 1 <= k <= 16. w_in == w_out is
 * allowed (in place); writing a new ring slot (w_out != w_in) is the
 * versioned-weights use. v and G are updated in place. n may be 0. */
int sprint_apply_update_sgd(const float* w_in, float* w_out, const float* const* bufs, int k, size_t n, float eta,
                            sprint_stream_t stream);
int sprint_apply_update_momentum(const float* w_in, float* w_out, float* v, const float* const* bufs, int k,
                                 size_t n, float eta, float nu, sprint_stream_t stream);
int sprint_apply_update_adagrad(const float* w_in, float* w_out, float* G, const float* const* bufs, int k, size_t n,
                                float eta, float eps, sprint_stream_t stream);

/* The parameter-server apply by rule: opt (sprint_opt) picks SGD, momentum,
 * Adagrad (as above; nu_or_eps = nu or eps) or Nesterov momentum
 *   v = nu*v - eta*S;   w_out = w_in + nu*v - eta*S
 * (the pipelined-training page's appendices train with "SGD with Nesterov
 * momentum" and print no formula: this is the usual form in the units of the
 * momentum rule above). weight_decay (lambda) adds L2 decay at the server:
 * S <- S + lambda*w_in before the rule (0: off, and the results equal the
 * sprint_apply_update_sgd / _momentum / _adagrad calls bit for bit). state: v
 * (momentum, Nesterov) or G (Adagrad), NULL for SGD. Arguments otherwise as
 * the calls above. */
int sprint_apply_update(int opt, const float* w_in, float* w_out, float* state, const float* const* bufs, int k,
                        size_t n, float eta, float nu_or_eps, float weight_decay, sprint_stream_t stream);

/* The same update over n_total elements by rule `opt` (sprint_opt; nu_or_eps
 * = nu for momentum and Nesterov, eps for Adagrad, unused for SGD; weight
 * decay as sprint_apply_update), bit for bit what sprint_apply_update over
 * n_total computes, whose first
 * rows*cols elements are a row-major [rows][cols] weight matrix that is also
 * written transposed: wT_out[c*rows + r] = w_out[r*cols + c] (device
 * [cols][rows]: the copy the input-gradient GEMMs read, written in the same
 * pass instead of reading W' back). The elements after the matrix (a layer's
 * bias, following its weights) are updated without a transpose, in the same
 * launch. state: v or G (device [n_total], in place; NULL for SGD). wT_out
 * must not overlap the other arguments; w_out may equal w_in. 1 <= k <= 16,
 * rows, cols >= 1, n_total >= rows*cols. */
int sprint_apply_update_t(int opt, const float* w_in, float* w_out, float* wT_out, float* state,
                          const float* const* bufs, int k, int rows, int cols, size_t n_total, float eta,
                          float nu_or_eps, float weight_decay, sprint_stream_t stream);

/* ------------------------------------------------------------------------
 * Staleness schedule (host only) — the delays of asynchronous SGD ([S] Sec. 1,
 * Fig. 1; [DB]: replicas fetch w, push dw). out[t*replicas + r] = delay of
 * replica r at step t, in {0..max_delay}: z = the (t*replicas + r)-th output of
 * SplitMix64 seeded with `seed` (Steele, Lea & Flood 2014), delay =
 * ((z >> 32) * (max_delay + 1)) >> 32. Replica r then computes its gradient
 * on W(max(0, t - delay)).
 * out: HOST int32 [steps*replicas]. */
int sprint_staleness_schedule(uint64_t seed, int steps, int replicas, int max_delay, int32_t* out);

#ifdef __cplusplus
}
#endif

#endif /* SPRINT_H */
