/*
 * cba.h -- C ABI of libcba: the backward pass of a darknet/caffe-style
 * convolutional layer (convolution + optional batch norm + activation) on
 * one NVIDIA GB300 (sm_103a).
 *
 * What one call computes (source pages cited by title and section):
 *
 *   delta'   = delta * f'(output)                    gradient_array, leaky
 *              f'(y) = (y > 0) ? 1 : 0.1, linear f' = 1
 *              ("YOLOv3反向传播原理 之 全流程源码分析" §3.1, §7)
 *   db      += sum_{n,p,q} delta'                    backward_bias (§3.1, §4)
 *   with batch norm (training-mode statistics mean, var; §4):
 *   dgamma  += sum_{n,p,q} delta' * x_norm           backward_scale_cpu
 *   dz       = normalize_delta(scale_bias(delta'))   mean_delta_cpu,
 *              variance_delta_cpu, normalize_delta_cpu; x_norm = (z - mean)
 *              / sqrt(var + eps)
 *   without batch norm: dz = delta'
 *   dW      += dz . im2col(x)^T                      gemm(0,1,...,1,...) of §3.1
 *   prev_delta (= or +=) col2im(W^T . dz) + residual gemm(1,0,...) + col2im_cpu
 *              of §3.1 / §3.2; residual = the shortcut-layer delta (§5)
 *
 * The batch-norm steps are evaluated in the algebraically equal form
 *   dz = a_k * delta' + b_k + c_k * (z - mean_k),
 *   a_k = gamma_k / sigma_k, b_k = -a_k * S1_k / m, c_k = -a_k * S2_k / (m sigma_k),
 *   sigma_k = sqrt(var_k + eps), S1 = sum delta', S2 = sum delta' * x_norm,
 * m = N*P*Q, which is also caffe's BatchNormLayer::Backward_cpu times gamma
 * ("BatchNorm 理解", Backward_cpu).
 *
 * Layouts: every tensor is contiguous fp32.  Activations are NCHW
 * (batch-major): x, residual, prev_delta are [N][C][H][W]; output, z, delta,
 * dz_out are [N][K][P][Q] with P = (H + 2 pad - R)/stride + 1 and
 * Q = (W + 2 pad - S)/stride + 1 (floor division, im2col_cpu of §3.2).
 * W and dW are [K][C][R][S]; gamma, mean, var, db, dgamma are [K].
 *
 * Ownership: every pointer is DEVICE memory owned by the caller.  The
 * library allocates nothing and frees nothing; scratch comes from the
 * caller's workspace (size from cba_workspace_bytes).  Calls are
 * stream-ordered and asynchronous: they enqueue kernels on `stream` (a
 * cudaStream_t; NULL = the legacy default stream) and return without
 * synchronising.  Two calls that share a workspace must not overlap in time.
 * cba_conv_bn_act_backward and its traced variant can be captured into a
 * CUDA graph (stream capture) and replayed on the same buffers; make one call
 * on the device before capturing (it sets per-kernel attributes).
 *
 * Errors: a negative return code; on any error nothing has been launched and
 * no output touched, except CBA_ERR_CUDA (a launch failed; the CUDA error is
 * cleared and recorded, see cba_last_cuda_error).  Device-side failures
 * (a bounded wait that ran out) are reported through cba_get_status.
 */
#ifndef CBA_H_
#define CBA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CBA_OK 0
#define CBA_ERR_ARG (-1)         /* bad dimension, NULL required pointer, P or Q <= 0 */
#define CBA_ERR_UNSUPPORTED (-2) /* shape beyond the library's limits (e.g. > 2^31 elements) */
#define CBA_ERR_ALIGN (-3)       /* a pointer not 16-byte aligned */
#define CBA_ERR_WORKSPACE (-4)   /* workspace NULL or smaller than cba_workspace_bytes() */
#define CBA_ERR_CUDA (-5)        /* a CUDA launch or runtime call failed */
#define CBA_ERR_DEVICE_TIMEOUT (-6) /* reported by cba_get_status: a device wait ran out */
#define CBA_ERR_SCRATCH_LIMIT (-7)  /* cba_bn_act_backward_noalloc: K > CBA_NOALLOC_MAX_K */

/* Activation of the layer; its gradient is evaluated on the output y, as the
 * *_gradient functions of "YOLOv3反向传播原理" §7 are (gradient_array, §3.1):
 *   LINEAR 1              LEAKY   y>0 ? 1 : .1       LOGISTIC (1-y)y
 *   RELU   [y>0]          RELIE   y>0 ? 1 : .01      RAMP     [y>0] + .1
 *   TANH   1 - y^2        PLSE    y<0 or y>1 ? .01 : .125
 *   ELU    [y>=0] + [y<0](y+1)    SELU [y>=0] 1.0507 + [y<0](y + 1.0507*1.6732)
 *   LHTAN  0<y<1 ? 1 : .001       HARDTAN -1<y<1 ? 1 : 0
 *   LOGGY  2(1-t)t, t = (y+1)/2   STAIR floor(y) == y ? 0 : 1
 * LINEAR and LEAKY are applied inside the reduction and GEMM operand passes;
 * the others by one extra elementwise pass that writes delta * f'(y) into the
 * workspace (cba_workspace_bytes counts it). */
typedef enum {
    CBA_ACT_LINEAR = 0, CBA_ACT_LEAKY = 1, CBA_ACT_LOGISTIC = 2, CBA_ACT_RELU = 3,
    CBA_ACT_RELIE = 4, CBA_ACT_RAMP = 5, CBA_ACT_TANH = 6, CBA_ACT_PLSE = 7, CBA_ACT_ELU = 8,
    CBA_ACT_SELU = 9, CBA_ACT_LHTAN = 10, CBA_ACT_HARDTAN = 11, CBA_ACT_LOGGY = 12,
    CBA_ACT_STAIR = 13
} cba_act_t;

/* Arithmetic of the two convolution GEMMs.  TF32: tensor cores (tcgen05,
 * inputs read as TF32, fp32 accumulation).  FFMA: fp32 fused multiply-add on
 * the CUDA cores.  The reductions and the BN transform are fp32 (with fp64
 * cross-block sums) in both modes. */
typedef enum { CBA_MATH_TF32 = 0, CBA_MATH_FFMA = 1 } cba_math_t;

typedef struct {
    int N, C, H, W;     /* layer input x: batch, channels, height, width */
    int K, R, S;        /* filters, kernel height, kernel width */
    int stride, pad;    /* the same in both spatial dimensions */
    int act;            /* cba_act_t */
    int batch_normalize;/* 0: no BN.  1: BN in training mode; mean/var are the batch
                           statistics ("YOLOv3反向传播原理" §4).  2: BN with frozen
                           statistics; mean/var are constants of the forward, so
                           the BN-input gradient is gamma * delta' / sqrt(var + eps)
                           (caffe use_global_stats, "BatchNorm 理解" Backward_cpu);
                           db and dgamma accumulate as in mode 1.  With BN, z,
                           gamma, mean, var and dgamma are used. */
    int accumulate;     /* prev_delta: 0 writes, 1 adds onto its contents */
    float eps;          /* BN epsilon inside the square root (1e-5 in darknet) */
    int math;           /* cba_math_t */
} cba_desc_t;

/* Bytes of scratch one call with this descriptor needs (0 if the descriptor is
 * invalid).  The workspace must be 256-byte aligned device memory. */
size_t cba_workspace_bytes(const cba_desc_t *d);

/* With CBA_WS_RECOMPUTE_Z: the bytes of a z-free call (BN on, z = NULL), which
 * recomputes z = conv(x, W) -- the pre-BN convolution output, stride and pad
 * of the descriptor, no bias; forward_convolutional_layer's W . im2col(x) of
 * "YOLOv3反向传播原理" §3.2 -- into the workspace before the backward.  With
 * flags = 0 the same as cba_workspace_bytes.  0 on an invalid descriptor or an
 * unknown flag. */
#define CBA_WS_RECOMPUTE_Z 1u
size_t cba_workspace_bytes_ex(const cba_desc_t *d, unsigned flags);

/* The backward of one conv(+BN)+activation layer; see the header comment.
 *   x        [N,C,H,W] layer input (darknet net.input); required
 *   output   [N,K,P,Q] post-activation output; required unless act = LINEAR
 *   z        [N,K,P,Q] pre-BN convolution output (darknet l.x); with BN, NULL
 *            recomputes it from x and W (the workspace must then hold
 *            cba_workspace_bytes_ex(d, CBA_WS_RECOMPUTE_Z) bytes); unused
 *            without BN
 *   delta    [N,K,P,Q] gradient at the output; required; NOT modified
 *   W        [K,C,R,S] weights; required
 *   gamma, mean, var [K] BN scale and statistics (batch_normalize 1: the
 *            batch's, biased variance; 2: the frozen ones); required iff BN
 *   residual [N,C,H,W] shortcut delta added into prev_delta; may be NULL
 *   dW       [K,C,R,S] += ; required
 *   db       [K]       += ; required
 *   dgamma   [K]       += ; required iff BN
 *   prev_delta [N,C,H,W] (= or += per accumulate); NULL skips the input
 *            gradient (darknet's `if (net.delta)` at the first layer)
 *   dz_out   [N,K,P,Q] optional debug copy of dz; usually NULL
 *   workspace, workspace_bytes: scratch, see cba_workspace_bytes
 *   stream   cudaStream_t to enqueue on
 * Returns CBA_OK or a negative CBA_ERR_* code. */
int cba_conv_bn_act_backward(const cba_desc_t *d, const float *x, const float *output,
                             const float *z, const float *delta, const float *W,
                             const float *gamma, const float *mean, const float *var,
                             const float *residual, float *dW, float *db, float *dgamma,
                             float *prev_delta, float *dz_out, void *workspace,
                             size_t workspace_bytes, void *stream);

/* Grouped convolution (the l.groups loop of backward_convolutional_layer,
 * "YOLOv3反向传播原理" §3.1): output channels in groups of K/groups, input
 * channels in groups of C/groups, output channel k meeting only the input
 * channels of its group.  W and dW are [K][C/groups][R][S]; every other
 * argument as for cba_conv_bn_act_backward (descriptor C and K are the totals,
 * both multiples of groups).  The call launches the same kernels as an
 * ungrouped one, once for all groups: the per-channel reductions do not
 * depend on the grouping, and the two convolution gradients run as the dense
 * K x C product with zero weights between groups (so their cost is that of
 * the ungrouped layer), dW receiving only the pairs within a group.  It needs
 * cba_workspace_bytes_grouped(d, groups, flags) bytes (flags as for
 * cba_workspace_bytes_ex: CBA_WS_RECOMPUTE_Z for calls without z).
 * groups = 1 is cba_conv_bn_act_backward.  CBA_ERR_ARG also when groups < 1
 * or does not divide C and K. */
int cba_conv_bn_act_backward_grouped(const cba_desc_t *d, int groups, const float *x,
                                     const float *output, const float *z, const float *delta,
                                     const float *W, const float *gamma, const float *mean,
                                     const float *var, const float *residual, float *dW,
                                     float *db, float *dgamma, float *prev_delta, float *dz_out,
                                     void *workspace, size_t workspace_bytes, void *stream);
size_t cba_workspace_bytes_grouped(const cba_desc_t *d, int groups, unsigned flags);
/* The same, for profiling: phase_events and launches as for
 * cba_conv_bn_act_backward_traced (below). */
int cba_conv_bn_act_backward_grouped_traced(const cba_desc_t *d, int groups, const float *x,
                                            const float *output, const float *z,
                                            const float *delta, const float *W,
                                            const float *gamma, const float *mean,
                                            const float *var, const float *residual, float *dW,
                                            float *db, float *dgamma, float *prev_delta,
                                            float *dz_out, void *workspace,
                                            size_t workspace_bytes, void *stream,
                                            void *const *phase_events, int *launches);

/* Same computation as cba_conv_bn_act_backward, for profiling.
 * phase_events: NULL, or an array of CBA_PHASE_EVENTS (5) cudaEvent_t created
 *   by the caller; the call records, all on `stream`:
 *     [0] before the reduction pass (after the workspace's counters are
 *         cleared; a call without z recomputes z after [0]),
 *     [1] after it: the per-channel coefficients are ready,
 *     [2] after the GEMM operand layout pass (dz written in the layouts the
 *         tensor-core GEMMs read, and x re-laid out where the weight gradient
 *         needs it; see cba_plan_info) -- right after [1] on the FFMA path,
 *         whose GEMMs transform delta as they load it,
 *     [3] after the weight gradient,
 *     [4] after the input gradient (right after [3] when prev_delta is NULL).
 *   Recording events between the kernels stops a kernel from starting while
 *   its predecessor drains, so traced calls can take slightly longer.
 * launches: NULL, or receives the number of kernels this call enqueued.
 * Return codes as cba_conv_bn_act_backward. */
int cba_conv_bn_act_backward_traced(const cba_desc_t *d, const float *x, const float *output,
                                    const float *z, const float *delta, const float *W,
                                    const float *gamma, const float *mean, const float *var,
                                    const float *residual, float *dW, float *db, float *dgamma,
                                    float *prev_delta, float *dz_out, void *workspace,
                                    size_t workspace_bytes, void *stream,
                                    void *const *phase_events, int *launches);

#define CBA_PHASE_EVENTS 5

/* Which kernels a call with this descriptor runs, and what its operand layout
 * pass moves: a host-side query that launches nothing (groups as for
 * cba_conv_bn_act_backward_grouped, 1 for an ungrouped layer; with_prev:
 * whether the call will compute prev_delta).  Fills *info and returns CBA_OK,
 * or CBA_ERR_ARG / CBA_ERR_UNSUPPORTED for a descriptor the backward call
 * would refuse.  The path depends on the descriptor and on whether the CUDA
 * driver offers tensor-map encoding (without a driver every call plans the
 * FFMA kernels). */
typedef enum {
    CBA_PATH_FFMA = 0,        /* both GEMMs on the CUDA cores, BN transform on load */
    CBA_PATH_TC_ROWS = 1,     /* tcgen05 TF32; weight gradient reads x rows by TMA
                                 (stride-1 3x3 and 1x1 layers whose input rows are
                                 16-byte strided; a 1x1 layer's plane is one row) */
    CBA_PATH_TC_BATCH_INNER = 2, /* tcgen05 TF32; weight gradient on batch-innermost
                                    copies of x and dz */
    CBA_PATH_TC_GEMM_1X1 = 3     /* tcgen05 TF32; 1x1 stride-1 unpadded layers with
                                    16-byte rows (H*W and C multiples of 4, one
                                    group): both gradients as plain TMA-fed GEMMs */
} cba_path_t;
typedef struct {
    int path;                      /* cba_path_t */
    long long layout_bytes_read;   /* the operand layout pass (phase events [1]..[2]) */
    long long layout_bytes_written;
} cba_plan_info_t;
int cba_plan_info(const cba_desc_t *d, int groups, int with_prev, cba_plan_info_t *info);

/* Reads (and clears) the device status word of a workspace after the work on
 * `stream` has finished: synchronises `stream`, then returns CBA_OK or
 * CBA_ERR_DEVICE_TIMEOUT (a bounded device wait ran out; the kernel stopped
 * early and its outputs are not valid), or CBA_ERR_CUDA. */
int cba_get_status(void *workspace, size_t workspace_bytes, void *stream);

/* Self-test of the bounded device wait: launches one block whose thread waits
 * on a barrier phase that never completes, with a limit of `timeout_us`
 * microseconds (1 .. 2,000,000).  The wait gives up and records
 * CBA_ERR_DEVICE_TIMEOUT in the workspace status (read it back with
 * cba_get_status).  Needs cba_workspace_bytes of any valid descriptor. */
int cba_selftest_bounded_wait(void *workspace, size_t workspace_bytes, unsigned timeout_us,
                              void *stream);

/* Largest K that cba_bn_act_backward_noalloc accepts (its static scratch). */
#define CBA_NOALLOC_MAX_K 16384

/* The activation-gradient and BN-backward pass of cba_conv_bn_act_backward
 * (db, dgamma and, optionally, dz) WITHOUT a workspace and without allocating.
 * No counterpart in the source pages: it exists for callers that cannot call
 * cudaMalloc where they run the backward and have no buffer to lend, e.g. a
 * plugin called from another runtime's enqueue hook (that runtime owns all
 * device memory and forbids allocation after start-up) or a latency-bounded
 * loop (cudaMalloc may synchronise the device).
 *
 * Scratch: one static 1 MiB device array inside the library, placed on every
 * device that loads the library and held until the process exits.  The first
 * call on each device looks up the array's address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  The
 * address is kept for the life of the process, so resetting the device
 * (cudaDeviceReset) after the first call is not supported.  All
 * calls on a device share the array and it keeps the last call's contents;
 * each call first clears the reduction's per-channel counters (4 * K bytes,
 * a memset on the stream) and writes every other word before reading it.
 * Calls that overlap on one device (other streams or host threads with no
 * ordering between them) race on it: order them, e.g. on one stream.
 *
 * Arguments as cba_conv_bn_act_backward (only N, K and the output size P, Q of
 * the descriptor matter; math is ignored):
 *   output [N,K,P,Q] required unless act = LINEAR; z, gamma, mean, var and
 *   dgamma required iff BN; delta required; db [K] += and dgamma [K] += ;
 *   dz_out [N,K,P,Q] receives dz when not NULL.  Device pointers, 16-byte
 *   aligned; stream = cudaStream_t on the device that holds delta (the call
 *   runs on that device).
 * Returns CBA_OK, CBA_ERR_ARG / CBA_ERR_ALIGN / CBA_ERR_UNSUPPORTED,
 * CBA_ERR_SCRATCH_LIMIT when K > CBA_NOALLOC_MAX_K (nothing is enqueued), or
 * CBA_ERR_CUDA. */
int cba_bn_act_backward_noalloc(const cba_desc_t *d, const float *output, const float *z,
                                const float *delta, const float *gamma, const float *mean,
                                const float *var, float *db, float *dgamma, float *dz_out,
                                void *stream);

/* ---- Backward of the data-movement layers next to the convolution ----
 * Same conventions as above: device pointers owned by the caller, enqueued on
 * `stream` (cudaStream_t, NULL = legacy default) without synchronising, no
 * allocation; on an error nothing is launched.  Returns CBA_OK or a code. */

/* YOLO layer ("YOLOv3反向传播原理 之 全流程源码分析" §2, backward_yolo_layer):
 * net_delta[i] += l_delta[i] for i < n (the layer's delta passed back with one
 * axpy of factor 1; n = batch * inputs).  l_delta and net_delta: fp32, n
 * elements each, not overlapping.  CBA_ERR_ARG: n < 0, or a NULL pointer with
 * n > 0. */
int cba_yolo_backward(const float *l_delta, float *net_delta, long long n, void *stream);

/* Most inputs a route layer may have in one call. */
#define CBA_ROUTE_MAX_INPUTS 8

/* Route layer (same page, §6, backward_route_layer).  Its output lays its
 * n_inputs inputs side by side per image: outputs = sum of input_sizes, and
 * route_delta is [batch][outputs].  For input i (offset_i = the sum of the
 * earlier sizes) and image j:
 *   input_deltas[i][j * input_sizes[i] + t] += route_delta[j * outputs + offset_i + t]
 * for t < input_sizes[i].  input_sizes and input_deltas are HOST arrays of
 * n_inputs entries; input_deltas[i] are DEVICE pointers ([batch][size_i] fp32),
 * pairwise disjoint and disjoint from route_delta.  CBA_ERR_ARG: batch < 1,
 * n_inputs outside 1..CBA_ROUTE_MAX_INPUTS, a size < 1, or a NULL pointer. */
int cba_route_backward(const float *route_delta, int batch, int n_inputs,
                       const long long *input_sizes, float *const *input_deltas, void *stream);

/* Max pooling ("LeNet反向过程" 第五层 Pooling, caffe PoolingLayer MAX): bottom
 * [N,C,H,W], top [N,C,PH,PW] with caffe's sizes PH = cba_pooled_size(H,
 * kernel_h, stride_h, pad_h) and PW likewise. */
typedef struct {
    int N, C, H, W;
    int kernel_h, kernel_w, stride_h, stride_w, pad_h, pad_w; /* 0 <= pad < kernel */
} cba_pool_desc_t;

/* caffe's pooled size: ceil((in + 2 pad - kernel) / stride) + 1, one less when
 * the last window would start in the bottom padding; -1 on bad arguments. */
int cba_pooled_size(int in, int kernel, int stride, int pad);

/* bottom_diff = 0, then bottom_diff[n][c][mask / W][mask % W] += top_diff for
 * every top element (mask[n][c][ph][pw] = h * W + w of the element the forward
 * took as the window's maximum).  Each bottom element is written once: it sums
 * the top gradients that point at it in ascending (ph, pw), the page's order.
 * A mask value outside its own window is ignored (never dereferenced).
 * top_diff fp32 and mask int32 [N,C,PH,PW], bottom_diff fp32 [N,C,H,W].
 * CBA_ERR_ARG: a non-positive size, kernel or stride, pad outside 0..kernel-1,
 * PH or PW < 1, a NULL pointer; CBA_ERR_UNSUPPORTED: N*C*H*W or N*C*PH*PW past
 * 2^62, H*W past 2^31. */
int cba_maxpool_backward(const cba_pool_desc_t *d, const float *top_diff, const int *mask,
                         float *bottom_diff, void *stream);

/* Human-readable text of a CBA_* code (static storage). */
const char *cba_error_string(int code);

/* The cudaError_t of the last CBA_ERR_CUDA in this process (0 if none). */
int cba_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int cba_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CBA_H_ */
