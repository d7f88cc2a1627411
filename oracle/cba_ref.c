/*
 * cba_ref.c -- the oracle: a plain, slow, obviously-correct CPU reference of the
 * backward pass of a darknet/caffe-style convolutional layer.
 *
 *   activation gradient -> batch-norm backward (bias, scale, mean_delta,
 *   variance_delta, normalize_delta) -> weight gradient -> input gradient
 *   -> shortcut-delta add;
 * and the backward of three adjacent data-movement layers: the YOLO layer's
 * delta copy, the route layer's split of its delta, max pooling's scatter.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's
 * CPU-baseline leg load this library; the product (the CUDA library) never
 * calls it, links it or includes anything from it, and it includes nothing
 * from the product.
 *
 * Precision: every intermediate and every output is a double.  The float
 * entry points take the same fp32 bits the GPU sees and widen them first.
 *
 * Sources, cited as page title + section:
 *   [YOLO]  "YOLOv3反向传播原理 之 全流程源码分析" (YOLOv3 back-propagation,
 *           full-flow source analysis): §1.1 initialisation, §3.1
 *           backward_convolutional_layer, §3.2 im2col_cpu / col2im_cpu / gemm,
 *           §4 batch_normalize backward, §5 shortcut layer, §6 route layer,
 *           §7 activations; §2 the YOLO layer.
 *   [LENET] "【caffe源码研究】第四章：完整案例源码篇(5)：LeNet反向过程"
 *           (caffe LeNet backward): 第四层 Convolution, 第五层 Pooling,
 *           第七层 ReLU.
 *   [BNU]   "BatchNorm 理解" (understanding BatchNorm): BatchNormLayer
 *           Forward_cpu / Backward_cpu.
 *
 * Layout (all tensors): NCHW, batch-major; element (b, f, i) of a [batch][n][size]
 * tensor sits at i + size*(f + n*b) -- the index printed in backward_scale_cpu,
 * [YOLO] §4.  Weights are [K][C][R][S]; the im2col row of (c, r, s) is
 * c*R*S + r*S + s, [YOLO] §3.2 im2col_cpu.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* activation codes: the same numbers as the library's cba_act_t */
#define REF_ACT_LINEAR 0
#define REF_ACT_LEAKY 1
#define REF_ACT_LOGISTIC 2
#define REF_ACT_RELU 3
#define REF_ACT_RELIE 4
#define REF_ACT_RAMP 5
#define REF_ACT_TANH 6
#define REF_ACT_PLSE 7
#define REF_ACT_ELU 8
#define REF_ACT_SELU 9
#define REF_ACT_LHTAN 10
#define REF_ACT_HARDTAN 11
#define REF_ACT_LOGGY 12
#define REF_ACT_STAIR 13

/* batch_normalize: 0 no BN, 1 training mode (batch statistics), 2 frozen
 * statistics (the given mean/var are constants of the forward) */
#define REF_BN_NONE 0
#define REF_BN_BATCH 1
#define REF_BN_FROZEN 2

/* ------------------------------------------------------------------ threads */

void cba_ref_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int cba_ref_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* --------------------------------------------------------------- geometry */

/* Output size of a convolution: (H + 2*pad - R)/stride + 1 with C integer
 * (floor) division, as height_col / width_col in [YOLO] §3.2 im2col_cpu. */
int cba_ref_out_size(int in, int ksize, int stride, int pad) {
    return (in + 2 * pad - ksize) / stride + 1;
}

/* ------------------------------------------------------------- activation */

/* Activation derivative evaluated on the activation's OUTPUT value y, as
 * gradient_array does ([YOLO] §3.1 calls gradient_array(l.output, ...)).  The
 * *_gradient functions of [YOLO] §7, each as a function of y:
 *   linear 1; leaky y>0 ? 1 : .1; logistic (1-y)y; relu [y>0];
 *   relie y>0 ? 1 : .01; ramp [y>0] + .1; tanh 1 - y^2;
 *   plse y<0 or y>1 ? .01 : .125; elu [y>=0] + [y<0](y+1);
 *   selu [y>=0] 1.0507 + [y<0](y + 1.0507*1.6732);
 *   lhtan 0<y<1 ? 1 : .001; hardtan -1<y<1 ? 1 : 0;
 *   loggy with t = (y+1)/2: 2(1-t)t; stair floor(y) == y ? 0 : 1. */
double cba_ref_activation_gradient(int act, double y) {
    switch (act) {
    case REF_ACT_LINEAR: return 1.0;
    case REF_ACT_LEAKY: return (y > 0) ? 1.0 : 0.1;
    case REF_ACT_LOGISTIC: return (1.0 - y) * y;
    case REF_ACT_RELU: return (y > 0) ? 1.0 : 0.0;
    case REF_ACT_RELIE: return (y > 0) ? 1.0 : 0.01;
    case REF_ACT_RAMP: return ((y > 0) ? 1.0 : 0.0) + 0.1;
    case REF_ACT_TANH: return 1.0 - y * y;
    case REF_ACT_PLSE: return (y < 0 || y > 1) ? 0.01 : 0.125;
    case REF_ACT_ELU: return (y >= 0) ? 1.0 : y + 1.0;
    case REF_ACT_SELU: return (y >= 0) ? 1.0507 : y + 1.0507 * 1.6732;
    case REF_ACT_LHTAN: return (y > 0 && y < 1) ? 1.0 : 0.001;
    case REF_ACT_HARDTAN: return (y > -1 && y < 1) ? 1.0 : 0.0;
    case REF_ACT_LOGGY: {
        const double t = (y + 1.0) / 2.0;
        return 2.0 * (1.0 - t) * t;
    }
    case REF_ACT_STAIR: return (floor(y) == y) ? 0.0 : 1.0;
    default: return NAN;
    }
}

/* gradient_array: delta[i] *= f'(output[i]) -- [YOLO] §3.1 / §7.
 * For the linear activation output may be NULL (its value is not needed). */
void cba_ref_gradient_array(const double *output, long n, int act, double *delta) {
    for (long i = 0; i < n; ++i) {
        double y = output ? output[i] : 0.0;
        delta[i] *= cba_ref_activation_gradient(act, y);
    }
}

/* ---------------------------------------------------- batch-norm backward */

/* backward_bias: bias_updates[f] += sum over batch and spatial of delta.
 * Its body is not printed; the prose of [YOLO] §4 says every delta of a
 * channel is summed into the shared bias gradient, and [YOLO] §3.1 calls it
 * with (l.bias_updates, l.delta, l.batch, l.n, k). */
void cba_ref_backward_bias(double *bias_updates, const double *delta, int batch, int n, int size) {
    for (int f = 0; f < n; ++f) {
        double sum = 0.0;
        for (int b = 0; b < batch; ++b)
            for (int i = 0; i < size; ++i) sum += delta[i + (long)size * (f + (long)n * b)];
        bias_updates[f] += sum;
    }
}

/* x_norm = (x - mean) / sqrt(var + eps): the normalised pre-BN output that the
 * forward pass caches (forward_batchnorm_layer, [YOLO] §4; the eps-inside-sqrt
 * placement follows the backward code of [YOLO] §4 and Forward_cpu of [BNU]). */
void cba_ref_x_norm(const double *x, const double *mean, const double *variance, double eps,
                    int batch, int filters, int spatial, double *x_norm) {
    for (int b = 0; b < batch; ++b)
        for (int f = 0; f < filters; ++f) {
            double sd = sqrt(variance[f] + eps);
            for (int k = 0; k < spatial; ++k) {
                long index = (long)b * filters * spatial + (long)f * spatial + k;
                x_norm[index] = (x[index] - mean[f]) / sd;
            }
        }
}

/* backward_scale_cpu: scale_updates[f] += sum delta * x_norm  ([YOLO] §4). */
void cba_ref_backward_scale(const double *x_norm, const double *delta, int batch, int n, int size,
                            double *scale_updates) {
    for (int f = 0; f < n; ++f) {
        double sum = 0.0;
        for (int b = 0; b < batch; ++b)
            for (int i = 0; i < size; ++i) {
                long index = i + (long)size * (f + (long)n * b);
                sum += delta[index] * x_norm[index];
            }
        scale_updates[f] += sum;
    }
}

/* scale_bias(delta, scales): delta *= scales[f]  (step 1 of [YOLO] §4). */
void cba_ref_scale_bias(double *delta, const double *scales, int batch, int n, int size) {
    for (int b = 0; b < batch; ++b)
        for (int f = 0; f < n; ++f)
            for (int i = 0; i < size; ++i) delta[i + (long)size * (f + (long)n * b)] *= scales[f];
}

/* mean_delta_cpu: mean_delta[f] = (sum delta) * (-1/sqrt(var[f] + eps))
 * ([YOLO] §4).  Written as printed: the term variance_delta * sum(-2(x-mean))/m
 * of the full derivative is not part of it (it is zero when mean is the batch
 * mean of x). */
void cba_ref_mean_delta(const double *delta, const double *variance, double eps, int batch,
                        int filters, int spatial, double *mean_delta) {
    for (int i = 0; i < filters; ++i) {
        double s = 0.0;
        for (int j = 0; j < batch; ++j)
            for (int k = 0; k < spatial; ++k) s += delta[(long)j * filters * spatial + (long)i * spatial + k];
        mean_delta[i] = s * (-1.0 / sqrt(variance[i] + eps));
    }
}

/* variance_delta_cpu: variance_delta[f] = sum delta*(x - mean[f])
 *                     * (-1/2) * (var[f] + eps)^(-3/2)   ([YOLO] §4). */
void cba_ref_variance_delta(const double *x, const double *delta, const double *mean,
                            const double *variance, double eps, int batch, int filters,
                            int spatial, double *variance_delta) {
    for (int i = 0; i < filters; ++i) {
        double s = 0.0;
        for (int j = 0; j < batch; ++j)
            for (int k = 0; k < spatial; ++k) {
                long index = (long)j * filters * spatial + (long)i * spatial + k;
                s += delta[index] * (x[index] - mean[i]);
            }
        variance_delta[i] = s * (-0.5 * pow(variance[i] + eps, -1.5));
    }
}

/* normalize_delta_cpu: delta = delta / sqrt(var + eps)
 *                            + variance_delta * 2 (x - mean) / (spatial*batch)
 *                            + mean_delta / (spatial*batch)   ([YOLO] §4). */
void cba_ref_normalize_delta(const double *x, const double *mean, const double *variance,
                             const double *mean_delta, const double *variance_delta, double eps,
                             int batch, int filters, int spatial, double *delta) {
    double m = (double)spatial * (double)batch;
    for (int j = 0; j < batch; ++j)
        for (int f = 0; f < filters; ++f)
            for (int k = 0; k < spatial; ++k) {
                long index = (long)j * filters * spatial + (long)f * spatial + k;
                delta[index] = delta[index] * 1.0 / sqrt(variance[f] + eps) +
                               variance_delta[f] * 2.0 * (x[index] - mean[f]) / m + mean_delta[f] / m;
            }
}

/* backward_batchnorm_layer in training mode, the page's step order ([YOLO] §4):
 * backward_bias -> backward_scale -> scale_bias -> mean_delta -> variance_delta
 * -> normalize_delta.  x is the pre-BN conv output (l.x), x_norm its normalised
 * form (l.x_norm). */
int cba_ref_backward_batchnorm(const double *x, const double *x_norm, const double *mean,
                               const double *variance, const double *scales, double eps, int batch,
                               int n, int size, double *delta, double *bias_updates,
                               double *scale_updates) {
    double *md = (double *)malloc(sizeof(double) * n);
    double *vd = (double *)malloc(sizeof(double) * n);
    if (!md || !vd) { free(md); free(vd); return -1; }
    cba_ref_backward_bias(bias_updates, delta, batch, n, size);
    cba_ref_backward_scale(x_norm, delta, batch, n, size, scale_updates);
    cba_ref_scale_bias(delta, scales, batch, n, size);
    cba_ref_mean_delta(delta, variance, eps, batch, n, size, md);
    cba_ref_variance_delta(x, delta, mean, variance, eps, batch, n, size, vd);
    cba_ref_normalize_delta(x, mean, variance, md, vd, eps, batch, n, size, delta);
    free(md);
    free(vd);
    return 0;
}

/* Frozen statistics: the mean and variance are constants of the forward (caffe's
 * use_global_stats_, [BNU] Backward_cpu, "use_global_stats_为真时" branch), so
 * the normalisation is the per-channel affine map (x - mean) / sqrt(var + eps)
 * and its gradient is the incoming gradient divided by sqrt(var + eps).  The
 * steps: backward_bias and backward_scale as in training mode ([YOLO] §4; the
 * Scale layer's bias and scale gradients in caffe), scale_bias (the product
 * with gamma, [YOLO] §4), then the division of the use_global_stats branch. */
int cba_ref_backward_batchnorm_frozen(const double *x_norm, const double *variance,
                                      const double *scales, double eps, int batch, int n,
                                      int size, double *delta, double *bias_updates,
                                      double *scale_updates) {
    cba_ref_backward_bias(bias_updates, delta, batch, n, size);
    cba_ref_backward_scale(x_norm, delta, batch, n, size, scale_updates);
    cba_ref_scale_bias(delta, scales, batch, n, size);
    for (int b = 0; b < batch; ++b)
        for (int f = 0; f < n; ++f) {
            const double sd = sqrt(variance[f] + eps);
            for (int i = 0; i < size; ++i) delta[i + (long)size * (f + (long)n * b)] /= sd;
        }
    return 0;
}

/* The second, independent formulation of the same gradient: caffe's
 * BatchNormLayer::Backward_cpu ([BNU]), which has no scale (a separate Scale
 * layer multiplies by gamma before it).  With Y = x_norm and dY = top_diff:
 *     dX = (dY - mean(dY) - mean(dY . Y) . Y) / sqrt(var + eps),
 * means taken over batch and spatial per channel.  The steps below follow the
 * order of the printed code: sum(dY.Y) -> broadcast and multiply by Y -> add
 * sum(dY) -> dY - (.)/m -> divide by sqrt(var+eps). */
void cba_ref_bn_backward_caffe(const double *top_diff, const double *x_norm, const double *variance,
                               double eps, int num, int channels, int spatial, double *bottom_diff) {
    double m = (double)num * (double)spatial;
    for (int c = 0; c < channels; ++c) {
        double s_dyy = 0.0, s_dy = 0.0;
        for (int n = 0; n < num; ++n)
            for (int i = 0; i < spatial; ++i) {
                long idx = ((long)n * channels + c) * spatial + i;
                s_dyy += top_diff[idx] * x_norm[idx];
            }
        for (int n = 0; n < num; ++n)
            for (int i = 0; i < spatial; ++i) {
                long idx = ((long)n * channels + c) * spatial + i;
                bottom_diff[idx] = s_dyy * x_norm[idx];
            }
        for (int n = 0; n < num; ++n)
            for (int i = 0; i < spatial; ++i) {
                long idx = ((long)n * channels + c) * spatial + i;
                s_dy += top_diff[idx];
            }
        for (int n = 0; n < num; ++n)
            for (int i = 0; i < spatial; ++i) {
                long idx = ((long)n * channels + c) * spatial + i;
                bottom_diff[idx] += s_dy;
                bottom_diff[idx] = top_diff[idx] - bottom_diff[idx] / m;
                bottom_diff[idx] /= sqrt(variance[c] + eps);
            }
    }
}

/* --------------------------------------------------- convolution gradients */

/* Weight gradient as direct nested loops (no im2col buffer):
 *   dW[k][c][r][s] += sum_{n,p,q} delta[n][k][p][q] * x[n][c][p*st + r - pad][q*st + s - pad],
 * input pixels outside the image are zero.  This is what
 * gemm(0,1,m,n,k,1,delta_i,k,col_i,k,1,dW,n) summed over the images computes
 * in [YOLO] §3.1 (col_i = im2col of image i, §3.2), and what
 * caffe_cpu_gemm(NoTrans, Trans, ..., 1., top_diff, bottom_data, 1., weight_diff)
 * computes in [LENET] 第四层 Convolution; both accumulate (beta = 1). */
/* With groups ([YOLO] §3.1, the l.groups loop of backward_convolutional_layer):
 * output channel k belongs to group g = k / (K/groups) and sees only the
 * input channels g*C/groups .. (g+1)*C/groups - 1; W and dW are
 * [K][C/groups][R][S]. */
void cba_ref_conv_wgrad_g(const double *delta, const double *x, int N, int C, int H, int W,
                          int K, int R, int S, int stride, int pad, int groups, double *dW) {
    int P = cba_ref_out_size(H, R, stride, pad), Q = cba_ref_out_size(W, S, stride, pad);
    const int Cg = C / groups, Kg = K / groups;
#pragma omp parallel for schedule(dynamic)
    for (int k = 0; k < K; ++k)
        for (int cg = 0; cg < Cg; ++cg)
            for (int r = 0; r < R; ++r)
                for (int s = 0; s < S; ++s) {
                    const int c = (k / Kg) * Cg + cg;
                    double acc = 0.0;
                    for (int n = 0; n < N; ++n)
                        for (int p = 0; p < P; ++p) {
                            int h = p * stride + r - pad;
                            if (h < 0 || h >= H) continue;
                            const double *drow = delta + (((long)n * K + k) * P + p) * Q;
                            const double *xrow = x + (((long)n * C + c) * H + h) * W;
                            for (int q = 0; q < Q; ++q) {
                                int w = q * stride + s - pad;
                                if (w < 0 || w >= W) continue;
                                acc += drow[q] * xrow[w];
                            }
                        }
                    dW[(((long)k * Cg + cg) * R + r) * S + s] += acc;
                }
}

void cba_ref_conv_wgrad(const double *delta, const double *x, int N, int C, int H, int W, int K,
                        int R, int S, int stride, int pad, double *dW) {
    cba_ref_conv_wgrad_g(delta, x, N, C, H, W, K, R, S, stride, pad, 1, dW);
}

/* Input gradient written as a scatter, the shape of col2im_cpu
 * ([YOLO] §3.2): for every column row (c, r, s) of W^T.delta and every output
 * position (p, q), the value sum_k W[k][c][r][s]*delta[n][k][p][q] is ADDED
 * into image pixel (p*st + r - pad, q*st + s - pad) when that pixel lies
 * inside the image (col2im_add_pixel).  dx must hold the values to add onto
 * (zeros for a plain result). */
/* With groups: input channel c of group g = c / (C/groups) receives only from
 * the output channels of group g, through W[k][c - g*C/groups][r][s]. */
void cba_ref_conv_dgrad_g(const double *delta, const double *Wt, int N, int C, int H, int W,
                          int K, int R, int S, int stride, int pad, int groups, double *dx) {
    int P = cba_ref_out_size(H, R, stride, pad), Q = cba_ref_out_size(W, S, stride, pad);
    const int Cg = C / groups, Kg = K / groups;
#pragma omp parallel for schedule(dynamic)
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < C; ++c)
            for (int r = 0; r < R; ++r)
                for (int s = 0; s < S; ++s)
                    for (int k = (c / Cg) * Kg; k < (c / Cg + 1) * Kg; ++k) {
                        double wv = Wt[(((long)k * Cg + c % Cg) * R + r) * S + s];
                        for (int p = 0; p < P; ++p) {
                            int h = p * stride + r - pad;
                            if (h < 0 || h >= H) continue;
                            const double *drow = delta + (((long)n * K + k) * P + p) * Q;
                            double *xrow = dx + (((long)n * C + c) * H + h) * W;
                            for (int q = 0; q < Q; ++q) {
                                int w = q * stride + s - pad;
                                if (w < 0 || w >= W) continue;
                                xrow[w] += wv * drow[q];
                            }
                        }
                    }
}

void cba_ref_conv_dgrad(const double *delta, const double *Wt, int N, int C, int H, int W, int K,
                        int R, int S, int stride, int pad, double *dx) {
    cba_ref_conv_dgrad_g(delta, Wt, N, C, H, W, K, R, S, stride, pad, 1, dx);
}

/* axpy_cpu: y += alpha * x  ([YOLO] §2).  The shortcut layer passes its delta
 * on with it, and shortcut_cpu with equal shapes and s1 = 1 is the same add
 * ([YOLO] §5). */
void cba_ref_axpy(long n, double alpha, const double *x, double *y) {
    for (long i = 0; i < n; ++i) y[i] += alpha * x[i];
}

/* ------------------------------------------------------------- full chain */

/* The whole backward of one conv(+BN)+activation layer, in the order of
 * backward_convolutional_layer ([YOLO] §3.1):
 *   1. gradient_array(output, act, delta)
 *   2. batch_normalize ? backward_batchnorm_layer : backward_bias
 *      (batch_normalize = 2: the frozen-statistics form above)
 *   3. dW += delta . im2col(x)^T          (always accumulates)
 *   4. if prev_delta: prev_delta (= or +=) col2im(W^T . delta) + residual
 * Inputs are not modified (delta is copied first).  dW, db, dgamma always
 * accumulate.  prev_delta: accumulate = 0 writes dgrad + residual,
 * accumulate = 1 adds dgrad + residual onto the values it holds.  residual
 * (the shortcut delta of [YOLO] §5) may be NULL; prev_delta NULL skips the
 * input gradient (the `if (net.delta)` test of [YOLO] §3.1); dz_out, if not
 * NULL, receives the BN-input gradient (the delta the GEMMs consume).
 * groups (the l.groups loop of backward_convolutional_layer, [YOLO] §3.1):
 * W and dW are [K][C/groups][R][S]; output channel k only meets the input
 * channels of its group (cba_ref_conv_wgrad_g, cba_ref_conv_dgrad_g); the BN
 * steps are per output channel and do not see the groups.
 * Returns 0, or -1 on a bad argument or an allocation failure. */
int cba_ref_conv_bn_act_backward_grouped_f64(
    int N, int C, int H, int W, int K, int R, int S, int stride, int pad, int groups, int act,
    int batch_normalize, int accumulate, double eps, const double *x, const double *output,
    const double *z, const double *delta, const double *Wt, const double *gamma,
    const double *mean, const double *var, const double *residual, double *dW, double *db,
    double *dgamma, double *prev_delta, double *dz_out) {
    if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || K <= 0 || R <= 0 || S <= 0 || stride <= 0 || pad < 0)
        return -1;
    if (groups < 1 || C % groups != 0 || K % groups != 0) return -1;
    if (batch_normalize < REF_BN_NONE || batch_normalize > REF_BN_FROZEN) return -1;
    if (act < REF_ACT_LINEAR || act > REF_ACT_STAIR) return -1;
    int P = cba_ref_out_size(H, R, stride, pad), Q = cba_ref_out_size(W, S, stride, pad);
    if (P <= 0 || Q <= 0) return -1;
    if (!x || !delta || !Wt || !dW || !db) return -1;
    if (act != REF_ACT_LINEAR && !output) return -1;
    if (batch_normalize && (!z || !gamma || !mean || !var || !dgamma)) return -1;
    long nout = (long)N * K * P * Q, nin = (long)N * C * H * W;
    double *d = (double *)malloc(sizeof(double) * nout);
    if (!d) return -1;
    memcpy(d, delta, sizeof(double) * nout);

    cba_ref_gradient_array(output, nout, act, d);
    if (batch_normalize) {
        double *xn = (double *)malloc(sizeof(double) * nout);
        if (!xn) { free(d); return -1; }
        cba_ref_x_norm(z, mean, var, eps, N, K, P * Q, xn);
        int rc = batch_normalize == REF_BN_FROZEN
                     ? cba_ref_backward_batchnorm_frozen(xn, var, gamma, eps, N, K, P * Q, d, db,
                                                         dgamma)
                     : cba_ref_backward_batchnorm(z, xn, mean, var, gamma, eps, N, K, P * Q, d,
                                                  db, dgamma);
        free(xn);
        if (rc) { free(d); return -1; }
    } else {
        cba_ref_backward_bias(db, d, N, K, P * Q);
    }
    if (dz_out) memcpy(dz_out, d, sizeof(double) * nout);

    cba_ref_conv_wgrad_g(d, x, N, C, H, W, K, R, S, stride, pad, groups, dW);

    if (prev_delta) {
        double *dx = (double *)calloc((size_t)nin, sizeof(double));
        if (!dx) { free(d); return -1; }
        cba_ref_conv_dgrad_g(d, Wt, N, C, H, W, K, R, S, stride, pad, groups, dx);
        if (residual) cba_ref_axpy(nin, 1.0, residual, dx);
        if (!accumulate)
            for (long i = 0; i < nin; ++i) prev_delta[i] = 0.0;
        cba_ref_axpy(nin, 1.0, dx, prev_delta);
        free(dx);
    }
    free(d);
    return 0;
}

int cba_ref_conv_bn_act_backward_f64(int N, int C, int H, int W, int K, int R, int S, int stride,
                                     int pad, int act, int batch_normalize, int accumulate,
                                     double eps, const double *x, const double *output,
                                     const double *z, const double *delta, const double *Wt,
                                     const double *gamma, const double *mean, const double *var,
                                     const double *residual, double *dW, double *db,
                                     double *dgamma, double *prev_delta, double *dz_out) {
    return cba_ref_conv_bn_act_backward_grouped_f64(N, C, H, W, K, R, S, stride, pad, 1, act,
                                                    batch_normalize, accumulate, eps, x, output,
                                                    z, delta, Wt, gamma, mean, var, residual, dW,
                                                    db, dgamma, prev_delta, dz_out);
}

static double *widen(const float *src, long n) {
    if (!src) return NULL;
    double *d = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    if (!d) return NULL;
    for (long i = 0; i < n; ++i) d[i] = (double)src[i];
    return d;
}

/* Same as cba_ref_conv_bn_act_backward_grouped_f64, on the float inputs the GPU sees
 * (widened exactly to double).  Outputs are double. */
int cba_ref_conv_bn_act_backward_grouped(int N, int C, int H, int W, int K, int R, int S,
                                         int stride, int pad, int groups, int act,
                                         int batch_normalize, int accumulate, float eps,
                                         const float *x, const float *output, const float *z,
                                         const float *delta, const float *Wt, const float *gamma,
                                         const float *mean, const float *var,
                                         const float *residual, double *dW, double *db,
                                         double *dgamma, double *prev_delta, double *dz_out) {
    if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || K <= 0 || R <= 0 || S <= 0 || stride <= 0 || pad < 0)
        return -1;
    if (groups < 1 || C % groups != 0 || K % groups != 0) return -1;
    int P = cba_ref_out_size(H, R, stride, pad), Q = cba_ref_out_size(W, S, stride, pad);
    if (P <= 0 || Q <= 0) return -1;
    long nout = (long)N * K * P * Q, nin = (long)N * C * H * W,
         nw = (long)K * (C / groups) * R * S;
    double *dx_ = widen(x, nin), *dout = widen(output, nout), *dz = widen(z, nout);
    double *dd = widen(delta, nout), *dWt = widen(Wt, nw), *dg = widen(gamma, K);
    double *dm = widen(mean, K), *dv = widen(var, K), *dres = widen(residual, nin);
    int rc = cba_ref_conv_bn_act_backward_grouped_f64(
        N, C, H, W, K, R, S, stride, pad, groups, act, batch_normalize, accumulate, (double)eps,
        dx_, dout, dz, dd, dWt, dg, dm, dv, dres, dW, db, dgamma, prev_delta, dz_out);
    free(dx_); free(dout); free(dz); free(dd); free(dWt); free(dg); free(dm); free(dv); free(dres);
    return rc;
}

int cba_ref_conv_bn_act_backward(int N, int C, int H, int W, int K, int R, int S, int stride,
                                 int pad, int act, int batch_normalize, int accumulate, float eps,
                                 const float *x, const float *output, const float *z,
                                 const float *delta, const float *Wt, const float *gamma,
                                 const float *mean, const float *var, const float *residual,
                                 double *dW, double *db, double *dgamma, double *prev_delta,
                                 double *dz_out) {
    return cba_ref_conv_bn_act_backward_grouped(N, C, H, W, K, R, S, stride, pad, 1, act,
                                                batch_normalize, accumulate, eps, x, output, z,
                                                delta, Wt, gamma, mean, var, residual, dW, db,
                                                dgamma, prev_delta, dz_out);
}

/* Steps 1-2 of the chain alone (activation gradient, then BN backward or
 * backward_bias), on the float inputs: dz receives the BN-input gradient the
 * convolution GEMMs consume, db and dgamma accumulate.  Returns 0 or -1. */
int cba_ref_backward_dz(int N, int K, int P, int Q, int act, int batch_normalize, float eps,
                        const float *output, const float *z, const float *delta,
                        const float *gamma, const float *mean, const float *var, double *dz,
                        double *db, double *dgamma) {
    if (N <= 0 || K <= 0 || P <= 0 || Q <= 0 || !delta || !dz || !db) return -1;
    if (batch_normalize < REF_BN_NONE || batch_normalize > REF_BN_FROZEN) return -1;
    if (act < REF_ACT_LINEAR || act > REF_ACT_STAIR) return -1;
    if (act != REF_ACT_LINEAR && !output) return -1;
    if (batch_normalize && (!z || !gamma || !mean || !var || !dgamma)) return -1;
    long nout = (long)N * K * P * Q;
    double *y = widen(output, nout);
    for (long i = 0; i < nout; ++i) dz[i] = (double)delta[i];
    cba_ref_gradient_array(y, nout, act, dz);
    free(y);
    if (!batch_normalize) {
        cba_ref_backward_bias(db, dz, N, K, P * Q);
        return 0;
    }
    double *zz = widen(z, nout), *g = widen(gamma, K), *m = widen(mean, K), *v = widen(var, K);
    double *xn = (double *)malloc(sizeof(double) * nout);
    int rc = -1;
    if (zz && g && m && v && xn) {
        cba_ref_x_norm(zz, m, v, (double)eps, N, K, P * Q, xn);
        rc = batch_normalize == REF_BN_FROZEN
                 ? cba_ref_backward_batchnorm_frozen(xn, v, g, (double)eps, N, K, P * Q, dz, db,
                                                     dgamma)
                 : cba_ref_backward_batchnorm(zz, xn, m, v, g, (double)eps, N, K, P * Q, dz, db,
                                              dgamma);
    }
    free(zz); free(g); free(m); free(v); free(xn);
    return rc;
}

/* -------------------------------------------- adjacent data-movement layers */

/* backward_yolo_layer ([YOLO] §2): the YOLO layer's delta goes to the previous
 * layer's delta with one axpy of factor 1 over batch * inputs elements. */
void cba_ref_yolo_backward(const double *l_delta, long n, double *net_delta) {
    cba_ref_axpy(n, 1.0, l_delta, net_delta);
}

/* backward_route_layer ([YOLO] §6): the route layer's output is its inputs laid
 * one after the other per image (outputs = sum of input_sizes values per image).
 * For input i and image j, input_sizes[i] values at offset_i + j * outputs of
 * the route delta are added onto input i's delta at j * input_sizes[i];
 * offset_i is the sum of the earlier inputs' sizes. */
void cba_ref_route_backward(const double *route_delta, int batch, int n, const int *input_sizes,
                            double *const *input_deltas) {
    long outputs = 0;
    for (int i = 0; i < n; ++i) outputs += input_sizes[i];
    long offset = 0;
    for (int i = 0; i < n; ++i) {
        const int size = input_sizes[i];
        for (int j = 0; j < batch; ++j)
            cba_ref_axpy(size, 1.0, route_delta + offset + (long)j * outputs,
                         input_deltas[i] + (long)j * size);
        offset += size;
    }
}

/* Pooled size of caffe's PoolingLayer (Reshape): ceil((in + 2 pad - k) / stride)
 * + 1, less one when the last window would start inside the bottom padding. */
int cba_ref_pooled_size(int in, int k, int stride, int pad) {
    int out = (int)ceil((double)(in + 2 * pad - k) / stride) + 1;
    if (pad > 0 && (out - 1) * stride >= in + pad) --out;
    return out;
}

/* PoolingLayer::Backward_cpu for MAX pooling ([LENET] 第五层 Pooling): the
 * bottom gradient starts at zero and, plane by plane (n, c) and top position
 * (ph, pw) in order, gets top_diff added at the bottom index the forward pass
 * recorded in mask (h * width + w within the plane). */
void cba_ref_maxpool_backward(const double *top_diff, const int *mask, int num, int channels,
                              int height, int width, int pooled_h, int pooled_w,
                              double *bottom_diff) {
    const long bottom_plane = (long)height * width, top_plane = (long)pooled_h * pooled_w;
    for (long i = 0; i < (long)num * channels * bottom_plane; ++i) bottom_diff[i] = 0.0;
    for (int n = 0; n < num; ++n)
        for (int c = 0; c < channels; ++c) {
            const long plane = (long)n * channels + c;
            const double *td = top_diff + plane * top_plane;
            const int *mk = mask + plane * top_plane;
            double *bd = bottom_diff + plane * bottom_plane;
            for (int ph = 0; ph < pooled_h; ++ph)
                for (int pw = 0; pw < pooled_w; ++pw) {
                    const int index = ph * pooled_w + pw;
                    bd[mk[index]] += td[index];
                }
        }
}

/* ----------------------------------------- sampled outputs at full sizes */

/* One weight-gradient element from its definition (gather form):
 *   sum_{n,p,q} dz[n][k][p][q] * x[n][c][p*st + r - pad][q*st + s - pad]
 * for each flat index idx[i] = ((k*C + c)*R + r)*S + s.  dz is the BN-input
 * gradient of the chain (dz_out of the full chain).  out[i] receives the sum
 * (the caller adds the prior dW value for accumulation). */
void cba_ref_wgrad_at(const double *dz, const float *x, int N, int C, int H, int W, int K, int R,
                      int S, int stride, int pad, const long *idx, long count, double *out) {
    int P = cba_ref_out_size(H, R, stride, pad), Q = cba_ref_out_size(W, S, stride, pad);
#pragma omp parallel for schedule(dynamic)
    for (long i = 0; i < count; ++i) {
        long t = idx[i];
        int s = (int)(t % S); t /= S;
        int r = (int)(t % R); t /= R;
        int c = (int)(t % C); t /= C;
        int k = (int)t;
        double acc = 0.0;
        for (int n = 0; n < N; ++n)
            for (int p = 0; p < P; ++p) {
                int h = p * stride + r - pad;
                if (h < 0 || h >= H) continue;
                for (int q = 0; q < Q; ++q) {
                    int w = q * stride + s - pad;
                    if (w < 0 || w >= W) continue;
                    acc += dz[(((long)n * K + k) * P + p) * Q + q] *
                           (double)x[(((long)n * C + c) * H + h) * W + w];
                }
            }
        out[i] = acc;
    }
}

/* One input-gradient element from the definition of the transposed
 * convolution (gather form, the other loop structure from the scatter above):
 *   sum_{k,r,s} W[k][c][r][s] * dz[n][k][p][q]  over the (r, s) for which
 *   p = (h + pad - r)/st and q = (w + pad - s)/st are exact and in range,
 * for each flat index idx[i] = ((n*C + c)*H + h)*W + w; then the shortcut
 * residual (may be NULL) and, when accumulate != 0, the prior value prev_in
 * (may be NULL when accumulate == 0) are added. */
void cba_ref_dgrad_at(const double *dz, const float *Wt, const float *residual,
                      const float *prev_in, int accumulate, int N, int C, int H, int W, int K,
                      int R, int S, int stride, int pad, const long *idx, long count, double *out) {
    int P = cba_ref_out_size(H, R, stride, pad), Q = cba_ref_out_size(W, S, stride, pad);
    (void)N; /* the batch index comes from idx */
#pragma omp parallel for schedule(dynamic)
    for (long i = 0; i < count; ++i) {
        long t = idx[i];
        int w = (int)(t % W); t /= W;
        int h = (int)(t % H); t /= H;
        int c = (int)(t % C); t /= C;
        int n = (int)t;
        double acc = 0.0;
        for (int r = 0; r < R; ++r) {
            int ph = h + pad - r;
            if (ph < 0 || ph % stride) continue;
            int p = ph / stride;
            if (p >= P) continue;
            for (int s = 0; s < S; ++s) {
                int qw = w + pad - s;
                if (qw < 0 || qw % stride) continue;
                int q = qw / stride;
                if (q >= Q) continue;
                for (int k = 0; k < K; ++k)
                    acc += (double)Wt[(((long)k * C + c) * R + r) * S + s] *
                           dz[(((long)n * K + k) * P + p) * Q + q];
            }
        }
        if (residual) acc += (double)residual[idx[i]];
        if (accumulate && prev_in) acc += (double)prev_in[idx[i]];
        out[i] = acc;
    }
}
