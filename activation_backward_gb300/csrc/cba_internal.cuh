// cba_internal.cuh -- shared declarations of libcba's translation units:
// the per-call plan (geometry, workspace carve-up, launch shapes), the
// per-channel coefficient record, the device status word, and small device
// helpers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/cba.h"

namespace cba {

constexpr int kNumSMs = 152;  // GB300: 2 dies x 76 SMs (the plan uses the queried value)

// Device status bits (workspace word 0).
constexpr unsigned kStatusTimeout = 1u;

// Per-channel BN-backward coefficients, written by the finalize kernel and
// read by every GEMM operand transform:
//   dz = a * delta' + b + c * (z - mu)
struct __align__(16) Coef {
    float a, b, c, mu;
};

struct Plan {
    // geometry
    int N, C, H, W, K, R, S, stride, pad, P, Q;
    int PQ, HW, RS, CRS;
    // grouped convolution: output channel k meets the Cg input channels of its
    // group k / Kg; W and dW are [K][Cg][R][S].  The GEMM kernels compute the
    // dense K x C product (the weights they read are zero between groups) and
    // the kernels that read W or write dW map (k, c) with w_off below.
    int groups, Cg, Kg;
    long long m;  // N*P*Q: elements per output channel
    int act, accumulate, math;  // act: the activation the main kernels apply
    int act_in;   // the descriptor's activation (cba_act_t)
    bool act_pre; // act_in is neither LINEAR nor LEAKY: a gradient_array pass writes
                  // delta * f'(output) to off_dprime and the main kernels run LINEAR
    int bn;  // 0 no BN, 1 batch statistics, 2 frozen statistics
    float eps;
    int num_sms;
    // reduction pass: a block sums red_pln whole (n, k) planes of one channel,
    // or one of red_pieces slices of each of them; red_groups = ceil(N /
    // red_pln); groups * pieces partials per channel
    int red_pln, red_groups, red_pieces;
    // SIMT wgrad split-K
    int wg_splits;
    long long wg_chunk;  // reduction positions per split (multiple of the K tile)
    // tensor-core path
    int use_tc2;  // tensor cores (TF32 tcgen05 kernels); else the FFMA kernels
    int use_wnb;  // (with use_tc2) the weight gradient on batch-innermost layouts
                  // (cba_wgrad_nb.cu): x and dz re-laid out at off_xn / off_dzn
    int use_g1;   // (with use_tc2) 1x1 layers as plain GEMMs (cba_gemm1x1.cu), with
                  // dz also in [N][K][H*W] order at off_dzt
    // workspace layout (byte offsets from the base)
    // off_cnt: per-channel arrival counters of the reduction (zeroed with the
    // status word at the start of every call; clear_bytes covers both)
    // off_wgacc: the TMA-fed weight gradient's tile accumulators, inside the
    // cleared prefix (zeroed with the counters)
    size_t off_status, off_cnt, off_wgacc, clear_bytes, off_red, off_coef, off_wgpart, off_dzc,
        off_wr, off_dprime, total;
    // z-free calls (BN without z): z = conv(x, W) goes to off_z; total_z bytes.
    // fwd_tc: the forward runs on the tensor cores as the input gradient of a
    // virtual convolution (forward_desc), whose workspace starts at 0
    size_t off_z, total_z;
    bool fwd_tc;
    size_t off_xn, off_dzn;  // batch-innermost x and dz (use_wnb)
    size_t off_dzt;          // dz in [N][K][H*W] order (use_g1)
};

// Builds the plan; returns CBA_OK or a CBA_ERR_* code.
int make_plan(const cba_desc_t *d, Plan *p, int groups = 1);

// Offset of W[k][c - g*Cg][rs] (g = k / Kg, the group of output channel k) in
// the [K][Cg][R*S] weight layout, or -1 when input channel c is not in that
// group.  With one group: (k * C + c) * RS + rs.
__host__ __device__ __forceinline__ long long w_off(int k, int c, int rs, int Cg, int Kg, int RS) {
    const int cl = c - (k / Kg) * Cg;
    if (cl < 0 || cl >= Cg) return -1;
    return ((long long)k * Cg + cl) * RS + rs;
}
// The reduction pass's block shape (red_pln, red_groups, red_pieces): about
// 3.5 blocks per SM, at most max_parts partials per channel.
void plan_reduction(Plan *p, long long max_parts);

// ---- launchers (each returns cudaSuccess or the launch error) ----
// The reduction pass: db, dgamma and the per-channel coefficients.
cudaError_t launch_reduce(const Plan &p, const float *delta, const float *output, const float *z,
                          const float *gamma, const float *mean, const float *var, float *db,
                          float *dgamma, void *ws, cudaStream_t st, int *launches);

// The input gradient's weight repack, W [K][Cg][R][S] -> wr [R][S][C][Kw]
// (cba_repack.cuh).
struct RepackJob {
    const float *W;
    float *wr;
    int K, C, R, S, Kw, Cg, Kg;
};
// dz_out may be the delta buffer itself (an in-place transform).
cudaError_t launch_dz_out(const Plan &p, const float *delta, const float *output, const float *z,
                          const void *ws, float *dz_out, cudaStream_t st);
// z = conv(x, W), the pre-BN convolution output (cba_fwd.cu).
cudaError_t launch_conv_forward(const Plan &p, const float *x, const float *W, float *z,
                                cudaStream_t st, int *launches);
// For stride 1, square kernels and pad <= R - 1: the forward is the input
// gradient of the virtual convolution with C and K swapped, H x W = P x Q, pad
// R - 1 - pad and the weights flipped and transposed.  Returns false when the
// descriptor does not have that form.
bool forward_desc(const cba_desc_t &d, cba_desc_t *virt);
// z through the tensor-core input gradient of the virtual convolution (plan
// pv); ws is the call's workspace (pv's regions from offset 0); Cg, Kg: the
// real layer's input / output channels per group.
cudaError_t launch_conv_forward_tc(const Plan &pv, const float *x, const float *W, void *ws,
                                   float *z, int Cg, int Kg, cudaStream_t st, int *launches);
// Data-movement layers (cba_layers.cu).
int pooled_size(int in, int k, int stride, int pad);
cudaError_t launch_yolo_backward(const float *l_delta, float *net_delta, long long n,
                                 cudaStream_t st);
cudaError_t launch_route_backward(const float *route, int batch, int n, const long long *sizes,
                                  float *const *deltas, cudaStream_t st);
cudaError_t launch_maxpool_backward(const cba_pool_desc_t &d, int PH, int PW, const float *top,
                                    const int *mask, float *bottom, cudaStream_t st);
// gradient_array for the activations other than LINEAR and LEAKY (p.act_in):
// dprime[i] = delta[i] * f'(output[i]).  dprime may be the delta buffer.
cudaError_t launch_gradient_array(const Plan &p, const float *delta, const float *output,
                                  float *dprime, cudaStream_t st, int *launches);
cudaError_t launch_wgrad_simt(const Plan &p, const float *x, const float *delta,
                              const float *output, const float *z, float *dW, void *ws,
                              cudaStream_t st, int *launches);
cudaError_t launch_dgrad_simt(const Plan &p, const float *Wt, const float *delta,
                              const float *output, const float *z, const float *residual,
                              float *prev, const void *ws, cudaStream_t st, int *launches);
cudaError_t launch_splitk_reduce(const Plan &p, const float *part, int splits, float *dW,
                                 cudaStream_t st, int *launches);
cudaError_t launch_selftest_wait(unsigned timeout_us, void *ws, cudaStream_t st);
// Records `e` as the last CUDA error of the library; returns CBA_ERR_CUDA.
int report_cuda_error(cudaError_t e);
bool tc2_supported(const Plan &p);
size_t tc2_dzc_bytes(const Plan &p);
size_t tc2_wr_bytes(const Plan &p);
// dz pass: dz written channels-last with its zero border (dzc_geom's layout),
// and, when dzt is not NULL, also in the input's [N][K][P][Q] order.
cudaError_t launch_dzc(const Plan &p, const float *delta, const float *output, const float *z,
                       const void *ws, float *dzc, cudaStream_t st, int *launches,
                       float *dzt = nullptr);
// prev = residual (+ prev when accumulating): the shortcut pre-pass before an
// input gradient that adds its result at the L2.
cudaError_t launch_prev_init(const Plan &p, const float *residual, float *prev, cudaStream_t st,
                             int *launches);

// The geometry the TMA kernels see and the channels-last dz copy's layout:
// dzc [N][Pp][Qpp][Kp], data at row offset bd_lo and column offset bq_lo (zero
// border elsewhere).
struct DzcGeom {
    int He, We, Pe, Qe, Kp, Pp, Qpp, bd_lo, bq_lo;
};
DzcGeom dzc_geom(const Plan &p);
// Dense row-major fp32 tensor map (dims[0] innermost) with the given box;
// 128-byte swizzle or none.  `tmap` points to a CUtensorMap.
bool tma_encode_f32(void *tmap, const void *base, int rank, const uint64_t *dims,
                    const uint32_t *box, bool swizzle128);
// The same with the swizzle span in bytes: 0 (none), 64 or 128.
bool tma_encode_f32_swz(void *tmap, const void *base, int rank, const uint64_t *dims,
                        const uint32_t *box, int swizzle_bytes);
// Weight gradient on batch-innermost layouts (cba_wgrad_nb.cu): xn
// [nc][H][W][C][nb] and dzn [nc][P][Q][K][nb] (nb = 16 or 32 images, zeros past
// N), written by launch_layouts; tile accumulators of wgrad_nb_acc_bytes,
// zeroed before the call.
bool wgrad_nb_supported(const Plan &p);
size_t wgrad_nb_acc_bytes(const Plan &p);
size_t wgrad_nb_xn_bytes(const Plan &p);
size_t wgrad_nb_dzn_bytes(const Plan &p);
// rep: NULL, or the input gradient's weight repack, done by extra blocks of
// the accumulator-apply launch (cba_repack.cuh).
cudaError_t launch_wgrad_nb(const Plan &p, const float *xn, const float *dzn, float *dW, void *ws,
                            float *acc, const RepackJob *rep, cudaStream_t st, int *launches);
// The layout pass of that weight gradient, one launch: dz batch-innermost
// (dzn), channels-last with its zero border when dzc is not NULL (the layout
// of dzc_geom, read by the input gradient), x batch-innermost (xn), and, when
// rep is not NULL, the input gradient's weight repack (cba_repack.cuh).
cudaError_t launch_layouts(const Plan &p, const float *delta, const float *output,
                           const float *z, const float *x, const void *ws, float *dzn,
                           float *dzc, float *xn, const RepackJob *rep, cudaStream_t st,
                           int *launches);
// Both gradients of 1x1 stride-1 unpadded layers as plain TMA-fed GEMMs
// (cba_gemm1x1.cu): dzt is dz in [N][K][H*W] order, dzc the channels-last copy,
// wr the repacked weights (written by the weight-gradient launch when rep is
// not NULL).
bool gemm1x1_supported(const Plan &p);
size_t gemm1x1_dzt_bytes(const Plan &p);
cudaError_t launch_gemm1x1_wgrad(const Plan &p, const float *dzt, const float *x, float *dW,
                                 const void *ws, const RepackJob *rep, cudaStream_t st,
                                 int *launches);
cudaError_t launch_gemm1x1_dgrad(const Plan &p, const float *wr, const float *dzc,
                                 const float *residual, float *prev, void *ws, cudaStream_t st,
                                 int *launches);
// Weight gradient with TMA-fed input rows (cba_wgrad4.cu).
bool wgrad_tc4_supported(const Plan &p);
size_t wgrad_tc4_ws_bytes(const Plan &p);  // tile accumulators (0 if the shape is not covered)
cudaError_t launch_wgrad_tc4(const Plan &p, const float *x, const float *dzc, float *dW,
                             void *ws, const RepackJob *rep, cudaStream_t st, int *launches);
// wr must already hold the repacked weights (the weight gradient's launch
// writes them).
cudaError_t launch_dgrad_tc2(const Plan &p, const float *dzc, const float *residual, float *prev,
                             void *ws, const float *wr, cudaStream_t st, int *launches);

// Launches `kern` with programmatic stream serialisation: it may be scheduled
// while the previous kernel in the stream is still finishing (that kernel's
// blocks call griddep_launch_dependents), and it calls griddep_wait before it
// touches memory its predecessors read or write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename T>
inline T *ws_at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}
template <typename T>
inline const T *ws_at(const void *ws, size_t off) {
    return reinterpret_cast<const T *>(static_cast<const char *>(ws) + off);
}

// ---- device helpers ----

// Activation derivative on the activation's output value (leaky: y > 0 -> 1,
// else 0.1; linear: 1).
template <int ACT>
__device__ __forceinline__ float act_grad(float y) {
    if constexpr (ACT == CBA_ACT_LEAKY) {
        return y > 0.f ? 1.f : 0.1f;
    } else {
        return 1.f;
    }
}

// The BN-input gradient of one element from its raw inputs and the channel's
// coefficients.  Without BN, dz = delta'.
template <int ACT, bool BN>
__device__ __forceinline__ float dz_of(float d, float y, float zv, const Coef &cf) {
    float dp = d * act_grad<ACT>(y);
    if constexpr (BN) {
        return fmaf(cf.a, dp, fmaf(cf.c, zv - cf.mu, cf.b));
    } else {
        return dp;
    }
}

}  // namespace cba
