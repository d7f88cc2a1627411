// cba_api.cu -- the C ABI of libcba: argument checks, the per-call plan and
// workspace carve-up, and the launch sequence
//   reduction pass -> finalize -> wgrad -> dgrad (if prev_delta)
// on the caller's stream.  Nothing here allocates, frees or synchronises
// (except cba_get_status, which exists to synchronise).
#include <cmath>
#include <cstdint>
#include <cstring>

#include "cba_internal.cuh"
#include "cba_repack.cuh"

namespace cba {

namespace {

int g_last_cuda_error = 0;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace

void plan_reduction(Plan *p, long long max_parts) {
    const long long target = (long long)p->num_sms * 7 / 2;
    const long long pa = p->PQ % 4 == 0 ? p->PQ / 4 : p->PQ;  // accesses per plane
    long long groups = std::max(1LL, std::min<long long>(p->N, ceil_div(target, p->K)));
    groups = std::min(groups, std::max(1LL, max_parts));
    long long pln = ceil_div(p->N, groups);
    groups = ceil_div(p->N, pln);
    long long pieces = 1;
    if (groups * p->K * 2 < target) {  // too few planes: slice them as well
        pieces = std::min(ceil_div(target, groups * p->K), std::max(1LL, pa / 256));
        pieces = std::max(1LL, std::min(pieces, max_parts / groups));
    }
    p->red_pln = (int)pln;
    p->red_groups = (int)groups;
    p->red_pieces = (int)pieces;
}

int make_plan(const cba_desc_t *d, Plan *p, int groups) {
    if (!d || !p) return CBA_ERR_ARG;
    std::memset(p, 0, sizeof(*p));
    if (d->N <= 0 || d->C <= 0 || d->H <= 0 || d->W <= 0 || d->K <= 0 || d->R <= 0 ||
        d->S <= 0 || d->stride <= 0 || d->pad < 0)
        return CBA_ERR_ARG;
    if (groups < 1 || d->C % groups != 0 || d->K % groups != 0) return CBA_ERR_ARG;
    if (d->act < CBA_ACT_LINEAR || d->act > CBA_ACT_STAIR) return CBA_ERR_ARG;
    if (d->math != CBA_MATH_TF32 && d->math != CBA_MATH_FFMA) return CBA_ERR_ARG;
    if (d->batch_normalize < 0 || d->batch_normalize > 2) return CBA_ERR_ARG;
    if (d->accumulate != 0 && d->accumulate != 1) return CBA_ERR_ARG;
    if (d->batch_normalize && !(std::isfinite(d->eps) && d->eps >= 0.f)) return CBA_ERR_ARG;
    const long long P = (long long)(d->H + 2LL * d->pad - d->R) / d->stride + 1;
    const long long Q = (long long)(d->W + 2LL * d->pad - d->S) / d->stride + 1;
    if (d->H + 2LL * d->pad - d->R < 0 || d->W + 2LL * d->pad - d->S < 0 || P <= 0 || Q <= 0)
        return CBA_ERR_ARG;
    const long long lim = (1LL << 31) - 1;
    const long long nin = (long long)d->N * d->C * d->H * d->W;
    const long long nout = (long long)d->N * d->K * P * Q;
    const long long nw = (long long)d->K * d->C * d->R * d->S;
    if (nin > lim || nout > lim || nw > lim || d->pad > (1 << 20) || d->stride > (1 << 20))
        return CBA_ERR_UNSUPPORTED;

    p->N = d->N; p->C = d->C; p->H = d->H; p->W = d->W; p->K = d->K; p->R = d->R; p->S = d->S;
    p->groups = groups; p->Cg = d->C / groups; p->Kg = d->K / groups;
    p->stride = d->stride; p->pad = d->pad; p->P = (int)P; p->Q = (int)Q;
    p->PQ = (int)(P * Q); p->HW = d->H * d->W; p->RS = d->R * d->S; p->CRS = d->C * p->RS;
    p->m = (long long)d->N * P * Q;
    p->act_in = d->act;
    p->act_pre = d->act != CBA_ACT_LINEAR && d->act != CBA_ACT_LEAKY;
    p->act = p->act_pre ? CBA_ACT_LINEAR : d->act;
    p->bn = d->batch_normalize; p->accumulate = d->accumulate;
    p->math = d->math; p->eps = d->eps;
    p->num_sms = kNumSMs;

    plan_reduction(p, 1LL << 30);

    // SIMT wgrad: split the reduction so that ~4 blocks per SM exist
    const long long tiles = ceil_div(p->K, 64) * ceil_div(p->CRS, 64);
    long long sw = std::max(1LL, ceil_div((long long)p->num_sms * 4, tiles));
    sw = std::min(sw, std::max(1LL, ceil_div(p->m, 256)));
    long long chunk = ceil_div(ceil_div(p->m, sw), 16) * 16;
    p->wg_chunk = chunk;
    p->wg_splits = (int)ceil_div(p->m, chunk);

    // tensor cores: the weight gradient with TMA-fed input rows where it
    // applies (stride-1 3x3 and 1x1 layers with 16-byte-strided input rows; it
    // needs no re-laid-out x and measured faster there), the batch-innermost
    // one everywhere else
    const bool tc_math = p->math == CBA_MATH_TF32 && tc2_supported(*p);
    // 1x1 stride-1 layers with 16-byte rows: both gradients as plain GEMMs
    p->use_g1 = tc_math && gemm1x1_supported(*p);
    const bool w4 = tc_math && !p->use_g1 && wgrad_tc4_supported(*p);
    p->use_wnb = tc_math && !p->use_g1 && !w4 && wgrad_nb_supported(*p);
    p->use_tc2 = p->use_g1 || w4 || p->use_wnb;

    // workspace carve-up
    size_t off = 0;
    p->off_status = off;
    off = align_up(off + 256, 256);
    p->off_cnt = off;
    off = align_up(off + sizeof(unsigned) * (size_t)p->K, 256);
    p->off_wgacc = off;
    if (p->use_tc2 && !p->use_g1)
        off = align_up(off + (p->use_wnb ? wgrad_nb_acc_bytes(*p) : wgrad_tc4_ws_bytes(*p)), 256);
    p->clear_bytes = off;
    p->off_red = off;
    off = align_up(off + sizeof(float) * 2 * (size_t)p->red_groups * p->red_pieces * p->K, 256);
    p->off_coef = off;
    off = align_up(off + sizeof(Coef) * (size_t)p->K, 256);
    p->off_wgpart = off;
    if (!p->use_tc2)  // split-K partials of the SIMT weight gradient
        off = align_up(off + sizeof(float) * (size_t)p->wg_splits * p->K * p->CRS, 256);
    p->off_dzc = off;
    if (p->use_tc2) off = align_up(off + tc2_dzc_bytes(*p), 256);
    p->off_wr = off;
    if (p->use_tc2) off = align_up(off + tc2_wr_bytes(*p), 256);
    p->off_dprime = off;
    if (p->act_pre) off = align_up(off + sizeof(float) * (size_t)nout, 256);
    p->off_xn = off;
    if (p->use_wnb) off = align_up(off + wgrad_nb_xn_bytes(*p), 256);
    p->off_dzn = off;
    if (p->use_wnb) off = align_up(off + wgrad_nb_dzn_bytes(*p), 256);
    p->off_dzt = off;
    if (p->use_g1) off = align_up(off + gemm1x1_dzt_bytes(*p), 256);
    p->total = off;
    p->off_z = off;
    p->fwd_tc = false;
    if (p->bn) {
        cba_desc_t dv;
        Plan pv;
        if (d->math == CBA_MATH_TF32 && forward_desc(*d, &dv) && make_plan(&dv, &pv) == CBA_OK &&
            pv.use_tc2) {
            p->fwd_tc = true;
            p->off_z = align_up(std::max(off, pv.total), 256);
        }
    }
    p->total_z = p->bn ? align_up(p->off_z + sizeof(float) * (size_t)nout, 256) : off;
    return CBA_OK;
}

}  // namespace cba

using namespace cba;

namespace {

inline bool misaligned(const void *ptr) {
    return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0;
}

int fail_cuda(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return CBA_ERR_CUDA;
}

// Makes the device that holds `ptr` (the call's data; the stream must belong
// to the same device) current for this library's runtime, which keeps its own
// per-thread current device.  Without a pointer, the stream's device.  The
// pointer query is also legal while the stream is being captured into a CUDA
// graph, where asking the stream for its device is not.
cudaError_t select_device(cudaStream_t stream, const void *ptr) {
    int dev = -1;
    cudaError_t e = cudaSuccess;
    if (ptr) {
        cudaPointerAttributes a;
        e = cudaPointerGetAttributes(&a, ptr);
        if (e == cudaSuccess) dev = a.device;
    } else if (stream) {
        e = cudaStreamGetDevice(stream, &dev);
    }
    if (e != cudaSuccess) return e;
    if (dev < 0) return cudaSuccess;
    int cur = -1;
    e = cudaGetDevice(&cur);
    if (e == cudaSuccess && cur != dev) e = cudaSetDevice(dev);
    return e;
}

}  // namespace

namespace cba {
int report_cuda_error(cudaError_t e) { return fail_cuda(e); }
}  // namespace cba

extern "C" {

size_t cba_workspace_bytes(const cba_desc_t *d) {
    Plan p;
    if (make_plan(d, &p) != CBA_OK) return 0;
    return p.total;
}

size_t cba_workspace_bytes_ex(const cba_desc_t *d, unsigned flags) {
    Plan p;
    if (make_plan(d, &p) != CBA_OK || (flags & ~(unsigned)CBA_WS_RECOMPUTE_Z)) return 0;
    return (flags & CBA_WS_RECOMPUTE_Z) ? p.total_z : p.total;
}

}  // extern "C"

namespace {

struct Tracer {
    void *const *ev;
    cudaStream_t st;
    cudaError_t mark(int i) const {
        if (!ev) return cudaSuccess;
        return cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st);
    }
};

int backward_impl(const cba_desc_t *d, const float *x, const float *output, const float *z,
                  const float *delta, const float *Wt, const float *gamma, const float *mean,
                  const float *var, const float *residual, float *dW, float *db, float *dgamma,
                  float *prev_delta, float *dz_out, void *workspace, size_t workspace_bytes,
                  void *stream, void *const *events, int *launches, int groups = 1) {
    Plan p;
    int rc = make_plan(d, &p, groups);
    if (rc != CBA_OK) return rc;
    if (!x || !delta || !Wt || !dW || !db) return CBA_ERR_ARG;
    if (p.act_in != CBA_ACT_LINEAR && !output) return CBA_ERR_ARG;
    if (p.bn && (!gamma || !mean || !var || !dgamma)) return CBA_ERR_ARG;
    const bool z_free = p.bn && !z;  // z = conv(x, W) is recomputed into the workspace
    const void *ptrs[] = {x, output, z, delta, Wt, gamma, mean, var, residual,
                          dW, db, dgamma, prev_delta, dz_out};
    for (const void *q : ptrs)
        if (misaligned(q)) return CBA_ERR_ALIGN;
    if (!workspace || workspace_bytes < (z_free ? p.total_z : p.total)) return CBA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CBA_ERR_ALIGN;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Tracer tr{events, st};
    int n_launch = 0;
    cudaGetLastError();  // the launches below report only their own errors
    cudaError_t e = select_device(st, delta);
    if (e != cudaSuccess) return fail_cuda(e);
    // status word, reduction counters and weight-gradient accumulators
    e = cudaMemsetAsync(workspace, 0, p.clear_bytes, st);
    if (e == cudaSuccess) e = tr.mark(0);
    if (e == cudaSuccess && z_free) {
        float *zbuf = ws_at<float>(workspace, p.off_z);
        cba_desc_t dv;
        Plan pv;
        if (p.fwd_tc && forward_desc(*d, &dv) && make_plan(&dv, &pv) == CBA_OK) {
            e = launch_conv_forward_tc(pv, x, Wt, workspace, zbuf, p.Cg, p.Kg, st, &n_launch);
            // the forward's scratch may overlap the reduction counters: zero them
            // again (the status word keeps what the forward set)
            if (e == cudaSuccess)
                e = cudaMemsetAsync(ws_at<char>(workspace, p.off_cnt), 0,
                                    p.clear_bytes - p.off_cnt, st);
        } else {
            e = launch_conv_forward(p, x, Wt, zbuf, st, &n_launch);
        }
        z = zbuf;
    }
    if (e == cudaSuccess && p.act_pre) {
        // activations other than linear and leaky: delta' first, then the main
        // kernels run in linear mode on it
        float *dprime = ws_at<float>(workspace, p.off_dprime);
        e = launch_gradient_array(p, delta, output, dprime, st, &n_launch);
        delta = dprime;
    }
    if (e == cudaSuccess)
        e = launch_reduce(p, delta, output, z, gamma, mean, var, db, dgamma, workspace, st,
                          &n_launch);
    if (e == cudaSuccess && dz_out) {
        e = launch_dz_out(p, delta, output, z, workspace, dz_out, st);
        ++n_launch;
    }
    if (e == cudaSuccess) e = tr.mark(1);
    if (p.use_tc2) {
        // the GEMM operand layouts: dz channels-last for the input gradient
        // (and for the weight gradient with TMA-fed rows); x and dz
        // batch-innermost for the other weight gradient
        float *dzc = ws_at<float>(workspace, p.off_dzc);
        float *xn = ws_at<float>(workspace, p.off_xn), *dzn = ws_at<float>(workspace, p.off_dzn);
        float *dzt = ws_at<float>(workspace, p.off_dzt);
        const RepackJob rep = make_repack_job(p, Wt, ws_at<float>(workspace, p.off_wr));
        const RepackJob *repp = prev_delta ? &rep : nullptr;
        if (p.use_g1) {
            // dz in the input's order for the weight gradient and channels-last
            // for the input gradient, then two plain GEMMs
            if (e == cudaSuccess)
                e = launch_dzc(p, delta, output, z, workspace, dzc, st, &n_launch, dzt);
            if (e == cudaSuccess) e = tr.mark(2);
            if (e == cudaSuccess)
                e = launch_gemm1x1_wgrad(p, dzt, x, dW, workspace, repp, st, &n_launch);
            if (e == cudaSuccess) e = tr.mark(3);
            if (e == cudaSuccess && prev_delta)
                e = launch_gemm1x1_dgrad(p, ws_at<float>(workspace, p.off_wr), dzc, residual,
                                         prev_delta, workspace, st, &n_launch);
            if (e == cudaSuccess) e = tr.mark(4);
            if (launches) *launches = n_launch;
            if (e != cudaSuccess) return fail_cuda(e);
            return CBA_OK;
        }
        // the tensor-core input gradient reads repacked weights: written by
        // extra blocks of the weight gradient's accumulator-apply launch, a
        // latency-bound kernel where they cost little; on the batch-innermost
        // path, for weights of at most 2 MB, by extra blocks of the layout pass
        // instead (measured: the LeNet and YOLO-head steps 4-7 us faster that
        // way, the 4.7 MB repacks of the 3x3 layers 1-3 us slower)
        const bool rep_layouts =
            p.use_wnb && repp && (long long)p.K * p.Cg * p.R * p.S * 4 <= (2LL << 20);
        if (p.use_wnb) {
            if (e == cudaSuccess)
                e = launch_layouts(p, delta, output, z, x, workspace, dzn,
                                   prev_delta ? dzc : nullptr, xn, rep_layouts ? repp : nullptr,
                                   st, &n_launch);
        } else if (e == cudaSuccess) {
            e = launch_dzc(p, delta, output, z, workspace, dzc, st, &n_launch);
        }
        if (e == cudaSuccess) e = tr.mark(2);
        if (e == cudaSuccess)
            e = p.use_wnb ? launch_wgrad_nb(p, xn, dzn, dW, workspace,
                                            ws_at<float>(workspace, p.off_wgacc),
                                            rep_layouts ? nullptr : repp, st, &n_launch)
                          : launch_wgrad_tc4(p, x, dzc, dW, workspace, repp, st, &n_launch);
        if (e == cudaSuccess) e = tr.mark(3);
        if (e == cudaSuccess && prev_delta)
            e = launch_dgrad_tc2(p, dzc, residual, prev_delta, workspace,
                                 ws_at<float>(workspace, p.off_wr), st, &n_launch);
    } else {
        // the SIMT kernels apply the BN transform while they load delta
        if (e == cudaSuccess) e = tr.mark(2);
        if (e == cudaSuccess) e = launch_wgrad_simt(p, x, delta, output, z, dW, workspace, st,
                                                    &n_launch);
        if (e == cudaSuccess) e = tr.mark(3);
        if (e == cudaSuccess && prev_delta)
            e = launch_dgrad_simt(p, Wt, delta, output, z, residual, prev_delta, workspace, st,
                                  &n_launch);
    }
    if (e == cudaSuccess) e = tr.mark(4);
    if (launches) *launches = n_launch;
    if (e != cudaSuccess) return fail_cuda(e);
    return CBA_OK;
}

}  // namespace

extern "C" {

int cba_conv_bn_act_backward_grouped(const cba_desc_t *d, int groups, const float *x,
                                     const float *output, const float *z, const float *delta,
                                     const float *Wt, const float *gamma, const float *mean,
                                     const float *var, const float *residual, float *dW,
                                     float *db, float *dgamma, float *prev_delta, float *dz_out,
                                     void *workspace, size_t workspace_bytes, void *stream) {
    return backward_impl(d, x, output, z, delta, Wt, gamma, mean, var, residual, dW, db, dgamma,
                         prev_delta, dz_out, workspace, workspace_bytes, stream, nullptr,
                         nullptr, groups);
}

int cba_conv_bn_act_backward_grouped_traced(const cba_desc_t *d, int groups, const float *x,
                                            const float *output, const float *z,
                                            const float *delta, const float *Wt,
                                            const float *gamma, const float *mean,
                                            const float *var, const float *residual, float *dW,
                                            float *db, float *dgamma, float *prev_delta,
                                            float *dz_out, void *workspace,
                                            size_t workspace_bytes, void *stream,
                                            void *const *phase_events, int *launches) {
    return backward_impl(d, x, output, z, delta, Wt, gamma, mean, var, residual, dW, db, dgamma,
                         prev_delta, dz_out, workspace, workspace_bytes, stream, phase_events,
                         launches, groups);
}

size_t cba_workspace_bytes_grouped(const cba_desc_t *d, int groups, unsigned flags) {
    Plan p;
    if (make_plan(d, &p, groups) != CBA_OK || (flags & ~(unsigned)CBA_WS_RECOMPUTE_Z)) return 0;
    return (flags & CBA_WS_RECOMPUTE_Z) ? p.total_z : p.total;
}

int cba_conv_bn_act_backward(const cba_desc_t *d, const float *x, const float *output,
                             const float *z, const float *delta, const float *Wt,
                             const float *gamma, const float *mean, const float *var,
                             const float *residual, float *dW, float *db, float *dgamma,
                             float *prev_delta, float *dz_out, void *workspace,
                             size_t workspace_bytes, void *stream) {
    return backward_impl(d, x, output, z, delta, Wt, gamma, mean, var, residual, dW, db, dgamma,
                         prev_delta, dz_out, workspace, workspace_bytes, stream, nullptr,
                         nullptr);
}

int cba_conv_bn_act_backward_traced(const cba_desc_t *d, const float *x, const float *output,
                                    const float *z, const float *delta, const float *Wt,
                                    const float *gamma, const float *mean, const float *var,
                                    const float *residual, float *dW, float *db, float *dgamma,
                                    float *prev_delta, float *dz_out, void *workspace,
                                    size_t workspace_bytes, void *stream,
                                    void *const *phase_events, int *launches) {
    return backward_impl(d, x, output, z, delta, Wt, gamma, mean, var, residual, dW, db, dgamma,
                         prev_delta, dz_out, workspace, workspace_bytes, stream, phase_events,
                         launches);
}

int cba_plan_info(const cba_desc_t *d, int groups, int with_prev, cba_plan_info_t *info) {
    if (!info) return CBA_ERR_ARG;
    Plan p;
    const int rc = make_plan(d, &p, groups);
    if (rc != CBA_OK) return rc;
    info->path = !p.use_tc2  ? CBA_PATH_FFMA
                 : p.use_g1  ? CBA_PATH_TC_GEMM_1X1
                 : p.use_wnb ? CBA_PATH_TC_BATCH_INNER
                             : CBA_PATH_TC_ROWS;
    info->layout_bytes_read = 0;
    info->layout_bytes_written = 0;
    if (p.use_tc2) {
        // dz from delta (or the delta' pass's output), output (leaky) and z (BN)
        const long long out = (long long)sizeof(float) * p.N * p.K * p.PQ;
        const int reads = 1 + (p.act == CBA_ACT_LEAKY ? 1 : 0) + (p.bn ? 1 : 0);
        info->layout_bytes_read = reads * out;
        const long long dzc = (long long)tc2_dzc_bytes(p);
        if (p.use_wnb) {
            info->layout_bytes_read += (long long)sizeof(float) * p.N * p.C * p.HW;  // x
            info->layout_bytes_written = (long long)wgrad_nb_dzn_bytes(p) +
                                         (long long)wgrad_nb_xn_bytes(p) + (with_prev ? dzc : 0);
        } else if (p.use_g1) {
            info->layout_bytes_written = dzc + (long long)gemm1x1_dzt_bytes(p);
        } else {
            info->layout_bytes_written = dzc;
        }
    }
    return CBA_OK;
}

int cba_get_status(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace || workspace_bytes < 256) return CBA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned word = 0;
    cudaError_t e = select_device(st, workspace);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(word), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail_cuda(e);
    return (word & kStatusTimeout) ? CBA_ERR_DEVICE_TIMEOUT : CBA_OK;
}

int cba_selftest_bounded_wait(void *workspace, size_t workspace_bytes, unsigned timeout_us,
                              void *stream) {
    if (!workspace || workspace_bytes < 256) return CBA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CBA_ERR_ALIGN;
    if (timeout_us < 1 || timeout_us > 2000000) return CBA_ERR_ARG;
    cudaGetLastError();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = select_device(st, workspace);
    if (e == cudaSuccess) e = launch_selftest_wait(timeout_us, workspace, st);
    if (e != cudaSuccess) return fail_cuda(e);
    return CBA_OK;
}

const char *cba_error_string(int code) {
    switch (code) {
    case CBA_OK: return "ok";
    case CBA_ERR_ARG: return "invalid argument (dimension, flag or required pointer)";
    case CBA_ERR_UNSUPPORTED: return "unsupported shape (beyond the library's limits)";
    case CBA_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case CBA_ERR_WORKSPACE: return "workspace missing or smaller than cba_workspace_bytes()";
    case CBA_ERR_CUDA: return "CUDA launch or runtime error (see cba_last_cuda_error)";
    case CBA_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out; outputs are not valid";
    case CBA_ERR_SCRATCH_LIMIT:
        return "K exceeds CBA_NOALLOC_MAX_K, the static scratch of cba_bn_act_backward_noalloc";
    default: return "unknown error code";
    }
}

int cba_last_cuda_error(void) { return g_last_cuda_error; }

int cba_version(void) { return 100; }

int cba_yolo_backward(const float *l_delta, float *net_delta, long long n, void *stream) {
    if (n < 0 || (n > 0 && (!l_delta || !net_delta))) return CBA_ERR_ARG;
    if (n == 0) return CBA_OK;
    cudaGetLastError();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = select_device(st, net_delta);
    if (e == cudaSuccess) e = launch_yolo_backward(l_delta, net_delta, n, st);
    return e == cudaSuccess ? CBA_OK : fail_cuda(e);
}

int cba_route_backward(const float *route_delta, int batch, int n_inputs,
                       const long long *input_sizes, float *const *input_deltas, void *stream) {
    if (!route_delta || batch < 1 || n_inputs < 1 || n_inputs > CBA_ROUTE_MAX_INPUTS ||
        !input_sizes || !input_deltas)
        return CBA_ERR_ARG;
    long long outputs = 0;
    for (int i = 0; i < n_inputs; ++i) {
        if (input_sizes[i] < 1 || !input_deltas[i]) return CBA_ERR_ARG;
        if (input_sizes[i] > (1LL << 50) || outputs > (1LL << 52)) return CBA_ERR_UNSUPPORTED;
        outputs += input_sizes[i];
    }
    if (outputs > (1LL << 62) / batch) return CBA_ERR_UNSUPPORTED;
    cudaGetLastError();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = select_device(st, route_delta);
    if (e == cudaSuccess)
        e = launch_route_backward(route_delta, batch, n_inputs, input_sizes, input_deltas, st);
    return e == cudaSuccess ? CBA_OK : fail_cuda(e);
}

int cba_pooled_size(int in, int kernel, int stride, int pad) {
    return pooled_size(in, kernel, stride, pad);
}

int cba_maxpool_backward(const cba_pool_desc_t *d, const float *top_diff, const int *mask,
                         float *bottom_diff, void *stream) {
    if (!d || !top_diff || !mask || !bottom_diff) return CBA_ERR_ARG;
    if (d->N < 1 || d->C < 1 || d->H < 1 || d->W < 1 || d->kernel_h < 1 || d->kernel_w < 1 ||
        d->stride_h < 1 || d->stride_w < 1 || d->pad_h < 0 || d->pad_w < 0 ||
        d->pad_h >= d->kernel_h || d->pad_w >= d->kernel_w)
        return CBA_ERR_ARG;
    const int PH = pooled_size(d->H, d->kernel_h, d->stride_h, d->pad_h);
    const int PW = pooled_size(d->W, d->kernel_w, d->stride_w, d->pad_w);
    if (PH < 1 || PW < 1) return CBA_ERR_ARG;
    const long long planes = (long long)d->N * d->C;
    if ((long long)d->H * d->W >= (1LL << 31) || (long long)PH * PW >= (1LL << 31) ||
        planes > (1LL << 62) / ((long long)d->H * d->W) ||
        planes > (1LL << 62) / ((long long)PH * PW))
        return CBA_ERR_UNSUPPORTED;
    cudaGetLastError();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = select_device(st, bottom_diff);
    if (e == cudaSuccess) e = launch_maxpool_backward(*d, PH, PW, top_diff, mask, bottom_diff, st);
    return e == cudaSuccess ? CBA_OK : fail_cuda(e);
}

}  // extern "C"
