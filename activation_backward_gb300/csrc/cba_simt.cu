// cba_simt.cu -- the two convolution gradients on the CUDA cores (fp32 FFMA).
//
// Used by CBA_MATH_FFMA (the 1e-5-accurate mode) and for shapes the tensor-core
// kernels do not take.  Both are implicit GEMMs: no im2col / col2im buffer is
// ever formed, and the BN/activation transform dz = a*delta' + b + c*(z - mu)
// is applied while the delta tile is loaded (the coefficients come from the
// reduction pass).
//
// wgrad: dW[k][crs] += sum_L dz[k][L] * col[crs][L], L = (n, p, q), the
//   gemm(0,1,...,beta=1) of backward_convolutional_layer ("YOLOv3反向传播原理
//   之 全流程源码分析" §3.1) over all images at once.  64x64 tiles, 16-deep
//   k-steps, 4x4 per thread; split over L into fp32 partials that a second
//   kernel adds into dW in a fixed order (fp64), so the result is
//   deterministic.
// dgrad: prev[n][c][h][w] = sum_{r,s,k} W[k][c][r][s] * dz[n][k][p][q] with
//   h = p*stride + r - pad, w = q*stride + s - pad -- the gather form of
//   col2im(W^T . dz) (§3.1, §3.2).  64 pixels x 64 channels per block; the
//   epilogue adds the shortcut residual and, if asked, the old prev_delta.
// Grouped layers (the l.groups loop of §3.1) run both as the dense product
// over all K x C channel pairs: dgrad reads zero for the weights between
// groups, and the split-K reduction adds only the pairs within a group to dW.
#include "cba_internal.cuh"

namespace cba {

namespace {

constexpr int TBM = 64, TBN = 64, TBK = 16, TTH = 256;

template <int ACT, bool BN>
__global__ void __launch_bounds__(TTH)
    wgrad_simt_kernel(const float *__restrict__ x, const float *__restrict__ delta,
                      const float *__restrict__ output, const float *__restrict__ z,
                      const Coef *__restrict__ coef, int C, int H, int W, int K, int R, int S,
                      int stride, int pad, int P, int Q, long long Ltot, long long chunk,
                      float *__restrict__ part) {
    __shared__ float As[TBK][TBM + 4];
    __shared__ float Bs[TBK][TBN + 4];
    const int PQ = P * Q, RS = R * S, CRS = C * RS;
    const int k0 = blockIdx.y * TBM, j0 = blockIdx.x * TBN;
    const long long L0 = (long long)blockIdx.z * chunk;
    const long long L1 = min(L0 + chunk, Ltot);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;

    // rows this thread loads: A rows k0 + ty + 16e, B rows j0 + ty + 16e
    Coef cf[4];
    int bc[4], br[4], bs[4];
    bool bok[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int k = k0 + ty + 16 * e;
        cf[e] = (k < K) ? coef[k] : Coef{0.f, 0.f, 0.f, 0.f};
        int crs = j0 + ty + 16 * e;
        bok[e] = crs < CRS;
        int cc = bok[e] ? crs : 0;
        bc[e] = cc / RS;
        br[e] = (cc % RS) / S;
        bs[e] = cc % S;
    }

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (long long L = L0; L < L1; L += TBK) {
        const long long Lp = L + tx;
        const bool vl = Lp < L1;
        const int n = vl ? (int)(Lp / PQ) : 0;
        const int jj = vl ? (int)(Lp - (long long)n * PQ) : 0;
        const int p = jj / Q, q = jj - (jj / Q) * Q;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = k0 + ty + 16 * e;
            float v = 0.f;
            if (vl && k < K) {
                const long long off = ((long long)n * K + k) * PQ + jj;
                float y = (ACT == CBA_ACT_LEAKY) ? __ldg(output + off) : 0.f;
                float zv = BN ? __ldg(z + off) : 0.f;
                v = dz_of<ACT, BN>(__ldg(delta + off), y, zv, cf[e]);
            }
            As[tx][ty + 16 * e] = v;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float v = 0.f;
            if (vl && bok[e]) {
                const int h = p * stride + br[e] - pad;
                const int w = q * stride + bs[e] - pad;
                if (h >= 0 && h < H && w >= 0 && w < W)
                    v = __ldg(x + (((long long)n * C + bc[e]) * H + h) * W + w);
            }
            Bs[tx][ty + 16 * e] = v;
        }
        __syncthreads();
#pragma unroll
        for (int l = 0; l < TBK; ++l) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[l][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[l][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *dst = part + (size_t)blockIdx.z * K * CRS;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = k0 + ty * 4 + i;
        if (k >= K) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int crs = j0 + tx * 4 + j;
            if (crs < CRS) dst[(size_t)k * CRS + crs] = acc[i][j];
        }
    }
}

// dW[i] += sum_s part[s][j], summed in a fixed order in fp64, where the
// partials are dense ([K][C*R*S], nel elements per split) and dW holds the
// pairs of one group ([K][Cg*R*S], ng elements): i = (k, cg, rs) reads
// j = (k, (k / Kg) * Cg + cg, rs).
__global__ void splitk_reduce_kernel(const float *__restrict__ part, int splits, long long nel,
                                     long long ng, int Cg, int Kg, int C, int RS,
                                     float *__restrict__ dW) {
    const long long CgRS = (long long)Cg * RS;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < ng;
         i += (long long)gridDim.x * blockDim.x) {
        const int k = (int)(i / CgRS);
        const long long j = (long long)k * C * RS + (long long)(k / Kg) * CgRS + (i - k * CgRS);
        double s = 0.0;
        for (int t = 0; t < splits; ++t) s += (double)part[(size_t)t * nel + j];
        dW[i] = (float)((double)dW[i] + s);
    }
}

template <int ACT, bool BN>
__global__ void __launch_bounds__(TTH)
    dgrad_simt_kernel(const float *__restrict__ Wt, const float *__restrict__ delta,
                      const float *__restrict__ output, const float *__restrict__ z,
                      const Coef *__restrict__ coef, int N, int C, int H, int W, int K, int R,
                      int S, int stride, int pad, int P, int Q, const float *__restrict__ residual,
                      float *__restrict__ prev, int accumulate, int Cg, int Kg) {
    __shared__ float As[TBK][TBM + 4];
    __shared__ float Bs[TBK][TBN + 4];
    const int HW = H * W, RS = R * S, KK = RS * K;
    const long long M = (long long)N * HW;
    const long long pix0 = (long long)blockIdx.x * TBM;
    const int c0 = blockIdx.y * TBN;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int pp = tid & 63, lrow = tid >> 6;  // loader: pixel pp, k-rows lrow + 4e

    const long long mypix = pix0 + pp;
    const bool pvalid = mypix < M;
    const int an = pvalid ? (int)(mypix / HW) : 0;
    const int ahw = pvalid ? (int)(mypix - (long long)an * HW) : 0;
    const int ah = ahw / W, aw = ahw - (ahw / W) * W;
    const int bcol = c0 + pp;

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int kk0 = 0; kk0 < KK; kk0 += TBK) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int l = lrow + 4 * e;
            const int kk = kk0 + l;
            float va = 0.f, vb = 0.f;
            if (kk < KK) {
                const int rs = kk / K, k = kk - (kk / K) * K;
                const int r = rs / S, s = rs - (rs / S) * S;
                if (pvalid) {
                    const int ph = ah + pad - r, pw = aw + pad - s;
                    if (ph >= 0 && pw >= 0 && (ph % stride) == 0 && (pw % stride) == 0) {
                        const int p = ph / stride, q = pw / stride;
                        if (p < P && q < Q) {
                            const long long off = (((long long)an * K + k) * P + p) * Q + q;
                            float y = (ACT == CBA_ACT_LEAKY) ? __ldg(output + off) : 0.f;
                            float zv = BN ? __ldg(z + off) : 0.f;
                            va = dz_of<ACT, BN>(__ldg(delta + off), y, zv, coef[k]);
                        }
                    }
                }
                if (bcol < C) {
                    const long long o = w_off(k, bcol, rs, Cg, Kg, RS);
                    if (o >= 0) vb = __ldg(Wt + o);
                }
            }
            As[l][pp] = va;
            Bs[l][pp] = vb;
        }
        __syncthreads();
#pragma unroll
        for (int l = 0; l < TBK; ++l) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[l][tx * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[l][ty * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long long pix = pix0 + tx * 4 + i;
        if (pix >= M) continue;
        const int n = (int)(pix / HW);
        const int hw = (int)(pix - (long long)n * HW);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + ty * 4 + j;
            if (c >= C) continue;
            const long long idx = ((long long)n * C + c) * HW + hw;
            float v = acc[i][j];
            if (residual) v += residual[idx];
            if (accumulate) v += prev[idx];
            prev[idx] = v;
        }
    }
}

}  // namespace

cudaError_t launch_wgrad_simt(const Plan &p, const float *x, const float *delta,
                              const float *output, const float *z, float *dW, void *ws,
                              cudaStream_t st, int *launches) {
    const Coef *coef = ws_at<Coef>(ws, p.off_coef);
    float *part = ws_at<float>(ws, p.off_wgpart);
    dim3 grid((p.CRS + TBN - 1) / TBN, (p.K + TBM - 1) / TBM, p.wg_splits);
    const bool leaky = p.act == CBA_ACT_LEAKY;
#define CBA_WG(A, B)                                                                             \
    wgrad_simt_kernel<A, B><<<grid, TTH, 0, st>>>(x, delta, output, z, coef, p.C, p.H, p.W, p.K, \
                                                  p.R, p.S, p.stride, p.pad, p.P, p.Q, p.m,     \
                                                  p.wg_chunk, part)
    if (p.bn) {
        if (leaky) CBA_WG(CBA_ACT_LEAKY, true);
        else CBA_WG(CBA_ACT_LINEAR, true);
    } else {
        if (leaky) CBA_WG(CBA_ACT_LEAKY, false);
        else CBA_WG(CBA_ACT_LINEAR, false);
    }
#undef CBA_WG
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
    return launch_splitk_reduce(p, part, p.wg_splits, dW, st, launches);
}

cudaError_t launch_splitk_reduce(const Plan &p, const float *part, int splits, float *dW,
                                 cudaStream_t st, int *launches) {
    const long long nel = (long long)p.K * p.CRS, ng = (long long)p.K * p.Cg * p.RS;
    int blocks = (int)std::min<long long>((ng + 255) / 256, (long long)p.num_sms * 8);
    splitk_reduce_kernel<<<blocks, 256, 0, st>>>(part, splits, nel, ng, p.Cg, p.Kg, p.C, p.RS,
                                                 dW);
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_dgrad_simt(const Plan &p, const float *Wt, const float *delta,
                              const float *output, const float *z, const float *residual,
                              float *prev, const void *ws, cudaStream_t st, int *launches) {
    const Coef *coef = ws_at<Coef>(ws, p.off_coef);
    const long long M = (long long)p.N * p.HW;
    dim3 grid((unsigned)((M + TBM - 1) / TBM), (p.C + TBN - 1) / TBN);
    const bool leaky = p.act == CBA_ACT_LEAKY;
#define CBA_DG(A, B)                                                                        \
    dgrad_simt_kernel<A, B><<<grid, TTH, 0, st>>>(Wt, delta, output, z, coef, p.N, p.C, p.H, \
                                                  p.W, p.K, p.R, p.S, p.stride, p.pad, p.P, \
                                                  p.Q, residual, prev, p.accumulate, p.Cg, \
                                                  p.Kg)
    if (p.bn) {
        if (leaky) CBA_DG(CBA_ACT_LEAKY, true);
        else CBA_DG(CBA_ACT_LINEAR, true);
    } else {
        if (leaky) CBA_DG(CBA_ACT_LEAKY, false);
        else CBA_DG(CBA_ACT_LINEAR, false);
    }
#undef CBA_DG
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace cba
