// cba_fwd.cu -- the convolution forward z = conv(x, W) (no bias), for calls
// that do not pass z, the pre-BN convolution output the BN backward reads
// (darknet's l.x, "YOLOv3反向传播原理 之 全流程源码分析" §3.1 / §4).  It is the
// forward_convolutional_layer product W . im2col(x) of that page (§3.2) as an
// implicit GEMM:
//   z[n][k][p][q] = sum_{c,r,s} W[k][c][r][s] x[n][c][p*st + r - pad][q*st + s - pad]
// with M = K output channels, N = the N*P*Q output positions, and the
// reduction over C*R*S; input pixels outside the image are zero.
//
// Register-tiled fp32 FMA: a 256-thread block computes 64 channels x 64
// positions (4 x 4 per thread) and walks the reduction in slices of 16,
// staging a W slice and an im2col slice of x in shared memory (double
// buffered: the loads of slice i + 1 are in registers while slice i is used).
#include <algorithm>
#include <cstdint>

#include "cba_internal.cuh"

namespace cba {

namespace {

constexpr int kFM = 64, kFN = 64, kFK = 16, kFThreads = 256;

struct FwdArgs {
    const float *x, *W;
    float *z;
    int C, H, Wd, K, R, S, stride, pad, P, Q, PQ, RS, CRS;
    int Cg, Kg;   // channels per group (W is [K][Cg][R][S])
    long long m;  // N * P * Q
};

__global__ void __launch_bounds__(kFThreads) conv_forward_kernel(const FwdArgs a) {
    __shared__ float As[2][kFK][kFM];      // W slice, [l][k]
    __shared__ float Bs[2][kFK][kFN + 4];  // im2col slice, [l][position]
    const int tid = threadIdx.x;
    const int k0 = blockIdx.y * kFM;
    const long long j0 = (long long)blockIdx.x * kFN;
    // loader roles: each thread stages 4 W values and 4 x values per slice
    const int a_k = tid >> 2, a_l = (tid & 3) * 4;     // W[k0 + a_k][l0 + a_l .. + 3]
    const int b_j = tid & 63, b_l = (tid >> 6) * 4;    // x column j0 + b_j, l0 + b_l .. + 3
    const long long jb = j0 + b_j;
    const bool jvalid = jb < a.m;
    int bn = 0, bp = 0, bq = 0;
    if (jvalid) {
        bn = (int)(jb / a.PQ);
        const int pq = (int)(jb - (long long)bn * a.PQ);
        bp = pq / a.Q;
        bq = pq - bp * a.Q;
    }
    const int h_base = bp * a.stride - a.pad, w_base = bq * a.stride - a.pad;
    const float *xn = a.x + (long long)bn * a.C * a.H * a.Wd;

    auto load = [&](int l0, float (&ra)[4], float (&rb)[4]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int l = l0 + a_l + e, k = k0 + a_k;
            float v = 0.f;
            if (l < a.CRS && k < a.K) {
                const int c = l / a.RS;
                const long long o = w_off(k, c, l - c * a.RS, a.Cg, a.Kg, a.RS);
                if (o >= 0) v = __ldg(a.W + o);
            }
            ra[e] = v;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int l = l0 + b_l + e;
            float v = 0.f;
            if (jvalid && l < a.CRS) {
                const int c = l / a.RS, rs = l - c * a.RS;
                const int r = rs / a.S, s = rs - r * a.S;
                const int h = h_base + r, w = w_base + s;
                if (h >= 0 && h < a.H && w >= 0 && w < a.Wd)
                    v = __ldg(xn + ((long long)c * a.H + h) * a.Wd + w);
            }
            rb[e] = v;
        }
    };
    auto store = [&](int buf, const float (&ra)[4], const float (&rb)[4]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) As[buf][a_l + e][a_k] = ra[e];
#pragma unroll
        for (int e = 0; e < 4; ++e) Bs[buf][b_l + e][b_j] = rb[e];
    };

    // compute roles: 16 x 16 threads, each 4 channels x 4 positions
    const int tk = (tid >> 4) * 4, tj = (tid & 15) * 4;
    float acc[4][4] = {};
    float ra[4], rb[4];
    load(0, ra, rb);
    store(0, ra, rb);
    __syncthreads();
    const int nslices = (a.CRS + kFK - 1) / kFK;
    for (int sl = 0; sl < nslices; ++sl) {
        const int buf = sl & 1;
        if (sl + 1 < nslices) load((sl + 1) * kFK, ra, rb);
#pragma unroll
        for (int l = 0; l < kFK; ++l) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = As[buf][l][tk + i];
#pragma unroll
            for (int i = 0; i < 4; ++i) bv[i] = Bs[buf][l][tj + i];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(av[i], bv[jj], acc[i][jj]);
        }
        if (sl + 1 < nslices) store(buf ^ 1, ra, rb);
        __syncthreads();
    }
    // z[n][k][p][q]
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const long long j = j0 + tj + jj;
        if (j >= a.m) continue;
        const int n = (int)(j / a.PQ);
        const int pq = (int)(j - (long long)n * a.PQ);
        float *zn = a.z + (long long)n * a.K * a.PQ + pq;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + tk + i;
            if (k < a.K) zn[(long long)k * a.PQ] = acc[i][jj];
        }
    }
}

// wr of the virtual convolution (K' = C, C' = K; [r][s][c'][k'], k' padded to
// Kw' = round4(K')): W'[k'][c'][r][s] = W[c'][k'][R-1-r][S-1-s], TF32-rounded
// (cvt.rna) as the input gradient's own weight repack rounds; zero between
// groups (Cg, Kg: the real layer's channels per group).
__global__ void __launch_bounds__(256)
    repack_flipped_kernel(const float *__restrict__ W, float *__restrict__ wr, int Kv, int Cv,
                          int R, int S, int Kw, int Cg, int Kg) {
    const long long total = (long long)R * S * Cv * Kw;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int kk = (int)(i % Kw);
        long long t = i / Kw;
        const int c = (int)(t % Cv);
        t /= Cv;
        const int s = (int)(t % S), r = (int)(t / S);
        float v = 0.f;
        const long long o =
            kk < Kv ? w_off(c, kk, (R - 1 - r) * S + (S - 1 - s), Cg, Kg, R * S) : -1;
        if (o >= 0) {
            uint32_t u;
            asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(W[o]));
            v = __uint_as_float(u);
        }
        wr[i] = v;
    }
}

}  // namespace

bool forward_desc(const cba_desc_t &d, cba_desc_t *v) {
    if (d.stride != 1 || d.R != d.S || d.pad > d.R - 1) return false;
    const long long P = (long long)d.H + 2LL * d.pad - d.R + 1;
    const long long Q = (long long)d.W + 2LL * d.pad - d.S + 1;
    if (P <= 0 || Q <= 0 || P > (1 << 30) || Q > (1 << 30)) return false;
    *v = d;
    v->C = d.K;          // the forward's output channels are the virtual input channels
    v->K = d.C;
    v->H = (int)P;
    v->W = (int)Q;
    v->pad = d.R - 1 - d.pad;
    v->act = CBA_ACT_LINEAR;
    v->batch_normalize = 0;
    v->accumulate = 0;   // z is written
    v->math = CBA_MATH_TF32;
    return true;
}

cudaError_t launch_conv_forward_tc(const Plan &pv, const float *x, const float *W, void *ws,
                                   float *z, int Cg, int Kg, cudaStream_t st, int *launches) {
    const int Kw = (pv.K + 3) / 4 * 4;
    float *wr = ws_at<float>(ws, pv.off_wr);
    const long long total = (long long)pv.R * pv.S * pv.C * Kw;
    const unsigned blocks = (unsigned)std::min<long long>((total + 255) / 256, 1024);
    repack_flipped_kernel<<<blocks, 256, 0, st>>>(W, wr, pv.K, pv.C, pv.R, pv.S, Kw, Cg, Kg);
    cudaError_t e = cudaGetLastError();
    *launches += 1;
    float *dzc = ws_at<float>(ws, pv.off_dzc);
    // x in the input gradient's channels-last, zero-bordered layout (the dz pass
    // with a linear activation and no BN passes its input through)
    if (e == cudaSuccess) e = launch_dzc(pv, x, nullptr, nullptr, ws, dzc, st, launches);
    if (e == cudaSuccess) e = launch_dgrad_tc2(pv, dzc, nullptr, z, ws, wr, st, launches);
    return e;
}

cudaError_t launch_conv_forward(const Plan &p, const float *x, const float *W, float *z,
                                cudaStream_t st, int *launches) {
    FwdArgs a;
    a.x = x; a.W = W; a.z = z;
    a.C = p.C; a.H = p.H; a.Wd = p.W; a.K = p.K; a.R = p.R; a.S = p.S;
    a.stride = p.stride; a.pad = p.pad; a.P = p.P; a.Q = p.Q; a.PQ = p.PQ; a.RS = p.RS;
    a.CRS = p.CRS; a.m = p.m; a.Cg = p.Cg; a.Kg = p.Kg;
    const long long gx = (p.m + kFN - 1) / kFN;
    if (gx > 0x7fffffffLL) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)gx, (unsigned)((p.K + kFM - 1) / kFM));
    conv_forward_kernel<<<grid, kFThreads, 0, st>>>(a);
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace cba
