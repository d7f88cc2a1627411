// cba_reduce.cu -- the per-channel reduction pass of the BN / bias backward.
//
// One read sweep over delta (and output for leaky, z for BN) produces, per
// output channel k,
//   S1_k = sum_{n,p,q} delta'          (bias_updates, backward_bias)
//   S2_k = sum_{n,p,q} delta' * x_norm (scale_updates, backward_scale_cpu)
// with delta' = delta * f'(output) and x_norm = (z - mean)/sqrt(var + eps)
// ("YOLOv3反向传播原理 之 全流程源码分析" §3.1, §4).  These two sums are the
// only reductions the BN backward needs: mean_delta, variance_delta and
// normalize_delta collapse into the per-channel affine map
//   dz = a*delta' + b + c*(z - mean),  a = gamma/sigma, b = -a*S1/m,
//   c = -a*S2/(m*sigma),  sigma = sqrt(var + eps),  m = N*P*Q,
// which the finalize kernel computes once per channel for the GEMMs.
//
// Pass A: grid (splits, K); each block sums a contiguous slice of channel k
// (16-byte vector loads when P*Q is a multiple of 4), fp32 per thread, warp
// shuffles, then fp64 across warps; one fp64 partial pair per block.
// Pass B: one thread per channel adds the partials in a fixed order (fp64),
// updates db / dgamma and writes the coefficients.  Deterministic.
#include "cba_internal.cuh"

namespace cba {

namespace {

constexpr int kRedThreads = 256;

template <int ACT, bool BN>
__device__ __forceinline__ void acc1(float d, float y, float zv, float mu, float rs, float &s1,
                                     float &s2) {
    float dp = d * act_grad<ACT>(y);
    s1 += dp;
    if constexpr (BN) s2 = fmaf(dp, (zv - mu) * rs, s2);
}

template <int ACT, bool BN, bool VEC>
__global__ void __launch_bounds__(kRedThreads)
    bn_reduce_kernel(const float *__restrict__ delta, const float *__restrict__ output,
                     const float *__restrict__ z, const float *__restrict__ mean,
                     const float *__restrict__ var, float eps, int K, int PQ, long long m,
                     int splits, double2 *__restrict__ part) {
    const int k = blockIdx.y;
    const int sp = blockIdx.x;
    float mu = 0.f, rs = 0.f;
    if constexpr (BN) {
        mu = mean[k];
        rs = (float)(1.0 / sqrt((double)var[k] + (double)eps));
    }
    long long lo = (m * sp) / splits, hi = (m * (sp + 1)) / splits;
    if constexpr (VEC) {
        lo &= ~3LL;
        hi = (sp == splits - 1) ? m : (hi & ~3LL);
    }
    float s1 = 0.f, s2 = 0.f;
    if (lo < hi) {
        const int n0 = (int)(lo / PQ), n1 = (int)((hi - 1) / PQ);
        for (int n = n0; n <= n1; ++n) {
            const long long pl = (long long)n * PQ;
            const int j0 = (int)max(lo - pl, 0LL);
            const int j1 = (int)min(hi - pl, (long long)PQ);
            const long long base = ((long long)n * K + k) * PQ;
            if constexpr (VEC) {
                const float4 *d4 = reinterpret_cast<const float4 *>(delta + base);
                const float4 *y4 = reinterpret_cast<const float4 *>(output + base);
                const float4 *z4 = reinterpret_cast<const float4 *>(z + base);
                int v0 = j0 >> 2, v1 = j1 >> 2;  // both multiples of 4 here
                int v = v0 + threadIdx.x;
                for (; v + kRedThreads < v1; v += 2 * kRedThreads) {
                    float4 da = __ldg(d4 + v), db = __ldg(d4 + v + kRedThreads);
                    float4 ya = make_float4(0, 0, 0, 0), yb = ya, za = ya, zb = ya;
                    if constexpr (ACT == CBA_ACT_LEAKY) {
                        ya = __ldg(y4 + v);
                        yb = __ldg(y4 + v + kRedThreads);
                    }
                    if constexpr (BN) {
                        za = __ldg(z4 + v);
                        zb = __ldg(z4 + v + kRedThreads);
                    }
                    acc1<ACT, BN>(da.x, ya.x, za.x, mu, rs, s1, s2);
                    acc1<ACT, BN>(da.y, ya.y, za.y, mu, rs, s1, s2);
                    acc1<ACT, BN>(da.z, ya.z, za.z, mu, rs, s1, s2);
                    acc1<ACT, BN>(da.w, ya.w, za.w, mu, rs, s1, s2);
                    acc1<ACT, BN>(db.x, yb.x, zb.x, mu, rs, s1, s2);
                    acc1<ACT, BN>(db.y, yb.y, zb.y, mu, rs, s1, s2);
                    acc1<ACT, BN>(db.z, yb.z, zb.z, mu, rs, s1, s2);
                    acc1<ACT, BN>(db.w, yb.w, zb.w, mu, rs, s1, s2);
                }
                for (; v < v1; v += kRedThreads) {
                    float4 da = __ldg(d4 + v);
                    float4 ya = make_float4(0, 0, 0, 0), za = ya;
                    if constexpr (ACT == CBA_ACT_LEAKY) ya = __ldg(y4 + v);
                    if constexpr (BN) za = __ldg(z4 + v);
                    acc1<ACT, BN>(da.x, ya.x, za.x, mu, rs, s1, s2);
                    acc1<ACT, BN>(da.y, ya.y, za.y, mu, rs, s1, s2);
                    acc1<ACT, BN>(da.z, ya.z, za.z, mu, rs, s1, s2);
                    acc1<ACT, BN>(da.w, ya.w, za.w, mu, rs, s1, s2);
                }
            } else {
                for (int j = j0 + threadIdx.x; j < j1; j += kRedThreads) {
                    float d = __ldg(delta + base + j);
                    float y = 0.f, zv = 0.f;
                    if constexpr (ACT == CBA_ACT_LEAKY) y = __ldg(output + base + j);
                    if constexpr (BN) zv = __ldg(z + base + j);
                    acc1<ACT, BN>(d, y, zv, mu, rs, s1, s2);
                }
            }
        }
    }
    // block reduction: warp shuffles in fp32, then fp64 across warps
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        if constexpr (BN) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    __shared__ float w1[kRedThreads / 32], w2[kRedThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        w1[warp] = s1;
        w2[warp] = s2;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t1 = 0.0, t2 = 0.0;
#pragma unroll
        for (int i = 0; i < kRedThreads / 32; ++i) {
            t1 += (double)w1[i];
            t2 += (double)w2[i];
        }
        part[(size_t)sp * K + k] = make_double2(t1, t2);
    }
}

__global__ void bn_finalize_kernel(const double2 *__restrict__ part, int splits, int K, long long m,
                                   const float *__restrict__ gamma, const float *__restrict__ mean,
                                   const float *__restrict__ var, float eps, int bn,
                                   float *__restrict__ db, float *__restrict__ dgamma,
                                   Coef *__restrict__ coef) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= K) return;
    double S1 = 0.0, S2 = 0.0;
    for (int s = 0; s < splits; ++s) {
        double2 v = part[(size_t)s * K + k];
        S1 += v.x;
        S2 += v.y;
    }
    db[k] = (float)((double)db[k] + S1);
    Coef cf;
    if (bn) {
        dgamma[k] = (float)((double)dgamma[k] + S2);
        const double sd = sqrt((double)var[k] + (double)eps);
        const double a = (double)gamma[k] / sd;
        cf.a = (float)a;
        cf.b = (float)(-a * S1 / (double)m);
        cf.c = (float)(-a * S2 / ((double)m * sd));
        cf.mu = mean[k];
    } else {
        cf.a = 1.f;
        cf.b = 0.f;
        cf.c = 0.f;
        cf.mu = 0.f;
    }
    coef[k] = cf;
}

template <int ACT, bool BN>
__global__ void dz_out_kernel(const float *__restrict__ delta, const float *__restrict__ output,
                              const float *__restrict__ z, const Coef *__restrict__ coef, int K,
                              int PQ, long long total, float *__restrict__ out) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int k = (int)((i / PQ) % K);
        const Coef cf = coef[k];
        float y = (ACT == CBA_ACT_LEAKY) ? output[i] : 0.f;
        float zv = BN ? z[i] : 0.f;
        out[i] = dz_of<ACT, BN>(delta[i], y, zv, cf);
    }
}

template <int ACT, bool BN>
void launch_reduce_t(const Plan &p, const float *delta, const float *output, const float *z,
                     const float *mean, const float *var, double2 *part, cudaStream_t st) {
    dim3 grid(p.red_splits, p.K);
    if (p.PQ % 4 == 0)
        bn_reduce_kernel<ACT, BN, true><<<grid, kRedThreads, 0, st>>>(
            delta, output, z, mean, var, p.eps, p.K, p.PQ, p.m, p.red_splits, part);
    else
        bn_reduce_kernel<ACT, BN, false><<<grid, kRedThreads, 0, st>>>(
            delta, output, z, mean, var, p.eps, p.K, p.PQ, p.m, p.red_splits, part);
}

}  // namespace

cudaError_t launch_reduce(const Plan &p, const float *delta, const float *output, const float *z,
                          const float *gamma, const float *mean, const float *var, float *db,
                          float *dgamma, void *ws, cudaStream_t st, int *launches) {
    double2 *part = ws_at<double2>(ws, p.off_red);
    Coef *coef = ws_at<Coef>(ws, p.off_coef);
    const bool leaky = p.act == CBA_ACT_LEAKY;
    if (p.bn) {
        if (leaky) launch_reduce_t<CBA_ACT_LEAKY, true>(p, delta, output, z, mean, var, part, st);
        else launch_reduce_t<CBA_ACT_LINEAR, true>(p, delta, output, z, mean, var, part, st);
    } else {
        if (leaky) launch_reduce_t<CBA_ACT_LEAKY, false>(p, delta, output, z, mean, var, part, st);
        else launch_reduce_t<CBA_ACT_LINEAR, false>(p, delta, output, z, mean, var, part, st);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bn_finalize_kernel<<<(p.K + 127) / 128, 128, 0, st>>>(part, p.red_splits, p.K, p.m, gamma,
                                                           mean, var, p.eps, p.bn, db, dgamma,
                                                           coef);
    *launches += 2;
    return cudaGetLastError();
}

cudaError_t launch_dz_out(const Plan &p, const float *delta, const float *output, const float *z,
                          const void *ws, float *dz_out, cudaStream_t st) {
    const Coef *coef = ws_at<Coef>(ws, p.off_coef);
    long long total = (long long)p.N * p.K * p.PQ;
    int blocks = (int)std::min<long long>((total + 255) / 256, (long long)p.num_sms * 8);
    const bool leaky = p.act == CBA_ACT_LEAKY;
    if (p.bn) {
        if (leaky)
            dz_out_kernel<CBA_ACT_LEAKY, true><<<blocks, 256, 0, st>>>(delta, output, z, coef, p.K,
                                                                      p.PQ, total, dz_out);
        else
            dz_out_kernel<CBA_ACT_LINEAR, true><<<blocks, 256, 0, st>>>(delta, output, z, coef,
                                                                       p.K, p.PQ, total, dz_out);
    } else {
        if (leaky)
            dz_out_kernel<CBA_ACT_LEAKY, false><<<blocks, 256, 0, st>>>(delta, output, z, coef,
                                                                       p.K, p.PQ, total, dz_out);
        else
            dz_out_kernel<CBA_ACT_LINEAR, false><<<blocks, 256, 0, st>>>(delta, output, z, coef,
                                                                        p.K, p.PQ, total, dz_out);
    }
    return cudaGetLastError();
}

}  // namespace cba
