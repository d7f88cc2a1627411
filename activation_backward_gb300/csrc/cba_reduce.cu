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
// One kernel, a few blocks per channel: each block sums a contiguous slice of
// its channel with 16-byte vector loads when P*Q is a multiple of 4 (many in
// flight), fp32 per thread, warp shuffles, fp64 across warps, one fp64
// partial pair per block.  The last block of a channel adds the partials in a
// fixed order (fp64), updates db / dgamma and writes the coefficients.
// Deterministic.  The per-channel arrival counters must be zero when the
// kernel starts; the last block of each channel resets its own.
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

// Per-channel finalisation from the S1, S2 totals: db += S1, dgamma += S2 and
// the coefficients of dz = a*delta' + b + c*(z - mu).
__device__ __forceinline__ void finalize_channel(int k, double S1, double S2, long long m,
                                                 const float *__restrict__ gamma,
                                                 const float *__restrict__ mean,
                                                 const float *__restrict__ var, float eps, int bn,
                                                 float *__restrict__ db,
                                                 float *__restrict__ dgamma,
                                                 Coef *__restrict__ coef) {
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

// One block reduces slot j of channel k: the contiguous range j * L .. (j+1)
// * L - 1 of the channel's m elements in (n, p, q) order (L = m / splits,
// taken in 16-byte quads when P*Q is a multiple of 4; the range crosses the
// per-image planes, each quad's address is computed on its own).  Few blocks
// (a couple per SM), each looping over its range: per iteration every thread
// issues U loads per tensor back to back (addresses clamped into the range,
// values past its end zeroed), so enough bytes stay in flight to keep HBM
// busy.  Sums in fp32 per thread, warp shuffles, fp64 across warps.  The fp64
// partial pair goes to part[j][k]; the block that finishes a channel's last
// slot (counted in cnt[k], which it resets) adds the partials in order j = 0,
// 1, ... and finalises the channel.  Deterministic.
template <int ACT, bool BN, bool VEC>
__global__ void __launch_bounds__(kRedThreads)
    bn_reduce_kernel(const float *__restrict__ delta, const float *__restrict__ output,
                     const float *__restrict__ z, const float *__restrict__ gamma,
                     const float *__restrict__ mean, const float *__restrict__ var, float eps,
                     int K, int PQ, long long m, int splits, double2 *__restrict__ part,
                     unsigned *__restrict__ cnt, float *__restrict__ db,
                     float *__restrict__ dgamma, Coef *__restrict__ coef) {
    constexpr int U = 4;  // loads per tensor per thread in flight
    const int k = (int)(blockIdx.x / splits), j = (int)(blockIdx.x - (blockIdx.x / splits) * splits);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // 1/sigma in fp64, once per block (fp64 is slow on this part: not per thread)
    __shared__ float rs_sh;
    if (BN && tid == 0) rs_sh = (float)(1.0 / sqrt((double)var[k] + (double)eps));
    __syncthreads();
    const float mu = BN ? mean[k] : 0.f, rs = BN ? rs_sh : 0.f;
    const int W = VEC ? 4 : 1;                     // elements per access
    const int mw = (int)(m / W);                   // accesses in the channel
    const int pqw = PQ / W;                        // accesses per plane
    const int g0 = (int)((long long)mw * j / splits), g1 = (int)((long long)mw * (j + 1) / splits);
    // this thread's accesses g = g0 + tid + 256 t: plane n, offset o, tracked
    // incrementally (one division up front)
    int g = g0 + tid;
    int n = g / pqw, o = g - (g / pqw) * pqw;
    const size_t plane_stride = (size_t)K * pqw;   // accesses between planes n, n+1
    float s1 = 0.f, s2 = 0.f;
    while (g < g1) {
        size_t idx[U];
        bool in[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            in[u] = g < g1;
            idx[u] = (size_t)n * plane_stride + (size_t)k * pqw + (size_t)(in[u] ? o : 0);
            g += kRedThreads;
            o += kRedThreads;
            while (o >= pqw) {
                o -= pqw;
                ++n;
            }
        }
        if constexpr (VEC) {
            float4 dd[U], yy[U], zz[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t i = in[u] ? idx[u] : idx[0];
                dd[u] = __ldg(reinterpret_cast<const float4 *>(delta) + i);
                if constexpr (ACT == CBA_ACT_LEAKY) yy[u] = __ldg(reinterpret_cast<const float4 *>(output) + i);
                if constexpr (BN) zz[u] = __ldg(reinterpret_cast<const float4 *>(z) + i);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!in[u]) dd[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if constexpr (ACT != CBA_ACT_LEAKY) yy[u] = dd[u];
                if constexpr (!BN) zz[u] = dd[u];
                acc1<ACT, BN>(dd[u].x, yy[u].x, zz[u].x, mu, rs, s1, s2);
                acc1<ACT, BN>(dd[u].y, yy[u].y, zz[u].y, mu, rs, s1, s2);
                acc1<ACT, BN>(dd[u].z, yy[u].z, zz[u].z, mu, rs, s1, s2);
                acc1<ACT, BN>(dd[u].w, yy[u].w, zz[u].w, mu, rs, s1, s2);
            }
        } else {
            float dd[U], yy[U], zz[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t i = in[u] ? idx[u] : idx[0];
                dd[u] = __ldg(delta + i);
                yy[u] = ACT == CBA_ACT_LEAKY ? __ldg(output + i) : 0.f;
                zz[u] = BN ? __ldg(z + i) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!in[u]) dd[u] = 0.f;
                acc1<ACT, BN>(dd[u], yy[u], zz[u], mu, rs, s1, s2);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        if constexpr (BN) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    __shared__ float w1[kRedThreads / 32], w2[kRedThreads / 32];
    __shared__ unsigned last;
    if (lane == 0) {
        w1[warp] = s1;
        w2[warp] = s2;
    }
    __syncthreads();
    if (tid == 0) {
        double t1 = 0.0, t2 = 0.0;
#pragma unroll
        for (int i = 0; i < kRedThreads / 32; ++i) {
            t1 += (double)w1[i];
            t2 += (double)w2[i];
        }
        part[(size_t)j * K + k] = make_double2(t1, t2);
        __threadfence();
        last = atomicAdd(cnt + k, 1u) == (unsigned)(splits - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!last || warp != 0) return;
    // the channel's last block: every partial is visible (fence + counter)
    __threadfence();
    double S1 = 0.0, S2 = 0.0;
    for (int s0 = 0; s0 < splits; s0 += 32) {
        double2 v = make_double2(0.0, 0.0);
        if (s0 + lane < splits) v = __ldcg(part + (size_t)(s0 + lane) * K + k);
        const int cntv = min(32, splits - s0);
        for (int i = 0; i < cntv; ++i) {  // in order of j
            S1 += __shfl_sync(0xffffffffu, v.x, i);
            S2 += __shfl_sync(0xffffffffu, v.y, i);
        }
    }
    if (lane == 0) {
        cnt[k] = 0u;  // ready for the next call
        finalize_channel(k, S1, S2, m, gamma, mean, var, eps, BN ? 1 : 0, db, dgamma, coef);
    }
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
                     const float *gamma, const float *mean, const float *var, double2 *part,
                     unsigned *cnt, float *db, float *dgamma, Coef *coef, cudaStream_t st) {
    const unsigned grid = (unsigned)((long long)p.K * p.red_splits);
    if (p.PQ % 4 == 0)
        bn_reduce_kernel<ACT, BN, true><<<grid, kRedThreads, 0, st>>>(
            delta, output, z, gamma, mean, var, p.eps, p.K, p.PQ, p.m, p.red_splits, part, cnt,
            db, dgamma, coef);
    else
        bn_reduce_kernel<ACT, BN, false><<<grid, kRedThreads, 0, st>>>(
            delta, output, z, gamma, mean, var, p.eps, p.K, p.PQ, p.m, p.red_splits, part, cnt,
            db, dgamma, coef);
}

}  // namespace

cudaError_t launch_reduce(const Plan &p, const float *delta, const float *output, const float *z,
                          const float *gamma, const float *mean, const float *var, float *db,
                          float *dgamma, void *ws, cudaStream_t st, int *launches) {
    double2 *part = ws_at<double2>(ws, p.off_red);
    unsigned *cnt = ws_at<unsigned>(ws, p.off_cnt);
    Coef *coef = ws_at<Coef>(ws, p.off_coef);
    const bool leaky = p.act == CBA_ACT_LEAKY;
#define CBA_RED(A, B) \
    launch_reduce_t<A, B>(p, delta, output, z, gamma, mean, var, part, cnt, db, dgamma, coef, st)
    if (p.bn) {
        if (leaky) CBA_RED(CBA_ACT_LEAKY, true);
        else CBA_RED(CBA_ACT_LINEAR, true);
    } else {
        if (leaky) CBA_RED(CBA_ACT_LEAKY, false);
        else CBA_RED(CBA_ACT_LINEAR, false);
    }
#undef CBA_RED
    *launches += 1;
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
