// One kernel.  A block sums one piece of one channel: a group of whole
// (n, k) planes, or, when there are too few plane groups to fill the GPU, one
// slice of each plane of the group.  Loads are 16-byte vectors when P*Q is a
// multiple of 4, three per tensor in flight per thread; sums in fp32 per
// thread, warp shuffles, fp32 across warps (a few thousand terms per block),
// one float2 partial per block.  The block that finishes a channel's last
// piece (counted in cnt[k], acquire-release, which it resets) adds the
// partials in a fixed order in fp64 and finalises the channel in fp32 (fp64
// division and square root are slow on this part, and the coefficients are
// fp32 anyway).  Deterministic.  The per-channel arrival counters must be
// zero when the kernel starts.

#include "cba_internal.cuh"
#include "cba_ptx.cuh"

namespace cba {

namespace {

constexpr int kRedThreads = 256;
constexpr int kRedU = 4;  // vector loads per tensor per thread in flight

template <int ACT, bool BN>
__device__ __forceinline__ void acc1(float d, float y, float zv, float mu, float rs, float &s1,
                                     float &s2) {
    float dp = d * act_grad<ACT>(y);
    s1 += dp;
    if constexpr (BN) s2 = fmaf(dp, (zv - mu) * rs, s2);
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// The per-channel inputs and running outputs of the finalisation, read by
// thread 0 of every block when it starts (their loads overlap the block's
// streaming, so the block that finalises the channel only waits for the other
// blocks' partials).
struct ChanIn {
    float db, dgamma, gamma, mean, var;
};

// Per-channel finalisation from the S1, S2 totals: db += S1, dgamma += S2 and
// the coefficients of dz = a*delta' + b + c*(z - mu).  bn: 0 no BN, 1 batch
// statistics, 2 frozen statistics (mean and var are constants of the forward:
// the gradient is gamma * delta' / sigma, b = c = 0; caffe's use_global_stats
// branch of BatchNormLayer::Backward_cpu, "BatchNorm 理解").
__device__ __forceinline__ void finalize_channel(int k, double S1, double S2, long long m,
                                                 const ChanIn &in, float eps, int bn,
                                                 float *__restrict__ db,
                                                 float *__restrict__ dgamma,
                                                 Coef *__restrict__ coef) {
    db[k] = (float)((double)in.db + S1);
    Coef cf;
    if (bn) {
        dgamma[k] = (float)((double)in.dgamma + S2);
        const float sd = sqrtf(in.var + eps);
        const float a = in.gamma / sd;
        const float s1m = (float)(S1 / (double)m), s2m = (float)(S2 / (double)m);
        cf.a = a;
        cf.b = bn == 2 ? 0.f : -a * s1m;
        cf.c = bn == 2 ? 0.f : -a * s2m / sd;
        cf.mu = in.mean;
    } else {
        cf.a = 1.f;
        cf.b = 0.f;
        cf.c = 0.f;
        cf.mu = 0.f;
    }
    coef[k] = cf;
}

// Block b < K * groups * pieces: channel k = b / (groups * pieces), its
// piece and group gq = b % (groups * pieces) (piece fastest).  Group g holds
// planes g * pln .. min(N, (g + 1) * pln) - 1; piece q covers accesses q * L ..
// (q + 1) * L - 1 of each of its planes (L = ceil(accesses per plane /
// pieces)).  The channels go in ascending order, so the last ones read are
// still in L2 when the dz pass, which walks the channels in descending order,
// starts.
template <int ACT, bool BN, bool VEC>
__global__ void __launch_bounds__(kRedThreads)
    bn_reduce_kernel(const float *__restrict__ delta, const float *__restrict__ output,
                     const float *__restrict__ z, const float *__restrict__ gamma,
                     const float *__restrict__ mean, const float *__restrict__ var, float eps,
                     int N, int K, int PQ, long long m, int pln, int groups, int pieces,
                     float2 *__restrict__ part, unsigned *__restrict__ cnt,
                     float *__restrict__ db, float *__restrict__ dgamma,
                     Coef *__restrict__ coef, int bn_mode) {
    ptx::griddep_wait();
    const int parts = groups * pieces;
    const int k = (int)(blockIdx.x / parts);
    const int gq = (int)(blockIdx.x - (unsigned)k * parts);
    const int q = gq % pieces, grp = gq / pieces;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float mu = BN ? mean[k] : 0.f;
    const float rs = BN ? rsqrtf(var[k] + eps) : 0.f;
    ChanIn cin{};
    if (tid == 0) {
        cin.db = db[k];
        if constexpr (BN) {
            cin.dgamma = dgamma[k];
            cin.gamma = gamma[k];
            cin.mean = mu;
            cin.var = var[k];
        }
    }
    constexpr int W = VEC ? 4 : 1;            // elements per access
    const int pa = PQ / W;                    // accesses per plane
    const int L = (pa + pieces - 1) / pieces;
    const int a0 = q * L, a1 = min(pa, a0 + L);
    const int n0 = grp * pln, n1 = min(N, n0 + pln);
    float s1 = 0.f, s2 = 0.f;
    // the block's accesses (planes n0 .. n1 - 1, accesses a0 .. a1 - 1 of each)
    // as one flat sequence, so that every round keeps kRedU loads per tensor in
    // flight in every thread even when a plane is shorter than the block
    const int La = a1 - a0;
    const int total = La > 0 ? (n1 - n0) * La : 0;
    for (int base = tid; base < total; base += kRedThreads * kRedU) {
        size_t off[kRedU];
        bool in[kRedU];
#pragma unroll
        for (int u = 0; u < kRedU; ++u) {
            const int f = base + u * kRedThreads;
            in[u] = f < total;
            const int ff = in[u] ? f : 0;
            const int pl = ff / La;
            off[u] = ((size_t)(n0 + pl) * K + k) * pa + (a0 + ff - pl * La);
        }
        if constexpr (VEC) {
            const float4 *D = reinterpret_cast<const float4 *>(delta);
            const float4 *Y = reinterpret_cast<const float4 *>(output);
            const float4 *Z = reinterpret_cast<const float4 *>(z);
            float4 dd[kRedU], yy[kRedU], zz[kRedU];
#pragma unroll
            for (int u = 0; u < kRedU; ++u) {
                dd[u] = __ldg(D + off[u]);
                if constexpr (ACT == CBA_ACT_LEAKY) yy[u] = __ldg(Y + off[u]);
                if constexpr (BN) zz[u] = __ldg(Z + off[u]);
            }
#pragma unroll
            for (int u = 0; u < kRedU; ++u) {
                if (!in[u]) dd[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if constexpr (ACT != CBA_ACT_LEAKY) yy[u] = dd[u];
                if constexpr (!BN) zz[u] = dd[u];
                acc1<ACT, BN>(dd[u].x, yy[u].x, zz[u].x, mu, rs, s1, s2);
                acc1<ACT, BN>(dd[u].y, yy[u].y, zz[u].y, mu, rs, s1, s2);
                acc1<ACT, BN>(dd[u].z, yy[u].z, zz[u].z, mu, rs, s1, s2);
                acc1<ACT, BN>(dd[u].w, yy[u].w, zz[u].w, mu, rs, s1, s2);
            }
        } else {
            float dd[kRedU], yy[kRedU], zz[kRedU];
#pragma unroll
            for (int u = 0; u < kRedU; ++u) {
                dd[u] = in[u] ? __ldg(delta + off[u]) : 0.f;
                yy[u] = ACT == CBA_ACT_LEAKY ? __ldg(output + off[u]) : 0.f;
                zz[u] = BN ? __ldg(z + off[u]) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kRedU; ++u) acc1<ACT, BN>(dd[u], yy[u], zz[u], mu, rs, s1, s2);
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
    // this block's loads are done: the dz pass may be scheduled (it still
    // waits for this grid to complete before it reads anything)
    ptx::griddep_launch_dependents();
    const int nparts = groups * pieces;
    if (tid == 0) {
        float t1 = 0.f, t2 = 0.f;
#pragma unroll
        for (int i = 0; i < kRedThreads / 32; ++i) {
            t1 += w1[i];
            t2 += w2[i];
        }
        part[(size_t)gq * K + k] = make_float2(t1, t2);
        // release: the partial is visible to whichever block sees the count
        // complete; acquire: that block sees every other block's partial
        last = atom_add_acq_rel(cnt + k, 1u) == (unsigned)(nparts - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!last || warp != 0) return;
    double S1 = 0.0, S2 = 0.0;
    for (int s0 = 0; s0 < nparts; s0 += 32) {
        float2 v = make_float2(0.f, 0.f);
        if (s0 + lane < nparts) v = __ldcg(part + (size_t)(s0 + lane) * K + k);
        const int cntv = min(32, nparts - s0);
        for (int i = 0; i < cntv; ++i) {  // in the partials' order
            S1 += (double)__shfl_sync(0xffffffffu, v.x, i);
            S2 += (double)__shfl_sync(0xffffffffu, v.y, i);
        }
    }
    if (lane == 0) {
        cnt[k] = 0u;  // ready for the next call
        finalize_channel(k, S1, S2, m, cin, eps, BN ? bn_mode : 0, db, dgamma, coef);
    }
}

template <int ACT, bool BN>
__global__ void dz_out_kernel(const float *delta, const float *__restrict__ output,
                              const float *__restrict__ z, const Coef *__restrict__ coef, int K,
                              int PQ, long long total, float *out) {  // out may be delta
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
                     const float *gamma, const float *mean, const float *var, float2 *part,
                     unsigned *cnt, float *db, float *dgamma, Coef *coef, cudaStream_t st) {
    const unsigned grid = (unsigned)((long long)p.K * p.red_groups * p.red_pieces);
    if (p.PQ % 4 == 0)
        bn_reduce_kernel<ACT, BN, true><<<grid, kRedThreads, 0, st>>>(
            delta, output, z, gamma, mean, var, p.eps, p.N, p.K, p.PQ, p.m, p.red_pln,
            p.red_groups, p.red_pieces, part, cnt, db, dgamma, coef, p.bn);
    else
        bn_reduce_kernel<ACT, BN, false><<<grid, kRedThreads, 0, st>>>(
            delta, output, z, gamma, mean, var, p.eps, p.N, p.K, p.PQ, p.m, p.red_pln,
            p.red_groups, p.red_pieces, part, cnt, db, dgamma, coef, p.bn);
}

}  // namespace

cudaError_t launch_reduce(const Plan &p, const float *delta, const float *output, const float *z,
                          const float *gamma, const float *mean, const float *var, float *db,
                          float *dgamma, void *ws, cudaStream_t st, int *launches) {
    float2 *part = ws_at<float2>(ws, p.off_red);
    unsigned *cnt = ws_at<unsigned>(ws, p.off_cnt);
    Coef *coef = ws_at<Coef>(ws, p.off_coef);
    const bool leaky = p.act == CBA_ACT_LEAKY;
#define CBA_RED(A, B) \
    launch_reduce_t<A, B>(p, delta, output, z, gamma, mean, var, part, cnt, db, dgamma, coef, \
                          st)
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

// The activation derivative on the output y for the activations other than
// LINEAR and LEAKY: the *_gradient functions of "YOLOv3反向传播原理" §7.
__device__ __forceinline__ float act_grad_other(int act, float y) {
    switch (act) {
    case CBA_ACT_LOGISTIC: return (1.f - y) * y;
    case CBA_ACT_RELU: return y > 0.f ? 1.f : 0.f;
    case CBA_ACT_RELIE: return y > 0.f ? 1.f : 0.01f;
    case CBA_ACT_RAMP: return (y > 0.f ? 1.f : 0.f) + 0.1f;
    case CBA_ACT_TANH: return 1.f - y * y;
    case CBA_ACT_PLSE: return (y < 0.f || y > 1.f) ? 0.01f : 0.125f;
    case CBA_ACT_ELU: return y >= 0.f ? 1.f : y + 1.f;
    case CBA_ACT_SELU: return y >= 0.f ? 1.0507f : y + 1.0507f * 1.6732f;
    case CBA_ACT_LHTAN: return (y > 0.f && y < 1.f) ? 1.f : 0.001f;
    case CBA_ACT_HARDTAN: return (y > -1.f && y < 1.f) ? 1.f : 0.f;
    case CBA_ACT_LOGGY: {
        const float t = (y + 1.f) * 0.5f;
        return 2.f * (1.f - t) * t;
    }
    case CBA_ACT_STAIR: return floorf(y) == y ? 0.f : 1.f;
    default: return 1.f;
    }
}

// gradient_array of backward_convolutional_layer ("YOLOv3反向传播原理" §3.1):
// dprime = delta * f'(output), 16-byte accesses (n4 of them) and a scalar tail.
__global__ void gradient_array_kernel(const float *delta, const float *__restrict__ output,
                                      float *dprime, long long n, int act) {  // dprime may be delta
    const long long n4 = n / 4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 d = reinterpret_cast<const float4 *>(delta)[i];
        const float4 y = __ldg(reinterpret_cast<const float4 *>(output) + i);
        reinterpret_cast<float4 *>(dprime)[i] =
            make_float4(d.x * act_grad_other(act, y.x), d.y * act_grad_other(act, y.y),
                        d.z * act_grad_other(act, y.z), d.w * act_grad_other(act, y.w));
    }
    for (long long i = 4 * n4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += stride)
        dprime[i] = delta[i] * act_grad_other(act, __ldg(output + i));
}

cudaError_t launch_gradient_array(const Plan &p, const float *delta, const float *output,
                                  float *dprime, cudaStream_t st, int *launches) {
    const long long n = (long long)p.N * p.K * p.PQ;
    const long long blocks = std::min<long long>((n / 4 + 255) / 256 + 1, (long long)p.num_sms * 8);
    gradient_array_kernel<<<(unsigned)blocks, 256, 0, st>>>(delta, output, dprime, n, p.act_in);
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
