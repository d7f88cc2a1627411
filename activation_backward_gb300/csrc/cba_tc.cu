// cba_tc.cu -- the two convolution gradients on the 5th-generation tensor
// cores (tcgen05.mma kind::tf32, fp32 accumulators in TMEM).
//
// Both kernels are implicit GEMMs with the same warp-specialised pipeline:
//
//   warps 0-7  operand producers: gather one 32-deep K slice of the A and B
//              tiles from global memory (the BN/activation transform
//              dz = a*delta' + b + c*(z - mu) applied on the fly, values
//              rounded to TF32), and store them in shared memory in the
//              K-major, 128-byte-swizzled layout the tensor core reads;
//              after the main loop the same warps are the epilogue (TMEM ->
//              registers -> global).
//   warp 8     allocates TMEM; its lane 0 issues the MMAs (4 per 32-deep
//              slice) and commits each stage back to the producers.
//
// Stages are handed over with mbarriers: `full` (256 producer arrivals) and
// `empty` (one tcgen05.commit).  Every wait is bounded in time; a wait that
// runs out sets the workspace status bit and an abort flag that the other
// roles poll, after which the block drains its MMAs, frees its TMEM and
// returns (no trap).
//
// wgrad:  D[k][crs] = sum_L dz[k][L] * col[crs][L] over a slice of the
//         positions L = (n, p, q) (split over blocks); tile 128 x BN; fp32
//         partials go to the workspace and are added into dW in a fixed order
//         ("YOLOv3反向传播原理 之 全流程源码分析" §3.1, gemm(0,1,...,beta=1)).
// dgrad:  D[pixel][c] = sum_{r,s,k} dz[n][k][p][q] * W[k][c][r][s] with
//         h = p*stride + r - pad, w = q*stride + s - pad -- col2im(W^T . dz)
//         of §3.1 / §3.2 written as a gather.  Output pixels are grouped by
//         (h mod stride, w mod stride) so that every block only visits the taps
//         that reach its pixels (no zero products for stride 2).  The epilogue
//         adds the shortcut residual (§5) and, if asked, the old prev_delta.
#include "cba_internal.cuh"
#include "cba_ptx.cuh"

namespace cba {

namespace {

constexpr int kStages = 4;
constexpr int kProducers = 256;                  // warps 0-7
constexpr int kThreads = kProducers + 32;        // + the MMA / TMEM warp
constexpr int kTileM = 128;
constexpr int kSliceK = 32;                      // fp32 elements per 128-byte row
constexpr uint32_t kTileABytes = kTileM * 128;   // 16 KiB
constexpr uint64_t kWaitLimitNs = 2000000000ull; // 2 s per wait

// Byte offset of element (row, kk), kk in [0, 32), of a K-major tile whose rows
// are 128 bytes and whose base is 1024-byte aligned: the 16-byte chunk index is
// XOR-ed with (row mod 8) (the 128-byte swizzle).
__device__ __forceinline__ uint32_t sw128(int row, int kk) {
    return (uint32_t)(row * 128 + ((((kk >> 2) ^ row) & 7) << 4) + ((kk & 3) << 2));
}

__device__ __forceinline__ float to_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

__device__ __forceinline__ void st_smem_f32(uint8_t *base, uint32_t off, float v) {
    *reinterpret_cast<float *>(base + off) = v;
}

struct Pipe {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t accum;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void pipe_init(Pipe &pp) {
    for (int s = 0; s < kStages; ++s) {
        ptx::mbar_init(ptx::smem_u32(&pp.full[s]), kProducers);
        ptx::mbar_init(ptx::smem_u32(&pp.empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&pp.accum), 1);
    pp.abort_flag = 0;
    ptx::fence_mbar_init();
}

// The MMA role (one thread): for every K slice wait until the producers have
// filled its stage, issue 4 MMAs of depth 8, and release the stage when they
// complete.  Ends with a commit on `accum`; the same thread then waits for it
// so that no MMA is in flight when the block frees its TMEM.
__device__ __forceinline__ void mma_role(Pipe &pp, uint8_t *smem, uint32_t stage_bytes,
                                         int nchunks, uint32_t tmem, uint32_t idesc,
                                         unsigned *status) {
    volatile int *abort_flag = &pp.abort_flag;
    for (int i = 0; i < nchunks; ++i) {
        const int s = i % kStages;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(&pp.full[s]), (uint32_t)(i / kStages) & 1u,
                                    abort_flag, status, kWaitLimitNs))
            break;
        ptx::tc_fence_after();
        const uint32_t a_base = ptx::smem_u32(smem + (size_t)s * stage_bytes);
        const uint32_t b_base = a_base + kTileABytes;
#pragma unroll
        for (int ks = 0; ks < kSliceK / 8; ++ks) {
            const uint64_t ad = ptx::smem_desc(a_base + ks * 32, 16, 1024, 2);
            const uint64_t bd = ptx::smem_desc(b_base + ks * 32, 16, 1024, 2);
            ptx::mma_tf32(tmem, ad, bd, idesc, (i > 0 || ks > 0) ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&pp.empty[s]));
    }
    ptx::mma_commit(ptx::smem_u32(&pp.accum));
    // wait for the MMAs even after an abort elsewhere (the TMEM is freed next)
    int no_abort = 0;
    ptx::mbar_wait_bounded(ptx::smem_u32(&pp.accum), 0, &no_abort, status, kWaitLimitNs);
}

// Producer-side wait for stage reuse (the i-th fill of stage i % kStages).
__device__ __forceinline__ bool producer_acquire(Pipe &pp, int i, unsigned *status) {
    if (i < kStages) return true;
    return ptx::mbar_wait_bounded(ptx::smem_u32(&pp.empty[i % kStages]),
                                  (uint32_t)(i / kStages - 1) & 1u, &pp.abort_flag, status,
                                  kWaitLimitNs);
}

__device__ __forceinline__ void producer_release(Pipe &pp, int i) {
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(ptx::smem_u32(&pp.full[i % kStages]));
}

// ------------------------------------------------------------------ wgrad

struct WgArgs {
    const float *x, *delta, *output, *z;
    const Coef *coef;
    float *part;  // [splits][K][CRS]
    unsigned *status;
    int C, H, W, K, R, S, stride, pad, P, Q, PQ, RS, CRS;
    long long L;          // N*P*Q
    long long split_len;  // positions per split, multiple of 32
    int bn;               // N tile, multiple of 32, <= 256
};

template <int ACT, bool BN>
__global__ void __launch_bounds__(kThreads, 1) wgrad_tc_kernel(const WgArgs a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ Pipe pp;
    __shared__ int tab_c[256], tab_rs[256];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int crs0 = blockIdx.x * a.bn, k0 = blockIdx.y * kTileM;
    const long long Ls0 = (long long)blockIdx.z * a.split_len;
    const long long Ls1 = min(Ls0 + a.split_len, a.L);
    const int nchunks = (int)((Ls1 - Ls0 + kSliceK - 1) / kSliceK);
    const uint32_t stage_bytes = kTileABytes + (uint32_t)a.bn * 128u;

    for (int i = tid; i < a.bn; i += kThreads) {
        const int crs = crs0 + i;
        const int cc = crs < a.CRS ? crs : 0;
        tab_c[i] = cc / a.RS;
        tab_rs[i] = ((cc % a.RS) / a.S) << 16 | (cc % a.S);
    }
    if (tid == 0) pipe_init(pp);
    const uint32_t ncols = a.bn <= 32 ? 32 : a.bn <= 64 ? 64 : a.bn <= 128 ? 128 : 256;
    if (warp == 8) {
        ptx::tmem_alloc(ptx::smem_u32(&pp.tmem_base), ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = pp.tmem_base;

    if (warp < 8) {
        Coef cf[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            const int k = k0 + warp * 16 + rr;
            cf[rr] = k < a.K ? a.coef[k] : Coef{0.f, 0.f, 0.f, 0.f};
        }
        int i = 0;
        for (; i < nchunks; ++i) {
            if (!producer_acquire(pp, i, a.status)) break;
            uint8_t *sa = smem + (size_t)(i % kStages) * stage_bytes;
            uint8_t *sb = sa + kTileABytes;
            const long long Lp = Ls0 + (long long)i * kSliceK + lane;
            const bool vl = Lp < Ls1;
            const int n = vl ? (int)(Lp / a.PQ) : 0;
            const int j = vl ? (int)(Lp - (long long)n * a.PQ) : 0;
            // A: dz rows k0 + warp*16 + rr, column = this lane's position
            {
                float dv[16], yv[16], zv[16];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    const int k = k0 + warp * 16 + rr;
                    dv[rr] = 0.f;
                    yv[rr] = 0.f;
                    zv[rr] = 0.f;
                    if (vl && k < a.K) {
                        const long long off = ((long long)n * a.K + k) * a.PQ + j;
                        dv[rr] = __ldg(a.delta + off);
                        if (ACT == CBA_ACT_LEAKY) yv[rr] = __ldg(a.output + off);
                        if (BN) zv[rr] = __ldg(a.z + off);
                    }
                }
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    const int row = warp * 16 + rr;
                    const float v = dz_of<ACT, BN>(dv[rr], yv[rr], zv[rr], cf[rr]);
                    st_smem_f32(sa, sw128(row, lane), to_tf32(v));
                }
            }
            // B: im2col rows crs0 + warp*rows_b + rr at this lane's position
            {
                const int p = j / a.Q, q = j - (j / a.Q) * a.Q;
                const int h0 = p * a.stride - a.pad, w0 = q * a.stride - a.pad;
                const float *xn = a.x + (long long)n * a.C * a.H * a.W;
                // rows warp, warp + 8, warp + 16, ... < bn (bn is a multiple of 32)
                for (int rb = 0; rb < a.bn; rb += 64) {
                    float xv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int row = rb + u * 8 + warp;
                        xv[u] = 0.f;
                        if (row < a.bn) {
                            const int rs = tab_rs[row];
                            const int h = h0 + (rs >> 16), w = w0 + (rs & 0xffff);
                            if (vl && crs0 + row < a.CRS && h >= 0 && h < a.H && w >= 0 &&
                                w < a.W)
                                xv[u] = __ldg(xn + ((long long)tab_c[row] * a.H + h) * a.W + w);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int row = rb + u * 8 + warp;
                        if (row < a.bn) st_smem_f32(sb, sw128(row, lane), to_tf32(xv[u]));
                    }
                }
            }
            producer_release(pp, i);
        }
        // epilogue: TMEM lanes 32*(warp%4)..+31, column half warp/4
        bool ok = (i == nchunks) &&
                  ptx::mbar_wait_bounded(ptx::smem_u32(&pp.accum), 0, &pp.abort_flag, a.status,
                                         kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
        if (ok) {
            ptx::tc_fence_after();
            const int quarter = warp & 3, half = warp >> 2;
            const int row = quarter * 32 + lane;
            const int k = k0 + row;
            const int cbeg = half * (a.bn >> 1), cend = cbeg + (a.bn >> 1);
            float *dst = a.part + ((size_t)blockIdx.z * a.K + (k < a.K ? k : 0)) * a.CRS + crs0;
            for (int col = cbeg; col < cend; col += 16) {
                float v[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col, v);
                ptx::tmem_ld_wait();
                if (k < a.K) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (crs0 + col + e < a.CRS) dst[col + e] = v[e];
                }
            }
        }
    } else if (lane == 0) {
        mma_role(pp, smem, stage_bytes, nchunks, tmem, ptx::idesc_tf32(kTileM, a.bn), a.status);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, ncols);
    }
}

// ------------------------------------------------------------------ dgrad

constexpr int kMaxClasses = 16;  // stride <= 4

struct DgArgs {
    const float *wt;  // [R*S][C][K]
    const float *delta, *output, *z;
    const Coef *coef;
    const float *residual;
    float *prev;
    unsigned *status;
    int N, C, H, W, K, R, S, stride, pad, P, Q, PQ;
    int accumulate, bn, kchunks, nclass;
    int tile0[kMaxClasses + 1];  // first M tile of each pixel class
    int hc[kMaxClasses], wc[kMaxClasses];
};

template <int ACT, bool BN>
__global__ void __launch_bounds__(kThreads, 1) dgrad_tc_kernel(const DgArgs a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ Pipe pp;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int cl = 0;
    while (cl + 1 < a.nclass && a.tile0[cl + 1] <= (int)blockIdx.x) ++cl;
    const int ph = cl / a.stride, pw = cl % a.stride;
    const int Hc = a.hc[cl], Wc = a.wc[cl];
    const long long Mc = (long long)a.N * Hc * Wc;
    const long long m0 = (long long)(blockIdx.x - a.tile0[cl]) * kTileM;
    const int c0 = blockIdx.y * a.bn;
    // taps that reach this class: r = (ph+pad) mod stride, + stride, ...
    const int r0 = (ph + a.pad) % a.stride, s0 = (pw + a.pad) % a.stride;
    const int nr = r0 < a.R ? (a.R - r0 + a.stride - 1) / a.stride : 0;
    const int ns = s0 < a.S ? (a.S - s0 + a.stride - 1) / a.stride : 0;
    const int nchunks = nr * ns * a.kchunks;
    const uint32_t stage_bytes = kTileABytes + (uint32_t)a.bn * 128u;

    if (tid == 0) pipe_init(pp);
    const uint32_t ncols = a.bn <= 32 ? 32 : a.bn <= 64 ? 64 : a.bn <= 128 ? 128 : 256;
    if (warp == 8) {
        ptx::tmem_alloc(ptx::smem_u32(&pp.tmem_base), ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = pp.tmem_base;

    if (warp < 8) {
        // A loader geometry: this thread fills pixel rows warp*16 + g*8 + (lane>>2)
        // and k columns 4*kk4 + (lane&3)
        const int psub = lane >> 2, ksub = lane & 3;
        bool pv[2];
        int pn[2], hq[2], wq[2];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const long long m = m0 + warp * 16 + g * 8 + psub;
            pv[g] = m < Mc;
            const long long mm = pv[g] ? m : 0;
            const int n = (int)(mm / ((long long)Hc * Wc));
            const int rem = (int)(mm - (long long)n * Hc * Wc);
            const int ii = rem / Wc, jj = rem - (rem / Wc) * Wc;
            pn[g] = n;
            hq[g] = ii * a.stride + ph + a.pad;
            wq[g] = jj * a.stride + pw + a.pad;
        }
        int i = 0;
        for (; i < nchunks; ++i) {
            if (!producer_acquire(pp, i, a.status)) break;
            uint8_t *sa = smem + (size_t)(i % kStages) * stage_bytes;
            uint8_t *sb = sa + kTileABytes;
            const int t = i / a.kchunks, kc = i - (i / a.kchunks) * a.kchunks;
            const int r = r0 + (t / ns) * a.stride, s = s0 + (t % ns) * a.stride;
            const int kb = kc * kSliceK;
            // A: dz at the tap-shifted position of each pixel
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int ph_ = hq[g] - r, pw_ = wq[g] - s;
                bool ok = pv[g] && ph_ >= 0 && pw_ >= 0;
                const int p = ok ? ph_ / a.stride : 0, q = ok ? pw_ / a.stride : 0;
                ok = ok && p < a.P && q < a.Q;
                const long long base = (long long)pn[g] * a.K * a.PQ + (long long)p * a.Q + q;
                float dv[8], yv[8], zv[8];
                Coef cf[8];
#pragma unroll
                for (int kk4 = 0; kk4 < 8; ++kk4) {
                    const int k = kb + kk4 * 4 + ksub;
                    dv[kk4] = 0.f;
                    yv[kk4] = 0.f;
                    zv[kk4] = 0.f;
                    cf[kk4] = Coef{0.f, 0.f, 0.f, 0.f};
                    if (ok && k < a.K) {
                        const long long off = base + (long long)k * a.PQ;
                        dv[kk4] = __ldg(a.delta + off);
                        if (ACT == CBA_ACT_LEAKY) yv[kk4] = __ldg(a.output + off);
                        if (BN) zv[kk4] = __ldg(a.z + off);
                        cf[kk4] = a.coef[k];
                    }
                }
                const int row = warp * 16 + g * 8 + psub;
#pragma unroll
                for (int kk4 = 0; kk4 < 8; ++kk4) {
                    const float v = dz_of<ACT, BN>(dv[kk4], yv[kk4], zv[kk4], cf[kk4]);
                    st_smem_f32(sa, sw128(row, kk4 * 4 + ksub), to_tf32(v));
                }
            }
            // B: W^T slice for tap (r, s): rows c, columns k
            {
                const float *wrow = a.wt + (long long)(r * a.S + s) * a.C * a.K;
                const int k = kb + lane;
                // rows warp, warp + 8, ... < bn (bn is a multiple of 32)
                for (int rb = 0; rb < a.bn; rb += 64) {
                    float wv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int row = rb + u * 8 + warp;
                        const int c = c0 + row;
                        wv[u] = (row < a.bn && c < a.C && k < a.K)
                                    ? __ldg(wrow + (long long)c * a.K + k) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int row = rb + u * 8 + warp;
                        if (row < a.bn) st_smem_f32(sb, sw128(row, lane), to_tf32(wv[u]));
                    }
                }
            }
            producer_release(pp, i);
        }
        // epilogue
        bool ok = (i == nchunks);
        if (ok && nchunks > 0)
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&pp.accum), 0, &pp.abort_flag, a.status,
                                        kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
        if (ok) {
            ptx::tc_fence_after();
            const int quarter = warp & 3, half = warp >> 2;
            const int row = quarter * 32 + lane;
            const long long m = m0 + row;
            const bool valid = m < Mc;
            const long long mm = valid ? m : 0;
            const int n = (int)(mm / ((long long)Hc * Wc));
            const int rem = (int)(mm - (long long)n * Hc * Wc);
            const int h = (rem / Wc) * a.stride + ph, w = (rem % Wc) * a.stride + pw;
            const long long HW = (long long)a.H * a.W;
            const long long pix = (long long)n * a.C * HW + (long long)h * a.W + w;
            const int cbeg = half * (a.bn >> 1), cend = cbeg + (a.bn >> 1);
            for (int col = cbeg; col < cend; col += 16) {
                float v[16];
                if (nchunks > 0) {
                    ptx::tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col, v);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = 0.f;
                }
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int c = c0 + col + e;
                        if (c < a.C) {
                            const long long idx = pix + (long long)c * HW;
                            float o = v[e];
                            if (a.residual) o += a.residual[idx];
                            if (a.accumulate) o += a.prev[idx];
                            a.prev[idx] = o;
                        }
                    }
                }
            }
        }
    } else if (lane == 0 && nchunks > 0) {
        mma_role(pp, smem, stage_bytes, nchunks, tmem, ptx::idesc_tf32(kTileM, a.bn), a.status);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, ncols);
    }
}

// W[k][c][r][s] -> wt[r*S + s][c][k]
__global__ void repack_w_kernel(const float *__restrict__ W, int K, int C, int RS,
                                float *__restrict__ wt) {
    const long long total = (long long)K * C * RS;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int rs = (int)(i % RS);
        const long long kc = i / RS;
        const int c = (int)(kc % C), k = (int)(kc / C);
        wt[((long long)rs * C + c) * K + k] = W[i];
    }
}

// One thread waits on a barrier phase nobody completes; the bounded wait must
// give up after timeout_us and set the status bit.
__global__ void selftest_wait_kernel(unsigned timeout_us, unsigned *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0, &abort_flag, status,
                               (uint64_t)timeout_us * 1000ull);
    }
    __syncthreads();
}

inline size_t tc_smem_bytes(int bn) {
    return (size_t)kStages * (kTileABytes + (size_t)bn * 128) + 1024;
}

template <typename Kern, typename Args>
cudaError_t launch_tc(Kern kern, dim3 grid, size_t smem, const Args &args, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(args);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const Plan &p) { return p.stride <= 4; }

void tc_plan(Plan &p) {
    // wgrad: N tiles over C*R*S (<= 256 wide, multiple of 32), M tiles of 128
    // output channels, the positions split so that about one block per SM runs
    const int nt = (p.CRS + 255) / 256;
    p.tc_wg_bn = ((p.CRS + nt - 1) / nt + 31) / 32 * 32;
    p.tc_wg_ntiles = (p.CRS + p.tc_wg_bn - 1) / p.tc_wg_bn;
    const int mt = (p.K + kTileM - 1) / kTileM;
    const long long chunks = (p.m + kSliceK - 1) / kSliceK;
    long long splits = std::max(1LL, (long long)p.num_sms / ((long long)nt * mt));
    splits = std::min(splits, chunks);
    const long long per = (chunks + splits - 1) / splits;
    p.tc_wg_chunk = per * kSliceK;
    p.tc_wg_splits = (int)((p.m + p.tc_wg_chunk - 1) / p.tc_wg_chunk);
    // dgrad: N tiles over C
    const int dn = (p.C + 255) / 256;
    p.tc_dg_bn = ((p.C + dn - 1) / dn + 31) / 32 * 32;
    p.tc_dg_ntiles = (p.C + p.tc_dg_bn - 1) / p.tc_dg_bn;
}

cudaError_t launch_wgrad_tc(const Plan &p, const float *x, const float *delta,
                            const float *output, const float *z, float *dW, void *ws,
                            cudaStream_t st, int *launches) {
    WgArgs a;
    a.x = x; a.delta = delta; a.output = output; a.z = z;
    a.coef = ws_at<Coef>(ws, p.off_coef);
    a.part = ws_at<float>(ws, p.off_wgpart);
    a.status = ws_at<unsigned>(ws, p.off_status);
    a.C = p.C; a.H = p.H; a.W = p.W; a.K = p.K; a.R = p.R; a.S = p.S;
    a.stride = p.stride; a.pad = p.pad; a.P = p.P; a.Q = p.Q; a.PQ = p.PQ; a.RS = p.RS;
    a.CRS = p.CRS; a.L = p.m; a.split_len = p.tc_wg_chunk; a.bn = p.tc_wg_bn;
    dim3 grid(p.tc_wg_ntiles, (p.K + kTileM - 1) / kTileM, p.tc_wg_splits);
    const size_t smem = tc_smem_bytes(a.bn);
    cudaError_t e;
    const bool leaky = p.act == CBA_ACT_LEAKY;
    if (p.bn)
        e = leaky ? launch_tc(wgrad_tc_kernel<CBA_ACT_LEAKY, true>, grid, smem, a, st)
                  : launch_tc(wgrad_tc_kernel<CBA_ACT_LINEAR, true>, grid, smem, a, st);
    else
        e = leaky ? launch_tc(wgrad_tc_kernel<CBA_ACT_LEAKY, false>, grid, smem, a, st)
                  : launch_tc(wgrad_tc_kernel<CBA_ACT_LINEAR, false>, grid, smem, a, st);
    if (e != cudaSuccess) return e;
    *launches += 1;
    return launch_splitk_reduce(p, a.part, p.tc_wg_splits, dW, st, launches);
}

cudaError_t launch_dgrad_tc(const Plan &p, const float *Wt, const float *delta,
                            const float *output, const float *z, const float *residual,
                            float *prev, void *ws, cudaStream_t st, int *launches) {
    float *wt = ws_at<float>(ws, p.off_wt);
    {
        const long long total = (long long)p.K * p.C * p.RS;
        const int blocks = (int)std::min<long long>((total + 255) / 256, (long long)p.num_sms * 4);
        repack_w_kernel<<<blocks, 256, 0, st>>>(Wt, p.K, p.C, p.RS, wt);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    DgArgs a;
    a.wt = wt; a.delta = delta; a.output = output; a.z = z;
    a.coef = ws_at<Coef>(ws, p.off_coef);
    a.residual = residual; a.prev = prev;
    a.status = ws_at<unsigned>(ws, p.off_status);
    a.N = p.N; a.C = p.C; a.H = p.H; a.W = p.W; a.K = p.K; a.R = p.R; a.S = p.S;
    a.stride = p.stride; a.pad = p.pad; a.P = p.P; a.Q = p.Q; a.PQ = p.PQ;
    a.accumulate = p.accumulate; a.bn = p.tc_dg_bn; a.kchunks = (p.K + kSliceK - 1) / kSliceK;
    a.nclass = p.stride * p.stride;
    int tiles = 0;
    for (int cl = 0; cl < a.nclass; ++cl) {
        const int ph = cl / p.stride, pw = cl % p.stride;
        a.hc[cl] = ph < p.H ? (p.H - ph + p.stride - 1) / p.stride : 0;
        a.wc[cl] = pw < p.W ? (p.W - pw + p.stride - 1) / p.stride : 0;
        a.tile0[cl] = tiles;
        const long long mc = (long long)p.N * a.hc[cl] * a.wc[cl];
        tiles += (int)((mc + kTileM - 1) / kTileM);
    }
    a.tile0[a.nclass] = tiles;
    if (tiles == 0) return cudaSuccess;
    dim3 grid(tiles, p.tc_dg_ntiles);
    const size_t smem = tc_smem_bytes(a.bn);
    cudaError_t e;
    const bool leaky = p.act == CBA_ACT_LEAKY;
    if (p.bn)
        e = leaky ? launch_tc(dgrad_tc_kernel<CBA_ACT_LEAKY, true>, grid, smem, a, st)
                  : launch_tc(dgrad_tc_kernel<CBA_ACT_LINEAR, true>, grid, smem, a, st);
    else
        e = leaky ? launch_tc(dgrad_tc_kernel<CBA_ACT_LEAKY, false>, grid, smem, a, st)
                  : launch_tc(dgrad_tc_kernel<CBA_ACT_LINEAR, false>, grid, smem, a, st);
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaSuccess;
}

cudaError_t launch_selftest_wait(unsigned timeout_us, void *ws, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(timeout_us, ws_at<unsigned>(ws, 0));
    return cudaGetLastError();
}

}  // namespace cba
