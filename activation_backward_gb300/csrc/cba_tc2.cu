// cba_tc2.cu -- tensor-core convolution gradients, TMEM-operand design.
//
// Both GEMMs put their A operand in tensor memory, written by 4 warps with
// tcgen05.st, and stream their B operand through shared memory with TMA
// (128-byte swizzle, K-major).  Writing A from registers makes any shift of
// the convolution taps free (no 16-byte alignment rule, no shared-memory
// traffic), and the tensor core then reads only B from shared memory.
//
// The BN-input gradient dz (activation derivative and normalize_delta of
// "YOLOv3反向传播原理 之 全流程源码分析" §4 applied to delta) is written once,
// TF32-rounded, by a memory-bound pass (`dz_materialize_kernel`) in
// [N][K][P][Qp] order (rows padded to Qp = Q rounded up to 4, so the rows are
// 16-byte strided for TMA); both GEMMs read it from there.  1x1 stride-1
// unpadded layers view each P x Q plane as one row of length P*Q.
//
// wgrad (dW[k][c][r][s] += sum_{n,p,q} dz[n][k][p][q] x[n][c][p*st+r-pad][q*st+s-pad],
//        the gemm(0,1,...) of §3.1):
//   TMEM lanes = (input channel c, kernel column s) pairs, columns = 32 output
//   columns q of one output row; the lane (c, s) holds x[n][c][h][q*st + s - pad]
//   for the input row h.  B = dz row p (128 output channels x 32 q) by TMA;
//   each input row h meets the output rows p = (h + pad - r)/st, one
//   accumulator D_r (128 x 128) per kernel row r.  dz rows live in a ring of
//   shared-memory slots and are loaded once per block.  The epilogue adds the
//   block's partial sums into dW in L2 with bulk async reductions.
// dgrad (prev[n][c][h][w] = sum_{r,s,k} W[k][c][r][s] dz[n][k][(h+pad-r)/st][(w+pad-s)/st],
//        col2im(W^T . dz) of §3.1 / §3.2 as a gather):
//   pixels of one stride phase class (h mod st, w mod st) on a grid of rows i
//   and columns jj; TMEM lanes = 128 consecutive grid positions, columns = 32
//   output channels k; the lane holds dz[n][k][i + dp_r][jj + min_dq] for
//   kernel row r.  B = W[k][c][r][s] for all kernel columns s of the class at
//   once (N = (s, c) pairs), so the MMA computes E[(i, q)][(s, c)] and the
//   epilogue finishes the column shift: prev(i, j) = sum_s E(i, j + dq_s)[s, c],
//   adds the shortcut residual (§5) and, if asked, the old prev_delta.
//
// All waits are bounded (2 s); see cba_ptx.cuh.
#include <cuda.h>

#include "cba_internal.cuh"
#include "cba_ptx.cuh"

namespace cba {

namespace {

constexpr uint64_t kLimitNs = 2000000000ull;

__device__ __forceinline__ float to_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

__host__ __device__ __forceinline__ int fdiv(int a, int b) {  // floor(a / b), b > 0
    return a >= 0 ? a / b : -((-a + b - 1) / b);
}
__host__ __device__ __forceinline__ int cdiv(int a, int b) { return -fdiv(-a, b); }

// ------------------------------------------------------ dz materialisation

template <int ACT, bool BN>
__global__ void dz_materialize_kernel(const float *__restrict__ delta,
                                      const float *__restrict__ output,
                                      const float *__restrict__ z, const Coef *__restrict__ coef,
                                      int K, int Pe, int Qe, int Qp, long long rows,
                                      float *__restrict__ dzt) {
    const int qv = Qp >> 2;
    const long long total = rows * qv;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / qv;
        const int q0 = (int)(i - row * qv) * 4;
        const int k = (int)((row / Pe) % K);
        const Coef cf = coef[k];
        const long long src = row * Qe;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int q = q0 + e;
            v[e] = 0.f;
            if (q < Qe) {
                const float y = (ACT == CBA_ACT_LEAKY) ? __ldg(output + src + q) : 0.f;
                const float zz = BN ? __ldg(z + src + q) : 0.f;
                v[e] = to_tf32(dz_of<ACT, BN>(__ldg(delta + src + q), y, zz, cf));
            }
        }
        reinterpret_cast<float4 *>(dzt)[i] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// W[k][c][r][s] -> wr[r][s][c][kk] (kk < Kw; zero for kk >= K), TF32-rounded.
__global__ void repack_wr_kernel(const float *__restrict__ W, int K, int C, int R, int S, int Kw,
                                 float *__restrict__ wr) {
    const long long total = (long long)R * S * C * Kw;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int kk = (int)(i % Kw);
        long long t = i / Kw;
        const int c = (int)(t % C);
        t /= C;
        const int s = (int)(t % S);
        const int r = (int)(t / S);
        wr[i] = kk < K ? to_tf32(W[(((long long)kk * C + c) * R + r) * S + s]) : 0.f;
    }
}

// ------------------------------------------------------------------ wgrad

constexpr int kW2Ring = 6;  // dz row tiles resident
constexpr int kW2NA = 4;    // A stages in TMEM (32 columns each)
constexpr int kW2Threads = 320;  // 8 producer warps, TMA warp, MMA warp

struct Wg2Args {
    const float *x;
    float *dW;
    unsigned *status;
    int C, He, We, K, R, S, RS, CRS, stride, pad, Pe, Qe;
    int ct;              // input channels per block (lanes = ct * S <= 128)
    int nk;              // output channels per block = MMA N (multiple of 32)
    int nqc;             // 32-wide output-column chunks per row
    int rows_per_split;  // input rows per block
    int splits_per_seg;
    int bulk;            // 1: bulk L2 reductions are aligned, 0: per-element atomics
    uint32_t ncols;      // TMEM columns allocated
};

struct W2Bars {
    uint64_t dz_full[kW2Ring], dz_empty[kW2Ring], a_full[kW2NA], a_empty[kW2NA], accum;
    uint32_t tmem_base;
    int abort_flag;
};

__global__ void __launch_bounds__(kW2Threads, 1)
    wgrad_tc2_kernel(const __grid_constant__ CUtensorMap tm, const Wg2Args a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ W2Bars sb;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k0 = blockIdx.x * a.nk;
    const int c0 = blockIdx.y * a.ct;
    const int ct_here = min(a.ct, a.C - c0);
    const int seg = blockIdx.z / a.splits_per_seg, split = blockIdx.z % a.splits_per_seg;
    const int n = seg / a.nqc, qc = seg % a.nqc;
    const int h0 = split * a.rows_per_split, h1 = min(a.He, h0 + a.rows_per_split);
    const int q_base = qc * 32;
    const int nsteps = (min(32, a.Qe - q_base) + 7) / 8;
    const uint32_t tile_bytes = (uint32_t)a.nk * 128u;
    const int st = a.stride, R = a.R;
    const int p_lo = max(0, cdiv(h0 - R + 1 + a.pad, st));
    const int p_hi = min(a.Pe - 1, fdiv(h1 - 1 + a.pad, st));
    const uint32_t a_col0 = (uint32_t)(R * a.nk);
    const uint32_t idesc = ptx::idesc_tf32(128, a.nk);

    if (tid == 0) {
        for (int i = 0; i < kW2Ring; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.dz_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.dz_empty[i]), 1);
        }
        for (int i = 0; i < kW2NA; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.a_full[i]), 128);
            ptx::mbar_init(ptx::smem_u32(&sb.a_empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&sb.accum), 1);
        sb.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 9) {
        ptx::tmem_alloc(ptx::smem_u32(&sb.tmem_base), a.ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sb.tmem_base;
    const bool has_work = h0 < h1 && p_lo <= p_hi;

    if (warp < 8) {
        // ---- A producers: two groups of 4 warps take alternate input rows and
        // load the next row of their group while storing the current one.
        // TMEM lane (c, s) holds x[n][c0+c][h][q*st + s - pad] for 32 q.
        const int grp = warp >> 2, wq = warp & 3;
        const int L = wq * 32 + lane;
        const int cl = L / a.S, s = L - (L / a.S) * a.S;
        const bool lv = cl < ct_here;
        const float *xb = a.x + ((long long)n * a.C + c0 + (lv ? cl : 0)) * a.He * a.We;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const int nrows = has_work ? h1 - h0 : 0;
        auto load_row = [&](float(&v)[32], int h) {
            const float *xr = xb + (long long)h * a.We;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int q = q_base + j;
                const int w = q * st + s - a.pad;
                v[j] = (lv && q < a.Qe && w >= 0 && w < a.We) ? to_tf32(__ldg(xr + w)) : 0.f;
            }
        };
        bool ok = true;
        float cur[32];
        if (grp < nrows) load_row(cur, h0 + grp);
        for (int t = grp; t < nrows; t += 2) {
            float nxt[32];
            if (t + 2 < nrows) load_row(nxt, h0 + t + 2);
            const int sa = t % kW2NA;
            if (t >= kW2NA)
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_empty[sa]),
                                            (uint32_t)(t / kW2NA - 1) & 1u, &sb.abort_flag,
                                            a.status, kLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            ptx::tmem_st32(tmem + lane_addr + a_col0 + (uint32_t)(sa * 32), cur);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&sb.a_full[sa]));
#pragma unroll
            for (int j = 0; j < 32; ++j) cur[j] = nxt[j];
        }
        // ---- epilogue: D_r[(c, s)][k] -> dW[k][c][r][s]; group g takes the
        // 32-wide output-channel chunks kc = g, g + 2, ...
        if (has_work && ok)
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &sb.abort_flag, a.status,
                                        kLimitNs);
        ok = __all_sync(0xffffffffu, ok) && has_work;
        if (ok) {
            ptx::tc_fence_after();
            const int pitch = ct_here * a.RS;  // floats per staged dW row segment
            float *stg = reinterpret_cast<float *>(ring) + grp * 32 * pitch;
            for (int kc = grp; kc * 32 < a.nk && k0 + kc * 32 < a.K; kc += 2) {
                const int krows = min(32, a.K - (k0 + kc * 32));
                for (int r = 0; r < R; ++r) {
                    // was accumulator r written by any input row of this block?
                    bool wr = false;
                    for (int h = h0; h < h1 && !wr; ++h) {
                        const int num = h - r + a.pad;
                        wr = num >= 0 && num % st == 0 && num / st >= p_lo && num / st <= p_hi;
                    }
                    float v[32];
                    if (wr) {
                        ptx::tmem_ld32(tmem + lane_addr + (uint32_t)(r * a.nk + kc * 32), v);
                        ptx::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0.f;
                    }
                    if (lv) {
                        if (a.bulk) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                stg[j * pitch + cl * a.RS + r * a.S + s] = v[j];
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < krows)
                                    atomicAdd(a.dW + ((long long)(k0 + kc * 32 + j) * a.C + c0 +
                                                      cl) * a.RS + r * a.S + s,
                                              v[j]);
                        }
                    }
                }
                if (a.bulk) {
                    ptx::fence_proxy_async_smem();
                    ptx::named_bar_sync(1 + grp, 128);
                    if (L < krows) {
                        ptx::bulk_reduce_add_f32(
                            a.dW + (long long)(k0 + kc * 32 + L) * a.CRS + (long long)c0 * a.RS,
                            ptx::smem_u32(stg + L * pitch), (uint32_t)pitch * 4u);
                        ptx::bulk_commit();
                        ptx::bulk_wait_read_all();
                    }
                    ptx::named_bar_sync(1 + grp, 128);
                }
            }
            if (a.bulk && L < 32) ptx::bulk_wait_all();
        }
    } else if (warp == 8) {
        // ---- TMA producer: dz rows p_lo..p_hi into the ring
        if (lane == 0 && has_work) {
            int issued = 0;
            for (int p = p_lo; p <= p_hi; ++p, ++issued) {
                const int seq = p - p_lo, slot = seq % kW2Ring;
                if (seq >= kW2Ring &&
                    !ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_empty[slot]),
                                            (uint32_t)(seq / kW2Ring - 1) & 1u, &sb.abort_flag,
                                            a.status, kLimitNs))
                    break;
                ptx::mbar_arrive_expect_tx(ptx::smem_u32(&sb.dz_full[slot]), tile_bytes);
                ptx::tma_load_4d(ptx::smem_u32(ring + (size_t)slot * tile_bytes), &tm, q_base, p,
                                 k0, n, ptx::smem_u32(&sb.dz_full[slot]));
            }
            // no copy may be in flight when the block exits
            int no_abort = 0;
            for (int seq = max(0, issued - kW2Ring); seq < issued; ++seq)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_full[seq % kW2Ring]),
                                       (uint32_t)(seq / kW2Ring) & 1u, &no_abort, a.status,
                                       kLimitNs);
        }
    } else {
        // ---- MMA issuer
        if (lane == 0 && has_work) {
            uint32_t written = 0;
            int p_rel = p_lo;
            int t = 0;
            bool ok = true;
            for (int h = h0; ok && h < h1; ++h, ++t) {
                const int sa = t % kW2NA;
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_full[sa]),
                                            (uint32_t)(t / kW2NA) & 1u, &sb.abort_flag, a.status,
                                            kLimitNs);
                if (!ok) break;
                ptx::tc_fence_after();
                for (int r = 0; r < R; ++r) {
                    const int num = h - r + a.pad;
                    if (num < 0 || num % st) continue;
                    const int p = num / st;
                    if (p < p_lo || p > p_hi) continue;
                    const int seq = p - p_lo, slot = seq % kW2Ring;
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_full[slot]),
                                                (uint32_t)(seq / kW2Ring) & 1u, &sb.abort_flag,
                                                a.status, kLimitNs);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint32_t b_base = ptx::smem_u32(ring + (size_t)slot * tile_bytes);
                    for (int ks = 0; ks < nsteps; ++ks) {
                        const uint64_t bd = ptx::smem_desc(b_base + ks * 32, 16, 1024, 2);
                        ptx::mma_tf32_ts(tmem + (uint32_t)(r * a.nk),
                                         tmem + a_col0 + (uint32_t)(sa * 32 + ks * 8), bd, idesc,
                                         ((written >> r) & 1u) || ks > 0 ? 1u : 0u);
                    }
                    written |= 1u << r;
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_u32(&sb.a_empty[sa]));
                while (p_rel <= p_hi && min(h1 - 1, p_rel * st - a.pad + R - 1) <= h) {
                    ptx::mma_commit(ptx::smem_u32(&sb.dz_empty[(p_rel - p_lo) % kW2Ring]));
                    ++p_rel;
                }
            }
            ptx::mma_commit(ptx::smem_u32(&sb.accum));
            int no_abort = 0;
            ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &no_abort, a.status, kLimitNs);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, a.ncols);
    }
}

// ------------------------------------------------------------------ dgrad

constexpr int kD2NA = 2;    // A stages in TMEM
constexpr int kD2Ring = 4;  // B stages in shared memory
constexpr int kD2Threads = 320;  // 8 producer warps, TMA warp, MMA warp
constexpr int kD2MaxTaps = 8;

struct Dg2Args {
    const float *dzt;
    const float *residual;
    float *prev;
    unsigned *status;
    int C, He, We, K, Pe, Qe, Qp, stride, accumulate;
    int ph, pw, Hc, Wc, Wx, min_dq, span;
    int nr, r_of[kD2MaxTaps], dp[kD2MaxTaps];
    int ns, s_of[kD2MaxTaps], dq[kD2MaxTaps];
    int c_tile, ncol, kchunks, T, total_tiles;
    long long total_pos;  // N * Hc * Wx
    uint32_t ncols;       // TMEM columns allocated
    uint32_t pitch;       // epilogue staging row pitch (floats)
};

struct D2Bars {
    uint64_t b_full[kD2Ring], b_empty[kD2Ring], a_full[kD2NA], a_empty[kD2NA], accum;
    uint32_t tmem_base;
    int abort_flag;
};

__global__ void __launch_bounds__(kD2Threads, 1)
    dgrad_tc2_kernel(const __grid_constant__ CUtensorMap tmw, const Dg2Args a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ D2Bars sb;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = blockIdx.y * a.c_tile;
    const int tstride = 128 - a.span;
    const int nstages = a.nr * a.kchunks;
    const uint32_t b_bytes = (uint32_t)a.ncol * 128u;
    const uint32_t a_col0 = (uint32_t)(a.T * a.ncol);
    const uint32_t idesc = ptx::idesc_tf32(128, a.ncol);

    if (tid == 0) {
        for (int i = 0; i < kD2Ring; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.b_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.b_empty[i]), 1);
        }
        for (int i = 0; i < kD2NA; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.a_full[i]), 256);
            ptx::mbar_init(ptx::smem_u32(&sb.a_empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&sb.accum), 1);
        sb.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 9) {
        ptx::tmem_alloc(ptx::smem_u32(&sb.tmem_base), a.ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sb.tmem_base;

    if (warp < 8) {
        // ---- A producers.  Work unit of a group per stage: with two tiles,
        // group g fills tile g (32 columns); with one tile, group g fills
        // columns 16g..16g+15.  Each group loads its next stage while storing
        // the current one.
        const int grp = warp >> 2, wq = warp & 3;
        const int L = wq * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const int tt = a.T == 2 ? grp : 0;
        const int j0 = a.T == 2 ? 0 : grp * 16;
        const int tile = blockIdx.x * a.T + tt;
        const long long g = (long long)tile * tstride + L;
        const bool gv = tile < a.total_tiles && g < a.total_pos;
        const long long gg = gv ? g : 0;
        const long long per_img = (long long)a.Hc * a.Wx;
        const int gn = (int)(gg / per_img);
        const int grem = (int)(gg - (long long)gn * per_img);
        const int gi = grem / a.Wx, gj = grem - (grem / a.Wx) * a.Wx;
        const long long kstride = (long long)a.Pe * a.Qp;
        auto load_stage = [&](float(&v)[32], int i) {
            const int ri = i / a.kchunks, kc = i - (i / a.kchunks) * a.kchunks;
            const int kb = kc * 32 + j0;
            const int p = gi + a.dp[ri], q = gj + a.min_dq;
            const bool pv = gv && p >= 0 && p < a.Pe && q >= 0 && q < a.Qe;
            const float *src = a.dzt + (((long long)gn * a.K + kb) * a.Pe + (pv ? p : 0)) * a.Qp +
                               (pv ? q : 0);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                v[j] = (pv && j < (a.T == 2 ? 32 : 16) && kb + j < a.K) ? __ldg(src + j * kstride)
                                                                         : 0.f;
        };
        bool ok = true;
        float cur[32];
        if (nstages > 0) load_stage(cur, 0);
        for (int i = 0; i < nstages; ++i) {
            float nxt[32];
            if (i + 1 < nstages) load_stage(nxt, i + 1);
            const int sa = i % kD2NA;
            if (i >= kD2NA)
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_empty[sa]),
                                            (uint32_t)(i / kD2NA - 1) & 1u, &sb.abort_flag,
                                            a.status, kLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t col = a_col0 + (uint32_t)((sa * a.T + tt) * 32 + j0);
            if (a.T == 2) {
                ptx::tmem_st32(tmem + lane_addr + col, cur);
            } else {
                float h16[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) h16[j] = cur[j];
                ptx::tmem_st16(tmem + lane_addr + col, h16);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&sb.a_full[sa]));
#pragma unroll
            for (int j = 0; j < 32; ++j) cur[j] = nxt[j];
        }
        // ---- epilogue.  Two tiles: group g finishes tile g with its own
        // staging.  One tile: both groups stage half the columns each, then
        // each writes half the output channels.
        if (ok && nstages > 0)
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &sb.abort_flag, a.status,
                                        kLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            ptx::tc_fence_after();
            const bool two = a.T == 2;
            float *stg = reinterpret_cast<float *>(ring) + (two ? grp * 128 * (int)a.pitch : 0);
            const int half = (a.ncol / 2 + 15) / 16 * 16;
            const int col_lo = two ? 0 : (grp == 0 ? 0 : half);
            const int col_hi = two ? a.ncol : (grp == 0 ? half : a.ncol);
            const int bar = two ? 1 + grp : 1, nthr = two ? 128 : 256;
            int col = col_lo;
            for (; col + 32 <= col_hi; col += 32) {
                float v[32];
                if (nstages > 0) {
                    ptx::tmem_ld32(tmem + lane_addr + (uint32_t)(tt * a.ncol + col), v);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) stg[L * a.pitch + col + j] = v[j];
            }
            if (col < col_hi) {  // 16-column tail
                float v[16];
                if (nstages > 0) {
                    ptx::tmem_ld16(tmem + lane_addr + (uint32_t)(tt * a.ncol + col), v);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) stg[L * a.pitch + col + j] = v[j];
            }
            ptx::named_bar_sync(bar, nthr);
            const bool out = gv && L < tstride && gj < a.Wc && gi < a.Hc;
            if (out) {
                const long long HW = (long long)a.He * a.We;
                const int h = gi * a.stride + a.ph, w = gj * a.stride + a.pw;
                const long long pix = (long long)gn * a.C * HW + (long long)h * a.We + w;
                const int ch_half = (a.c_tile + 1) / 2;
                const int cl_lo = two ? 0 : (grp == 0 ? 0 : ch_half);
                const int cl_hi = two ? a.c_tile : (grp == 0 ? ch_half : a.c_tile);
                for (int cl = cl_lo; cl < cl_hi && c0 + cl < a.C; ++cl) {
                    float v = 0.f;
                    for (int si = 0; si < a.ns; ++si)
                        v += stg[(L + a.dq[si] - a.min_dq) * a.pitch + si * a.c_tile + cl];
                    const long long idx = pix + (long long)(c0 + cl) * HW;
                    if (a.residual) v += a.residual[idx];
                    if (a.accumulate) v += a.prev[idx];
                    a.prev[idx] = v;
                }
            }
        }
    } else if (warp == 8) {
        // ---- TMA producer: W slices (all kernel columns of the class) per stage
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nstages; ++i, ++issued) {
                const int slot = i % kD2Ring;
                if (i >= kD2Ring &&
                    !ptx::mbar_wait_bounded(ptx::smem_u32(&sb.b_empty[slot]),
                                            (uint32_t)(i / kD2Ring - 1) & 1u, &sb.abort_flag,
                                            a.status, kLimitNs))
                    break;
                const int ri = i / a.kchunks, kc = i - (i / a.kchunks) * a.kchunks;
                ptx::mbar_arrive_expect_tx(ptx::smem_u32(&sb.b_full[slot]), b_bytes);
                for (int si = 0; si < a.ns; ++si)
                    ptx::tma_load_4d(ptx::smem_u32(ring + (size_t)slot * b_bytes +
                                                   (size_t)si * a.c_tile * 128),
                                     &tmw, kc * 32, c0, a.s_of[si], a.r_of[ri],
                                     ptx::smem_u32(&sb.b_full[slot]));
            }
            int no_abort = 0;
            for (int i = max(0, issued - kD2Ring); i < issued; ++i)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.b_full[i % kD2Ring]),
                                       (uint32_t)(i / kD2Ring) & 1u, &no_abort, a.status,
                                       kLimitNs);
        }
    } else {
        // ---- MMA issuer
        if (lane == 0 && nstages > 0) {
            bool ok = true;
            for (int i = 0; ok && i < nstages; ++i) {
                const int sa = i % kD2NA, slot = i % kD2Ring;
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_full[sa]),
                                            (uint32_t)(i / kD2NA) & 1u, &sb.abort_flag, a.status,
                                            kLimitNs) &&
                     ptx::mbar_wait_bounded(ptx::smem_u32(&sb.b_full[slot]),
                                            (uint32_t)(i / kD2Ring) & 1u, &sb.abort_flag,
                                            a.status, kLimitNs);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t b_base = ptx::smem_u32(ring + (size_t)slot * b_bytes);
                for (int tt = 0; tt < a.T; ++tt) {
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t bd = ptx::smem_desc(b_base + ks * 32, 16, 1024, 2);
                        ptx::mma_tf32_ts(tmem + (uint32_t)(tt * a.ncol),
                                         tmem + a_col0 + (uint32_t)((sa * a.T + tt) * 32 + ks * 8),
                                         bd, idesc, (i > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                ptx::mma_commit(ptx::smem_u32(&sb.a_empty[sa]));
                ptx::mma_commit(ptx::smem_u32(&sb.b_empty[slot]));
            }
            ptx::mma_commit(ptx::smem_u32(&sb.accum));
            int no_abort = 0;
            ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &no_abort, a.status, kLimitNs);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, a.ncols);
    }
}

// -------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// fp32 4-D tensor (d0 innermost, dense strides), box b0..b3, 128-byte swizzle
bool encode_4d(CUtensorMap *m, const void *base, const uint64_t (&d)[4], const uint32_t (&b)[4]) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {d[0], d[1], d[2], d[3]};
    cuuint64_t strides[3] = {d[0] * 4, d[0] * d[1] * 4, d[0] * d[1] * d[2] * 4};
    cuuint32_t box[4] = {b[0], b[1], b[2], b[3]};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline uint32_t pow2_cols(int need) {
    uint32_t c = 32;
    while ((int)c < need) c <<= 1;
    return c;
}

}  // namespace

// Geometry the v2 kernels work in: 1x1 stride-1 unpadded layers are viewed as
// one row per plane.
struct V2Geom {
    int He, We, Pe, Qe, Qp;
};
static V2Geom v2_geom(const Plan &p) {
    V2Geom g;
    const bool flat = p.R == 1 && p.S == 1 && p.stride == 1 && p.pad == 0;
    g.He = flat ? 1 : p.H;
    g.We = flat ? p.H * p.W : p.W;
    g.Pe = flat ? 1 : p.P;
    g.Qe = flat ? p.P * p.Q : p.Q;
    g.Qp = (g.Qe + 3) / 4 * 4;
    return g;
}

bool tc2_supported(const Plan &p) {
    const V2Geom g = v2_geom(p);
    if (p.stride > 4 || p.R > kD2MaxTaps || p.S > kD2MaxTaps) return false;
    if ((long long)p.N * p.K * g.Pe * g.Qp >= (1LL << 31)) return false;
    // dgrad column shift span must leave room in a 128-row tile
    if ((p.S - 1) / p.stride + 1 > 32) return false;
    return encode_fn() != nullptr;
}

size_t tc2_dzt_bytes(const Plan &p) {
    const V2Geom g = v2_geom(p);
    return sizeof(float) * (size_t)p.N * p.K * g.Pe * g.Qp;
}

size_t tc2_wr_bytes(const Plan &p) {
    return sizeof(float) * (size_t)p.R * p.S * p.C * ((p.K + 3) / 4 * 4);
}

cudaError_t launch_dz_materialize(const Plan &p, const float *delta, const float *output,
                                  const float *z, const void *ws, float *dzt, cudaStream_t st,
                                  int *launches) {
    const V2Geom g = v2_geom(p);
    const Coef *coef = ws_at<Coef>(ws, p.off_coef);
    const long long rows = (long long)p.N * p.K * g.Pe;
    const long long total = rows * (g.Qp / 4);
    const int blocks = (int)std::min<long long>((total + 255) / 256, (long long)p.num_sms * 16);
    const bool leaky = p.act == CBA_ACT_LEAKY;
#define CBA_DZM(A, B)                                                                            \
    dz_materialize_kernel<A, B><<<blocks, 256, 0, st>>>(delta, output, z, coef, p.K, g.Pe, g.Qe, \
                                                        g.Qp, rows, dzt)
    if (p.bn) {
        if (leaky) CBA_DZM(CBA_ACT_LEAKY, true);
        else CBA_DZM(CBA_ACT_LINEAR, true);
    } else {
        if (leaky) CBA_DZM(CBA_ACT_LEAKY, false);
        else CBA_DZM(CBA_ACT_LINEAR, false);
    }
#undef CBA_DZM
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_wgrad_tc2(const Plan &p, const float *x, const float *dzt, float *dW,
                             void *ws, cudaStream_t st, int *launches) {
    const V2Geom g = v2_geom(p);
    Wg2Args a;
    a.x = x;
    a.dW = dW;
    a.status = ws_at<unsigned>(ws, p.off_status);
    a.C = p.C; a.He = g.He; a.We = g.We; a.K = p.K; a.R = p.R; a.S = p.S;
    a.RS = p.RS; a.CRS = p.CRS; a.stride = p.stride; a.pad = p.pad; a.Pe = g.Pe; a.Qe = g.Qe;
    // lanes = (c, s) pairs; channels per block a multiple of 4 (aligned dW segments)
    int ct = 128 / p.S;
    if (ct >= 4) ct &= ~3;
    ct = std::max(1, std::min(ct, p.C));
    const int mtiles = (p.C + ct - 1) / ct;
    a.ct = (p.C + mtiles - 1) / mtiles;
    if (a.ct >= 4 && a.ct * p.S <= 128) a.ct = std::min((a.ct + 3) / 4 * 4, 128 / p.S);
    // output channels per block: R accumulators of nk columns + 4 A stages of 32 <= 512
    int nk_cap = ((512 - kW2NA * 32) / p.R) / 32 * 32;
    nk_cap = std::max(32, std::min(256, nk_cap));
    const int ktiles = (p.K + nk_cap - 1) / nk_cap;
    a.nk = std::min(nk_cap, ((p.K + ktiles - 1) / ktiles + 31) / 32 * 32);
    a.ncols = pow2_cols(p.R * a.nk + kW2NA * 32);
    if (a.ncols > 512) return cudaErrorNotSupported;
    a.nqc = (g.Qe + 31) / 32;
    const long long segs = (long long)p.N * a.nqc;
    const long long units = (long long)((p.C + a.ct - 1) / a.ct) * ((p.K + a.nk - 1) / a.nk) * segs;
    int sps = (int)std::max(1LL, std::min<long long>(g.He, (long long)p.num_sms / units));
    a.rows_per_split = (g.He + sps - 1) / sps;
    a.splits_per_seg = (g.He + a.rows_per_split - 1) / a.rows_per_split;
    const int ct_last = p.C - ((p.C + a.ct - 1) / a.ct - 1) * a.ct;
    a.bulk = (p.CRS % 4 == 0) && ((a.ct * p.RS) % 4 == 0) && ((ct_last * p.RS) % 4 == 0);
    // each producer group stages 32 rows of its dW segment in the ring
    if ((long long)2 * 32 * a.ct * p.RS * 4 > (long long)kW2Ring * a.nk * 128) a.bulk = 0;

    CUtensorMap tm;
    const uint64_t d[4] = {(uint64_t)g.Qp, (uint64_t)g.Pe, (uint64_t)p.K, (uint64_t)p.N};
    const uint32_t b[4] = {32, 1, (uint32_t)a.nk, 1};
    if (!encode_4d(&tm, dzt, d, b)) return cudaErrorInvalidValue;
    const size_t smem = (size_t)kW2Ring * a.nk * 128 + 1024;
    cudaError_t e = cudaFuncSetAttribute(wgrad_tc2_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.K + a.nk - 1) / a.nk, (p.C + a.ct - 1) / a.ct, (unsigned)(segs * a.splits_per_seg));
    wgrad_tc2_kernel<<<grid, kW2Threads, smem, st>>>(tm, a);
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_dgrad_tc2(const Plan &p, const float *Wt, const float *dzt,
                             const float *residual, float *prev, void *ws, float *wr,
                             cudaStream_t st, int *launches) {
    const V2Geom g = v2_geom(p);
    const int Kw = (p.K + 3) / 4 * 4;
    {
        const long long total = (long long)p.R * p.S * p.C * Kw;
        const int blocks = (int)std::min<long long>((total + 255) / 256, (long long)p.num_sms * 8);
        repack_wr_kernel<<<blocks, 256, 0, st>>>(Wt, p.K, p.C, p.R, p.S, Kw, wr);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    const int sdv = p.stride;
    for (int cl = 0; cl < sdv * sdv; ++cl) {
        Dg2Args a;
        a.dzt = dzt; a.residual = residual; a.prev = prev;
        a.status = ws_at<unsigned>(ws, p.off_status);
        a.C = p.C; a.He = g.He; a.We = g.We; a.K = p.K; a.Pe = g.Pe; a.Qe = g.Qe; a.Qp = g.Qp;
        a.stride = sdv; a.accumulate = p.accumulate;
        a.ph = cl / sdv; a.pw = cl % sdv;
        a.Hc = a.ph < g.He ? (g.He - a.ph + sdv - 1) / sdv : 0;
        a.Wc = a.pw < g.We ? (g.We - a.pw + sdv - 1) / sdv : 0;
        if (a.Hc == 0 || a.Wc == 0) continue;
        a.nr = 0;
        for (int r = (a.ph + p.pad) % sdv; r < p.R; r += sdv) {
            a.r_of[a.nr] = r;
            a.dp[a.nr] = (a.ph + p.pad - r) / sdv;
            ++a.nr;
        }
        a.ns = 0;
        int mn = 1 << 30, mx = -(1 << 30);
        for (int s = (a.pw + p.pad) % sdv; s < p.S; s += sdv) {
            a.s_of[a.ns] = s;
            a.dq[a.ns] = (a.pw + p.pad - s) / sdv;
            mn = std::min(mn, a.dq[a.ns]);
            mx = std::max(mx, a.dq[a.ns]);
            ++a.ns;
        }
        if (a.ns == 0) { mn = 0; mx = 0; }
        a.min_dq = mn;
        a.span = mx - mn;
        a.Wx = a.Wc + a.span;
        const int ns1 = std::max(1, a.ns);
        // (s, c) columns per block <= 256, c_tile a multiple of 16
        int cap = std::max(16, (256 / ns1) / 16 * 16);
        const int ctiles = (p.C + cap - 1) / cap;
        a.c_tile = std::min(cap, ((p.C + ctiles - 1) / ctiles + 15) / 16 * 16);
        a.ncol = ns1 * a.c_tile;
        a.kchunks = (p.K + 31) / 32;
        a.T = (2 * a.ncol + 2 * kD2NA * 32 <= 512) ? 2 : 1;
        a.ncols = pow2_cols(a.T * a.ncol + a.T * kD2NA * 32);
        if (a.ncols > 512) return cudaErrorNotSupported;
        a.total_pos = (long long)p.N * a.Hc * a.Wx;
        const int tstride = 128 - a.span;
        a.total_tiles = (int)((a.total_pos + tstride - 1) / tstride);
        a.pitch = (uint32_t)a.ncol + 1;
        if (a.ns == 0) a.nr = 0;  // no kernel column reaches this class

        CUtensorMap tmw;
        const uint64_t d[4] = {(uint64_t)Kw, (uint64_t)p.C, (uint64_t)p.S, (uint64_t)p.R};
        const uint32_t b[4] = {32, (uint32_t)a.c_tile, 1, 1};
        if (!encode_4d(&tmw, wr, d, b)) return cudaErrorInvalidValue;
        const size_t ring = (size_t)kD2Ring * a.ncol * 128;
        const size_t stage = (size_t)a.T * 128 * a.pitch * 4;  // one staging area per tile
        const size_t smem = std::max(ring, stage) + 1024;
        cudaError_t e = cudaFuncSetAttribute(dgrad_tc2_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        dim3 grid((unsigned)((a.total_tiles + a.T - 1) / a.T), (p.C + a.c_tile - 1) / a.c_tile);
        dgrad_tc2_kernel<<<grid, kD2Threads, smem, st>>>(tmw, a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    return cudaSuccess;
}

}  // namespace cba
