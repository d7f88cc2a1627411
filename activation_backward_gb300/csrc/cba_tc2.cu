// cba_tc2.cu -- the input gradient on the tensor cores, and the dz pass that
// feeds it.
//
// dz pass (`dzc_kernel`): the BN-input gradient dz (activation derivative and
// normalize_delta of "YOLOv3反向传播原理 之 全流程源码分析" §4, applied to delta
// with the per-channel coefficients of the reduction pass), TF32-rounded and
// written channels-last, dzc[n][pp][qq][k] on a grid of Pp x Qpp positions: the
// data sits at row offset bd_lo and column offset bq_lo and a zero border
// surrounds it, wide enough for every row and column shift below.  1x1
// stride-1 unpadded layers view each P x Q plane as one row of length P*Q.
//
// Input gradient (prev[n][c][h][w] = sum_{r,s,k} W[k][c][r][s] dz[n][k][p][q]
// with h = p*st + r - pad, w = q*st + s - pad: col2im(W^T . dz) of §3.1 / §3.2
// written as a gather).  Output pixels are split into stride phase classes
// (h mod st, w mod st); within a class the kernel rows r and columns s that
// reach it give row shifts dp_r and column shifts dq_s on dz's grid.  One GEMM
// per class:
//   A (M = 128 grid positions x 32 channels k per step) is a TMA box of dzc,
//     started dp_r rows further on for kernel row r: every tap shift is a
//     tensor-map coordinate, no thread touches an operand;
//   B (N = the class's kernel columns s times a tile of input channels c) is
//     a box of the repacked weights wr[r][s][c][k] (written by extra blocks of
//     the reduction pass);
//   D[position][(s, c)] accumulates over r and k in TMEM.  The epilogue
//     finishes the column shifts, prev(i, j) = sum_s D(i, j + dq_s)[s, c]
//     (a warp hands the lanes at its edge to its neighbour through shared
//     memory), and adds the shortcut delta (§5) and, when accumulating, the
//     old prev_delta -- or, for layers with either, adds its result at the L2
//     onto prev, which `prev_init_kernel` has first set to residual (+ prev).
// `dgrad_tc4_kernel` is persistent, one block per SM, with two TMEM
// accumulators so that a tile's epilogue overlaps the next tile's MMAs;
// `dgrad_tc4_classes_kernel` runs the classes of a strided layer side by side
// in one launch (each class on its own share of the SMs, in proportion to its
// work), so that the small classes do not each leave most of the GPU idle;
// `dgrad_tc3_kernel` (one tile pair per block) takes the classes whose column
// span or kernel-column count is past what the persistent kernel's halo and
// TMEM budget hold.
//
// All waits are bounded (2 s); see cba_ptx.cuh.
#include <cuda.h>

#include <cstring>
#include <vector>

#include "cba_internal.cuh"
#include "cba_ptx.cuh"

namespace cba {

namespace {

constexpr uint64_t kLimitNs = 2000000000ull;
constexpr int kD2MaxTaps = 8;  // kernel rows / columns per stride phase class

__device__ __forceinline__ float to_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}


// ------------------------------------------------------------ dz pass

// dz in the channels-last layout only: dzc [N][Pp][Qpp][Kp] with a zero border
// of bd_lo / bq_lo rows / columns before the data (zeros after it too, and in
// the channels K .. Kp-1).  Block (bx, n * Pp + pp, kz): bx < nqc transposes
// output columns 32 bx .. 32 bx + 31 of row pp - bd_lo for the 64 channels
// 64 kz .. 64 kz + 63 through shared memory (each thread reads 4 consecutive
// columns of one channel from each input, and writes 4 consecutive channels
// of one column as a float4).  The first and last column chunks of a row also
// write its left and right border columns.
template <int ACT, bool BN, bool VEC>
__global__ void __launch_bounds__(256)
    dzc_kernel(const float *__restrict__ delta, const float *__restrict__ output,
               const float *__restrict__ z, const Coef *__restrict__ coef, int K, int Pe, int Qe,
               int Kp, int Pp, int Qpp, int bd_lo, int bq_lo, int nqc, float *__restrict__ dzc,
               float *__restrict__ dzt) {
    ptx::griddep_wait();  // the coefficients come from the reduction pass
    __shared__ float tile[32][65];
    const int t = threadIdx.x;
    const int n = blockIdx.y / Pp, pp = blockIdx.y - (blockIdx.y / Pp) * Pp, p = pp - bd_lo;
    // channel chunks in descending order: the reduction pass read the high
    // channels last, so they are the ones still in L2
    const int k0 = (gridDim.z - 1 - blockIdx.z) * 64;
    float *rowp = dzc + ((size_t)n * Pp + pp) * Qpp * Kp;
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
    {  // border columns: the left ones with the first column chunk, the right ones with the last
        const int nl = blockIdx.x == 0 ? bq_lo : 0;
        const int nr = (int)blockIdx.x == nqc - 1 ? Qpp - bq_lo - Qe : 0;
        for (int i = t; i < (nl + nr) * 16; i += 256) {
            const int c = i >> 4, kc = k0 + (i & 15) * 4;
            const int pq = c < nl ? c : bq_lo + Qe + (c - nl);
            if (kc < Kp) *reinterpret_cast<float4 *>(rowp + (size_t)pq * Kp + kc) = zero4;
        }
    }
    const int q0 = blockIdx.x * 32;
    if (p < 0 || p >= Pe) {  // zero border row
        for (int i = t; i < 32 * 16; i += 256) {
            const int qq = i >> 4, kc = k0 + (i & 15) * 4;
            if (q0 + qq < Qe && kc < Kp)
                *reinterpret_cast<float4 *>(rowp + (size_t)(q0 + qq + bq_lo) * Kp + kc) = zero4;
        }
        return;
    }
    {
        const int kk = t >> 3, q4 = t & 7;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int kl = kk + 32 * pass, k = k0 + kl;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (k < K) {
                const size_t base = (((size_t)n * K + k) * Pe + p) * Qe;
                const Coef cf = coef[k];
                float d[4], y[4], zz[4];
                if (VEC && q0 + 4 * q4 < Qe) {  // rows 16-byte aligned, Qe a multiple of 4
                    const size_t o = base + q0 + 4 * q4;
                    const float4 d4 = __ldg(reinterpret_cast<const float4 *>(delta + o));
                    d[0] = d4.x; d[1] = d4.y; d[2] = d4.z; d[3] = d4.w;
                    if constexpr (ACT == CBA_ACT_LEAKY) {
                        const float4 y4 = __ldg(reinterpret_cast<const float4 *>(output + o));
                        y[0] = y4.x; y[1] = y4.y; y[2] = y4.z; y[3] = y4.w;
                    } else {
                        y[0] = y[1] = y[2] = y[3] = 0.f;
                    }
                    if constexpr (BN) {
                        const float4 z4 = __ldg(reinterpret_cast<const float4 *>(z + o));
                        zz[0] = z4.x; zz[1] = z4.y; zz[2] = z4.z; zz[3] = z4.w;
                    } else {
                        zz[0] = zz[1] = zz[2] = zz[3] = 0.f;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int q = q0 + 4 * q4 + e;
                        const bool in = !VEC && q < Qe;
                        d[e] = in ? __ldg(delta + base + q) : 0.f;
                        y[e] = (ACT == CBA_ACT_LEAKY && in) ? __ldg(output + base + q) : 0.f;
                        zz[e] = (BN && in) ? __ldg(z + base + q) : 0.f;
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = to_tf32(dz_of<ACT, BN>(d[e], y[e], zz[e], cf));
                if (dzt != nullptr) {  // dz in the input's own [N][K][Pe][Qe] order too
                    const int q = q0 + 4 * q4;
                    if (VEC) {
                        if (q < Qe)
                            *reinterpret_cast<float4 *>(dzt + base + q) =
                                make_float4(v[0], v[1], v[2], v[3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (q + e < Qe) dzt[base + q + e] = v[e];
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) tile[4 * q4 + e][kl] = v[e];
        }
    }
    __syncthreads();
    ptx::griddep_launch_dependents();  // the weight gradient may be scheduled
    {
        const int qq = t >> 4, k4 = t & 15;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int ql = qq + 16 * pass, q = q0 + ql, kc = k0 + 4 * k4;
            if (q < Qe && kc < Kp)
                *reinterpret_cast<float4 *>(rowp + (size_t)(q + bq_lo) * Kp + kc) =
                    make_float4(tile[ql][4 * k4], tile[ql][4 * k4 + 1], tile[ql][4 * k4 + 2],
                                tile[ql][4 * k4 + 3]);
        }
    }
}

// ------------------------------------------------------------------ dgrad

constexpr int kD3Stages = 3;
constexpr int kD3Threads = 320;  // TMA warp, MMA warp, 8 epilogue warps

struct Dg3Args {
    float *prev;
    unsigned *status;
    int C, He, We, Pp, Qpp, bd_lo, bq_lo, stride;
    // red_add: prev already holds what the output is added to (the residual,
    // plus its old value when accumulating; written by prev_init_kernel): the
    // output is added at the L2.  Otherwise it is stored.
    int red_add;
    int ph, pw, Hc, Wc, min_dq, span;
    int nr, r_of[kD2MaxTaps], dp[kD2MaxTaps];
    int ns, s_of[kD2MaxTaps], dq[kD2MaxTaps];
    int c_tile, ncol, kchunks, total_tiles;
    long long total_pos;  // N * Pp * Qpp padded positions
    uint32_t ncols;       // TMEM columns allocated (2 * ncol, power of 2)
};

struct D3Bars {
    uint64_t full[kD3Stages], empty[kD3Stages], accum;
    uint32_t tmem_base;
    int abort_flag;
};

// Output of one pixel (one staging lane): for each of its cl_hi channels, the
// sum over the class's kernel columns of the staged E values at lane offsets
// dq[si] (column-major staging, 128 lanes per column), stored or added at the
// L2 (red_add).
__device__ __forceinline__ void dgrad_out_lane(const float *__restrict__ sl,
                                               float *__restrict__ prev, long long pix,
                                               long long HW, int c0, int cl_hi, int c_tile, int ns,
                                               const int (&dq)[kD2MaxTaps], int red_add) {
    for (int cl = 0; cl < cl_hi; cl += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = 0.f;
        for (int si = 0; si < ns; ++si) {
            const float *sc = sl + dq[si] + (si * c_tile + cl) * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (cl + u < cl_hi) v[u] += sc[u * 128];
        }
        if (red_add) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (cl + u < cl_hi) ptx::red_add_f32(prev + pix + (long long)(c0 + cl + u) * HW, v[u]);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (cl + u < cl_hi) prev[pix + (long long)(c0 + cl + u) * HW] = v[u];
        }
    }
}

// Two 128-row tiles per block share every B stage.  A tiles come straight
// from the channels-last zero-bordered dz (TMA, rows shifted by dp*Qpp for
// kernel row r); no thread touches an operand.
__global__ void __launch_bounds__(kD3Threads, 1)
    dgrad_tc3_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmw,
                     const Dg3Args a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ D3Bars sb;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = blockIdx.y * a.c_tile;
    const int tstride = 128 - a.span;
    const int nstages = a.nr * a.kchunks;
    const uint32_t b_bytes = (uint32_t)a.ncol * 128u;
    const uint32_t stage_bytes = 2u * 16384u + b_bytes;
    const uint32_t idesc = ptx::idesc_tf32(128, a.ncol);
    long long m0[2];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) m0[tt] = (long long)(blockIdx.x * 2 + tt) * tstride + a.min_dq;

    if (tid == 0) {
        for (int i = 0; i < kD3Stages; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&sb.accum), 1);
        sb.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&sb.tmem_base), a.ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sb.tmem_base;

    if (warp == 0) {
        // ---- TMA producer: per stage (kernel row r, 32 output channels k):
        // A of both tiles and the W slices of all kernel columns of the class
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nstages; ++i, ++issued) {
                const int slot = i % kD3Stages;
                if (i >= kD3Stages &&
                    !ptx::mbar_wait_bounded(ptx::smem_u32(&sb.empty[slot]),
                                            (uint32_t)(i / kD3Stages - 1) & 1u, &sb.abort_flag,
                                            a.status, kLimitNs))
                    break;
                const int ri = i / a.kchunks, kc = i - (i / a.kchunks) * a.kchunks;
                const uint32_t bar = ptx::smem_u32(&sb.full[slot]);
                uint8_t *st = smem + (size_t)slot * stage_bytes;
                ptx::mbar_arrive_expect_tx(bar, stage_bytes);
#pragma unroll
                for (int tt = 0; tt < 2; ++tt)
                    ptx::tma_load_2d(ptx::smem_u32(st + tt * 16384), &tma, kc * 32,
                                     (int)(m0[tt] + (long long)a.dp[ri] * a.Qpp), bar);
                for (int si = 0; si < a.ns; ++si)
                    ptx::tma_load_4d(ptx::smem_u32(st + 32768 + (size_t)si * a.c_tile * 128), &tmw,
                                     kc * 32, c0, a.s_of[si], a.r_of[ri], bar);
            }
            int no_abort = 0;
            for (int i = max(0, issued - kD3Stages); i < issued; ++i)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.full[i % kD3Stages]),
                                       (uint32_t)(i / kD3Stages) & 1u, &no_abort, a.status,
                                       kLimitNs);
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0 && nstages > 0) {
            bool ok = true;
            for (int i = 0; ok && i < nstages; ++i) {
                const int slot = i % kD3Stages;
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.full[slot]),
                                            (uint32_t)(i / kD3Stages) & 1u, &sb.abort_flag,
                                            a.status, kLimitNs);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t base = ptx::smem_u32(smem + (size_t)slot * stage_bytes);
                for (int tt = 0; tt < 2; ++tt) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ad = ptx::smem_desc(base + tt * 16384 + ks * 32, 16, 1024, 2);
                        const uint64_t bd = ptx::smem_desc(base + 32768 + ks * 32, 16, 1024, 2);
                        ptx::mma_tf32(tmem + (uint32_t)(tt * a.ncol), ad, bd, idesc,
                                      (i > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                ptx::mma_commit(ptx::smem_u32(&sb.empty[slot]));
            }
            ptx::mma_commit(ptx::smem_u32(&sb.accum));
            int no_abort = 0;
            ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &no_abort, a.status, kLimitNs);
        }
    } else {
        // ---- epilogue (warps 2-9, two groups; warp & 3 is the TMEM lane
        // quarter): E -> column-major staging (each group half the columns) ->
        // shifted sum over the kernel columns (each group half the channels)
        // -> prev_delta (stored, or added at the L2)
        const int eg = (warp - 2) >> 2, wq = warp & 3;
        const int L = wq * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        bool ok = true;
        if (nstages > 0)
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &sb.abort_flag, a.status,
                                        kLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            ptx::tc_fence_after();
            float *stg = reinterpret_cast<float *>(smem);
            const long long HW = (long long)a.He * a.We;
            const long long plane = (long long)a.Pp * a.Qpp;
            const int half = (a.ncol / 2 + 15) / 16 * 16;
            const int col_lo = eg == 0 ? 0 : half, col_hi = eg == 0 ? half : a.ncol;
            const int cl_all = min(a.c_tile, a.C - c0);
            const int ch_half = (cl_all + 1) / 2;
            for (int tt = 0; tt < 2; ++tt) {
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
                    for (int j = 0; j < 32; ++j) stg[(col + j) * 128 + L] = v[j];
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
                    for (int j = 0; j < 16; ++j) stg[(col + j) * 128 + L] = v[j];
                }
                ptx::named_bar_sync(1, 256);
                // home lane L: padded position m = m0 + L - min_dq
                const long long m = m0[tt] + L - a.min_dq;
                const int tile = blockIdx.x * 2 + tt;
                bool out = L < tstride && tile < a.total_tiles && m >= 0 && m < a.total_pos;
                int n = 0, i = 0, j = 0;
                if (out) {
                    n = (int)(m / plane);
                    const int rem = (int)(m - (long long)n * plane);
                    i = rem / a.Qpp - a.bd_lo;
                    j = rem % a.Qpp - a.bq_lo;
                    out = i >= 0 && i < a.Hc && j >= 0 && j < a.Wc;
                }
                if (out) {
                    const int h = i * a.stride + a.ph, w = j * a.stride + a.pw;
                    const long long pix = (long long)n * a.C * HW + (long long)h * a.We + w;
                    int dqr[kD2MaxTaps];
#pragma unroll
                    for (int si = 0; si < kD2MaxTaps; ++si) dqr[si] = a.dq[si] - a.min_dq;
                    const int cb = eg == 0 ? 0 : ch_half, ce = eg == 0 ? ch_half : cl_all;
                    dgrad_out_lane(stg + L + cb * 128, a.prev, pix, HW, c0 + cb, ce - cb,
                                   a.c_tile, a.ns, dqr, a.red_add);
                }
                ptx::named_bar_sync(1, 256);
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, a.ncols);
    }
}

// Persistent input gradient: the CTA loops over work units (one 128-position
// tile of one channel tile), with two TMEM accumulators so that the
// epilogue of unit i runs while the MMAs of unit i + 1 do.  Per stage (kernel
// row r, kpb chunks of 32 output channels k): A = the dzc rows of the tile
// shifted by dp_r, B = the W slices of all the class's kernel columns; each
// is one TMA copy when the chunks and slices are consecutive (a copy costs
// the issuing SM a fixed time whatever its size, so few large copies keep
// the tensor pipe fed).  Epilogue: each warp takes 16 channels of its 32
// positions, loads E[., (s, c)] for its kernel columns s from TMEM, shifts it
// down by dq_s lanes with warp shuffles (the lanes past the warp come from
// the next warp through a small shared-memory halo, double-buffered so that
// one barrier per chunk suffices), sums over s and stores prev_delta or adds
// it at the L2.
constexpr int kD4Stages = 6;
constexpr int kD4Threads = 352;  // A TMA warp, MMA warp, 8 epilogue warps, W TMA warp
constexpr int kD4MaxClasses = 4;  // stride phase classes in one launch (stride <= 2)
constexpr int kD4Slots = 6;      // TMEM loads (16 columns each) one epilogue warp has in flight
constexpr int kD4HaloLanes = 4;  // lanes a warp passes to the warp below (the class's column span)
constexpr int kD4LdBatch = 2;    // TMEM loads in flight per wait in the flat 1x1 epilogue

struct D4Args {
    Dg3Args g;
    int ctiles;        // channel tiles
    int total_units;   // total_tiles * ctiles
    int nst;           // pipeline stages in use
    int w_one;         // W slices of the class in one copy
    int kpb;           // 32-channel chunks of k per stage (1, or 2 with 3-D / 5-D copies)
    int kst;           // stages per kernel row: ceil(kchunks / kpb)
    uint32_t halo_off; // byte offset of the epilogue halo in shared memory
};

struct D4Bars {
    uint64_t full[kD4Stages], empty[kD4Stages], acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
};

// One epilogue batch of dgrad_tc4 for a warp: NB chunks of 16 channels (the
// group's chunks t0 .. t0 + NB - 1) times the NS kernel columns of the class,
// all TMEM loads in flight together.  Publishes lanes 0 .. span-1 of every
// slot to the halo, meets the group at a barrier, shifts every column down by
// its dq with warp shuffles (the top lanes from the next warp's halo), sums
// the columns and writes the NB chunks.  `release` arrives on the unit's
// accumulator-empty barrier right after the loads.
struct D4Epi {
    uint32_t tbase;       // TMEM address of this warp's lanes in the unit's accumulator
    int c_tile, eg, wq, lane, span;
    const int *dqr;
    float *hpar;          // this batch's halo parity
    long long pix, HW;
    int c0, cl_all;
    bool out;
    float *prev;
    int red_add;
};

template <int NS, int NB>
__device__ __forceinline__ void d4_epilogue_batch(const D4Epi &E, int t0, uint64_t *release) {
    constexpr int NV = NS * NB;
    constexpr size_t kHSlot = (size_t)16 * kD4HaloLanes;
    float v[NV][16];
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        const int cc = E.eg + 2 * (t0 + q / NS);
        ptx::tmem_ld16(E.tbase + (uint32_t)((q % NS) * E.c_tile + cc * 16), v[q]);
    }
    ptx::tmem_ld_wait();
    if (release) {
        // the unit's last loads are done: the MMAs may reuse the buffer
        ptx::tc_fence_before();
        __syncwarp();
        if (E.lane == 0) ptx::mbar_arrive(ptx::smem_u32(release));
    }
    if (E.lane < E.span) {
        // value-major ([e][lane]) so that the reads below touch distinct banks
        float *hw = E.hpar + (size_t)(E.eg * 4 + E.wq) * kD4Slots * kHSlot;
#pragma unroll
        for (int q = 0; q < NV; ++q)
#pragma unroll
            for (int e = 0; e < 16; ++e) hw[q * kHSlot + e * kD4HaloLanes + E.lane] = v[q][e];
    }
    ptx::named_bar_sync(1 + E.eg, 128);
    const float *hn = E.hpar + (size_t)(E.eg * 4 + ((E.wq + 1) & 3)) * kD4Slots * kHSlot;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        const int dsh = E.dqr[q % NS];
        if (dsh != 0) {  // warp-uniform
#pragma unroll
            for (int e = 0; e < 16; ++e) v[q][e] = __shfl_down_sync(0xffffffffu, v[q][e], dsh);
            // the top dsh lanes take the next warp's lanes 0 .. dsh-1
            if (E.lane + dsh >= 32) {
                const int hl = E.lane + dsh - 32;
#pragma unroll
                for (int e = 0; e < 16; ++e) v[q][e] = hn[q * kHSlot + e * kD4HaloLanes + hl];
            }
        }
        if (q % NS != 0) {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[q - q % NS][e] += v[q][e];
        }
    }
    if (E.out) {
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            const int cc = E.eg + 2 * (t0 + t);
            const int nvalid = min(16, E.cl_all - cc * 16);
            const long long idx0 = E.pix + (long long)(E.c0 + cc * 16) * E.HW;
            if (E.red_add) {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (e < nvalid) ptx::red_add_f32(E.prev + idx0 + (long long)e * E.HW, v[t * NS][e]);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (e < nvalid) E.prev[idx0 + (long long)e * E.HW] = v[t * NS][e];
            }
        }
    }
}

// A batch of nb (1 .. kD4Slots / NS) chunks; nb = 0 only releases.
template <int NS>
__device__ __forceinline__ void d4_epilogue_nb(const D4Epi &E, int t0, int nb, uint64_t *release) {
    constexpr int BCH = kD4Slots / NS;
    if (nb <= 0) {
        if (release) {
            ptx::tc_fence_before();
            __syncwarp();
            if (E.lane == 0) ptx::mbar_arrive(ptx::smem_u32(release));
        }
        return;
    }
    if constexpr (BCH >= 6) { if (nb == 6) { d4_epilogue_batch<NS, 6>(E, t0, release); return; } }
    if constexpr (BCH >= 5) { if (nb == 5) { d4_epilogue_batch<NS, 5>(E, t0, release); return; } }
    if constexpr (BCH >= 4) { if (nb == 4) { d4_epilogue_batch<NS, 4>(E, t0, release); return; } }
    if constexpr (BCH >= 3) { if (nb == 3) { d4_epilogue_batch<NS, 3>(E, t0, release); return; } }
    if constexpr (BCH >= 2) { if (nb == 2) { d4_epilogue_batch<NS, 2>(E, t0, release); return; } }
    d4_epilogue_batch<NS, 1>(E, t0, release);
}

// The persistent input-gradient GEMM of one stride phase class, run by block
// bid of the class's nblk blocks.
__device__ __forceinline__ void dgrad_tc4_body(const CUtensorMap *tma, const CUtensorMap *tmw,
                                               const CUtensorMap *tmw1, const D4Args &d, int bid,
                                               int nblk) {
    const Dg3Args &a = d.g;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ D4Bars sb;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tstride = 128 - a.span;
    const int nstages = a.nr * d.kst;
    const uint32_t a_bytes = (uint32_t)d.kpb * 16384u;
    const uint32_t b_chunk = (uint32_t)a.ncol * 128u;  // one k-chunk of the W slices
    const uint32_t b_bytes = (uint32_t)d.kpb * b_chunk;
    const uint32_t stage_bytes = a_bytes + b_bytes;
    const int nunits = d.total_units > bid
                           ? (d.total_units - 1 - bid) / nblk + 1
                           : 0;

    if (tid == 0) {
        for (int i = 0; i < kD4Stages; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.full[i]), 2);  // the A and the W issuer
            ptx::mbar_init(ptx::smem_u32(&sb.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.acc_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.acc_empty[i]), 8);  // the 8 epilogue warps
        }
        ptx::mbar_init(ptx::smem_u32(&sb.drain), 1);
        sb.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&sb.tmem_base), a.ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sb.tmem_base;
    // dzc, wr and prev are touched only after the previous kernels completed
    ptx::griddep_wait();

    if (warp == 0 || warp == 10) {
        // ---- TMA: warp 0 the A tiles, warp 10 the W slices
        if (lane == 0) {
            const bool wside = warp == 10;
            int gs = 0;  // global stage counter
            bool ok = true;
            for (int i = 0; ok && i < nunits; ++i) {
                const int u = bid + i * nblk;
                const int ct = u / a.total_tiles, tile = u - ct * a.total_tiles;
                const int c0 = ct * a.c_tile;
                const long long m0 = (long long)tile * tstride + a.min_dq;
                for (int st = 0; st < nstages; ++st, ++gs) {
                    const int slot = gs % d.nst;
                    if (gs >= d.nst)
                        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.empty[slot]),
                                                    (uint32_t)(gs / d.nst - 1) & 1u,
                                                    &sb.abort_flag, a.status, kLimitNs);
                    if (!ok) break;
                    const int ri = st / d.kst, kc = (st - ri * d.kst) * d.kpb;
                    const uint32_t bar = ptx::smem_u32(&sb.full[slot]);
                    uint8_t *sp = smem + (size_t)slot * stage_bytes;
                    const int row = (int)(m0 + (long long)a.dp[ri] * a.Qpp);
                    if (!wside) {
                        ptx::mbar_arrive_expect_tx(bar, a_bytes);
                        if (d.kpb == 1)
                            ptx::tma_load_2d(ptx::smem_u32(sp), tma, kc * 32, row, bar);
                        else
                            ptx::tma_load_3d(ptx::smem_u32(sp), tma, 0, row, kc, bar);
                    } else {
                        ptx::mbar_arrive_expect_tx(bar, b_bytes);
                        if (d.kpb > 1)
                            ptx::tma_load_5d(ptx::smem_u32(sp + a_bytes), tmw, 0, c0, a.s_of[0],
                                             kc, a.r_of[ri], bar);
                        else if (d.w_one)
                            ptx::tma_load_4d(ptx::smem_u32(sp + a_bytes), tmw, kc * 32, c0,
                                             a.s_of[0], a.r_of[ri], bar);
                        else
                            for (int si = 0; si < a.ns; ++si)
                                ptx::tma_load_4d(
                                    ptx::smem_u32(sp + a_bytes + (size_t)si * a.c_tile * 128),
                                    tmw1, kc * 32, c0, a.s_of[si], a.r_of[ri], bar);
                    }
                }
            }
            int no_abort = 0;
            for (int i = max(0, gs - d.nst); i < gs; ++i)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.full[i % d.nst]),
                                       (uint32_t)(i / d.nst) & 1u, &no_abort, a.status, kLimitNs);
        }
    } else if (warp == 1) {
        // ---- MMA issue: unit i into accumulator i & 1
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_tf32(128, a.ncol);
            int gs = 0;
            bool ok = true;
            for (int i = 0; ok && i < nunits; ++i) {
                const int b = i & 1;
                if (i >= 2)
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.acc_empty[b]),
                                                (uint32_t)((i >> 1) - 1) & 1u, &sb.abort_flag,
                                                a.status, kLimitNs);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t dtm = tmem + (uint32_t)(b * a.ncol);
                for (int st = 0; st < nstages; ++st, ++gs) {
                    const int slot = gs % d.nst;
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.full[slot]),
                                                (uint32_t)(gs / d.nst) & 1u, &sb.abort_flag,
                                                a.status, kLimitNs);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint32_t base = ptx::smem_u32(smem + (size_t)slot * stage_bytes);
                    const uint64_t ad0 = ptx::smem_desc(base, 16, 1024, 2);
                    const uint64_t bd0 = ptx::smem_desc(base + a_bytes, 16, 1024, 2);
                    for (int j = 0; j < d.kpb; ++j) {
                        // descriptor start addresses count 16-byte units
                        const uint64_t ad = ad0 + (uint64_t)(j * (16384 >> 4));
                        const uint64_t bd = bd0 + (uint64_t)(j * (b_chunk >> 4));
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            ptx::mma_tf32(dtm, ad + 2 * ks, bd + 2 * ks, idesc,
                                          (st > 0 || j > 0 || ks > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(ptx::smem_u32(&sb.empty[slot]));
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_u32(&sb.acc_full[b]));
            }
            if (!ok) {
                *reinterpret_cast<volatile int *>(&sb.abort_flag) = 1;
                __threadfence_block();
            }
            // drain: every MMA issued has finished before TMEM is released
            ptx::mma_commit(ptx::smem_u32(&sb.drain));
            int no_abort = 0;
            ptx::mbar_wait_bounded(ptx::smem_u32(&sb.drain), 0, &no_abort, a.status, kLimitNs);
        }
    } else {
        // ---- epilogue: group eg of 4 warps (one per TMEM lane quarter) takes
        // the 16-channel chunks cc = eg, eg + 2, ... of the unit's channels,
        // a batch of whole chunks at a time: every TMEM load of the batch is in
        // flight together, the accumulator is released after the unit's last
        // loads, and one barrier per batch publishes the halo.
        const int eg = (warp - 2) >> 2, wq = warp & 3;
        const int L = wq * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const long long HW = (long long)a.He * a.We;
        const long long plane = (long long)a.Pp * a.Qpp;
        const int span = a.span, ns = a.ns;
        // halo[par][eg][wq][slot][16][4]: lanes 0 .. span-1 (span <= 4) of each
        // warp, for the warp below; par alternates with the group's batches
        float *halo = reinterpret_cast<float *>(smem + d.halo_off);
        constexpr size_t kHSlot = (size_t)16 * kD4HaloLanes;
        int dqr[kD2MaxTaps];
#pragma unroll
        for (int si = 0; si < kD2MaxTaps; ++si) dqr[si] = a.dq[si] - a.min_dq;
        const int bch = ns > 0 ? max(1, kD4Slots / ns) : 1;  // chunks per batch
        // the plane-per-image form of 1x1 stride-1 layers: a tile's positions are
        // consecutive in memory within each image, in aligned groups of 4
        const bool flat4 = ns == 1 && span == 0 && a.He == 1 && a.stride == 1 && a.Hc == 1 &&
                           a.bq_lo == 0 && a.Qpp == a.We && HW % 4 == 0 && tstride % 4 == 0;
        int par = 0;
        bool ok = true;
        for (int i = 0; ok && i < nunits; ++i) {
            const int b = i & 1;
            const int u = bid + i * nblk;
            const int ct = u / a.total_tiles, tile = u - ct * a.total_tiles;
            const int c0 = ct * a.c_tile;
            const int cl_all = min(a.c_tile, a.C - c0);
            const int gch = ((cl_all + 15) / 16 - eg + 1) / 2;  // this group's chunks
            // this lane's output pixel (padded position m = tile * tstride + L)
            const long long m = (long long)tile * tstride + L;
            bool out = L < tstride && m < a.total_pos;
            long long pix = 0;
            if (out) {
                const int n = (int)(m / plane);
                const int rem = (int)(m - (long long)n * plane);
                const int ii = rem / a.Qpp - a.bd_lo, jj = rem % a.Qpp - a.bq_lo;
                out = ii >= 0 && ii < a.Hc && jj >= 0 && jj < a.Wc;
                pix = (long long)n * a.C * HW + (long long)(ii * a.stride + a.ph) * a.We +
                      (jj * a.stride + a.pw);
            }
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.acc_full[b]), (uint32_t)(i >> 1) & 1u,
                                        &sb.abort_flag, a.status, kLimitNs);
            // the group's 4 warps agree before the halo barriers below
            ok = ptx::named_bar_and(1 + eg, 128, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            D4Epi E;
            E.tbase = tmem + lane_addr + (uint32_t)(b * a.ncol);
            E.c_tile = a.c_tile; E.eg = eg; E.wq = wq; E.lane = lane; E.span = span;
            E.dqr = dqr; E.pix = pix; E.HW = HW; E.c0 = c0; E.cl_all = cl_all; E.out = out;
            E.prev = a.prev; E.red_add = a.red_add;
            if (flat4) {
                // one plane of positions per image (1x1, stride 1; HW a multiple
                // of 4, at least 32): the warp's 32 positions x 16 channels of a
                // chunk go from TMEM through its staging rows [16][32] in shared
                // memory, then out as float4 along the positions: each memory
                // instruction of the warp moves four whole 128-byte rows instead
                // of 32 scalars spread over a channel plane each.  The TMEM loads
                // go kD4LdBatch chunks at a time before one wait: while the next
                // unit's MMAs run a TMEM load waits behind them, and a wait per
                // chunk cost ~1.5 us each.
                float *stg = halo + (warp - 2) * 512;
                const long long mw = (long long)tile * tstride + wq * 32;  // lane 0's position
                // lane -> (channel row e = k * 4 + lane / 8, positions p4 .. p4 + 3),
                // k = 0 .. 3; the global offset of each, without the channel
                const int p4 = (lane & 7) * 4;
                const long long m = mw + p4;
                const bool mv = m < a.total_pos;
                const long long nimg = m / HW;
                const long long pbase = nimg * a.C * HW + (m - nimg * HW);
                for (int t0 = 0; t0 < gch; t0 += kD4LdBatch) {
                    const int nb = min(kD4LdBatch, gch - t0);
                    float vb[kD4LdBatch][16];
#pragma unroll
                    for (int j = 0; j < kD4LdBatch; ++j)
                        if (j < nb) ptx::tmem_ld16(E.tbase + (uint32_t)((eg + 2 * (t0 + j)) * 16), vb[j]);
                    ptx::tmem_ld_wait();
                    if (t0 + nb >= gch) {  // the unit's last loads: the MMAs may reuse it
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sb.acc_empty[b]));
                    }
#pragma unroll
                    for (int j = 0; j < kD4LdBatch; ++j) {
                        if (j >= nb) break;
                        const int cc = eg + 2 * (t0 + j);
                        const int nvalid = min(16, cl_all - cc * 16);
                        __syncwarp();  // the previous chunk's rows have been read
#pragma unroll
                        for (int e = 0; e < 16; ++e) stg[e * 32 + lane] = vb[j][e];
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int e = k * 4 + (lane >> 3);
                            if (!mv || e >= nvalid) continue;
                            const float4 val = *reinterpret_cast<const float4 *>(stg + e * 32 + p4);
                            float *o = a.prev + pbase + (long long)(c0 + cc * 16 + e) * HW;
                            if (a.red_add) ptx::red_add_v4_f32(o, val);
                            else *reinterpret_cast<float4 *>(o) = val;
                        }
                    }
                }
                if (gch <= 0) {  // no chunk for this group: release at once
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sb.acc_empty[b]));
                }
                continue;
            }
            // every other form (the 1x1 layers whose planes are not 16-byte
            // rows included): kD4Slots / ns chunks of TMEM loads per wait
            int t0 = 0;
            do {  // at least once, so that the accumulator is always released
                const int nb = min(bch, gch - t0);
                uint64_t *rel = t0 + bch >= gch ? &sb.acc_empty[b] : nullptr;
                E.hpar = halo + (size_t)par * 8 * kD4Slots * kHSlot;
                switch (ns) {
                case 1: d4_epilogue_nb<1>(E, t0, nb, rel); break;
                case 2: d4_epilogue_nb<2>(E, t0, nb, rel); break;
                case 3: d4_epilogue_nb<3>(E, t0, nb, rel); break;
                case 4: d4_epilogue_nb<4>(E, t0, nb, rel); break;
                case 5: d4_epilogue_nb<5>(E, t0, nb, rel); break;
                case 6: d4_epilogue_nb<6>(E, t0, nb, rel); break;
                default:  // no kernel tap reaches this class: the gradient is 0
                    d4_epilogue_nb<1>(E, t0, 0, rel);
                    for (int t = t0; out && !a.red_add && t < t0 + nb; ++t) {
                        const int cc = eg + 2 * t;
                        for (int e = 0; e < 16 && cc * 16 + e < cl_all; ++e)
                            a.prev[pix + (long long)(c0 + cc * 16 + e) * HW] = 0.f;
                    }
                    break;
                }
                t0 += bch;
                par ^= 1;
            } while (t0 < gch);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, a.ncols);
    }
}

__global__ void __launch_bounds__(kD4Threads, 1)
    dgrad_tc4_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmw,
                     const __grid_constant__ CUtensorMap tmw1, const D4Args d) {
    dgrad_tc4_body(&tma, &tmw, &tmw1, d, (int)blockIdx.x, (int)gridDim.x);
}

// All stride phase classes of a layer in one launch: blocks first[c] ..
// first[c + 1] - 1 run class c (its own tensor maps and arguments, copied to
// shared memory), each class's block count in proportion to its work, so
// that the classes run side by side instead of one launch after another.
struct D4Classes {
    CUtensorMap tma[kD4MaxClasses], tmw[kD4MaxClasses], tmw1[kD4MaxClasses];
    D4Args d[kD4MaxClasses];
    int first[kD4MaxClasses + 1];
    int ncls;
};

__global__ void __launch_bounds__(kD4Threads, 1)
    dgrad_tc4_classes_kernel(const __grid_constant__ D4Classes m) {
    __shared__ D4Args sd;
    int cls = 0;
    while (cls + 1 < m.ncls && (int)blockIdx.x >= m.first[cls + 1]) ++cls;
    if (threadIdx.x == 0) sd = m.d[cls];
    __syncthreads();
    dgrad_tc4_body(&m.tma[cls], &m.tmw[cls], &m.tmw1[cls], sd, (int)blockIdx.x - m.first[cls],
                   m.first[cls + 1] - m.first[cls]);
}

// -------------------------------------------------------------- host side

// prev = residual (+ prev when accumulating), before the input gradient adds
// its result to prev at the L2: a streaming pass, so that the input
// gradient's epilogue reads nothing.  n elements; float4 where aligned.
__global__ void __launch_bounds__(256)
    prev_init_kernel(float *__restrict__ prev, const float *__restrict__ residual, long long n,
                     int accumulate) {
    ptx::griddep_wait();
    const long long n4 = n / 4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    float4 *p4 = reinterpret_cast<float4 *>(prev);
    const float4 *r4 = reinterpret_cast<const float4 *>(residual);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 r = __ldg(r4 + i);
        if (accumulate) {
            const float4 o = p4[i];
            r.x += o.x; r.y += o.y; r.z += o.z; r.w += o.w;
        }
        p4[i] = r;
    }
    for (long long i = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += stride)
        prev[i] = residual[i] + (accumulate ? prev[i] : 0.f);
    ptx::griddep_launch_dependents();
}

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

// One thread waits on a barrier phase that nothing completes: the bounded wait
// must give up after timeout_us and set the status bit.
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

}  // namespace

// Geometry the TMEM/TMA kernels work in.  1x1 stride-1 unpadded layers are
// viewed as one row per plane.  The channels-last dz copy carries a zero border
// wide enough for every row shift dp and column shift dq of every stride
// phase class of the input gradient.
struct V2Geom {
    int He, We, Pe, Qe, Qp;
    int Kp, Pp, Qpp, bd_lo, bq_lo;
};

struct ClassTaps {
    int Hc, Wc, nr, ns, r_of[kD2MaxTaps], dp[kD2MaxTaps], s_of[kD2MaxTaps], dq[kD2MaxTaps];
    int min_dq, max_dq, min_dp, max_dp;
};

static ClassTaps class_taps(const Plan &p, int He, int We, int cl) {
    ClassTaps c;
    const int sd = p.stride, ph = cl / sd, pw = cl % sd;
    c.Hc = ph < He ? (He - ph + sd - 1) / sd : 0;
    c.Wc = pw < We ? (We - pw + sd - 1) / sd : 0;
    c.nr = c.ns = 0;
    c.min_dp = c.min_dq = 1 << 30;
    c.max_dp = c.max_dq = -(1 << 30);
    for (int r = (ph + p.pad) % sd; r < p.R && c.nr < kD2MaxTaps; r += sd) {
        c.r_of[c.nr] = r;
        c.dp[c.nr] = (ph + p.pad - r) / sd;
        c.min_dp = std::min(c.min_dp, c.dp[c.nr]);
        c.max_dp = std::max(c.max_dp, c.dp[c.nr]);
        ++c.nr;
    }
    for (int s = (pw + p.pad) % sd; s < p.S && c.ns < kD2MaxTaps; s += sd) {
        c.s_of[c.ns] = s;
        c.dq[c.ns] = (pw + p.pad - s) / sd;
        c.min_dq = std::min(c.min_dq, c.dq[c.ns]);
        c.max_dq = std::max(c.max_dq, c.dq[c.ns]);
        ++c.ns;
    }
    if (c.nr == 0 || c.ns == 0) {  // no kernel tap reaches this class
        c.nr = c.ns = 0;
        c.min_dp = c.max_dp = c.min_dq = c.max_dq = 0;
    }
    return c;
}

static V2Geom v2_geom(const Plan &p) {
    V2Geom g;
    const bool flat = p.R == 1 && p.S == 1 && p.stride == 1 && p.pad == 0;
    g.He = flat ? 1 : p.H;
    g.We = flat ? p.H * p.W : p.W;
    g.Pe = flat ? 1 : p.P;
    g.Qe = flat ? p.P * p.Q : p.Q;
    g.Qp = (g.Qe + 3) / 4 * 4;
    g.Kp = (p.K + 3) / 4 * 4;
    int blo = 0, bhi = 0, qlo = 0, qhi = 0;
    for (int cl = 0; cl < p.stride * p.stride; ++cl) {
        const ClassTaps c = class_taps(p, g.He, g.We, cl);
        if (c.Hc == 0 || c.Wc == 0 || c.nr == 0) continue;
        blo = std::max(blo, -c.min_dp);
        bhi = std::max(bhi, c.Hc - 1 + c.max_dp - (g.Pe - 1));
        qlo = std::max(qlo, -c.min_dq);
        qhi = std::max(qhi, c.Wc - 1 + c.max_dq - (g.Qe - 1));
    }
    g.bd_lo = blo;
    g.bq_lo = qlo;
    g.Pp = g.Pe + blo + bhi;
    g.Qpp = g.Qe + qlo + qhi;
    return g;
}

DzcGeom dzc_geom(const Plan &p) {
    const V2Geom g = v2_geom(p);
    DzcGeom d;
    d.He = g.He; d.We = g.We; d.Pe = g.Pe; d.Qe = g.Qe;
    d.Kp = g.Kp; d.Pp = g.Pp; d.Qpp = g.Qpp; d.bd_lo = g.bd_lo; d.bq_lo = g.bq_lo;
    return d;
}

bool tma_encode_f32_swz(void *tmap, const void *base, int rank, const uint64_t *dims,
                        const uint32_t *box, int swizzle_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rank < 1 || rank > 5) return false;
    CUtensorMapSwizzle sw;
    switch (swizzle_bytes) {
    case 0: sw = CU_TENSOR_MAP_SWIZZLE_NONE; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return false;
    }
    cuuint64_t d[5], strides[4];
    cuuint32_t b[5], es[5];
    uint64_t stride = 4;
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i > 0) strides[i - 1] = stride;
        stride *= dims[i];
    }
    return fn(static_cast<CUtensorMap *>(tmap), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank,
              const_cast<void *>(base), d, strides, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_encode_f32(void *tmap, const void *base, int rank, const uint64_t *dims,
                    const uint32_t *box, bool swizzle128) {
    return tma_encode_f32_swz(tmap, base, rank, dims, box, swizzle128 ? 128 : 0);
}

bool tc2_supported(const Plan &p) {
    if (p.stride > 4 || p.R > kD2MaxTaps || p.S > kD2MaxTaps) return false;
    const V2Geom g = v2_geom(p);
    if ((long long)p.N * g.Pp * g.Qpp * g.Kp >= (1LL << 31)) return false;
    if ((long long)p.N * g.Pp > 65535) return false;  // grid.z of the dz pass
    // the input gradient's column shifts must leave room in a 128-row tile
    if ((p.S - 1) / p.stride + 1 > 32) return false;
    return encode_fn() != nullptr;
}

size_t tc2_dzc_bytes(const Plan &p) {
    const V2Geom g = v2_geom(p);
    return sizeof(float) * (size_t)p.N * g.Pp * g.Qpp * g.Kp;
}

size_t tc2_wr_bytes(const Plan &p) {
    return sizeof(float) * (size_t)p.R * p.S * p.C * ((p.K + 3) / 4 * 4);
}

cudaError_t launch_dzc(const Plan &p, const float *delta, const float *output, const float *z,
                       const void *ws, float *dzc, cudaStream_t st, int *launches, float *dzt) {
    const V2Geom g = v2_geom(p);
    const Coef *coef = ws_at<Coef>(ws, p.off_coef);
    const bool leaky = p.act == CBA_ACT_LEAKY;
    const int nqc = (g.Qe + 31) / 32;
    dim3 grid((unsigned)nqc, (unsigned)(p.N * g.Pp), (unsigned)((g.Kp + 63) / 64));
    cudaError_t e = cudaSuccess;
#define CBA_DZC(A, B)                                                                          \
    do {                                                                                       \
        if (g.Qe % 4 == 0)                                                                     \
            e = launch_pdl(dzc_kernel<A, B, true>, grid, dim3(256), 0, st, delta, output, z,   \
                           coef, p.K, g.Pe, g.Qe, g.Kp, g.Pp, g.Qpp, g.bd_lo, g.bq_lo, nqc,   \
                           dzc, dzt);                                                          \
        else                                                                                   \
            e = launch_pdl(dzc_kernel<A, B, false>, grid, dim3(256), 0, st, delta, output, z,  \
                           coef, p.K, g.Pe, g.Qe, g.Kp, g.Pp, g.Qpp, g.bd_lo, g.bq_lo, nqc,   \
                           dzc, dzt);                                                          \
    } while (0)
    if (p.bn) {
        if (leaky) CBA_DZC(CBA_ACT_LEAKY, true);
        else CBA_DZC(CBA_ACT_LINEAR, true);
    } else {
        if (leaky) CBA_DZC(CBA_ACT_LEAKY, false);
        else CBA_DZC(CBA_ACT_LINEAR, false);
    }
#undef CBA_DZC
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_prev_init(const Plan &p, const float *residual, float *prev, cudaStream_t st,
                             int *launches) {
    const long long n = (long long)p.N * p.C * p.H * p.W;
    const unsigned blocks =
        (unsigned)std::min<long long>((n / 4 + 255) / 256 + 1, (long long)p.num_sms * 8);
    cudaError_t e = launch_pdl(prev_init_kernel, dim3(blocks), dim3(256), 0, st, prev, residual, n,
                               p.accumulate);
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaSuccess;
}

cudaError_t launch_dgrad_tc2(const Plan &p, const float *dzc, const float *residual, float *prev,
                             void *ws, const float *wr_c, cudaStream_t st, int *launches) {
    const V2Geom g = v2_geom(p);
    const int Kw = (p.K + 3) / 4 * 4;
    float *wr = const_cast<float *>(wr_c);  // tensor maps take a non-const base; only read
    const long long total_pos = (long long)p.N * g.Pp * g.Qpp;
    CUtensorMap tma;
    {
        EncodeTiledFn fn = encode_fn();
        if (!fn) return cudaErrorNotSupported;
        cuuint64_t dims[2] = {(cuuint64_t)g.Kp, (cuuint64_t)total_pos};
        cuuint64_t strides[1] = {(cuuint64_t)g.Kp * 4};
        cuuint32_t box[2] = {32, 128};
        cuuint32_t es[2] = {1, 1};
        if (fn(&tma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(dzc), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // With a residual or accumulation, prev is set to residual (+ old prev)
    // first and every class adds its result to it at the L2 (red_add).
    const bool red_add = residual != nullptr || p.accumulate != 0;
    if (residual) {
        cudaError_t e = launch_prev_init(p, residual, prev, st, launches);
        if (e != cudaSuccess) return e;
    }
    // the classes that take the persistent kernel, launched together below
    struct Tc4Class {
        D4Args d4;
        CUtensorMap tma4, tmw4, tmw;
        size_t smem;
        long long unit_work;  // (stages per unit + 1) x W columns per stage
    };
    std::vector<Tc4Class> tc4;
    for (int cl = 0; cl < p.stride * p.stride; ++cl) {
        const ClassTaps c = class_taps(p, g.He, g.We, cl);
        if (c.Hc == 0 || c.Wc == 0) continue;
        Dg3Args a;
        a.prev = prev;
        a.red_add = red_add ? 1 : 0;
        a.status = ws_at<unsigned>(ws, p.off_status);
        a.C = p.C; a.He = g.He; a.We = g.We; a.Pp = g.Pp; a.Qpp = g.Qpp;
        a.bd_lo = g.bd_lo; a.bq_lo = g.bq_lo; a.stride = p.stride;
        a.ph = cl / p.stride; a.pw = cl % p.stride; a.Hc = c.Hc; a.Wc = c.Wc;
        a.nr = c.nr; a.ns = c.ns;
        for (int i = 0; i < kD2MaxTaps; ++i) {
            a.r_of[i] = c.r_of[i]; a.dp[i] = c.dp[i]; a.s_of[i] = c.s_of[i]; a.dq[i] = c.dq[i];
        }
        a.min_dq = c.min_dq;
        a.span = c.max_dq - c.min_dq;
        const int ns1 = std::max(1, a.ns);
        // (s, c) columns per block <= 256, c_tile a multiple of 16
        const int cap = std::max(16, (256 / ns1) / 16 * 16);
        const int ctiles = (p.C + cap - 1) / cap;
        a.c_tile = std::min(cap, ((p.C + ctiles - 1) / ctiles + 15) / 16 * 16);
        a.ncol = ns1 * a.c_tile;
        a.ncols = 32;
        while ((int)a.ncols < 2 * a.ncol) a.ncols <<= 1;
        if (a.ncols > 512) return cudaErrorNotSupported;
        a.kchunks = (p.K + 31) / 32;
        a.total_pos = total_pos;
        const int tstride = 128 - a.span;
        a.total_tiles = (int)((total_pos + tstride - 1) / tstride);

        CUtensorMap tmw;
        const uint64_t d[4] = {(uint64_t)Kw, (uint64_t)p.C, (uint64_t)p.S, (uint64_t)p.R};
        const uint32_t b[4] = {32, (uint32_t)a.c_tile, 1, 1};
        if (!encode_4d(&tmw, wr, d, b)) return cudaErrorInvalidValue;

        // persistent, double-buffered kernel when the halo and two
        // accumulators fit
        if (a.span <= kD4HaloLanes && a.ns <= kD4Slots && 2 * a.ncol <= 512) {
            D4Args d4;
            d4.g = a;
            d4.ctiles = (p.C + a.c_tile - 1) / a.c_tile;
            d4.total_units = a.total_tiles * d4.ctiles;
            d4.w_one = a.ns == 1 || p.stride == 1;
            const size_t halo_bytes = (size_t)2 * 8 * kD4Slots * kD4HaloLanes * 16 * 4;
            const size_t cap = 232448 - 2048;  // dynamic shared memory, room for the static part
            CUtensorMap tma4 = tma, tmw4;
            // Two k-chunks per stage in one A copy (3-D view: chunk, position,
            // channel in chunk) and one W copy (5-D view: r, chunk, s, c, k)
            // when the channel pitch is whole chunks and the slices are
            // adjacent: half the copies of one chunk per stage, which measured
            // faster at equal bytes in flight.
            d4.kpb = 1;
            if (Kw % 32 == 0 && g.Kp % 32 == 0 && a.kchunks >= 2 && d4.w_one) {
                const size_t ps2 = 2 * (16384 + (size_t)a.ncol * 128);
                if (2 * ps2 + halo_bytes + 1024 <= cap) {
                    EncodeTiledFn fn = encode_fn();
                    cuuint64_t ad[3] = {32, (cuuint64_t)total_pos, (cuuint64_t)(g.Kp / 32)};
                    cuuint64_t as[2] = {(cuuint64_t)g.Kp * 4, 128};
                    cuuint32_t ab[3] = {32, 128, 2}, es[5] = {1, 1, 1, 1, 1};
                    cuuint64_t wd[5] = {32, (cuuint64_t)p.C, (cuuint64_t)p.S, (cuuint64_t)(Kw / 32),
                                        (cuuint64_t)p.R};
                    cuuint64_t ws5[4] = {(cuuint64_t)Kw * 4, (cuuint64_t)p.C * Kw * 4, 128,
                                         (cuuint64_t)p.S * p.C * Kw * 4};
                    cuuint32_t wb[5] = {32, (cuuint32_t)a.c_tile, (cuuint32_t)std::max(1, a.ns), 2, 1};
                    CUtensorMap t3, t5;
                    if (fn(&t3, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(dzc), ad, as,
                           ab, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
                        fn(&t5, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, wr, wd, ws5, wb, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
                        d4.kpb = 2;
                        tma4 = t3;
                        tmw4 = t5;
                    }
                }
            }
            d4.kst = (a.kchunks + d4.kpb - 1) / d4.kpb;
            const size_t per_stage = (size_t)d4.kpb * (16384 + (size_t)a.ncol * 128);
            d4.nst = (int)std::min<size_t>(kD4Stages, (cap - halo_bytes - 1024) / per_stage);
            if (d4.nst >= 2) {
                d4.halo_off = (uint32_t)(d4.nst * per_stage);
                const size_t smem4 = d4.halo_off + halo_bytes + 1024;
                if (d4.kpb == 1) {
                    // all the class's kernel columns in one box
                    const uint32_t bn[4] = {32, (uint32_t)a.c_tile,
                                            (uint32_t)(d4.w_one ? std::max(1, a.ns) : 1), 1};
                    if (!encode_4d(&tmw4, wr, d, bn)) return cudaErrorInvalidValue;
                }
                Tc4Class t;
                t.d4 = d4;
                t.tma4 = tma4;
                t.tmw4 = tmw4;
                t.tmw = tmw;
                t.smem = smem4;
                // (+ 1 stage for the epilogue: a class no tap reaches still
                // writes its zeros)
                t.unit_work = ((long long)a.nr * d4.kst * d4.kpb + 1) * a.ncol;
                tc4.push_back(t);
                continue;
            }
        }
        const size_t pipe = (size_t)kD3Stages * (32768 + (size_t)a.ncol * 128);
        const size_t stage = (size_t)a.ncol * 128 * 4;  // epilogue staging
        const size_t smem = std::max(pipe, stage) + 1024;
        cudaError_t e = cudaFuncSetAttribute(dgrad_tc3_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        dim3 grid((unsigned)((a.total_tiles + 1) / 2), (p.C + a.c_tile - 1) / a.c_tile);
        dgrad_tc3_kernel<<<grid, kD3Threads, smem, st>>>(tma, tmw, a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    const int ntc4 = (int)tc4.size();
    if (ntc4 == 0) return cudaSuccess;
    size_t smem = 0;
    for (int k = 0; k < ntc4; ++k) smem = std::max(smem, tc4[k].smem);
    // blocks per class: in proportion to its work (units x unit work), at
    // least one and at most one per unit, the total within one per SM; the
    // SMs left over go one at a time to the class that would finish last
    int blocks[kD4MaxClasses];
    bool together = ntc4 > 1 && ntc4 <= kD4MaxClasses;
    if (together) {
        long double total = 0;
        for (int k = 0; k < ntc4; ++k) total += (long double)tc4[k].d4.total_units * tc4[k].unit_work;
        int used = 0;
        for (int k = 0; k < ntc4; ++k) {
            const long double share =
                total > 0 ? p.num_sms * (long double)tc4[k].d4.total_units * tc4[k].unit_work / total
                          : 1;
            blocks[k] = (int)std::max<long long>(
                1, std::min<long long>(tc4[k].d4.total_units, (long long)share));
            used += blocks[k];
        }
        together = used <= p.num_sms;
        auto finish = [&](int k, int b) {
            return (long long)((tc4[k].d4.total_units + b - 1) / b) * tc4[k].unit_work;
        };
        while (together && used < p.num_sms) {
            int worst = -1;
            for (int k = 0; k < ntc4; ++k)
                if (blocks[k] < tc4[k].d4.total_units &&
                    (worst < 0 || finish(k, blocks[k]) > finish(worst, blocks[worst])))
                    worst = k;
            if (worst < 0) break;
            ++blocks[worst];
            ++used;
        }
    }
    if (!together) {
        for (int k = 0; k < ntc4; ++k) {
            cudaError_t e = cudaFuncSetAttribute(
                dgrad_tc4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc4[k].smem);
            if (e != cudaSuccess) return e;
            const int grid4 = std::max(1, std::min(p.num_sms, tc4[k].d4.total_units));
            e = launch_pdl(dgrad_tc4_kernel, dim3(grid4), dim3(kD4Threads), tc4[k].smem, st,
                           tc4[k].tma4, tc4[k].tmw4, tc4[k].tmw, tc4[k].d4);
            if (e == cudaSuccess) e = cudaGetLastError();
            if (e != cudaSuccess) return e;
            *launches += 1;
        }
        return cudaSuccess;
    }
    D4Classes m;
    std::memset(&m, 0, sizeof(m));
    m.ncls = ntc4;
    m.first[0] = 0;
    for (int k = 0; k < ntc4; ++k) {
        m.tma[k] = tc4[k].tma4;
        m.tmw[k] = tc4[k].tmw4;
        m.tmw1[k] = tc4[k].tmw;
        m.d[k] = tc4[k].d4;
        m.first[k + 1] = m.first[k] + blocks[k];
    }
    cudaError_t e = cudaFuncSetAttribute(dgrad_tc4_classes_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(dgrad_tc4_classes_kernel, dim3(m.first[ntc4]), dim3(kD4Threads), smem, st, m);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaSuccess;
}

cudaError_t launch_selftest_wait(unsigned timeout_us, void *ws, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(timeout_us, ws_at<unsigned>(ws, 0));
    return cudaGetLastError();
}

}  // namespace cba
