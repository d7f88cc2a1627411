// cba_gemm1x1.cu -- both convolution gradients of a 1x1, stride-1, unpadded
// layer as plain TMA-fed GEMMs ("YOLOv3反向传播原理 之 全流程源码分析" §3.1:
// with a 1x1 kernel im2col(x) is x itself, so gemm(0,1,...) and gemm(1,0,...)
// need no column buffer and no tap shifts).
//
//   weight gradient  dW[k][c] += sum_{n,hw} dz[n][k][hw] * x[n][c][hw]
//                    D[k][c]: A = dz in NCHW order (k rows, hw contiguous),
//                    B = x (c rows, hw contiguous); the contraction runs over
//                    the (image, 32-position chunk) pairs of a block's range.
//   input gradient   prev[n][c][hw] (=, or += at the L2) sum_k W[k][c] dz[n][k][hw]
//                    D[c][hw]: A = the repacked weights wr[c][k], B = the
//                    channels-last dz copy dzc[n*HW + hw][k]; one image's
//                    positions per tile.
//
// Both operands are K-major boxes of 32 fp32 (128 bytes, 128-byte swizzle)
// loaded by TMA; the MMA is tcgen05 kind::tf32 with M = 128 and N = 256, the
// accumulator in TMEM.  The output leaves through TMA too: the epilogue warps
// move 32 x 32 boxes of the accumulator through swizzled shared memory and
// store them (prev) or add them at the L2 (dW, and prev when it already holds
// the shortcut delta or its old value), so the weight gradient needs no tile
// accumulators and no apply pass.  The grid is persistent: a block walks its
// units (output tiles, or tile and contraction range) with two TMEM
// accumulators, so a unit's epilogue overlaps the next unit's MMAs.
//
// Roles: warps 0 and 6 issue the TMA loads (A and B), warp 1 owns TMEM and
// issues the MMAs, warps 2-5 (one per TMEM lane quarter) run the epilogue.  Every wait is
// bounded (2 s); on a timeout the block sets the workspace status bit, stops,
// waits (bounded) for its copies in flight, frees its TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "cba_internal.cuh"
#include "cba_ptx.cuh"
#include "cba_repack.cuh"

namespace cba {

namespace {

constexpr uint64_t kG1LimitNs = 2000000000ull;
constexpr int kG1Threads = 224;  // A TMA warp, MMA warp, 4 epilogue warps, B TMA warp
constexpr int kG1N = 256;                      // MMA N: positions (dgrad) or channels (wgrad)
constexpr int kG1Stages = 4;
constexpr uint32_t kG1ABytes = 128u * 128u;    // 128 rows x 32 fp32
constexpr uint32_t kG1BBytes = kG1N * 128u;    // 256 rows x 32 fp32
constexpr uint32_t kG1StageBytes = kG1ABytes + kG1BBytes;
constexpr uint32_t kG1EpiBytes = 2u * 32u * 128u;  // two 32 x 32 boxes per epilogue warp

struct G1Args {
    int mode;       // 0 input gradient, 1 weight gradient
    int units;      // total units
    int kchunks;    // dgrad: 32-wide k chunks per unit
    int HW, nhc;    // positions per image, 32-position chunks per image
    int mtiles, ntiles;  // dgrad: c tiles, positions tiles per image; wgrad: k tiles, c tiles
    long long items;     // wgrad: N * nhc (image, chunk) pairs, split over units
    int splits;          // wgrad: contraction ranges per tile
    int red_add;         // dgrad: add at the L2 instead of storing
    int mrows, ncols;    // output extent: rows (C, or K) and columns (HW, or C)
    unsigned *status;
};

struct G1Bars {
    uint64_t full[kG1Stages], empty[kG1Stages];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// The unit u's coordinates.  dgrad: (n, position tile, c tile), c fastest;
// wgrad: (tile, split) with the contraction range [g0, g1) of (n, chunk) pairs.
struct G1Unit {
    int m0, n0, img;        // output tile origin (rows m0, columns n0); dgrad image
    long long g0, g1;       // wgrad contraction range; dgrad: 0 .. kchunks
};

__device__ __forceinline__ G1Unit g1_unit(const G1Args &a, int u) {
    G1Unit r;
    if (a.mode == 0) {
        const int ct = u % a.mtiles;
        const int rest = u / a.mtiles;
        const int ht = rest % a.ntiles;
        r.img = rest / a.ntiles;
        r.m0 = ct * 128;
        r.n0 = ht * kG1N;
        r.g0 = 0;
        r.g1 = a.kchunks;
    } else {
        const int split = u % a.splits, tile = u / a.splits;
        const int kt = tile / a.ntiles, ct = tile % a.ntiles;
        r.img = 0;
        r.m0 = kt * 128;
        r.n0 = ct * kG1N;
        r.g0 = (long long)split * a.items / a.splits;
        r.g1 = (long long)(split + 1) * a.items / a.splits;
    }
    return r;
}

}  // namespace

namespace {

__global__ void __launch_bounds__(kG1Threads, 1)
    gemm1x1_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                   const __grid_constant__ CUtensorMap tmo, const G1Args a, const RepackJob rep,
                   int nrep) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ G1Bars sb;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nunits =
        a.units > (int)blockIdx.x ? (a.units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (tid == 0) {
        for (int i = 0; i < kG1Stages; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.full[i]), 2);  // the A and the B issuer
            ptx::mbar_init(ptx::smem_u32(&sb.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.acc_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.acc_empty[i]), 4);  // the 4 epilogue warps
        }
        ptx::mbar_init(ptx::smem_u32(&sb.drain), 1);
        sb.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&sb.tmem_base), 2 * kG1N);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sb.tmem_base;
    // the operands (dz copies, repacked weights) come from the previous kernels
    ptx::griddep_wait();

    if (warp == 0 || warp == 6) {
        // ---- TMA: warp 0 the A boxes, warp 6 the B boxes of every contraction
        // chunk (one issuing thread starts a box every few hundred cycles, so
        // the two operands get a thread each)
        if (lane == 0) {
            const bool bside = warp == 6;
            int gs = 0;
            bool ok = true;
            for (int i = 0; ok && i < nunits; ++i) {
                const G1Unit un = g1_unit(a, (int)blockIdx.x + i * (int)gridDim.x);
                for (long long g = un.g0; ok && g < un.g1; ++g, ++gs) {
                    const int slot = gs % kG1Stages;
                    if (gs >= kG1Stages)
                        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.empty[slot]),
                                                    (uint32_t)(gs / kG1Stages - 1) & 1u,
                                                    &sb.abort_flag, a.status, kG1LimitNs);
                    if (!ok) break;
                    const uint32_t sp = ptx::smem_u32(smem + (size_t)slot * kG1StageBytes);
                    const uint32_t bar = ptx::smem_u32(&sb.full[slot]);
                    ptx::mbar_arrive_expect_tx(bar, bside ? kG1BBytes : kG1ABytes);
                    if (a.mode == 0) {
                        const int kc = (int)g * 32;
                        if (!bside) ptx::tma_load_2d(sp, &tma, kc, un.m0, bar);  // wr (k, c)
                        else ptx::tma_load_2d(sp + kG1ABytes, &tmb, kc, un.img * a.HW + un.n0, bar);
                    } else {
                        const int n = (int)(g / a.nhc), hc = (int)(g - (long long)n * a.nhc);
                        if (!bside) ptx::tma_load_3d(sp, &tma, hc * 32, un.m0, n, bar);  // dz (hw, k, n)
                        else ptx::tma_load_3d(sp + kG1ABytes, &tmb, hc * 32, un.n0, n, bar);  // x
                    }
                }
            }
            // no copy may be in flight when the block exits
            int no_abort = 0;
            for (int v = gs > kG1Stages ? gs - kG1Stages : 0; v < gs; ++v)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.full[v % kG1Stages]),
                                       (uint32_t)(v / kG1Stages) & 1u, &no_abort, a.status,
                                       kG1LimitNs);
        }
    } else if (warp == 1) {
        // ---- MMA issue: unit i into accumulator i & 1, 4 MMAs (K = 8) per chunk
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_tf32(128, kG1N);
            int gs = 0;
            bool ok = true;
            for (int i = 0; ok && i < nunits; ++i) {
                const int b = i & 1;
                if (i >= 2)
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.acc_empty[b]),
                                                (uint32_t)((i >> 1) - 1) & 1u, &sb.abort_flag,
                                                a.status, kG1LimitNs);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t dtm = tmem + (uint32_t)(b * kG1N);
                const G1Unit un = g1_unit(a, (int)blockIdx.x + i * (int)gridDim.x);
                bool first = true;
                for (long long g = un.g0; ok && g < un.g1; ++g, ++gs) {
                    const int slot = gs % kG1Stages;
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.full[slot]),
                                                (uint32_t)(gs / kG1Stages) & 1u, &sb.abort_flag,
                                                a.status, kG1LimitNs);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint32_t base = ptx::smem_u32(smem + (size_t)slot * kG1StageBytes);
                    const uint64_t ad = ptx::smem_desc(base, 16, 1024, 2);
                    const uint64_t bd = ptx::smem_desc(base + kG1ABytes, 16, 1024, 2);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)  // descriptor addresses count 16-byte units
                        ptx::mma_tf32(dtm, ad + 2 * ks, bd + 2 * ks, idesc,
                                      (first && ks == 0) ? 0u : 1u);
                    first = false;
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
            ptx::mbar_wait_bounded(ptx::smem_u32(&sb.drain), 0, &no_abort, a.status, kG1LimitNs);
        }
    } else if (warp >= 2 && warp <= 5) {
        // ---- epilogue: warp w reads TMEM lanes 32 (w & 3) .. + 31 (rows of D).
        // Each 32-column box goes through swizzled shared memory (row = lane,
        // 16-byte chunk j of a row at j ^ (row & 7): conflict-free writes) to
        // one TMA store or L2 reduce-add; two boxes per warp in flight.
        const int wq = warp & 3;
        const int et = tid - 64;  // thread index among the 128 epilogue threads
        uint8_t *ebuf = smem + (size_t)kG1Stages * kG1StageBytes + (size_t)(warp - 2) * kG1EpiBytes;
        if (a.mode == 1 && nrep > 0 && rep.W != nullptr) {
            // the input gradient's weight repack, a tile or so per block, while
            // the first unit's MMAs run (the epilogue buffers are still idle)
            repack_part_group(rep, (int)blockIdx.x, nrep,
                              reinterpret_cast<float *>(smem + (size_t)kG1Stages * kG1StageBytes),
                              et, 128, 1);
        }
        bool ok = true;
        int nbox = 0;
        for (int i = 0; ok && i < nunits; ++i) {
            const int b = i & 1;
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.acc_full[b]), (uint32_t)(i >> 1) & 1u,
                                        &sb.abort_flag, a.status, kG1LimitNs);
            if (ok) ok = *reinterpret_cast<volatile int *>(&sb.abort_flag) == 0;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const G1Unit un = g1_unit(a, (int)blockIdx.x + i * (int)gridDim.x);
            const bool has = un.g1 > un.g0;
            const int row0 = un.m0 + wq * 32;
            const uint32_t tb = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(b * kG1N);
            for (int cg = 0; cg < kG1N / 32; cg += 2) {
                float v[2][32];
                ptx::tmem_ld32(tb + (uint32_t)(cg * 32), v[0]);
                ptx::tmem_ld32(tb + (uint32_t)((cg + 1) * 32), v[1]);
                ptx::tmem_ld_wait();
                if (cg + 2 >= kG1N / 32) {  // the unit's last loads: the MMAs may reuse it
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sb.acc_empty[b]));
                }
                if (!has || row0 >= a.mrows) continue;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int col = un.n0 + (cg + j) * 32;
                    if (col >= a.ncols) continue;  // past the image's positions / the channels
                    uint8_t *buf = ebuf + (size_t)(nbox & 1) * 4096;
                    if (nbox >= 2) {  // the box stored from this buffer before has been read
                        if (lane == 0) ptx::bulk_wait_read_1();
                        __syncwarp();
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<float4 *>(buf + lane * 128 + ((q ^ (lane & 7)) * 16)) =
                            make_float4(v[j][4 * q], v[j][4 * q + 1], v[j][4 * q + 2],
                                        v[j][4 * q + 3]);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t src = ptx::smem_u32(buf);
                        if (a.mode == 0) {
                            if (a.red_add) ptx::tma_reduce_add_3d(&tmo, src, col, row0, un.img);
                            else ptx::tma_store_3d(&tmo, src, col, row0, un.img);
                        } else {
                            ptx::tma_reduce_add_2d(&tmo, src, col, row0);
                        }
                        ptx::bulk_commit();
                    }
                    ++nbox;
                }
            }
        }
        if (lane == 0) ptx::bulk_wait_all();  // every store complete before the block exits
        __syncwarp();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::griddep_launch_dependents();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 2 * kG1N);
    }
}

}  // namespace

namespace {

constexpr size_t kG1Smem =
    (size_t)kG1Stages * kG1StageBytes + 4u * kG1EpiBytes + 1024;  // + alignment slack

// One dense fp32 tensor map with a 32-float inner box and 128-byte swizzle.
bool g1_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
            const uint32_t *box) {
    return tma_encode_f32_swz(m, base, rank, dims, box, 128);
}

cudaError_t g1_launch(const G1Args &a, const CUtensorMap &ta, const CUtensorMap &tb,
                      const CUtensorMap &to, const RepackJob &job, int nrep, int grid,
                      cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(gemm1x1_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kG1Smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(gemm1x1_kernel, dim3(grid), dim3(kG1Threads), kG1Smem, st, ta, tb, to, a, job,
                   nrep);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool gemm1x1_supported(const Plan &p) {
    if (p.R != 1 || p.S != 1 || p.stride != 1 || p.pad != 0 || p.groups != 1) return false;
    // TMA rows of x, dz, prev (HW floats), dW (C), wr (Kw) and dzc (Kp) must
    // be 16-byte strided
    if (p.HW % 4 != 0 || p.C % 4 != 0) return false;
    if ((long long)p.N * p.HW >= (1LL << 31)) return false;
    return kG1Smem <= 227 * 1024 && tc2_supported(p);
}

size_t gemm1x1_dzt_bytes(const Plan &p) {
    return sizeof(float) * (size_t)p.N * p.K * p.HW;
}

cudaError_t launch_gemm1x1_wgrad(const Plan &p, const float *dzt, const float *x, float *dW,
                                 const void *ws, const RepackJob *rep, cudaStream_t st,
                                 int *launches) {
    G1Args a{};
    a.mode = 1;
    a.HW = p.HW;
    a.nhc = (p.HW + 31) / 32;
    a.mtiles = (p.K + 127) / 128;
    a.ntiles = (p.C + kG1N - 1) / kG1N;
    a.items = (long long)p.N * a.nhc;
    const int tiles = a.mtiles * a.ntiles;
    a.splits = (int)std::max(1LL, std::min<long long>(a.items, std::max(1, p.num_sms / tiles)));
    a.units = tiles * a.splits;
    a.mrows = p.K;
    a.ncols = p.C;
    a.status = ws_at<unsigned>(const_cast<void *>(ws), p.off_status);
    CUtensorMap ta, tb, to;
    {
        const uint64_t d[3] = {(uint64_t)p.HW, (uint64_t)p.K, (uint64_t)p.N};
        const uint32_t b[3] = {32, 128, 1};
        if (!g1_map(&ta, dzt, 3, d, b)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t d[3] = {(uint64_t)p.HW, (uint64_t)p.C, (uint64_t)p.N};
        const uint32_t b[3] = {32, (uint32_t)kG1N, 1};
        if (!g1_map(&tb, x, 3, d, b)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t d[2] = {(uint64_t)p.C, (uint64_t)p.K};
        const uint32_t b[2] = {32, 32};
        if (!g1_map(&to, dW, 2, d, b)) return cudaErrorInvalidValue;
    }
    const int grid = std::max(1, std::min(a.units, p.num_sms));
    const RepackJob job = rep ? *rep : RepackJob{};
    cudaError_t e = g1_launch(a, ta, tb, to, job, rep ? grid : 0, grid, st);
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaSuccess;
}

cudaError_t launch_gemm1x1_dgrad(const Plan &p, const float *wr, const float *dzc,
                                 const float *residual, float *prev, void *ws, cudaStream_t st,
                                 int *launches) {
    // with a residual or accumulation, prev first holds residual (+ old prev)
    // and the products are added to it at the L2
    const bool red_add = residual != nullptr || p.accumulate != 0;
    if (residual) {
        cudaError_t e = launch_prev_init(p, residual, prev, st, launches);
        if (e != cudaSuccess) return e;
    }
    const int Kw = (p.K + 3) / 4 * 4;
    G1Args a{};
    a.mode = 0;
    a.HW = p.HW;
    a.kchunks = (p.K + 31) / 32;
    a.mtiles = (p.C + 127) / 128;
    a.ntiles = (p.HW + kG1N - 1) / kG1N;
    a.units = p.N * a.ntiles * a.mtiles;
    a.red_add = red_add ? 1 : 0;
    a.mrows = p.C;
    a.ncols = p.HW;
    a.status = ws_at<unsigned>(ws, p.off_status);
    CUtensorMap ta, tb, to;
    {
        const uint64_t d[2] = {(uint64_t)Kw, (uint64_t)p.C};
        const uint32_t b[2] = {32, 128};
        if (!g1_map(&ta, wr, 2, d, b)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t d[2] = {(uint64_t)Kw, (uint64_t)p.N * p.HW};
        const uint32_t b[2] = {32, (uint32_t)kG1N};
        if (!g1_map(&tb, dzc, 2, d, b)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t d[3] = {(uint64_t)p.HW, (uint64_t)p.C, (uint64_t)p.N};
        const uint32_t b[3] = {32, 32, 1};
        if (!g1_map(&to, prev, 3, d, b)) return cudaErrorInvalidValue;
    }
    const int grid = std::max(1, std::min(a.units, p.num_sms));
    cudaError_t e = g1_launch(a, ta, tb, to, RepackJob{}, 0, grid, st);
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaSuccess;
}

}  // namespace cba
