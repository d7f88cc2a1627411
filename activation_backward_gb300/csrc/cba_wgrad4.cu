// cba_wgrad4.cu -- weight gradient with both operands fed by TMA tiles
// (dW[k][c][r][s] += sum_{n,p,q} dz[n][k][p][q] x[n][c][p + r - pad][q + s - pad],
// the gemm(0,1,...) of "YOLOv3反向传播原理 之 全流程源码分析" §3.1 over the
// im2col_cpu columns of §3.2, without the column buffer).
//
// Substituting w = q + s - pad moves the kernel-column shift from x onto dz:
//   dW[k][c][r][s] = sum_{n,p,w} dz[n][k][p][w - s + pad] * x[n][c][p + r - pad][w].
// A block owns 128 output channels k (MMA M, TMEM lanes) and cb input
// channels c, and walks a range of (n, 32-wide column chunk w0, output row p)
// items.  Per item:
//   A_s = dz[n][k0..k0+127][p][w0 + j - s + pad], j < 32: the dz row shifted
//         by each kernel column s, written into TMEM by producer warps from a
//         TMA-staged tile of the channels-last, zero-bordered dz copy;
//   B   = x rows p - pad .. p - pad + R - 1 of channels c0..c0+cb, columns
//         w0..w0+31: R consecutive rows of a TMA ring (128-byte swizzle,
//         K-major), so one MMA covers all kernel rows with N = R * cb;
//   D_s[k][(r, c)] += A_s * B^T, one accumulator per kernel column s.
// The ring keeps every x row once; rows that wrap around the ring end are
// also stored in R - 1 mirror slots after it, so any R consecutive rows are
// contiguous.  Padding rows and columns come from TMA's zero fill.
// The epilogue permutes D_s into dW's [c][r][s] order through shared memory
// and adds each dW row segment in L2 with one bulk async reduction.
//
// Roles: warp 0 issues TMA, warp 1 issues MMAs, warps 2-9 (two groups of
// four, one warp per TMEM lane quarter, alternating items) write the A
// operand and then run the epilogue.  Every wait is bounded (2 s); on a
// timeout the block sets the workspace status bit and stops.
#include <cuda.h>

#include "cba_internal.cuh"
#include "cba_ptx.cuh"

namespace cba {

namespace {

constexpr uint64_t kW4LimitNs = 2000000000ull;
constexpr int kW4Threads = 320;
constexpr int kW4MaxNR = 8;   // x ring rows (mirror slots come on top)
constexpr int kW4ND = 4;      // dz ring slots (even: each producer group owns half)
constexpr int kW4Stages = 2;  // A stages in TMEM (one per producer group)

struct W4Args {
    float *dW;
    unsigned *status;
    int K, C, RS, CRS;
    int Pe, pad, nwc, Wx;
    int bq_lo, bd_lo;
    int kbox;                // channels per dz box
    int wdz;                 // dz columns per box (32 + S - 1)
    int cb;                  // input channels per block
    int nctile;              // c tiles
    int ctas_per_tile;
    int items_per_tile;      // N * nwc * Pe
    int nr;                  // x ring rows
    uint32_t xslot_bytes;    // cb * 128
    uint32_t dz_bytes;       // wdz * kbox * 4
    uint32_t dz_stride;      // ring slot stride (128-byte multiple)
    uint32_t dz_off;         // byte offset of the dz ring
    int pitch;               // floats per staged dW row (16-byte multiple, 4 mod 32)
    int bulk;                // 1: bulk reductions aligned
};

struct W4Bars {
    uint64_t x_full[kW4MaxNR], x_empty[kW4MaxNR];
    uint64_t dz_full[kW4ND], dz_empty[kW4ND];
    uint64_t a_full[kW4Stages], a_empty[kW4Stages], accum;
    uint32_t tmem_base;
    int abort_flag;
};

struct Item {
    int n, w0, p, seg;
};

__device__ __forceinline__ Item decode(const W4Args &a, int i) {
    Item it;
    const int per_n = a.nwc * a.Pe;
    it.n = i / per_n;
    const int rem = i - it.n * per_n;
    const int wc = rem / a.Pe;
    it.p = rem - wc * a.Pe;
    it.w0 = wc * 32;
    it.seg = it.n * a.nwc + wc;
    return it;
}

template <int R, int S>
__global__ void __launch_bounds__(kW4Threads, 1)
    wgrad_tc4_kernel(const __grid_constant__ CUtensorMap tmx,
                     const __grid_constant__ CUtensorMap tmdz, const W4Args a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ W4Bars sb;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x / a.ctas_per_tile, split = blockIdx.x % a.ctas_per_tile;
    const int k0 = (tile / a.nctile) * 128, c0 = (tile % a.nctile) * a.cb;
    const int i0 = (int)((long long)split * a.items_per_tile / a.ctas_per_tile);
    const int i1 = (int)((long long)(split + 1) * a.items_per_tile / a.ctas_per_tile);
    const bool has_work = i1 > i0;
    const int N = R * a.cb;                                    // MMA N
    const uint32_t acol0 = (uint32_t)(S * N);                  // first A column
    uint8_t *xring = smem;
    uint8_t *dzring = smem + a.dz_off;

    if (tid == 0) {
        for (int i = 0; i < kW4MaxNR; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.x_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.x_empty[i]), 1);
        }
        for (int i = 0; i < kW4ND; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.dz_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.dz_empty[i]), 128);
        }
        for (int i = 0; i < kW4Stages; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.a_full[i]), 128);
            ptx::mbar_init(ptx::smem_u32(&sb.a_empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&sb.accum), 1);
        sb.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&sb.tmem_base), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sb.tmem_base;

    if (warp == 0) {
        // ---- TMA: x rows into the ring (and its mirror slots), dz tiles
        if (lane == 0 && has_work) {
            int t_row = 0, seg = -1, h_next = 0, j = 0;
            bool ok = true;
            for (int i = i0; ok && i < i1; ++i, ++j) {
                const Item it = decode(a, i);
                if (it.seg != seg) {
                    seg = it.seg;
                    h_next = it.p - a.pad;
                }
                const int h_top = it.p - a.pad + R - 1;
                for (; ok && h_next <= h_top; ++h_next, ++t_row) {
                    const int slot = t_row % a.nr;
                    if (t_row >= a.nr)
                        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.x_empty[slot]),
                                                    (uint32_t)(t_row / a.nr - 1) & 1u,
                                                    &sb.abort_flag, a.status, kW4LimitNs);
                    if (!ok) break;
                    const bool mirror = slot < R - 1;
                    const uint32_t bar = ptx::smem_u32(&sb.x_full[slot]);
                    ptx::mbar_arrive_expect_tx(bar, a.xslot_bytes * (mirror ? 2u : 1u));
                    ptx::tma_load_4d(ptx::smem_u32(xring + (size_t)slot * a.xslot_bytes), &tmx,
                                     it.w0, h_next, c0, it.n, bar);
                    if (mirror)
                        ptx::tma_load_4d(
                            ptx::smem_u32(xring + (size_t)(a.nr + slot) * a.xslot_bytes), &tmx,
                            it.w0, h_next, c0, it.n, bar);
                }
                if (!ok) break;
                const int ds = j % kW4ND;
                if (j >= kW4ND)
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_empty[ds]),
                                                (uint32_t)(j / kW4ND - 1) & 1u, &sb.abort_flag,
                                                a.status, kW4LimitNs);
                if (!ok) break;
                const uint32_t bar = ptx::smem_u32(&sb.dz_full[ds]);
                ptx::mbar_arrive_expect_tx(bar, a.dz_bytes);
                // columns w0 - (S - 1 - pad) .. w0 + 31 + pad of dz row p
                ptx::tma_load_4d(ptx::smem_u32(dzring + (size_t)ds * a.dz_stride), &tmdz, k0,
                                 it.w0 - (S - 1 - a.pad) + a.bq_lo, it.p + a.bd_lo, it.n, bar);
            }
            // no copy may be in flight when the block exits
            int no_abort = 0;
            for (int t = max(0, t_row - a.nr); t < t_row; ++t)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.x_full[t % a.nr]),
                                       (uint32_t)(t / a.nr) & 1u, &no_abort, a.status,
                                       kW4LimitNs);
            for (int jj = max(0, j - kW4ND); jj < j; ++jj)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_full[jj % kW4ND]),
                                       (uint32_t)(jj / kW4ND) & 1u, &no_abort, a.status,
                                       kW4LimitNs);
        }
    } else if (warp == 1) {
        // ---- MMA issue (one thread)
        if (lane == 0 && has_work) {
            const uint32_t idesc = ptx::idesc_tf32(128, N);
            const uint64_t bd0 = ptx::smem_desc(ptx::smem_u32(xring), 16, 1024, 2);
            const uint32_t slot_units = a.xslot_bytes >> 4;
            int t_row = 0, seg = -1, h_next = 0, t_seg = 0, h_first = 0, t_ready = 0, j = 0;
            bool ok = true;
            for (int i = i0; ok && i < i1; ++i, ++j) {
                const Item it = decode(a, i);
                if (it.seg != seg) {
                    seg = it.seg;
                    h_next = h_first = it.p - a.pad;
                    t_seg = t_row;
                }
                const int h_top = it.p - a.pad + R - 1;
                t_row += h_top - h_next + 1;
                h_next = h_top + 1;
                const int t_ws = t_seg + (it.p - a.pad - h_first);  // window's first row
                while (ok && t_ready < t_ws + R) {
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.x_full[t_ready % a.nr]),
                                                (uint32_t)(t_ready / a.nr) & 1u,
                                                &sb.abort_flag, a.status, kW4LimitNs);
                    ++t_ready;
                }
                const int stage = j & 1;
                if (ok)
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_full[stage]),
                                                (uint32_t)(j >> 1) & 1u, &sb.abort_flag,
                                                a.status, kW4LimitNs);
                if (!ok) break;
                ptx::tc_fence_after();
                const int nks = min(4, (a.Wx - it.w0 + 7) >> 3);
                const uint64_t bd = bd0 + (uint64_t)((uint32_t)(t_ws % a.nr) * slot_units);
                const uint32_t a_tm = tmem + acol0 + (uint32_t)(stage * S * 32);
#pragma unroll
                for (int s = 0; s < S; ++s) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        if (ks < nks)
                            ptx::mma_tf32_ts(tmem + (uint32_t)(s * N), a_tm + s * 32 + ks * 8,
                                             bd + 2 * ks, idesc, (j > 0 || ks > 0) ? 1u : 0u);
                }
                ptx::mma_commit(ptx::smem_u32(&sb.a_empty[stage]));
                // x rows the next item does not use
                bool seg_end = i + 1 >= i1;
                if (!seg_end) seg_end = decode(a, i + 1).seg != seg;
                const int nrel = seg_end ? R : 1;
                for (int u = 0; u < nrel; ++u)
                    ptx::mma_commit(ptx::smem_u32(&sb.x_empty[(t_ws + u) % a.nr]));
            }
            if (!ok) {  // the epilogue must not take the drain below for a result
                *reinterpret_cast<volatile int *>(&sb.abort_flag) = 1;
                __threadfence_block();
            }
            // drain: every MMA issued has finished before TMEM is released
            ptx::mma_commit(ptx::smem_u32(&sb.accum));
            int no_abort = 0;
            ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &no_abort, a.status, kW4LimitNs);
        }
    } else {
        // ---- A producers: group g writes the items j = g, g + 2, ... into
        // TMEM stage g.  Thread = TMEM lane kl = output channel k0 + kl.
        const int g = (warp - 2) >> 2, quarter = warp & 3;
        const int kl = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const bool kv = kl < a.kbox;
        bool ok = true;
        for (int j = g; has_work && i0 + j < i1; j += 2) {
            const int ds = j % kW4ND;
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_full[ds]),
                                        (uint32_t)(j / kW4ND) & 1u, &sb.abort_flag, a.status,
                                        kW4LimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            constexpr int WDZ = 32 + S - 1;
            float v[WDZ];
            const float *tilep = reinterpret_cast<const float *>(dzring + (size_t)ds * a.dz_stride);
#pragma unroll
            for (int jj = 0; jj < WDZ; ++jj) v[jj] = kv ? tilep[jj * a.kbox + kl] : 0.f;
            ptx::mbar_arrive(ptx::smem_u32(&sb.dz_empty[ds]));
            if (j >= 2)
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_empty[g]),
                                            (uint32_t)((j >> 1) - 1) & 1u, &sb.abort_flag,
                                            a.status, kW4LimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t a_tm = tmem + lane_addr + acol0 + (uint32_t)(g * S * 32);
#pragma unroll
            for (int s = 0; s < S; ++s) {
                // A_s[j] = dz[w0 + j - s + pad] = tile[j + S - 1 - s]
                float w[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) w[q] = v[q + S - 1 - s];
                ptx::tmem_st32(a_tm + (uint32_t)(s * 32), w);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&sb.a_full[g]));
        }
        // ---- epilogue: D_s[k][(r, c)] -> staged dW rows [c][r][s] -> L2
        if (has_work && ok)
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &sb.abort_flag, a.status,
                                        kW4LimitNs);
        if (ok) ok = *reinterpret_cast<volatile int *>(&sb.abort_flag) == 0;
        ok = __all_sync(0xffffffffu, ok) && has_work;
        // both groups agree before the ring memory is reused for staging
        ok = ptx::named_bar_and(1, 256, ok);
        if (ok) {
            ptx::tc_fence_after();
            float *stg = reinterpret_cast<float *>(smem);
            const int cvalid = min(a.cb, a.C - c0);
            const int ngrp = (cvalid + 3) >> 2;
            float *row = stg + (size_t)kl * a.pitch;
            for (int cg = g; cg < ngrp; cg += 2) {
                float vals[4 * R * S];
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int s = 0; s < S; ++s) {
                        float t4[4];
                        ptx::tmem_ld4(tmem + lane_addr + (uint32_t)(s * N + r * a.cb + cg * 4),
                                      t4);
#pragma unroll
                        for (int e = 0; e < 4; ++e) vals[e * R * S + r * S + s] = t4[e];
                    }
                }
                ptx::tmem_ld_wait();
                float4 *dst = reinterpret_cast<float4 *>(row + cg * 4 * R * S);
#pragma unroll
                for (int u = 0; u < R * S; ++u)
                    dst[u] = make_float4(vals[4 * u], vals[4 * u + 1], vals[4 * u + 2],
                                         vals[4 * u + 3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar_sync(1, 256);
            const bool krow = g == 0 && k0 + kl < a.K;
            if (krow) {
                float *dst = a.dW + (long long)(k0 + kl) * a.CRS + (long long)c0 * a.RS;
                const int nel = cvalid * a.RS;
                if (a.bulk) {
                    ptx::bulk_reduce_add_f32(dst, ptx::smem_u32(row), (uint32_t)nel * 4u);
                    ptx::bulk_commit();
                    ptx::bulk_wait_all();
                } else {
                    for (int e = 0; e < nel; ++e) atomicAdd(dst + e, row[e]);
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool wgrad_tc4_supported(const Plan &p, const float *x) {
    if (p.stride != 1) return false;
    const bool k3 = p.R == 3 && p.S == 3, k1 = p.R == 1 && p.S == 1;
    if (!k3 && !k1) return false;
    if (p.pad > p.S - 1) return false;
    const DzcGeom g = dzc_geom(p);
    if (g.We % 4 != 0) return false;  // x rows must be 16-byte strided for TMA
    if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) return false;
    if ((long long)p.N * ((g.We + 31) / 32) * g.Pe >= (1LL << 31)) return false;
    return true;
}

cudaError_t launch_wgrad_tc4(const Plan &p, const float *x, const float *dzc, float *dW,
                             void *ws, cudaStream_t st, int *launches) {
    const DzcGeom g = dzc_geom(p);
    W4Args a;
    a.dW = dW;
    a.status = ws_at<unsigned>(ws, p.off_status);
    a.K = p.K; a.C = p.C; a.RS = p.RS; a.CRS = p.CRS;
    a.Pe = g.Pe; a.pad = p.pad; a.nwc = (g.We + 31) / 32; a.Wx = g.We;
    a.bq_lo = g.bq_lo; a.bd_lo = g.bd_lo;
    a.kbox = std::min(128, g.Kp);
    a.wdz = 32 + p.S - 1;
    // input channels per block: N = R * cb <= 256 and the S accumulators plus
    // two A stages within 512 TMEM columns; cb a multiple of 8
    int cb_cap = p.R == 1 ? 256 : 32;
    int cb = std::min(cb_cap, (p.C + 7) / 8 * 8);
    if ((p.R * cb) % 16 != 0) cb = (cb + 15) / 16 * 16;
    if (p.S * p.R * cb + kW4Stages * p.S * 32 > 512 || p.R * cb > 256) return cudaErrorNotSupported;
    a.cb = cb;
    a.nctile = (p.C + cb - 1) / cb;
    const int ktiles = (p.K + 127) / 128;
    const int ntiles = ktiles * a.nctile;
    a.items_per_tile = p.N * a.nwc * g.Pe;
    a.ctas_per_tile = std::max(1, std::min(a.items_per_tile, p.num_sms / ntiles));
    a.xslot_bytes = (uint32_t)cb * 128u;
    a.dz_bytes = (uint32_t)(a.wdz * a.kbox * 4);
    a.dz_stride = (a.dz_bytes + 127u) / 128u * 128u;
    // shared memory: x ring (nr + R - 1 slots), dz ring; the staging area
    // for the epilogue reuses it
    const size_t budget = 220 * 1024;
    const size_t dz_ring = (size_t)kW4ND * a.dz_stride;
    int nr = kW4MaxNR;
    while (nr > p.R && (size_t)(nr + p.R - 1) * a.xslot_bytes + dz_ring > budget) --nr;
    if ((size_t)(nr + p.R - 1) * a.xslot_bytes + dz_ring > budget || nr < p.R)
        return cudaErrorNotSupported;
    a.nr = nr;
    a.dz_off = (uint32_t)((size_t)(nr + p.R - 1) * a.xslot_bytes);
    int pitch = cb * p.RS;
    pitch = (pitch + 3) / 4 * 4;
    while (pitch % 32 != 4) pitch += 4;
    a.pitch = pitch;
    const size_t main_bytes = (size_t)a.dz_off + dz_ring;
    const size_t stage_bytes = (size_t)128 * pitch * 4;
    const size_t smem = std::max(main_bytes, stage_bytes) + 1024;
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    const int cvalid_last = p.C - (a.nctile - 1) * cb;
    a.bulk = (p.CRS % 4 == 0) && ((cb * p.RS) % 4 == 0) && ((cvalid_last * p.RS) % 4 == 0) &&
             ((reinterpret_cast<uintptr_t>(dW) & 15u) == 0);

    alignas(64) CUtensorMap tmx, tmdz;
    {
        const uint64_t d[4] = {(uint64_t)g.We, (uint64_t)g.He, (uint64_t)p.C, (uint64_t)p.N};
        const uint32_t b[4] = {32, 1, (uint32_t)cb, 1};
        if (!tma_encode_f32(&tmx, x, 4, d, b, true)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t d[4] = {(uint64_t)g.Kp, (uint64_t)g.Qpp, (uint64_t)g.Pp, (uint64_t)p.N};
        const uint32_t b[4] = {(uint32_t)a.kbox, (uint32_t)a.wdz, 1, 1};
        if (!tma_encode_f32(&tmdz, dzc, 4, d, b, false)) return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)(ntiles * a.ctas_per_tile));
    cudaError_t e;
    if (p.R == 3) {
        e = cudaFuncSetAttribute(wgrad_tc4_kernel<3, 3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        wgrad_tc4_kernel<3, 3><<<grid, kW4Threads, smem, st>>>(tmx, tmdz, a);
    } else {
        e = cudaFuncSetAttribute(wgrad_tc4_kernel<1, 1>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        wgrad_tc4_kernel<1, 1><<<grid, kW4Threads, smem, st>>>(tmx, tmdz, a);
    }
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace cba
