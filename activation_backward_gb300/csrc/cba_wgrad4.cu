// cba_wgrad4.cu -- weight gradient with both operands fed by TMA tiles
// (dW[k][c][r][s] += sum_{n,p,q} dz[n][k][p][q] x[n][c][p + r - pad][q + s - pad],
// the gemm(0,1,...) of "YOLOv3反向传播原理 之 全流程源码分析" §3.1 over the
// im2col_cpu columns of §3.2, without the column buffer).
//
// Substituting w = q + s - pad moves the kernel-column shift from x onto dz:
//   dW[k][c][r][s] = sum_{n,p,w} dz[n][k][p][w - s + pad] * x[n][c][p + r - pad][w].
// A block owns one tile (128 output channels k = MMA M = TMEM lanes, cb
// input channels c, one kernel column s) and walks a range of
// (n, 32-wide column chunk w0, output row p) items.  Per item:
//   A = dz[n][k0..k0+127][p][w0 - s + pad + j], j < 32: a TMA tile of the
//       channels-last, zero-bordered dz copy (its column offset is free: the
//       column is not the innermost dimension there), moved into TMEM by the
//       producer warps (one 32-column store per lane);
//   B = x rows p - pad .. p - pad + R - 1 of channels c0..c0+cb, columns
//       w0..w0+31: R consecutive rows of a TMA ring (128-byte swizzle,
//       K-major), so one MMA covers all kernel rows, N = R * cb;
//   D[k][(r, c)] += A * B^T  (4 MMAs of K = 8).
// The ring keeps every x row once; rows that wrap around its end are also
// stored in R - 1 mirror slots after it, so any R consecutive rows are
// contiguous.  Padding rows and columns come from TMA's zero fill.
// Each block adds its tile into a per-tile accumulator in the workspace with
// one bulk reduce-add (the L2 does the adds, in arrival order); a second
// kernel adds the accumulators into dW.
//
// Roles: warp 0 issues the x-row TMA loads, warp 10 the dz-tile TMA loads
// (one issuing thread costs a few hundred cycles per copy, so the two streams
// get a thread each), warp 1 issues MMAs, warps 2-9 (two groups of four, one
// warp per TMEM lane quarter, alternating items) move dz into TMEM, check
// that the item's x rows have landed, and then run the epilogue.  The MMA
// thread waits once and commits once per item.  Every wait is bounded
// (2 s); on a timeout the block sets the workspace status bit and stops.
#include <cuda.h>

#include "cba_internal.cuh"
#include "cba_ptx.cuh"
#include "cba_repack.cuh"

namespace cba {

namespace {

constexpr uint64_t kW4LimitNs = 2000000000ull;
constexpr int kW4Threads = 352;
constexpr int kW4MaxNR = 16;  // x ring rows (mirror slots come on top)
constexpr int kW4MaxND = 4;   // dz ring slots
// TMA loads take about a microsecond to land, so the rings are as deep as
// shared memory allows: enough loads stay in flight to cover that latency.
constexpr int kW4NA = 4;      // A stages in TMEM (even), one item pair (64 columns) each
constexpr int kW4Done = 16;   // pair-completion barriers (a ring; lag stays below 16)

struct W4Geom {
    bool ok;
    int cb, N, nctile, ktiles, ntiles, cpt, items, nwc, grid, kbox, nr, nd;
    uint32_t xslot_bytes, dz_bytes, dz_stride, dz_off;
    size_t smem, acc_bytes;
};

struct W4Args {
    float *acc;              // [tile][N][128] tile accumulators (zeroed before the call)
    unsigned *status;
    int S, Pe, pad, nwc, Wx;
    int bq_lo, bd_lo;
    int kbox;                // channels per dz box
    int cb, N;               // input channels per block, MMA N = R * cb
    int nctile;              // c tiles
    int cpt;                 // blocks per tile
    int items_per_tile;      // N * nwc * Pe
    int nr;                  // x ring rows
    int nd;                  // dz ring slots
    uint32_t xslot_bytes;    // cb * 128
    uint32_t dz_bytes;       // 32 * kbox * 4
    uint32_t dz_stride;      // ring slot stride (128-byte multiple)
    uint32_t dz_off;         // byte offset of the dz ring
};

struct W4Bars {
    uint64_t x_full[kW4MaxNR];
    uint64_t dz_full[kW4MaxND], dz_empty[kW4MaxND];
    uint64_t a_full[kW4NA], done[kW4Done], accum;
    uint32_t tmem_base;
    int abort_flag;
};

struct Item {
    int n, w0, p;
};

__device__ __forceinline__ Item decode(const W4Args &a, int i) {
    Item it;
    const int per_n = a.nwc * a.Pe;
    it.n = i / per_n;
    const int rem = i - it.n * per_n;
    const int wc = rem / a.Pe;
    it.p = rem - wc * a.Pe;
    it.w0 = wc * 32;
    return it;
}

// Item bookkeeping shared by the roles.  Items advance incrementally (p
// fastest, then the column chunk, then n).  x rows form one sequence t: a
// segment (fixed n and column chunk) loads R rows for its first item and one
// more per further item, and item j's window is rows t_ws(j) .. t_ws(j)+R-1.
// Items go through the tensor core in pairs (2m, 2m + 1), which share a TMEM
// stage, one wait and one commit: pair m's MMAs complete done[m % kW4Done];
// the MMA thread waits only for a_full, which the producers signal once the
// pair's A operands are in TMEM and its x rows have landed.
template <int R>
__global__ void __launch_bounds__(kW4Threads, 1)
    wgrad_tc4_kernel(const __grid_constant__ CUtensorMap tmx,
                     const __grid_constant__ CUtensorMap tmdz, const W4Args a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ W4Bars sb;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x / a.cpt, split = blockIdx.x % a.cpt;
    const int s = tile % a.S, kc = tile / a.S;
    const int k0 = (kc / a.nctile) * 128, c0 = (kc % a.nctile) * a.cb;
    const int i0 = (int)((long long)split * a.items_per_tile / a.cpt);
    const int i1 = (int)((long long)(split + 1) * a.items_per_tile / a.cpt);
    const bool has_work = i1 > i0;
    const int cnt = has_work ? i1 - i0 : 0;
    const uint32_t acol0 = (uint32_t)a.N;  // first A column (accumulator at 0)
    uint8_t *xring = smem;
    uint8_t *dzring = smem + a.dz_off;

    if (tid == 0) {
        for (int i = 0; i < kW4MaxNR; ++i) ptx::mbar_init(ptx::smem_u32(&sb.x_full[i]), 1);
        for (int i = 0; i < kW4Done; ++i) ptx::mbar_init(ptx::smem_u32(&sb.done[i]), 1);
        for (int i = 0; i < kW4MaxND; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.dz_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.dz_empty[i]), 4);  // one arrival per warp
        }
        for (int i = 0; i < kW4NA; ++i) ptx::mbar_init(ptx::smem_u32(&sb.a_full[i]), 4);
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
    // dzc and the partials are touched only after the previous kernels completed
    ptx::griddep_wait();

    if (warp == 0) {
        // ---- TMA: x rows into the ring (and its mirror slots), dz tiles
        if (lane == 0 && has_work) {
            Item it = decode(a, i0);
            int wc = it.w0 >> 5;
            int t_row = 0, h_next = it.p - a.pad, j_seg_end = -1;
            int last_user[kW4MaxNR];  // per ring slot: last item reading the row held
            int j = 0;
            bool ok = true;
            for (; j < cnt; ++j) {
                if (j > j_seg_end) j_seg_end = j + min(cnt - j, a.Pe - it.p) - 1;
                const int h_top = it.p - a.pad + R - 1;
                for (; h_next <= h_top; ++h_next, ++t_row) {
                    const int slot = t_row % a.nr;
                    if (t_row >= a.nr) {
                        const int u = last_user[slot] >> 1;  // pair of the last user
                        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.done[u % kW4Done]),
                                                    (uint32_t)(u / kW4Done) & 1u, &sb.abort_flag,
                                                    a.status, kW4LimitNs);
                    }
                    if (!ok) break;
                    // the row sits at window position h - (p - pad) of item j
                    last_user[slot] = min(j + (h_next - (it.p - a.pad)), j_seg_end);
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
                if (++it.p == a.Pe) {  // next item; a new segment restarts the x rows
                    it.p = 0;
                    if (++wc == a.nwc) {
                        wc = 0;
                        ++it.n;
                    }
                    it.w0 = wc * 32;
                    h_next = -a.pad;
                }
            }
            // no copy may be in flight when the block exits
            int no_abort = 0;
            for (int t = max(0, t_row - a.nr); t < t_row; ++t)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.x_full[t % a.nr]),
                                       (uint32_t)(t / a.nr) & 1u, &no_abort, a.status,
                                       kW4LimitNs);
        }
    } else if (warp == 10) {
        // ---- TMA: dz tiles, one per item
        if (lane == 0 && has_work) {
            Item it = decode(a, i0);
            int wc = it.w0 >> 5;
            int j = 0, ds = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (; j < cnt; ++j) {
                if (j >= a.nd)
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_empty[ds]), ph ^ 1u,
                                                &sb.abort_flag, a.status, kW4LimitNs);
                if (!ok) break;
                const uint32_t bar = ptx::smem_u32(&sb.dz_full[ds]);
                ptx::mbar_arrive_expect_tx(bar, a.dz_bytes);
                // dz columns w0 - s + pad .. + 31 of row p
                ptx::tma_load_4d(ptx::smem_u32(dzring + (size_t)ds * a.dz_stride), &tmdz, k0,
                                 it.w0 - s + a.pad + a.bq_lo, it.p + a.bd_lo, it.n, bar);
                if (++ds == a.nd) {
                    ds = 0;
                    ph ^= 1u;
                }
                if (++it.p == a.Pe) {
                    it.p = 0;
                    if (++wc == a.nwc) {
                        wc = 0;
                        ++it.n;
                    }
                    it.w0 = wc * 32;
                }
            }
            // no copy may be in flight when the block exits
            int no_abort = 0;
            for (int jj = max(0, j - a.nd); jj < j; ++jj)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_full[jj % a.nd]),
                                       (uint32_t)(jj / a.nd) & 1u, &no_abort, a.status,
                                       kW4LimitNs);
        }
    } else if (warp == 1) {
        // ---- MMA issue (one thread): per item pair one wait, 2 x nks MMAs
        // (operands hoisted) and one commit
        if (lane == 0 && has_work) {
            const uint32_t idesc = ptx::idesc_tf32(128, a.N);
            const uint64_t bd0 = ptx::smem_desc(ptx::smem_u32(xring), 16, 1024, 2);
            const uint32_t slot_units = a.xslot_bytes >> 4;
            Item it = decode(a, i0);
            int wc = it.w0 >> 5;
            const int nks_last = min(4, (a.Wx - (a.nwc - 1) * 32 + 7) >> 3);
            int t_ws = 0;
            bool ok = true;
            for (int m = 0; 2 * m < cnt; ++m) {
                const int stage = m % kW4NA;
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_full[stage]),
                                            (uint32_t)(m / kW4NA) & 1u, &sb.abort_flag,
                                            a.status, kW4LimitNs);
                if (!ok) break;
                ptx::tc_fence_after();
                const int nitems = min(2, cnt - 2 * m);
                for (int e = 0; e < nitems; ++e) {
                    const uint64_t bd = bd0 + (uint64_t)((uint32_t)(t_ws % a.nr) * slot_units);
                    const uint32_t a_tm = tmem + acol0 + (uint32_t)(stage * 64 + e * 32);
                    ptx::mma_tf32_ts(tmem, a_tm, bd, idesc, (m > 0 || e > 0) ? 1u : 0u);
                    if (wc + 1 < a.nwc || nks_last == 4) {
#pragma unroll
                        for (int ks = 1; ks < 4; ++ks)
                            ptx::mma_tf32_ts(tmem, a_tm + ks * 8, bd + 2 * ks, idesc, 1u);
                    } else {
                        for (int ks = 1; ks < nks_last; ++ks)
                            ptx::mma_tf32_ts(tmem, a_tm + ks * 8, bd + 2 * ks, idesc, 1u);
                    }
                    t_ws += it.p + 1 == a.Pe ? R : 1;
                    if (++it.p == a.Pe) {
                        it.p = 0;
                        if (++wc == a.nwc) wc = 0;
                    }
                }
                ptx::mma_commit(ptx::smem_u32(&sb.done[m % kW4Done]));
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
        // ---- A producers: group g takes the item pairs m = g, g + 2, ...;
        // pair m goes to TMEM stage m % kW4NA (item 2m in its first 32
        // columns, item 2m + 1 in the next 32).  Thread = TMEM lane kl =
        // output channel k0 + kl.
        const int g = (warp - 2) >> 2, quarter = warp & 3;
        const int kl = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const bool kv = kl < a.kbox;
        int p = has_work ? decode(a, i0).p : 0;
        int t_ws = 0, t_ready = 0;  // x rows this warp has seen land (lane 0)
        bool ok = true;
        for (int m = 0; 2 * m < cnt; ++m) {
            const int nitems = min(2, cnt - 2 * m);
            const int t_lo = t_ws;  // rows the pair needs: t_lo .. t_hi - 1
            int t_hi = 0;
            for (int e = 0; e < nitems; ++e) {
                t_hi = t_ws + R;
                t_ws += p + 1 == a.Pe ? R : 1;
                if (++p == a.Pe) p = 0;
            }
            if ((m & 1) != g) continue;
            if (m >= kW4NA)  // the stage was last read by pair m - kW4NA
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.done[(m - kW4NA) % kW4Done]),
                                            (uint32_t)((m - kW4NA) / kW4Done) & 1u,
                                            &sb.abort_flag, a.status, kW4LimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            for (int e = 0; e < nitems; ++e) {
                const int j = 2 * m + e;
                const int ds = j % a.nd;
                ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.dz_full[ds]),
                                            (uint32_t)(j / a.nd) & 1u, &sb.abort_flag,
                                            a.status, kW4LimitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                float v[32];
                const float *tilep =
                    reinterpret_cast<const float *>(dzring + (size_t)ds * a.dz_stride);
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = kv ? tilep[q * a.kbox + kl] : 0.f;
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sb.dz_empty[ds]));
                ptx::tmem_st32(tmem + lane_addr + acol0 + (uint32_t)((m % kW4NA) * 64 + e * 32),
                               v);
            }
            if (!ok) break;
            // the pair's x rows must have landed before the MMA may start
            if (lane == 0) {
                for (int t = max(t_ready, t_lo); ok && t < t_hi; ++t)
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.x_full[t % a.nr]),
                                                (uint32_t)(t / a.nr) & 1u, &sb.abort_flag,
                                                a.status, kW4LimitNs);
                t_ready = t_hi;
            }
            ok = __all_sync(0xffffffffu, __shfl_sync(0xffffffffu, ok, 0));
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            if (!ok) break;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sb.a_full[m % kW4NA]));
        }
        // ---- epilogue: D[k][col] -> shared memory [col][k] (the x ring is idle
        // once every MMA has completed), then one bulk reduce-add of the tile
        // into acc[tile]
        if (has_work && ok)
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &sb.abort_flag, a.status,
                                        kW4LimitNs);
        if (ok) ok = *reinterpret_cast<volatile int *>(&sb.abort_flag) == 0;
        ok = __all_sync(0xffffffffu, ok) && has_work;
        float *stage = reinterpret_cast<float *>(smem);
        if (ok) {
            ptx::tc_fence_after();
            // this group's 16-column chunks g, g + 2, ..., four TMEM loads per wait
            for (int c0 = g; c0 * 16 < a.N; c0 += 8) {
                float v[4][16];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if ((c0 + 2 * j) * 16 < a.N)
                        ptx::tmem_ld16(tmem + lane_addr + (uint32_t)((c0 + 2 * j) * 16), v[j]);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if ((c0 + 2 * j) * 16 < a.N) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            stage[((c0 + 2 * j) * 16 + e) * 128 + kl] = v[j][e];
                    }
            }
            ptx::fence_proxy_async_smem();  // the bulk copy reads these writes
        }
        ok = ptx::named_bar_and(1, 256, ok);  // the eight epilogue warps
        if (ok && warp == 2 && lane == 0) {
            ptx::bulk_reduce_add_f32(a.acc + (size_t)tile * a.N * 128, ptx::smem_u32(stage),
                                     (uint32_t)(a.N * 128 * sizeof(float)));
            ptx::bulk_commit();
            ptx::bulk_wait_read_all();  // shared memory is read before the block exits
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::griddep_launch_dependents();  // the accumulator apply may be scheduled
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// dW[k][cg][r][s] += acc[tile][r * cb + c_local][k_local]: the tile
// accumulators (tile = (k tile * nctile + c tile) * S + s) added into dW, one
// thread per (k, cg, r), which adds its S contiguous dW elements (coalesced
// along the warp) from S accumulator entries (scattered reads that hit the
// L2); 32-bit index arithmetic, computed once per thread.  The input channel
// of group-local index cg is c = (k / Kg) * Cg + cg (dense: Cg = C, Kg = K).
// The first nrep blocks transpose the input gradient's weight repack instead
// (see cba_repack.cuh), beside the apply blocks.
__global__ void __launch_bounds__(256)
    wgrad_acc_apply_kernel(const float *__restrict__ acc, int N, int cb, int S, int nctile,
                           int R, int Cg, int Kg, int nrows, float *__restrict__ dW, int napply,
                           RepackJob rep, int nrep) {
    ptx::griddep_wait();  // the accumulators come from the weight-gradient kernel
    if ((int)blockIdx.x < nrep) {
        repack_part(rep, (int)blockIdx.x, nrep);
        return;
    }
    const int ab = (int)blockIdx.x - nrep;  // apply block
    const size_t tile_stride = (size_t)N * 128;
    for (int row = ab * (int)blockDim.x + (int)threadIdx.x; row < nrows;
         row += napply * (int)blockDim.x) {
        const int kc = row / R, r = row - kc * R;  // row = (k * Cg + cg) * R + r
        const int k = kc / Cg, cg = kc - k * Cg;
        const int c = cg + (k / Kg) * Cg;
        const int kt = k >> 7, kl = k & 127;
        const int ct = c / cb, cl = c - ct * cb;
        const float *ap = acc + (size_t)(kt * nctile + ct) * S * tile_stride +
                          ((size_t)r * cb + cl) * 128 + kl;
        float *wp = dW + (size_t)row * S;
        for (int s0 = 0; s0 < S; s0 += 4) {
            float av[4], wv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (s0 + u < S) {
                    av[u] = ap[(size_t)(s0 + u) * tile_stride];
                    wv[u] = wp[s0 + u];
                }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (s0 + u < S) wp[s0 + u] = wv[u] + av[u];
        }
    }
}

W4Geom w4_geom(const Plan &p) {
    W4Geom w{};
    w.ok = false;
    if (p.stride != 1) return w;
    if (!((p.R == 3 && p.S == 3) || (p.R == 1 && p.S == 1))) return w;
    if (p.pad > p.S - 1) return w;
    const DzcGeom g = dzc_geom(p);
    if (g.We % 4 != 0) return w;  // x rows must be 16-byte strided for TMA
    // input channels per block: N = R * cb a multiple of 16, at most 256
    const int cap = p.R == 1 ? 256 : 64;
    w.cb = std::min(cap, (p.C + 15) / 16 * 16);
    w.N = p.R * w.cb;
    if (w.N > 256 || w.N % 16 != 0 || w.N + kW4NA * 64 > 512) return w;
    w.nctile = (p.C + w.cb - 1) / w.cb;
    w.ktiles = (p.K + 127) / 128;
    w.ntiles = w.ktiles * w.nctile * p.S;
    w.nwc = (g.We + 31) / 32;
    const long long items = (long long)p.N * w.nwc * g.Pe;
    if (items >= (1LL << 31)) return w;
    w.items = (int)items;
    w.cpt = std::max(1, std::min(w.items, p.num_sms / w.ntiles));
    w.grid = w.ntiles * w.cpt;
    w.kbox = std::min(128, g.Kp);
    w.xslot_bytes = (uint32_t)w.cb * 128u;
    w.dz_bytes = (uint32_t)(32 * w.kbox * 4);
    w.dz_stride = (w.dz_bytes + 127u) / 128u * 128u;
    // shared memory: dz ring, x ring with its mirror slots; as deep as fits,
    // at least 4 dz slots and R + 2 x rows
    const size_t budget = 224 * 1024;
    int nd = kW4MaxND, nr = kW4MaxNR;
    auto bytes = [&](int d, int r) {
        return (size_t)d * w.dz_stride + (size_t)(r + p.R - 1) * w.xslot_bytes;
    };
    while (bytes(nd, nr) > budget && (nr > 8 || nd > 4) && nr > p.R + 2) {
        if (nd > 4 && (nr <= 8 || nd * (size_t)w.dz_stride > (size_t)nr * w.xslot_bytes)) --nd;
        else --nr;
    }
    while (bytes(nd, nr) > budget && nr > p.R + 2) --nr;
    while (bytes(nd, nr) > budget && nd > 2) --nd;
    if (bytes(nd, nr) > budget) return w;
    w.nr = nr;
    w.nd = nd;
    const size_t dz_ring = (size_t)nd * w.dz_stride;
    w.dz_off = (uint32_t)((size_t)(nr + p.R - 1) * w.xslot_bytes);
    // the epilogue stages a whole tile ([N][128] fp32) in the same memory
    w.smem = std::max((size_t)w.dz_off + dz_ring, (size_t)w.N * 128 * sizeof(float)) + 1024;
    if (w.smem > 227 * 1024) return w;
    w.acc_bytes = (size_t)w.ntiles * w.N * 128 * sizeof(float);
    w.ok = true;
    return w;
}

}  // namespace

size_t wgrad_tc4_ws_bytes(const Plan &p) {
    const W4Geom w = w4_geom(p);
    return w.ok ? w.acc_bytes : 0;
}

bool wgrad_tc4_supported(const Plan &p) {
    // int32 dW row index of the accumulator apply
    return w4_geom(p).ok && (long long)p.K * p.Cg * p.R < (1LL << 31);
}

cudaError_t launch_wgrad_tc4(const Plan &p, const float *x, const float *dzc, float *dW,
                             void *ws, const RepackJob *rep, cudaStream_t st, int *launches) {
    const W4Geom w = w4_geom(p);
    if (!w.ok) return cudaErrorNotSupported;
    const DzcGeom g = dzc_geom(p);
    W4Args a;
    a.acc = ws_at<float>(ws, p.off_wgacc);
    a.status = ws_at<unsigned>(ws, p.off_status);
    a.S = p.S; a.Pe = g.Pe; a.pad = p.pad; a.nwc = w.nwc; a.Wx = g.We;
    a.bq_lo = g.bq_lo; a.bd_lo = g.bd_lo;
    a.kbox = w.kbox; a.cb = w.cb; a.N = w.N; a.nctile = w.nctile; a.cpt = w.cpt;
    a.items_per_tile = w.items; a.nr = w.nr; a.nd = w.nd;
    a.xslot_bytes = w.xslot_bytes; a.dz_bytes = w.dz_bytes; a.dz_stride = w.dz_stride;
    a.dz_off = w.dz_off;

    alignas(64) CUtensorMap tmx, tmdz;
    {
        const uint64_t d[4] = {(uint64_t)g.We, (uint64_t)g.He, (uint64_t)p.C, (uint64_t)p.N};
        const uint32_t b[4] = {32, 1, (uint32_t)w.cb, 1};
        if (!tma_encode_f32(&tmx, x, 4, d, b, true)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t d[4] = {(uint64_t)g.Kp, (uint64_t)g.Qpp, (uint64_t)g.Pp, (uint64_t)p.N};
        const uint32_t b[4] = {(uint32_t)w.kbox, 32, 1, 1};
        if (!tma_encode_f32(&tmdz, dzc, 4, d, b, false)) return cudaErrorInvalidValue;
    }
    cudaError_t e;
    if (p.R == 3) {
        e = cudaFuncSetAttribute(wgrad_tc4_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)w.smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(wgrad_tc4_kernel<3>, dim3(w.grid), dim3(kW4Threads), w.smem, st, tmx, tmdz,
                       a);
    } else {
        e = cudaFuncSetAttribute(wgrad_tc4_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)w.smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(wgrad_tc4_kernel<1>, dim3(w.grid), dim3(kW4Threads), w.smem, st, tmx, tmdz,
                       a);
    }
    if (e != cudaSuccess) return e;
    const int nrows = p.K * p.Cg * p.R;  // dW rows of S elements, < 2^31 (wgrad_tc4_supported)
    const unsigned ablocks = (unsigned)std::min<long long>((nrows + 255) / 256, p.num_sms * 32LL);
    const RepackJob job = rep ? *rep : RepackJob{};
    const int nrep = rep ? (int)std::min<long long>(repack_tiles(*rep), 4LL * p.num_sms) : 0;
    e = launch_pdl(wgrad_acc_apply_kernel, dim3(ablocks + nrep), dim3(256), 0, st,
                   (const float *)a.acc, w.N, w.cb, p.S, w.nctile, p.R, p.Cg, p.Kg, nrows, dW,
                   (int)ablocks, job, nrep);
    if (e != cudaSuccess) return e;
    *launches += 2;
    return cudaGetLastError();
}

}  // namespace cba
