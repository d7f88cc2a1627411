// cba_wgrad_nb.cu -- weight gradient on batch-innermost operand layouts
// (dW[k][c][r][s] += sum_{n,p,q} dz[n][k][p][q] x[n][c][p*st + r - pad][q*st + s - pad],
// the gemm(0,1,...) of "YOLOv3反向传播原理 之 全流程源码分析" §3.1 over the
// im2col_cpu columns of §3.2, without the column buffer).
//
// The contraction runs over (n, p, q).  Both operands are laid out with the
// batch innermost, in chunks of nb = 16 or 32 images:
//   xn  [nc][H][W][C][nb]   x, TF32-rounded, zeros for images past N
//   dzn [nc][P][Q][K][nb]   the BN-input gradient dz, TF32-rounded
// so one output position (p, q) with its nb images is one K-major operand
// row per channel (nb * 4 = 64 or 128 bytes, 64- or 128-byte swizzle), and
// every tap shift (r, s) and the stride move only the pixel coordinates,
// which are not the innermost dimension: TMA loads them at any offset, and
// padding is TMA's zero fill.  No thread touches an operand.
//
// A block owns one tile (KT k-tiles of 128 output channels = MMA M, cb input
// channels, one kernel row r) and a range of contraction items (one output
// position with its nb images each).  Per item:
//   A = dzn[(j, p, q)][k0 .. k0 + 127][nb]       a slot of the A ring
//   B = xn[j][h = p*st + r - pad][w0 .. w0 + S - 1][c0 .. c0 + cb - 1][nb]
//       with w0 = q*st - pad: S consecutive pixels of the pixel ring, whose
//       rows (s, c) are contiguous, so one MMA of N = S * cb covers all S
//       kernel columns; the first pixels of the ring are mirrored after its
//       end, so a window that wraps is still contiguous
//   D[k][(s, c)] += A * B^T   (nb / 8 MMAs of K = 8 per k-tile)
// Consecutive items of an output row share S - st of their pixels, so the
// pixel ring loads st new pixels per item.  Each block adds its D tile into a
// per-tile accumulator in the workspace with bulk reduce-adds (the L2 sums
// the blocks of a tile); a second kernel adds the accumulators into dW.
//
// Roles: warp 0 issues the A loads, warp 2 the pixel loads, warp 1 the MMAs
// (one thread), warps 4-7 run the epilogue (TMEM lanes 0-127).  Every wait is
// bounded (2 s); on a timeout the block sets the workspace status bit and
// stops.
#include <cuda.h>

#include <algorithm>

#include "cba_internal.cuh"
#include "cba_ptx.cuh"
#include "cba_repack.cuh"

namespace cba {

namespace {

constexpr uint64_t kWnLimitNs = 2000000000ull;
constexpr int kWnThreads = 256;
constexpr int kWnMaxNA = 8;   // A ring slots
constexpr int kWnMaxNG = 8;   // pixel-ring groups (the mirror comes on top)

__device__ __forceinline__ float rna_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// ------------------------------------------------------- layout passes

template <int ACT, bool BN>
struct DzSrc {
    const float *delta, *output, *z;
    const Coef *coef;
    __device__ __forceinline__ float operator()(long long off, int k) const {
        const float y = (ACT == CBA_ACT_LEAKY) ? __ldg(output + off) : 0.f;
        const float zz = BN ? __ldg(z + off) : 0.f;
        return dz_of<ACT, BN>(__ldg(delta + off), y, zz, coef[k]);
    }
    // four consecutive elements (off a multiple of 4), TF32-rounded
    __device__ __forceinline__ float4 load4(long long off, int k) const {
        const float4 d = __ldg(reinterpret_cast<const float4 *>(delta + off));
        const float4 y = (ACT == CBA_ACT_LEAKY) ? __ldg(reinterpret_cast<const float4 *>(output + off))
                                                : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 zz = BN ? __ldg(reinterpret_cast<const float4 *>(z + off))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        const Coef cf = coef[k];
        return make_float4(rna_tf32(dz_of<ACT, BN>(d.x, y.x, zz.x, cf)),
                           rna_tf32(dz_of<ACT, BN>(d.y, y.y, zz.y, cf)),
                           rna_tf32(dz_of<ACT, BN>(d.z, y.z, zz.z, cf)),
                           rna_tf32(dz_of<ACT, BN>(d.w, y.w, zz.w, cf)));
    }
};

// Four consecutive elements of x (off a multiple of 4), TF32-rounded.
__device__ __forceinline__ float4 x_load4(const float *x, long long off) {
    const float4 v = __ldg(reinterpret_cast<const float4 *>(x + off));
    return make_float4(rna_tf32(v.x), rna_tf32(v.y), rna_tf32(v.z), rna_tf32(v.w));
}

// Loads the (NB images of chunk j) x (8 channels c0 ..) x (32 positions pos0 ..)
// tile of src [N][CH][PLANE] into tile[position][channel * NB + image]
// (TF32-rounded, zeros past N, CH and PLANE).  VEC: PLANE a multiple of 4, float4
// reads along the positions.  Every load of the thread is issued before the
// first store to shared memory.
template <int NB, bool VEC, class Load1, class Load4>
__device__ __forceinline__ void bi_load_tile(Load1 load1, Load4 load4, int N, int CH, int PLANE,
                                             int j, int c0, int pos0, float (*tile)[8 * NB + 1]) {
    const int t = threadIdx.x;
    if constexpr (VEC) {
        constexpr int PER4 = NB * 8 * 8 / 256;
        float4 v[PER4];
#pragma unroll
        for (int u = 0; u < PER4; ++u) {
            const int e = t + u * 256;
            const int q4 = e & 7, rc = e >> 3;
            const int n = j * NB + (rc >> 3), c = c0 + (rc & 7), pp = pos0 + 4 * q4;
            v[u] = (n < N && c < CH && pp < PLANE) ? load4(((long long)n * CH + c) * PLANE + pp, c)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < PER4; ++u) {
            const int e = t + u * 256;
            const int q4 = e & 7, rc = e >> 3;
            const int col = (rc & 7) * NB + (rc >> 3);
            tile[4 * q4 + 0][col] = v[u].x;
            tile[4 * q4 + 1][col] = v[u].y;
            tile[4 * q4 + 2][col] = v[u].z;
            tile[4 * q4 + 3][col] = v[u].w;
        }
    } else {
        constexpr int PER = NB * 8 * 32 / 256;
        float v[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = t + u * 256;
            const int pos = e & 31, rc = e >> 5;
            const int n = j * NB + (rc >> 3), c = c0 + (rc & 7), pp = pos0 + pos;
            v[u] = (n < N && c < CH && pp < PLANE)
                       ? rna_tf32(load1(((long long)n * CH + c) * PLANE + pp, c))
                       : 0.f;
        }
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = t + u * 256;
            const int rc = e >> 5;
            tile[e & 31][(rc & 7) * NB + (rc >> 3)] = v[u];
        }
    }
}

// Writes the tile batch-innermost: dst [nc][PLANE][CH][NB], for each position
// the 8 channels x NB images contiguous.
template <int NB>
__device__ __forceinline__ void bi_store_tile(const float (*tile)[8 * NB + 1], int CH, int PLANE,
                                              int j, int c0, int pos0, float *__restrict__ dst) {
    const int ncl = min(8, CH - c0);
    for (int e = threadIdx.x; e < 32 * 8 * NB; e += 256) {
        const int pos = e / (8 * NB), vv = e % (8 * NB);
        const int pp = pos0 + pos;
        if (pp < PLANE && vv < ncl * NB)
            dst[(((long long)j * PLANE + pp) * CH + c0) * NB + vv] = tile[pos][vv];
    }
}

// The layout pass of the batch-innermost weight gradient, one launch.  Blocks,
// in this order (a 1-D grid):
//   dz tiles:  dzn [nc][PQ][K][NB] batch-innermost (weight gradient) and, with
//              DZC, dzc [N][Pp][Qpp][Kp] channels-last with a zero border of
//              bd_lo / bq_lo rows / columns (input gradient; channels K .. Kp-1
//              zero).  Channel chunks in descending order: the reduction pass
//              read the high channels last, so they are the ones still in L2.
//   x tiles:   xn [nc][HW][C][NB] (TF32-rounded).
//   border:    one (image, row) of dzc per block: a border row zeroed whole, an
//              inner row at its bq_lo left and Qpp - bq_lo - Qe right columns.
struct LayoutArgs {
    int N, K, Kp, PQ, Qe, Pp, Qpp, Pe, bd_lo, bq_lo;
    int kchunks, npx_dz, ndz;      // dz: channel chunks of 8 (over Kp), position chunks, blocks
    int C, HW, xchunks, npx_x, nx;  // x: channel chunks, position chunks, blocks
    int nborder;                    // border rows (0 without dzc or border)
    int nrep;                       // weight-repack blocks (0: none)
    RepackJob rep;
    const float *x;
    float *dzn, *dzc, *xn;
};

template <int NB, int ACT, bool BN, bool DZC, bool VEC, bool XVEC>
__global__ void __launch_bounds__(256) layouts_kernel(DzSrc<ACT, BN> src, LayoutArgs la) {
    ptx::griddep_wait();  // the coefficients come from the reduction pass
    __shared__ float tile[32][8 * NB + 1];
    const int t = threadIdx.x;
    int bid = (int)blockIdx.x;
    if (bid < la.ndz) {
        const int px = bid % la.npx_dz, py = bid / la.npx_dz;
        const int j = py / la.kchunks, k0 = (la.kchunks - 1 - py % la.kchunks) * 8;
        const int pos0 = px * 32;
        bi_load_tile<NB, VEC>(
            [&](long long off, int k) { return src(off, k); },
            [&](long long off, int k) { return src.load4(off, k); }, la.N, la.K, la.PQ, j, k0,
            pos0, tile);
        __syncthreads();
        ptx::griddep_launch_dependents();
        bi_store_tile<NB>(tile, la.K, la.PQ, j, k0, pos0, la.dzn);
        if constexpr (DZC) {
            // dzc: for each (image, position), the 8 channels as two float4 (Kp
            // and k0 are multiples of 4)
            const int nk4 = min(2, (la.Kp - k0) / 4);
            for (int e = t; e < 32 * NB; e += 256) {
                const int pos = e & 31, nl = e >> 5;
                const int n = j * NB + nl, pp = pos0 + pos;
                if (n >= la.N || pp >= la.PQ) continue;
                const int pr = pp / la.Qe, qc = pp - pr * la.Qe;
                float4 *out = reinterpret_cast<float4 *>(
                    la.dzc +
                    (((long long)n * la.Pp + la.bd_lo + pr) * la.Qpp + la.bq_lo + qc) * la.Kp + k0);
                for (int h = 0; h < nk4; ++h)
                    out[h] = make_float4(tile[pos][(4 * h + 0) * NB + nl],
                                         tile[pos][(4 * h + 1) * NB + nl],
                                         tile[pos][(4 * h + 2) * NB + nl],
                                         tile[pos][(4 * h + 3) * NB + nl]);
            }
        }
        return;
    }
    bid -= la.ndz;
    if (bid < la.nx) {
        const int px = bid % la.npx_x, py = bid / la.npx_x;
        const int j = py / la.xchunks, c0 = (py % la.xchunks) * 8;
        const int pos0 = px * 32;
        const float *x = la.x;
        bi_load_tile<NB, XVEC>([&](long long off, int) { return __ldg(x + off); },
                               [&](long long off, int) { return x_load4(x, off); }, la.N, la.C,
                               la.HW, j, c0, pos0, tile);
        __syncthreads();
        ptx::griddep_launch_dependents();
        bi_store_tile<NB>(tile, la.C, la.HW, j, c0, pos0, la.xn);
        return;
    }
    bid -= la.nx;
    if (bid < la.nborder) {
        ptx::griddep_launch_dependents();
        if constexpr (DZC) {
            const int row = bid % la.Pp;
            float4 *base = reinterpret_cast<float4 *>(la.dzc + (long long)bid * la.Qpp * la.Kp);
            const int k4 = la.Kp / 4;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < la.bd_lo || row >= la.bd_lo + la.Pe) {
                for (int i = t; i < la.Qpp * k4; i += 256) base[i] = z;
                return;
            }
            const int nl = la.bq_lo, nr = la.Qpp - la.bq_lo - la.Qe;
            for (int i = t; i < (nl + nr) * k4; i += 256) {
                const int c = i / k4, kk = i - c * k4;
                const int col = c < nl ? c : la.bq_lo + la.Qe + (c - nl);
                base[col * k4 + kk] = z;
            }
        }
        return;
    }
    bid -= la.nborder;
    if (bid < la.nrep) {
        // the input gradient's weight repack (cba_repack.cuh), through this
        // block's tile buffer
        ptx::griddep_launch_dependents();
        repack_part_group(la.rep, bid, la.nrep, &tile[0][0], t, 256, 1);
    }
}

}  // namespace

namespace {

struct WnArgs {
    float *acc;             // [unit][KT][cols][128] tile accumulators (zeroed before the call)
    unsigned *status;
    int P, Q, R, S, stride, pad;
    int ctiles, KT, cb, cols;  // cols = S * cb = the MMA's N
    int stages;             // epilogue stages in shared memory: KT, or 1 (reused)
    int splits;             // blocks per tile
    long long items;        // nc * P * Q
    int Qa, NA;             // positions per A box, A ring slots
    int G, NG;              // pixels per group, pixel-ring groups (mirror group after them)
    int mirror;             // 1 when S > 1 (a window may wrap the ring)
    uint32_t rb;            // operand row bytes (nb * 4)
    uint32_t swz;           // shared-memory descriptor swizzle code
    uint32_t a_pos_bytes;   // 128 * rb: one position of one k-tile
    uint32_t a_slot_bytes;  // KT * Qa * a_pos_bytes
    uint32_t pix_bytes;     // cb * rb
    uint32_t grp_bytes;     // G * pix_bytes
    uint32_t b_off;         // byte offset of the pixel ring
};

struct WnBars {
    uint64_t a_full[kWnMaxNA], a_empty[kWnMaxNA];
    uint64_t b_full[kWnMaxNG], b_empty[kWnMaxNG];
    uint64_t accum;
    uint32_t tmem_base;
    int abort_flag;
};

// Items are output positions in (j, p, q) order, q fastest; a run is the
// part of one output row (j, p) inside a block's range.  Every role walks
// the runs the same way: A boxes of up to Qa positions from the start of each
// run, pixel groups of G pixels from the run's first window.
struct Run {
    long long row;  // j * P + p
    int qa, qb;     // positions qa .. qb - 1 of the row
};

__device__ __forceinline__ Run run_at(long long i, long long i1, int Q) {
    Run u;
    u.row = i / Q;
    u.qa = (int)(i - u.row * Q);
    u.qb = (int)(min(i1, (u.row + 1) * Q) - u.row * Q);
    return u;
}

template <int NB>
__global__ void __launch_bounds__(kWnThreads, 1)
    wgrad_nb_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                    const WnArgs a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ WnBars sb;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
    const int r = unit % a.R;
    const int ct = (unit / a.R) % a.ctiles;
    const int kt = unit / (a.R * a.ctiles);
    const int k0 = kt * a.KT * 128, c0 = ct * a.cb;
    const long long i0 = split * a.items / a.splits, i1 = (split + 1) * a.items / a.splits;
    const bool has_work = i1 > i0;
    uint8_t *aring = smem;
    uint8_t *bring = smem + a.b_off;
    const int ring_pix = a.NG * a.G;  // pixel slots before the mirror

    if (tid == 0) {
        for (int i = 0; i < kWnMaxNA; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.a_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.a_empty[i]), 1);
        }
        for (int i = 0; i < kWnMaxNG; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sb.b_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sb.b_empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&sb.accum), 1);
        sb.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        const uint32_t need = (uint32_t)(a.KT * a.cols);
        uint32_t ncols = 32;
        while (ncols < need) ncols <<= 1;
        ptx::tmem_alloc(ptx::smem_u32(&sb.tmem_base), ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sb.tmem_base;
    // the operand layouts come from the previous kernels
    ptx::griddep_wait();

    if (warp == 0) {
        // ---- A loads: boxes of up to Qa positions x KT k-tiles
        if (lane == 0 && has_work) {
            int slot = 0, issued = 0;
            uint32_t ph = 0;  // parity of the slot's previous release
            bool ok = true;
            for (long long i = i0; ok && i < i1;) {
                const Run rn = run_at(i, i1, a.Q);
                const int j = (int)(rn.row / a.P), p = (int)(rn.row - (long long)j * a.P);
                for (int q = rn.qa; q < rn.qb; q += a.Qa) {
                    if (issued >= a.NA)
                        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_empty[slot]), ph,
                                                    &sb.abort_flag, a.status, kWnLimitNs);
                    if (!ok) break;
                    const uint32_t bar = ptx::smem_u32(&sb.a_full[slot]);
                    ptx::mbar_arrive_expect_tx(bar, a.a_slot_bytes);
                    for (int t = 0; t < a.KT; ++t)
                        ptx::tma_load_4d(ptx::smem_u32(aring + (size_t)slot * a.a_slot_bytes +
                                                       (size_t)t * a.Qa * a.a_pos_bytes),
                                         &tma, 0, k0 + t * 128, q, j * a.P + p, bar);
                    ++issued;
                    if (++slot == a.NA) {
                        slot = 0;
                        if (issued > a.NA) ph ^= 1u;
                    }
                }
                i = rn.row * a.Q + rn.qb;
            }
            // no copy may be in flight when the block exits: wait for the last
            // min(issued, NA) copies (slot, phase counted back from the end)
            int no_abort = 0;
            for (int v = issued > a.NA ? issued - a.NA : 0; v < issued; ++v)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_full[v % a.NA]),
                                       (uint32_t)((v / a.NA) & 1), &no_abort, a.status,
                                       kWnLimitNs);
        }
    } else if (warp == 2) {
        // ---- pixel loads: per run, groups of G pixels from its first window
        if (lane == 0 && has_work) {
            int gs = 0, issued = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (long long i = i0; ok && i < i1;) {
                const Run rn = run_at(i, i1, a.Q);
                const int j = (int)(rn.row / a.P), p = (int)(rn.row - (long long)j * a.P);
                const int h = p * a.stride + r - a.pad;
                const int wa = rn.qa * a.stride - a.pad;
                const int npix = (rn.qb - 1 - rn.qa) * a.stride + a.S;
                const int ng = (npix + a.G - 1) / a.G;
                for (int g = 0; g < ng; ++g) {
                    if (issued >= a.NG)
                        ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.b_empty[gs]), ph,
                                                    &sb.abort_flag, a.status, kWnLimitNs);
                    if (!ok) break;
                    const bool mir = a.mirror && gs == 0;
                    const uint32_t bar = ptx::smem_u32(&sb.b_full[gs]);
                    ptx::mbar_arrive_expect_tx(bar, a.grp_bytes * (mir ? 2u : 1u));
                    ptx::tma_load_5d(ptx::smem_u32(bring + (size_t)gs * a.grp_bytes), &tmb, 0, c0,
                                     wa + g * a.G, h, j, bar);
                    if (mir)
                        ptx::tma_load_5d(ptx::smem_u32(bring + (size_t)a.NG * a.grp_bytes), &tmb,
                                         0, c0, wa + g * a.G, h, j, bar);
                    ++issued;
                    if (++gs == a.NG) {
                        gs = 0;
                        if (issued > a.NG) ph ^= 1u;
                    }
                }
                i = rn.row * a.Q + rn.qb;
            }
            int no_abort = 0;
            for (int v = issued > a.NG ? issued - a.NG : 0; v < issued; ++v)
                ptx::mbar_wait_bounded(ptx::smem_u32(&sb.b_full[v % a.NG]),
                                       (uint32_t)((v / a.NG) & 1), &no_abort, a.status,
                                       kWnLimitNs);
        }
    } else if (warp == 1) {
        // ---- MMA issue (one thread): per item KT x NB/8 MMAs of N = S * cb;
        // an A slot is released after its last position, a pixel group once
        // no later window of the run reaches it.  The loop keeps only
        // incremental counters (ring slots, parities, the window's ring pixel)
        // and adds 16-byte offsets to two precomputed descriptors.
        if (lane == 0 && has_work) {
            constexpr int KS = NB / 8;  // K = 8 steps per operand row
            const uint32_t idesc = ptx::idesc_tf32(128, a.cols);
            const uint32_t sbo = 8 * a.rb;
            const uint64_t da0 = ptx::smem_desc(ptx::smem_u32(aring), 16, sbo, a.swz);
            const uint64_t db0 = ptx::smem_desc(ptx::smem_u32(bring), 16, sbo, a.swz);
            const uint32_t a_slot16 = a.a_slot_bytes >> 4, a_pos16 = a.a_pos_bytes >> 4;
            const uint32_t a_t16 = ((uint32_t)a.Qa * a.a_pos_bytes) >> 4, pix16 = a.pix_bytes >> 4;
            int a_slot = 0, g_wslot = 0, g_rslot = 0, ps_run = 0;
            uint32_t a_ph = 0, g_wph = 0;
            bool ok = true, first = true;
            for (long long i = i0; ok && i < i1;) {
                const Run rn = run_at(i, i1, a.Q);
                const int npix = (rn.qb - 1 - rn.qa) * a.stride + a.S;
                const int ng = (npix + a.G - 1) / a.G;
                int waited = 0, released = 0;  // groups of this run
                int ps = ps_run;               // ring pixel of the item's window
                int u0 = 0;                    // run pixel of the item's window
                for (int qbox = rn.qa; ok && qbox < rn.qb; qbox += a.Qa) {
                    ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.a_full[a_slot]), a_ph,
                                                &sb.abort_flag, a.status, kWnLimitNs);
                    const int qend = min(qbox + a.Qa, rn.qb);
                    uint32_t a_off = (uint32_t)a_slot * a_slot16;
                    for (int q = qbox; ok && q < qend; ++q, a_off += a_pos16) {
                        for (; ok && waited * a.G < u0 + a.S; ++waited) {
                            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.b_full[g_wslot]), g_wph,
                                                        &sb.abort_flag, a.status, kWnLimitNs);
                            if (++g_wslot == a.NG) {
                                g_wslot = 0;
                                g_wph ^= 1u;
                            }
                        }
                        if (!ok) break;
                        ptx::tc_fence_after();
                        const uint64_t db = db0 + (uint64_t)((uint32_t)ps * pix16);
                        for (int t = 0; t < a.KT; ++t) {
                            const uint64_t da = da0 + (uint64_t)(a_off + (uint32_t)t * a_t16);
#pragma unroll
                            for (int ks = 0; ks < KS; ++ks)
                                ptx::mma_tf32(tmem + (uint32_t)(t * a.cols), da + 2 * ks,
                                              db + 2 * ks, idesc, (first && ks == 0) ? 0u : 1u);
                        }
                        first = false;
                        u0 += a.stride;
                        ps += a.stride;
                        while (ps >= ring_pix) ps -= ring_pix;
                        // groups that end before the next window are done
                        for (; released < ng && (released + 1) * a.G <= u0; ++released) {
                            ptx::mma_commit(ptx::smem_u32(&sb.b_empty[g_rslot]));
                            if (++g_rslot == a.NG) g_rslot = 0;
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit(ptx::smem_u32(&sb.a_empty[a_slot]));
                    if (++a_slot == a.NA) {
                        a_slot = 0;
                        a_ph ^= 1u;
                    }
                }
                if (!ok) break;
                for (; released < ng; ++released) {  // the rest of the run's groups
                    ptx::mma_commit(ptx::smem_u32(&sb.b_empty[g_rslot]));
                    if (++g_rslot == a.NG) g_rslot = 0;
                }
                ps_run += ng * a.G;
                while (ps_run >= ring_pix) ps_run -= ring_pix;
                i = rn.row * a.Q + rn.qb;
            }
            if (!ok) {  // the epilogue must not take the drain below for a result
                *reinterpret_cast<volatile int *>(&sb.abort_flag) = 1;
                __threadfence_block();
            }
            // drain: every MMA issued has finished before TMEM is released
            ptx::mma_commit(ptx::smem_u32(&sb.accum));
            int no_abort = 0;
            ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &no_abort, a.status, kWnLimitNs);
        }
    } else if (warp >= 4) {
        // ---- epilogue: D[k][col] of each k-tile -> shared memory [col][k] (the
        // rings are idle once every MMA has completed; each k-tile has its own
        // stage, so the bulk reduce-add of one overlaps the staging of the
        // next), then one bulk reduce-add of the tile into its accumulator.
        // The TMEM loads go four at a time before one wait.
        const int wq = warp & 3;
        const int kl = wq * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        bool ok = has_work;
        if (ok)
            ok = ptx::mbar_wait_bounded(ptx::smem_u32(&sb.accum), 0, &sb.abort_flag, a.status,
                                        kWnLimitNs);
        if (ok) ok = *reinterpret_cast<volatile int *>(&sb.abort_flag) == 0;
        ok = __all_sync(0xffffffffu, ok);
        const int nld = a.cols / 16;  // 16-column TMEM loads per k-tile
        for (int t = 0; t < a.KT; ++t) {
            const int si = t % a.stages;
            float *stage = reinterpret_cast<float *>(smem) + (size_t)si * a.cols * 128;
            if (t >= a.stages) {  // the stage's previous reduce-add has read it
                if (warp == 4 && lane == 0) ptx::bulk_wait_read_all();
                ptx::named_bar_sync(1, 128);
            }
            if (ok) {
                ptx::tc_fence_after();
                for (int c0 = 0; c0 < nld; c0 += 4) {
                    float v[4][16];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (c0 + j < nld)
                            ptx::tmem_ld16(tmem + lane_addr + (uint32_t)(t * a.cols + (c0 + j) * 16),
                                           v[j]);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (c0 + j < nld) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                stage[((c0 + j) * 16 + e) * 128 + kl] = v[j][e];
                        }
                }
                ptx::fence_proxy_async_smem();  // the bulk copy reads these writes
            }
            ok = ptx::named_bar_and(1, 128, ok);
            if (ok && warp == 4 && lane == 0) {
                ptx::bulk_reduce_add_f32(a.acc + ((size_t)unit * a.KT + t) * a.cols * 128,
                                         ptx::smem_u32(stage),
                                         (uint32_t)(a.cols * 128 * sizeof(float)));
                ptx::bulk_commit();
            }
        }
        if (warp == 4 && lane == 0) ptx::bulk_wait_read_all();  // before the block exits
        ptx::named_bar_sync(1, 128);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::griddep_launch_dependents();  // the accumulator apply may be scheduled
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        const uint32_t need = (uint32_t)(a.KT * a.cols);
        uint32_t ncols = 32;
        while (ncols < need) ncols <<= 1;
        ptx::tmem_dealloc(tmem, ncols);
    }
}

// dW[k][cg][r][s] += acc[unit][t][s * cb + cl][kl] with unit = (kt * ctiles +
// ct) * R + r, k = (kt * KT + t) * 128 + kl, c = ct * cb + cl, where c = (k /
// Kg) * Cg + cg is the input channel of group-local index cg (dense: Cg = C):
// one thread per (k, cg, r), which adds its S contiguous dW elements
// (coalesced along the warp) from S accumulator entries (scattered reads that
// hit the L2); 32-bit index arithmetic, computed once per thread.
// The first nrep blocks transpose the input gradient's weight repack instead
// (rep; see cba_repack.cuh): first, so that they run beside the apply blocks
// rather than after them.
__global__ void __launch_bounds__(256)
    wgrad_nb_apply_kernel(const float *__restrict__ acc, int KT, int cols, int cb, int S, int R,
                          int ctiles, int Cg, int Kg, int nrows, float *__restrict__ dW,
                          int napply, RepackJob rep, int nrep) {
    ptx::griddep_wait();  // the accumulators come from the weight-gradient kernel
    if ((int)blockIdx.x < nrep) {
        repack_part(rep, (int)blockIdx.x, nrep);
        return;
    }
    const int ab = (int)blockIdx.x - nrep;  // apply block
    const size_t unit_stride = (size_t)KT * cols * 128;  // one unit's accumulators
    for (int row = ab * (int)blockDim.x + (int)threadIdx.x; row < nrows;
         row += napply * (int)blockDim.x) {
        const int kc = row / R, r = row - kc * R;  // row = (k * Cg + cg) * R + r
        const int k = kc / Cg, cg = kc - k * Cg;
        const int c = cg + (k / Kg) * Cg;
        const int kt = k / (128 * KT), t = (k >> 7) - kt * KT, kl = k & 127;
        const int ct = c / cb, cl = c - ct * cb;
        const float *ap = acc + (size_t)((kt * ctiles + ct) * R + r) * unit_stride +
                          ((size_t)t * cols + cl) * 128 + kl;
        float *wp = dW + (size_t)row * S;
        // batches of 8 kernel columns: every load of a batch before its adds
        for (int s0 = 0; s0 < S; s0 += 8) {
            float av[8], wv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (s0 + u < S) {
                    av[u] = ap[(size_t)(s0 + u) * cb * 128];
                    wv[u] = wp[s0 + u];
                }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (s0 + u < S) wp[s0 + u] = wv[u] + av[u];
        }
    }
}

}  // namespace

namespace {

struct WnGeom {
    bool ok;
    int nb, nc, cb, cols, KT, ktiles, ctiles, units, splits, grid;
    long long items;
    int Qa, NA, G, NG;
    int stages;  // epilogue stages (one per k-tile when they fit)
    uint32_t rb, a_pos_bytes, a_slot_bytes, pix_bytes, grp_bytes, b_off;
    size_t smem, acc_bytes, xn_bytes, dzn_bytes;
};

WnGeom wn_geom(const Plan &p) {
    WnGeom w{};
    w.ok = false;
    if (p.S > 16 || p.R > 64) return w;
    w.nb = p.N <= 16 ? 16 : 32;
    w.nc = (p.N + w.nb - 1) / w.nb;
    w.rb = (uint32_t)w.nb * 4;
    // input channels per block: a multiple of 16 with S * cb <= 256 (one MMA),
    // the one that pads C least (the larger on a tie)
    const int cap = (256 / p.S) / 16 * 16;
    if (cap < 16) return w;
    int best = 16;
    long long best_pad = (long long)((p.C + 15) / 16) * 16;
    for (int cb = 32; cb <= cap; cb += 16) {
        const long long pad = (long long)((p.C + cb - 1) / cb) * cb;
        if (pad <= best_pad) {
            best = cb;
            best_pad = pad;
        }
    }
    w.cb = best;
    w.cols = p.S * w.cb;
    // two k-tiles per block share every pixel when both accumulators fit
    w.KT = (p.K > 128 && 2 * w.cols <= 512) ? 2 : 1;
    w.ktiles = (p.K + 128 * w.KT - 1) / (128 * w.KT);
    w.ctiles = (p.C + w.cb - 1) / w.cb;
    const long long units = (long long)w.ktiles * w.ctiles * p.R;
    w.items = (long long)w.nc * p.P * p.Q;
    if (units >= (1 << 20) || w.items >= (1LL << 40)) return w;
    w.units = (int)units;
    w.splits = (int)std::max(1LL, std::min(w.items, (long long)(p.num_sms / w.units)));
    w.grid = w.units * w.splits;
    // A boxes and pixel groups of at least 32 KB (positions per box, pixels
    // per group; a window of S pixels spans at most two groups): an issuing
    // thread's cost per barrier wait and copy, not the bytes in flight, sets
    // the copy rate, so fewer, larger copies per position keep the MMAs fed
    // (the residual block's 3x3 weight-gradient phase: 117 us with 16 KB of
    // dz rows per box and 16 KB pixel groups, 103 with 32 KB boxes, 99 with
    // 32 KB groups as well)
    w.a_pos_bytes = 128u * w.rb;
    w.Qa = std::max(1, (int)(32768 / w.a_pos_bytes));
    w.a_slot_bytes = (uint32_t)w.KT * w.Qa * w.a_pos_bytes;
    w.pix_bytes = (uint32_t)w.cb * w.rb;
    w.G = std::max({p.S - 1, 1, (int)((32768 + w.pix_bytes - 1) / w.pix_bytes)});
    if (w.G > 256) return w;
    w.grp_bytes = (uint32_t)w.G * w.pix_bytes;
    const size_t budget = 226 * 1024;  // 227 KB less the alignment slack
    const int mirror = p.S > 1 ? 1 : 0;
    int na = kWnMaxNA, ng = kWnMaxNG;
    auto bytes = [&](int a_, int g_) {
        return (size_t)a_ * w.a_slot_bytes + (size_t)(g_ + mirror) * w.grp_bytes;
    };
    while (bytes(na, ng) > budget && (na > 2 || ng > 2)) {
        if (na > 2 && (ng <= 2 || (size_t)na * w.a_slot_bytes >= (size_t)ng * w.grp_bytes)) --na;
        else --ng;
    }
    if (bytes(na, ng) > budget) return w;
    w.NA = na;
    w.NG = ng;
    w.b_off = (uint32_t)((size_t)na * w.a_slot_bytes);
    // epilogue stages: one per k-tile when they fit, else one reused
    const size_t stage1 = (size_t)w.cols * 128 * sizeof(float);
    w.stages = (std::max(bytes(na, ng), (size_t)w.KT * stage1) + 1024 <= 227 * 1024) ? w.KT : 1;
    w.smem = std::max(bytes(na, ng), (size_t)w.stages * stage1) + 1024;
    if (w.smem > 227 * 1024) return w;
    w.acc_bytes = (size_t)w.units * w.KT * w.cols * 128 * sizeof(float);
    w.xn_bytes = sizeof(float) * (size_t)w.nc * w.nb * p.H * p.W * p.C;
    w.dzn_bytes = sizeof(float) * (size_t)w.nc * w.nb * p.P * p.Q * p.K;
    w.ok = true;
    return w;
}

template <int NB, int ACT, bool BN>
cudaError_t launch_layouts_t(const Plan &p, const DzcGeom &g, const float *delta,
                             const float *output, const float *z, const Coef *coef,
                             const LayoutArgs &la, unsigned blocks, cudaStream_t st) {
    const DzSrc<ACT, BN> src{delta, output, z, coef};
    const bool vec = p.PQ % 4 == 0, xvec = p.HW % 4 == 0;
    auto kern = la.dzc ? (vec ? (xvec ? layouts_kernel<NB, ACT, BN, true, true, true>
                                      : layouts_kernel<NB, ACT, BN, true, true, false>)
                              : (xvec ? layouts_kernel<NB, ACT, BN, true, false, true>
                                      : layouts_kernel<NB, ACT, BN, true, false, false>))
                       : (vec ? (xvec ? layouts_kernel<NB, ACT, BN, false, true, true>
                                      : layouts_kernel<NB, ACT, BN, false, true, false>)
                              : (xvec ? layouts_kernel<NB, ACT, BN, false, false, true>
                                      : layouts_kernel<NB, ACT, BN, false, false, false>));
    (void)g;
    return launch_pdl(kern, dim3(blocks), dim3(256), 0, st, src, la);
}

template <int NB>
cudaError_t launch_layouts_nb(const Plan &p, const DzcGeom &g, const float *delta,
                              const float *output, const float *z, const Coef *coef,
                              const LayoutArgs &la, unsigned blocks, cudaStream_t st) {
    const bool leaky = p.act == CBA_ACT_LEAKY;
    if (p.bn)
        return leaky ? launch_layouts_t<NB, CBA_ACT_LEAKY, true>(p, g, delta, output, z, coef, la,
                                                                  blocks, st)
                     : launch_layouts_t<NB, CBA_ACT_LINEAR, true>(p, g, delta, output, z, coef,
                                                                   la, blocks, st);
    return leaky ? launch_layouts_t<NB, CBA_ACT_LEAKY, false>(p, g, delta, output, z, coef, la,
                                                               blocks, st)
                 : launch_layouts_t<NB, CBA_ACT_LINEAR, false>(p, g, delta, output, z, coef, la,
                                                                blocks, st);
}

}  // namespace

bool wgrad_nb_supported(const Plan &p) {
    const WnGeom w = wn_geom(p);
    if (!w.ok) return false;
    // int32 indices of the layout pass and its 1-D grid
    const DzcGeom g = dzc_geom(p);
    const long long blocks = (long long)w.nc * ((p.PQ + 31) / 32) * ((g.Kp + 7) / 8) +
                             (long long)w.nc * ((p.HW + 31) / 32) * ((p.C + 7) / 8) +
                             (long long)p.N * g.Pp + 4LL * p.num_sms;  // + weight-repack blocks
    if (blocks >= (1LL << 31)) return false;
    if ((long long)p.N * g.Pp >= (1LL << 31)) return false;
    // int32 dW row index of the accumulator apply
    if ((long long)p.K * p.Cg * p.R >= (1LL << 31)) return false;
    return true;
}

size_t wgrad_nb_acc_bytes(const Plan &p) {
    const WnGeom w = wn_geom(p);
    return w.ok ? w.acc_bytes : 0;
}

size_t wgrad_nb_xn_bytes(const Plan &p) {
    const WnGeom w = wn_geom(p);
    return w.ok ? w.xn_bytes : 0;
}

size_t wgrad_nb_dzn_bytes(const Plan &p) {
    const WnGeom w = wn_geom(p);
    return w.ok ? w.dzn_bytes : 0;
}

cudaError_t launch_layouts(const Plan &p, const float *delta, const float *output,
                           const float *z, const float *x, const void *ws, float *dzn,
                           float *dzc, float *xn, const RepackJob *rep, cudaStream_t st,
                           int *launches) {
    const WnGeom w = wn_geom(p);
    if (!w.ok) return cudaErrorNotSupported;
    const DzcGeom g = dzc_geom(p);
    const int nc = (p.N + w.nb - 1) / w.nb;
    LayoutArgs la{};
    la.N = p.N; la.K = p.K; la.Kp = g.Kp; la.PQ = p.PQ; la.Qe = g.Qe; la.Pp = g.Pp;
    la.Qpp = g.Qpp; la.Pe = g.Pe; la.bd_lo = g.bd_lo; la.bq_lo = g.bq_lo;
    la.kchunks = (g.Kp + 7) / 8;
    la.npx_dz = (p.PQ + 31) / 32;
    la.C = p.C; la.HW = p.HW;
    la.xchunks = (p.C + 7) / 8;
    la.npx_x = (p.HW + 31) / 32;
    la.x = x; la.dzn = dzn; la.dzc = dzc; la.xn = xn;
    const long long ndz = (long long)la.npx_dz * nc * la.kchunks;
    const long long nx = (long long)la.npx_x * nc * la.xchunks;
    const long long nborder =
        (dzc && (g.Pp != g.Pe || g.Qpp != g.Qe)) ? (long long)p.N * g.Pp : 0;
    const long long nrep = rep ? std::min<long long>(repack_tiles(*rep), 4LL * p.num_sms) : 0;
    if (ndz + nx + nborder + nrep >= (1LL << 31)) return cudaErrorInvalidValue;
    la.ndz = (int)ndz; la.nx = (int)nx; la.nborder = (int)nborder;
    la.nrep = (int)nrep;
    la.rep = rep ? *rep : RepackJob{};
    const unsigned blocks = (unsigned)(ndz + nx + nborder + nrep);
    const Coef *coef = ws_at<Coef>(ws, p.off_coef);
    cudaError_t e = w.nb == 16
                        ? launch_layouts_nb<16>(p, g, delta, output, z, coef, la, blocks, st)
                        : launch_layouts_nb<32>(p, g, delta, output, z, coef, la, blocks, st);
    if (e != cudaSuccess) return e;
    ++*launches;
    return cudaSuccess;
}

cudaError_t launch_wgrad_nb(const Plan &p, const float *xn, const float *dzn, float *dW, void *ws,
                            float *acc, const RepackJob *rep, cudaStream_t st, int *launches) {
    const WnGeom w = wn_geom(p);
    if (!w.ok) return cudaErrorNotSupported;
    WnArgs a;
    a.acc = acc;
    a.status = ws_at<unsigned>(ws, p.off_status);
    a.P = p.P; a.Q = p.Q; a.R = p.R; a.S = p.S; a.stride = p.stride; a.pad = p.pad;
    a.ctiles = w.ctiles; a.KT = w.KT; a.cb = w.cb; a.cols = w.cols; a.splits = w.splits;
    a.stages = w.stages;
    a.items = w.items; a.Qa = w.Qa; a.NA = w.NA; a.G = w.G; a.NG = w.NG;
    a.mirror = p.S > 1 ? 1 : 0;
    a.rb = w.rb;
    a.swz = w.nb == 16 ? 4u : 2u;  // 64-byte or 128-byte swizzle
    a.a_pos_bytes = w.a_pos_bytes; a.a_slot_bytes = w.a_slot_bytes;
    a.pix_bytes = w.pix_bytes; a.grp_bytes = w.grp_bytes; a.b_off = w.b_off;
    const size_t smem = w.smem;

    alignas(64) CUtensorMap tma, tmb;
    const int swz_bytes = (int)w.rb;  // the row is exactly one swizzle span
    {
        const uint64_t d[4] = {(uint64_t)w.nb, (uint64_t)p.K, (uint64_t)p.Q,
                               (uint64_t)w.nc * p.P};
        const uint32_t b[4] = {(uint32_t)w.nb, 128, (uint32_t)w.Qa, 1};
        if (!tma_encode_f32_swz(&tma, dzn, 4, d, b, swz_bytes)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t d[5] = {(uint64_t)w.nb, (uint64_t)p.C, (uint64_t)p.W, (uint64_t)p.H,
                               (uint64_t)w.nc};
        const uint32_t b[5] = {(uint32_t)w.nb, (uint32_t)w.cb, (uint32_t)w.G, 1, 1};
        if (!tma_encode_f32_swz(&tmb, xn, 5, d, b, swz_bytes)) return cudaErrorInvalidValue;
    }
    auto kern = w.nb == 16 ? wgrad_nb_kernel<16> : wgrad_nb_kernel<32>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(w.grid), dim3(kWnThreads), smem, st, tma, tmb, a);
    if (e != cudaSuccess) return e;
    const int nrows = p.K * p.Cg * p.R;  // dW rows of S elements, < 2^31 (wgrad_nb_supported)
    const unsigned ablocks = (unsigned)std::min<long long>((nrows + 255) / 256, p.num_sms * 32LL);
    const RepackJob job = rep ? *rep : RepackJob{};
    const int nrep = rep ? (int)std::min<long long>(repack_tiles(*rep), 4LL * p.num_sms) : 0;
    e = launch_pdl(wgrad_nb_apply_kernel, dim3(ablocks + nrep), dim3(256), 0, st,
                   (const float *)acc, w.KT, w.cols, w.cb, p.S, p.R, w.ctiles, p.Cg, p.Kg, nrows,
                   dW, (int)ablocks, job, nrep);
    if (e != cudaSuccess) return e;
    *launches += 2;
    return cudaGetLastError();
}

}  // namespace cba
