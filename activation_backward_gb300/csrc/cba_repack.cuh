// cba_repack.cuh -- the input gradient's weight repack, W[k][c - g*Cg][r][s]
// -> wr[r][s][c][k] (TF32-rounded, k padded to Kw with zeros, zero where input
// channel c is outside output channel k's group), as 32 x 32 tiles that
// threads of another kernel transpose through shared memory: the idle
// epilogue warps of the 1x1 plain GEMM while its MMAs run; extra blocks of
// the batch-innermost layout pass for weights of at most 2 MB; else extra
// blocks of the weight gradient's accumulator-apply launch, which is
// latency-bound.  (Inside the memory-bound reduction pass the tiles delayed
// its streaming by several microseconds.)
#pragma once

#include "cba_internal.cuh"
#include "cba_ptx.cuh"

namespace cba {

inline RepackJob make_repack_job(const Plan &p, const float *W, float *wr) {
    return RepackJob{W, wr, p.K, p.C, p.R, p.S, (p.K + 3) / 4 * 4, p.Cg, p.Kg};
}

inline long long repack_tiles(const RepackJob &j) {
    return (long long)((j.Kw + 31) / 32) * ((j.C * j.R * j.S + 31) / 32);
}

// Tiles rb, rb + nrep, ... of the repack (32 output channels k x 32 flattened
// (c, r, s)): reads coalesced along (c, r, s), writes along k.  Every thread
// of the block (blockDim.x a multiple of 32, at most 1024) takes part.
__device__ __forceinline__ void repack_part(const RepackJob &j, int rb, int nrep) {
    __shared__ float tile[32][33];
    const int CRS = j.C * j.R * j.S, RS = j.R * j.S;
    const int tk = (j.Kw + 31) / 32, tc = (CRS + 31) / 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5, rows = blockDim.x >> 5;
    for (int t = rb; t < tk * tc; t += nrep) {
        const int k0 = (t / tc) * 32, q0 = (t % tc) * 32;
        for (int r = ty; r < 32; r += rows) {
            const int k = k0 + r, q = q0 + tx;
            float v = 0.f;
            if (k < j.K && q < CRS) {
                const int c = q / RS;
                const long long o = w_off(k, c, q - c * RS, j.Cg, j.Kg, RS);
                if (o >= 0) {
                    uint32_t u;
                    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(j.W[o]));
                    v = __uint_as_float(u);
                }
            }
            tile[r][tx] = v;
        }
        __syncthreads();
        for (int r = ty; r < 32; r += rows) {
            const int q = q0 + r, k = k0 + tx;
            if (q < CRS && k < j.Kw) {
                const int c = q / RS, rs = q - c * RS;  // rs = r * S + s
                j.wr[((long long)rs * j.C + c) * j.Kw + k] = tile[tx][r];
            }
        }
        __syncthreads();
    }
}

// The same, run by a group of `nthreads` threads (a multiple of 32; `t` is a
// thread's index in the group) that synchronise on named barrier `bar`, with
// the 32 x 33 tile in `tile` (shared memory): for kernels whose other warps
// are busy with other roles.
__device__ __forceinline__ void repack_part_group(const RepackJob &j, int rb, int nrep, float *tile,
                                                  int t, int nthreads, int bar) {
    const int CRS = j.C * j.R * j.S, RS = j.R * j.S;
    const int tk = (j.Kw + 31) / 32, tc = (CRS + 31) / 32;
    const int tx = t & 31, ty = t >> 5, rows = nthreads >> 5;
    for (int u = rb; u < tk * tc; u += nrep) {
        const int k0 = (u / tc) * 32, q0 = (u % tc) * 32;
        for (int r = ty; r < 32; r += rows) {
            const int k = k0 + r, q = q0 + tx;
            float v = 0.f;
            if (k < j.K && q < CRS) {
                const int c = q / RS;
                const long long o = w_off(k, c, q - c * RS, j.Cg, j.Kg, RS);
                if (o >= 0) {
                    uint32_t w;
                    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(w) : "f"(j.W[o]));
                    v = __uint_as_float(w);
                }
            }
            tile[r * 33 + tx] = v;
        }
        ptx::named_bar_sync(bar, nthreads);
        for (int r = ty; r < 32; r += rows) {
            const int q = q0 + r, k = k0 + tx;
            if (q < CRS && k < j.Kw) {
                const int c = q / RS, rs = q - c * RS;
                j.wr[((long long)rs * j.C + c) * j.Kw + k] = tile[tx * 33 + r];
            }
        }
        ptx::named_bar_sync(bar, nthreads);
    }
}

}  // namespace cba
