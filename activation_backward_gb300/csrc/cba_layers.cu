// cba_layers.cu -- the backward of three data-movement layers that sit next to
// the convolution in the networks of the pages:
//   * the YOLO layer ("YOLOv3反向传播原理 之 全流程源码分析" §2): its delta is
//     added onto the previous layer's delta (one axpy of factor 1);
//   * the route layer (same page, §6): its output lays its inputs side by side
//     per image, so its delta is split back and added onto each input's delta;
//   * max pooling ("LeNet反向过程", 第五层 Pooling): each top gradient goes to the
//     bottom element the forward recorded in the mask.  The page scatters top
//     by top; here each bottom element gathers, in ascending top position (the
//     page's loop order), the top gradients whose mask points at it.  The gather
//     writes every bottom element once (no atomics, deterministic) and never
//     indexes memory with a mask value.
// All three are HBM-bound: 16-byte accesses where the sizes allow, grids of a
// few blocks per SM with grid-stride loops.
#include <algorithm>
#include <cstdint>

#include "cba_internal.cuh"

namespace cba {

namespace {

constexpr int kLThreads = 256;

inline unsigned grid_for(long long work, int per_sm = 8) {
    const long long blocks = (work + kLThreads - 1) / kLThreads;
    return (unsigned)std::max<long long>(1, std::min<long long>(blocks, (long long)kNumSMs * per_sm));
}

__global__ void __launch_bounds__(kLThreads)
    yolo_backward_kernel(const float *__restrict__ l_delta, float *__restrict__ net_delta,
                         long long n, int vec) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long t0 = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    long long done = 0;
    if (vec) {
        const long long n4 = n / 4;
        const float4 *l4 = reinterpret_cast<const float4 *>(l_delta);
        float4 *d4 = reinterpret_cast<float4 *>(net_delta);
        for (long long i = t0; i < n4; i += stride) {
            const float4 a = __ldg(l4 + i);
            float4 b = d4[i];
            b.x += a.x; b.y += a.y; b.z += a.z; b.w += a.w;
            d4[i] = b;
        }
        done = 4 * n4;
    }
    for (long long i = done + t0; i < n; i += stride) net_delta[i] += __ldg(l_delta + i);
}

struct RouteArgs {
    const float *route;              // [batch][outputs]
    float *dst[CBA_ROUTE_MAX_INPUTS];  // input i's delta, [batch][size[i]]
    long long size[CBA_ROUTE_MAX_INPUTS];
    long long off[CBA_ROUTE_MAX_INPUTS];  // offset of input i within an image's row
    int n;
    long long outputs, total;        // total = batch * outputs
};

// One element (or one group of 4, when every size and offset is a multiple of
// 4) of the route delta per thread: image j = e / outputs, position t = e %
// outputs falls in input i with off[i] <= t < off[i] + size[i].
__global__ void __launch_bounds__(kLThreads) route_backward_kernel(const RouteArgs a, int vec) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    const int w = vec ? 4 : 1;
    const long long units = a.total / w;
    for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < units; u += stride) {
        const long long e = u * w;
        const long long j = e / a.outputs, t = e - j * a.outputs;
        int i = 0;
        while (i + 1 < a.n && t >= a.off[i + 1]) ++i;
        float *d = a.dst[i] + j * a.size[i] + (t - a.off[i]);
        if (vec) {
            const float4 r = __ldg(reinterpret_cast<const float4 *>(a.route + e));
            float4 v = *reinterpret_cast<float4 *>(d);
            v.x += r.x; v.y += r.y; v.z += r.z; v.w += r.w;
            *reinterpret_cast<float4 *>(d) = v;
        } else {
            *d += __ldg(a.route + e);
        }
    }
}

// Division of n < 2^31 by a divisor fixed for a launch, with one multiply-high,
// an add and a shift: Granlund and Montgomery, "Division by invariant integers
// using multiplication" (PLDI 1994), the round-up multiplier with
// l = ceil(log2 d):  m = floor(2^32 (2^l - d) / d) + 1,  q = (mulhi(n, m) + n) >> l.
// n < 2^31 keeps mulhi(n, m) + n below 2^32.
struct FastDiv {
    uint32_t d, mul, shift;
};

inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return FastDiv{d, (uint32_t)m, l};
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return (__umulhi(n, f.mul) + n) >> f.shift;
}

struct PoolArgs {
    const float *top;  // [N*C][PH][PW]
    const int *mask;   // [N*C][PH][PW]: h * W + w of the window's recorded maximum
    float *bottom;     // [N*C][H][W]
    int H, W, PH, PW, kh, kw, sh, sw, ph, pw;
    long long total;   // N * C * H * W
    FastDiv seg, fw, fsh, fsw;  // by the thread units per plane, W, stride_h, stride_w
};

// Top rows whose window covers bottom row h: the window of top row p is rows
// p*s - pad .. p*s - pad + k - 1, so p*s <= h + pad and p*s >= h + pad - k + 1.
__device__ __forceinline__ void covering(int h, int k, int s, int pad, int P, int &lo, int &hi) {
    const int a = h + pad - k + 1;
    lo = a > 0 ? (a + s - 1) / s : 0;
    hi = min(P - 1, (h + pad) / s);
}
__device__ __forceinline__ void covering(int h, int k, const FastDiv &s, int pad, int P, int &lo,
                                         int &hi) {
    const int a = h + pad - k + 1;
    lo = a > 0 ? (int)fdiv((uint32_t)(a + (int)s.d - 1), s) : 0;
    hi = min(P - 1, (int)fdiv((uint32_t)(h + pad), s));
}

// EPT consecutive bottom elements of one row per thread (4 when W is a
// multiple of 4: one 16-byte store).  CH x CW bounds the windows that cover an
// element (ceil(kernel / stride) per axis): with them fixed, every mask and top
// load of the thread's elements is issued before the first compare, so a
// thread keeps many loads in flight; CH = CW = 0 walks the windows at run time.
// Either way an element sums its top gradients in ascending (ph, pw).
// SMALL: fewer than 2^31 thread units and 2^31 elements per plane, so the
// index arithmetic runs on 32-bit values with FastDiv; else 64-bit division.
template <int CH, int CW, int EPT, bool SMALL>
__global__ void __launch_bounds__(kLThreads) maxpool_backward_kernel(const PoolArgs a) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    const int hw_n = a.H * a.W, phw = a.PH * a.PW;
    const long long units = a.total / EPT;
    for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < units; u += stride) {
        long long plane;
        int hw0, h, w0, p0, p1;
        if constexpr (SMALL) {
            const uint32_t pl = fdiv((uint32_t)u, a.seg);
            hw0 = ((int)u - (int)(pl * a.seg.d)) * EPT;
            h = (int)fdiv((uint32_t)hw0, a.fw);
            plane = pl;
            covering(h, a.kh, a.fsh, a.ph, a.PH, p0, p1);
        } else {
            const long long b0 = u * EPT;
            plane = b0 / hw_n;
            hw0 = (int)(b0 - plane * hw_n);
            h = hw0 / a.W;
            covering(h, a.kh, a.sh, a.ph, a.PH, p0, p1);
        }
        w0 = hw0 - h * a.W;
        const long long b0 = plane * hw_n + hw0;
        const int *mk = a.mask + plane * phw;
        const float *tp = a.top + plane * phw;
        float acc[EPT];
        if constexpr (CH > 0) {
            int m[EPT][CH][CW];
            float t[EPT][CH][CW];
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                int q0, q1;
                if constexpr (SMALL) covering(w0 + e, a.kw, a.fsw, a.pw, a.PW, q0, q1);
                else covering(w0 + e, a.kw, a.sw, a.pw, a.PW, q0, q1);
#pragma unroll
                for (int i = 0; i < CH; ++i)
#pragma unroll
                    for (int j = 0; j < CW; ++j) {
                        const bool ok = p0 + i <= p1 && q0 + j <= q1;
                        const int idx = ok ? (p0 + i) * a.PW + q0 + j : 0;
                        m[e][i][j] = ok ? __ldg(mk + idx) : -1;
                        t[e][i][j] = ok ? __ldg(tp + idx) : 0.f;
                    }
            }
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                acc[e] = 0.f;
#pragma unroll
                for (int i = 0; i < CH; ++i)
#pragma unroll
                    for (int j = 0; j < CW; ++j)
                        if (m[e][i][j] == hw0 + e) acc[e] += t[e][i][j];
            }
        } else {
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                int q0, q1;
                covering(w0 + e, a.kw, a.sw, a.pw, a.PW, q0, q1);
                acc[e] = 0.f;
                for (int p = p0; p <= p1; ++p)
                    for (int q = q0; q <= q1; ++q) {
                        const int idx = p * a.PW + q;
                        const int mv = __ldg(mk + idx);
                        const float tv = __ldg(tp + idx);
                        if (mv == hw0 + e) acc[e] += tv;
                    }
            }
        }
        if constexpr (EPT == 4)
            *reinterpret_cast<float4 *>(a.bottom + b0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        else
            a.bottom[b0] = acc[0];
    }
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int pooled_size(int in, int k, int stride, int pad) {
    const long long span = (long long)in + 2LL * pad - k;
    if (in <= 0 || k <= 0 || stride <= 0 || pad < 0 || span < 0) return -1;
    long long out = (span + stride - 1) / stride + 1;
    if (pad > 0 && (out - 1) * stride >= (long long)in + pad) --out;
    return out > 0 && out < (1LL << 31) ? (int)out : -1;
}

cudaError_t launch_yolo_backward(const float *l_delta, float *net_delta, long long n,
                                 cudaStream_t st) {
    const int vec = aligned16(l_delta) && aligned16(net_delta);
    yolo_backward_kernel<<<grid_for(vec ? n / 4 + 1 : n), kLThreads, 0, st>>>(l_delta, net_delta,
                                                                             n, vec);
    return cudaGetLastError();
}

cudaError_t launch_route_backward(const float *route, int batch, int n, const long long *sizes,
                                  float *const *deltas, cudaStream_t st) {
    RouteArgs a{};
    a.route = route;
    a.n = n;
    long long off = 0;
    bool vec = aligned16(route);
    for (int i = 0; i < n; ++i) {
        a.dst[i] = deltas[i];
        a.size[i] = sizes[i];
        a.off[i] = off;
        off += sizes[i];
        vec = vec && sizes[i] % 4 == 0 && aligned16(deltas[i]);
    }
    a.outputs = off;
    a.total = off * batch;
    route_backward_kernel<<<grid_for(vec ? a.total / 4 : a.total), kLThreads, 0, st>>>(a, vec ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_maxpool_backward(const cba_pool_desc_t &d, int PH, int PW, const float *top,
                                    const int *mask, float *bottom, cudaStream_t st) {
    PoolArgs a;
    a.top = top; a.mask = mask; a.bottom = bottom;
    a.H = d.H; a.W = d.W; a.PH = PH; a.PW = PW;
    a.kh = d.kernel_h; a.kw = d.kernel_w; a.sh = d.stride_h; a.sw = d.stride_w;
    a.ph = d.pad_h; a.pw = d.pad_w;
    a.total = (long long)d.N * d.C * d.H * d.W;
    const int ch = (d.kernel_h + d.stride_h - 1) / d.stride_h;
    const int cw = (d.kernel_w + d.stride_w - 1) / d.stride_w;
    const bool v4 = d.W % 4 == 0 && aligned16(bottom);
    const long long units = v4 ? a.total / 4 : a.total;
    const bool small = units < (1LL << 31);
    a.seg = make_fastdiv((uint32_t)(v4 ? d.H * d.W / 4 : d.H * d.W));
    a.fw = make_fastdiv((uint32_t)d.W);
    a.fsh = make_fastdiv((uint32_t)d.stride_h);
    a.fsw = make_fastdiv((uint32_t)d.stride_w);
    const unsigned grid = grid_for(units);
#define CBA_POOL(CH, CW)                                                                      \
    do {                                                                                      \
        if (v4 && small)                                                                      \
            maxpool_backward_kernel<CH, CW, 4, true><<<grid, kLThreads, 0, st>>>(a);          \
        else if (v4)                                                                          \
            maxpool_backward_kernel<CH, CW, 4, false><<<grid, kLThreads, 0, st>>>(a);         \
        else if (small)                                                                       \
            maxpool_backward_kernel<CH, CW, 1, true><<<grid, kLThreads, 0, st>>>(a);          \
        else                                                                                  \
            maxpool_backward_kernel<CH, CW, 1, false><<<grid, kLThreads, 0, st>>>(a);         \
    } while (0)
    if (ch == 1 && cw == 1) CBA_POOL(1, 1);
    else if (ch == 2 && cw == 2) CBA_POOL(2, 2);
    else if (ch <= 3 && cw <= 3) CBA_POOL(3, 3);
    else CBA_POOL(0, 0);
#undef CBA_POOL
    return cudaGetLastError();
}

}  // namespace cba
