// cba_noalloc.cu -- cba_bn_act_backward_noalloc: the activation-gradient and
// BN-backward pass (bias and scale gradients, optionally the BN-input
// gradient dz) for callers that cannot allocate device memory.
//
// Who needs it: code that may not call cudaMalloc where it runs the backward
// and has no buffer of its own to lend as a workspace.  Examples are a plugin
// called from another runtime's enqueue hook, where that runtime owns all
// device memory and forbids allocation after start-up, and a latency-bounded
// loop.  In both cases cudaMalloc can implicitly synchronise the device and
// its latency is unbounded.
//
// The pass needs a small scratch for its per-block partial sums and
// per-channel coefficients.  Here the scratch is one file-scope __device__
// array, kScratchBytes (1 MiB), placed on every device that loads this
// library and held there until the process exits.  The entry point allocates
// nothing: the only CUDA calls are cudaGetSymbolAddress (once per device), one
// memset and the kernel launches on the stream, and the device/stream queries
// that select the device.
//
// Scratch contents: every call shares the one array per device, and the array
// keeps whatever the last call left in it.  Only the per-channel arrival
// counters of the reduction must start at zero, so every call first clears
// them (a memset of 4 * K bytes on the stream, not an allocation).  Every
// other word is written before it is read in the same call: each reduction
// block writes its partial before the channel's last block reads them all,
// and that block writes the coefficients before the dz kernel reads them.
// Calls that overlap on one device (two streams, or two host threads, with no
// ordering between them) race on the array; the caller must order them, e.g.
// by using one stream.
#include <mutex>

#include "cba_internal.cuh"

namespace cba {

namespace {

constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

inline size_t align256(size_t v) { return (v + 255) / 256 * 256; }

inline bool misaligned16(const void *ptr) {
    return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0;
}

// The device the call runs on: the device that holds `ptr` (the call's data;
// the stream must belong to the same device), made current for this
// library's runtime.  The pointer query is also legal while the stream is
// being captured into a CUDA graph, where asking the stream for its device is
// not; the stream is asked only when there is no pointer.
cudaError_t current_device_for(cudaStream_t stream, const void *ptr, int *dev) {
    cudaError_t e = cudaSuccess;
    int want = -1;
    if (ptr) {
        cudaPointerAttributes a;
        e = cudaPointerGetAttributes(&a, ptr);
        if (e == cudaSuccess) want = a.device;
    } else if (stream) {
        e = cudaStreamGetDevice(stream, &want);
    }
    if (e != cudaSuccess) return e;
    int cur = -1;
    e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    if (want >= 0 && want != cur) {
        e = cudaSetDevice(want);
        cur = want;
    }
    *dev = cur;
    return e;
}

// Set-up, once per device with that device current: the device address of the
// scratch array.  The first call on each device does this, and the address is
// kept for the life of the process: a cudaDeviceReset after that first call
// (which may place the array elsewhere) is not supported.
cudaError_t scratch_for_device(int dev, void **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (!ptr || (reinterpret_cast<uintptr_t>(ptr) & 255u) != 0) return cudaErrorInvalidSymbol;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace cba

extern "C" int cba_bn_act_backward_noalloc(const cba_desc_t *d, const float *output,
                                           const float *z, const float *delta,
                                           const float *gamma, const float *mean,
                                           const float *var, float *db, float *dgamma,
                                           float *dz_out, void *stream) {
    using namespace cba;
    Plan p;
    int rc = make_plan(d, &p);
    if (rc != CBA_OK) return rc;
    if (!delta || !db) return CBA_ERR_ARG;
    if (p.act_in != CBA_ACT_LINEAR && !output) return CBA_ERR_ARG;
    // activations other than linear and leaky need a buffer for delta': dz_out
    if (p.act_pre && !dz_out) return CBA_ERR_UNSUPPORTED;
    if (p.bn && (!z || !gamma || !mean || !var || !dgamma)) return CBA_ERR_ARG;
    const void *ptrs[] = {output, z, delta, gamma, mean, var, db, dgamma, dz_out};
    for (const void *q : ptrs)
        if (misaligned16(q)) return CBA_ERR_ALIGN;
    if (p.K > CBA_NOALLOC_MAX_K) return CBA_ERR_SCRATCH_LIMIT;

    // scratch layout: arrival counters [K] at 0, coefficients [K], then the
    // partials [groups * pieces][K]
    const size_t cnt_bytes = align256(sizeof(unsigned) * (size_t)p.K);
    const size_t coef_bytes = align256(sizeof(Coef) * (size_t)p.K);
    const size_t part_unit = sizeof(float) * 2 * (size_t)p.K;  // one partial per channel
    const long long fit = (long long)((kScratchBytes - cnt_bytes - coef_bytes) / part_unit);
    if (fit < 1) return CBA_ERR_SCRATCH_LIMIT;  // unreachable with K <= CBA_NOALLOC_MAX_K
    plan_reduction(&p, fit);
    p.off_cnt = 0;
    p.off_coef = cnt_bytes;
    p.off_red = cnt_bytes + coef_bytes;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();  // the launches below report only their own errors
    int dev = -1;
    cudaError_t e = current_device_for(st, delta, &dev);
    if (e != cudaSuccess) return report_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return CBA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    e = scratch_for_device(dev, &scratch);
    if (e != cudaSuccess) return report_cuda_error(e);
    int n_launch = 0;
    e = cudaMemsetAsync(scratch, 0, cnt_bytes, st);  // the reduction's arrival counters
    if (e == cudaSuccess && p.act_pre) {
        // delta' into dz_out; the reduction reads it and the dz pass then
        // transforms it in place
        e = launch_gradient_array(p, delta, output, dz_out, st, &n_launch);
        delta = dz_out;
    }
    if (e == cudaSuccess)
        e = launch_reduce(p, delta, output, z, gamma, mean, var, db, dgamma, scratch, st,
                          &n_launch);
    if (e == cudaSuccess && dz_out) e = launch_dz_out(p, delta, output, z, scratch, dz_out, st);
    if (e != cudaSuccess) return report_cuda_error(e);
    return CBA_OK;
}
