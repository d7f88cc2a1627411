// cba_tc.cu -- tensor-core (tcgen05, TF32) convolution gradients.
#include "cba_internal.cuh"
#include "cba_ptx.cuh"

namespace cba {

namespace {

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

}  // namespace

bool tc_supported(const Plan &p) {
    (void)p;
    return false;
}

cudaError_t launch_wgrad_tc(const Plan &p, const float *x, const float *delta,
                            const float *output, const float *z, float *dW, void *ws,
                            cudaStream_t st, int *launches) {
    (void)launches;
    (void)p; (void)x; (void)delta; (void)output; (void)z; (void)dW; (void)ws; (void)st;
    return cudaErrorNotSupported;
}

cudaError_t launch_dgrad_tc(const Plan &p, const float *Wt, const float *delta,
                            const float *output, const float *z, const float *residual,
                            float *prev, void *ws, cudaStream_t st, int *launches) {
    (void)launches;
    (void)p; (void)Wt; (void)delta; (void)output; (void)z; (void)residual; (void)prev; (void)ws;
    (void)st;
    return cudaErrorNotSupported;
}

cudaError_t launch_selftest_wait(unsigned timeout_us, void *ws, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(timeout_us, ws_at<unsigned>(ws, 0));
    return cudaGetLastError();
}

}  // namespace cba
