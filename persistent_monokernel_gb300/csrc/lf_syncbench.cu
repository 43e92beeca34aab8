// lf_syncbench.cu -- microbenchmark of the two grid synchronisation schemes
// the decode kernel can use between dependent stages: a one-hop readiness
// flag (a gpu-scope release by one CTA, an acquire poll by another) and an
// arrival-counter grid barrier.  The pages measure both on MI300X
// (shivam2003.com, "KOG LaneFormer-2B & the monokernel", section
// "Cross-GPU synchronization without atomics"); this measures them on the
// GPU the library runs on.
#include <cuda_runtime.h>

#include "../../include/lf.h"
#include "lf_internal.cuh"
#include "lf_ptx.cuh"

namespace lfk {
namespace {

constexpr long long kProbeTimeoutNs = 1000000000LL;

// Spin until *ctr >= target or the timeout; false on timeout (the flag at
// err is then set and every CTA stops at its next wait).
__device__ bool probe_wait(const unsigned *ctr, unsigned target, unsigned *err)
{
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned it = 0;; ++it) {
        if ((int)(ld_acquire(ctr) - target) >= 0) return true;
        if ((it & 63u) == 63u) {
            if (ld_relaxed(err)) return false;
            if ((long long)(globaltimer_ns() - t0) > kProbeTimeoutNs) {
                atomicExch(err, 1u);
                return false;
            }
        }
    }
}

// mode 0: a token travels round the ring of CTAs `iters` times; each hop is a
// release add on the next CTA's flag and an acquire poll by that CTA.
// mode 1: `iters` grid barriers on one arrival counter.
// One thread per CTA works; out[0] = elapsed ns seen by CTA 0, out[1] = error.
__global__ void lf_sync_probe(int mode, int iters, unsigned *flags, unsigned *err, unsigned long long *out)
{
    if (threadIdx.x != 0) return;
    const unsigned P = gridDim.x, b = blockIdx.x;
    const unsigned long long t0 = globaltimer_ns();
    if (mode == 0) {
        unsigned *mine = flags + (size_t)b * CNT_STRIDE;
        unsigned *next = flags + (size_t)((b + 1) % P) * CNT_STRIDE;
        for (int r = 0; r < iters; ++r) {
            if (b != 0 || r > 0) {
                if (!probe_wait(mine, (unsigned)r + (b == 0 ? 0u : 1u), err)) return;
            }
            red_release_add(next, 1u);
        }
        if (b == 0 && !probe_wait(mine, (unsigned)iters, err)) return;
    } else {
        for (int r = 0; r < iters; ++r) {
            red_release_add(flags, 1u);
            if (!probe_wait(flags, (unsigned)(r + 1) * P, err)) return;
        }
    }
    if (b == 0) out[0] = globaltimer_ns() - t0;
}

}  // namespace
}  // namespace lfk

extern "C" LF_API lf_status lf_sync_latency(int32_t mode, int32_t n_ctas, int32_t iters, double *ns_out)
{
    if (!ns_out || (mode != 0 && mode != 1) || n_ctas < 2 || iters < 1) return LF_ERR_INVALID_ARG;
    int dev = 0, sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return LF_ERR_CUDA;
    if (n_ctas > sm) return LF_ERR_NOT_RESIDENT;
    const size_t words = (size_t)n_ctas * lfk::CNT_STRIDE + 64;
    unsigned *buf = nullptr;
    if (cudaMalloc(&buf, words * sizeof(unsigned)) != cudaSuccess) return LF_ERR_OUT_OF_MEMORY;
    unsigned *flags = buf, *err = buf + (size_t)n_ctas * lfk::CNT_STRIDE;
    unsigned long long *out = reinterpret_cast<unsigned long long *>(err + 32);
    cudaError_t e = cudaMemset(buf, 0, words * sizeof(unsigned));
    int m = mode, it = iters;
    void *args[] = {&m, &it, &flags, &err, &out};
    if (e == cudaSuccess)
        e = cudaLaunchCooperativeKernel((const void *)lfk::lf_sync_probe, dim3(n_ctas), dim3(32), args, 0, nullptr);
    unsigned long long res[2] = {0, 0};
    unsigned errv = 0;
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(res, out, sizeof(res), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&errv, err, sizeof(errv), cudaMemcpyDeviceToHost);
    cudaFree(buf);
    if (e != cudaSuccess) return LF_ERR_CUDA;
    if (errv) return LF_ERR_TIMEOUT;
    const double events = mode == 0 ? (double)iters * n_ctas : (double)iters;
    *ns_out = (double)res[0] / events;
    return LF_OK;
}
