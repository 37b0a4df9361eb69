// bench_read.cu -- helpers around the method, not part of it:
//   * a read-only streaming probe for the benchmark: every SM runs a few CTAs
//     that stream 16-byte vectors with eight loads in flight per thread, so
//     the only limit is the memory system's read bandwidth;
//   * a self-test of the bounded mbarrier wait every ring of the kernels uses:
//     one CTA waits on a barrier nothing arrives at, gives up after the given
//     limit and records SPEC_DEV_WAIT_TIMEOUT in the workspace status word,
//     exactly as a kernel whose copy never landed would.
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_bench.h"
#include "spec_verify.h"
#include "device_common.cuh"
#include "internal.h"

namespace {

constexpr int THREADS = 512;
constexpr int CTAS_PER_SM = 4;
constexpr int INFLIGHT = 8;

__global__ void __launch_bounds__(THREADS) read_kernel(const uint4 *__restrict__ p, size_t n,
                                                       uint32_t *sink)
{
    uint32_t acc = 0;
    const size_t stride = (size_t)gridDim.x * THREADS;
    size_t i = (size_t)blockIdx.x * THREADS + threadIdx.x;
    for (; i + (INFLIGHT - 1) * stride < n; i += INFLIGHT * stride) {
        uint4 v[INFLIGHT];
#pragma unroll
        for (int j = 0; j < INFLIGHT; ++j)
            v[j] = __ldcs(p + i + j * stride);
#pragma unroll
        for (int j = 0; j < INFLIGHT; ++j)
            acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
    }
    for (; i < n; i += stride) {
        const uint4 v = __ldcs(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ uint32_t wacc[THREADS / 32];
    if ((threadIdx.x & 31) == 0)
        wacc[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t a = 0;
        for (int w = 0; w < THREADS / 32; ++w)
            a ^= wacc[w];
        sink[blockIdx.x] = a;
    }
}

// One thread waits on a fresh mbarrier that no thread arrives at.
__global__ void wait_selftest_kernel(spec_dev::WsHeader *hdr, unsigned long long limit_ns)
{
    __shared__ unsigned long long bar;
    spec_dev::mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!spec_dev::mbar_wait_for(&bar, 0, limit_ns))
        atomicExch(&hdr->status, SPEC_DEV_WAIT_TIMEOUT);
}

int grid_size()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    return sms * CTAS_PER_SM;
}

}  // namespace

extern "C" {

int32_t spec_bench_read_sink_words(void)
{
    return grid_size();
}

int32_t spec_bench_read(const void *buf, size_t bytes, uint32_t *sink, void *stream)
{
    if (!buf || !sink || (reinterpret_cast<uintptr_t>(buf) & 15) || (bytes & 15))
        return SPEC_EINVAL;
    const int grid = grid_size();
    if (grid <= 0)
        return SPEC_ECUDA;
    read_kernel<<<grid, THREADS, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint4 *>(buf), bytes / 16, sink);
    return cudaPeekAtLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int32_t spec_selftest_wait_timeout_noalloc(uint64_t limit_ns, void *stream)
{
    void *ws = nullptr;
    const int rc = spec_internal::noalloc_scratch(&ws);
    if (rc != SPEC_OK)
        return rc;
    return spec_selftest_wait_timeout(ws, limit_ns, stream);
}

int32_t spec_selftest_wait_timeout(void *workspace, uint64_t limit_ns, void *stream)
{
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15) || limit_ns == 0 ||
        limit_ns > 100000000ull)
        return SPEC_EINVAL;
    wait_selftest_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<spec_dev::WsHeader *>(workspace), (unsigned long long)limit_ns);
    return cudaPeekAtLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // extern "C"
