// Device copies of host-resident inputs for sdm_write_read_host: one kernel reads every input
// array straight from its mapped page-locked host pages (16-byte loads, four in flight per
// thread) and writes the workspace's device copy. For the several 1-8 MB arrays of a call this
// moves the bytes faster than one copy-engine transfer per array.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

__global__ void __launch_bounds__(512) k_host_copy(HostCopyTable t) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (int a = 0; a < t.n; ++a) {
        const uint4 *s = t.src[a];
        uint4 *d = t.dst[a];
        const long long n = t.n16[a];
        for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += 4 * stride) {
            uint4 x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const long long j = i + k * stride;
                if (j < n) x[k] = s[j];
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const long long j = i + k * stride;
                if (j < n) d[j] = x[k];
            }
        }
    }
}

}  // namespace

cudaError_t launch_host_copy(const HostCopyTable &t, cudaStream_t st) {
    k_host_copy<<<4 * kRefSms, 512, 0, st>>>(t);
    return cudaGetLastError();
}

}  // namespace sdm
