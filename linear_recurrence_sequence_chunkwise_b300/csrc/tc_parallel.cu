// tc_parallel.cu -- tensor-core (tcgen05) kernel of the parallel form (placeholder until written).
#include "common.cuh"

namespace ret {
namespace { __device__ unsigned g_err_parallel; }
cudaError_t launch_parallel_tc(const void*, const void*, const void*, void*, int, int, int, int,
                               int, int, const HeadConsts&, unsigned, cudaStream_t) {
    return cudaErrorNotSupported;
}
unsigned read_clear_error_tc_parallel(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_parallel, sizeof(h), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return 0;
    cudaMemcpyToSymbolAsync(g_err_parallel, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}
}  // namespace ret
