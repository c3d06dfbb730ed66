// tc_chunkwise.cu -- tensor-core (tcgen05) kernel of the chunkwise form (placeholder until written).
#include "common.cuh"

namespace ret {
namespace { __device__ unsigned g_err_chunkwise; }
cudaError_t launch_chunkwise_tc(const void*, const void*, const void*, void*, int, int, int, int,
                                int, int, int, const HeadConsts&, const float*, float*,
                                cudaStream_t) {
    return cudaErrorNotSupported;
}
unsigned read_clear_error_tc_chunkwise(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_chunkwise, sizeof(h), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return 0;
    cudaMemcpyToSymbolAsync(g_err_chunkwise, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}
}  // namespace ret
