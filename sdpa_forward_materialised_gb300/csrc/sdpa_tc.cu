// sdpa_tc.cu -- tensor-core (tcgen05) kernels; placeholder until they land.
#include "internal.h"

namespace sdpa {

__device__ unsigned int g_status_word;

bool tc_supports(const Problem&, bool, const char** why) {
    *why = "tensor-core kernels are not built yet";
    return false;
}

cudaError_t launch_tc(const Problem&, bool, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t status_read_and_clear(cudaStream_t stream, unsigned int* value) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_status_word, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace sdpa
