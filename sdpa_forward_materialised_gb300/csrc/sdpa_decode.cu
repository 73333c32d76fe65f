// sdpa_decode.cu -- split-KV decode kernel; placeholder until it lands.
#include "internal.h"

namespace sdpa {

bool decode_supports(const Problem&, const char** why) {
    *why = "decode kernel is not built yet";
    return false;
}

cudaError_t launch_decode(const Problem&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace sdpa
