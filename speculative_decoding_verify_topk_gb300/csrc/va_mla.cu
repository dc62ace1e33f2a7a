// Absorbed-MLA prefix kernel (tcgen05 / TMEM): not built yet; planning never
// selects the MLA path while mla_available() is false.
#include "va_common.cuh"

namespace va {

bool mla_available() { return false; }

cudaError_t launch_prefix_mla(const Args&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace va
