// Tensor-core (tcgen05 / TMEM / TMA) block attention for bf16 -- placeholder
// until the kernel lands: covers no sizes, so AUTO selects the SIMT kernel.
#include "dflash_device.cuh"

namespace dflash {

bool tc_supports(const AttnParams&) { return false; }

cudaError_t launch_tc_attn(const AttnParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace dflash
