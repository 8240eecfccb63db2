// Instantiations of the split-KV partial kernel for E4M3 pools (query fp32 / bf16, head dim 64 / 128 / 256).
#include "decode_kernels.cuh"

namespace nbx {
NBX_DECODE_FOR_POOL(E4M3)
}  // namespace nbx
