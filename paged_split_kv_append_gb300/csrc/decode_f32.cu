// Instantiations of the split-KV partial kernel for F32 pools (query fp32 / bf16, head dim 64 / 128 / 256).
#include "decode_kernels.cuh"

namespace nbx {
NBX_DECODE_FOR_POOL(F32)
}  // namespace nbx
