// Prefill W4A16 GEMM (M > 8) on the 5th-generation tensor cores.
// Placeholder until the tcgen05 kernel lands: reports "not supported".
#include "internal.h"

namespace w4 {

cudaError_t run_prefill(float *, const uint16_t *, const uint32_t *, const uint16_t *, int, int,
                        int, int, cudaStream_t)
{
    return cudaErrorNotSupported;
}

} // namespace w4
