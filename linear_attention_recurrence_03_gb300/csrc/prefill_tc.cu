// prefill_tc.cu -- chunked GDN prefill on the tcgen05 tensor cores (bf16 operands,
// fp32 accumulation in tensor memory, fp32 state).
#include "internal.h"

namespace gdn {

// Status bits set by kernels of this file when a bounded wait runs out.
__device__ uint32_t g_tc_status = 0;

uint32_t prefill_tc_take_status() {
    uint32_t bits = 0;
    if (cudaMemcpyFromSymbol(&bits, g_tc_status, sizeof(bits)) != cudaSuccess) return 0;
    if (bits != 0) {
        const uint32_t zero = 0;
        cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(zero));
    }
    return bits;
}

}  // namespace gdn
