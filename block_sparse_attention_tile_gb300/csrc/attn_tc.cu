// tcgen05 tensor-core attention kernels (filled in below the stubs).
#include "common.cuh"

namespace bsa {

bsa_status tc_block_attention(const void*, const void*, const void*, int, int, const int32_t*,
                              const int32_t*, int, int, const int32_t*, const int32_t*, int,
                              const void*, const void*, float, void*, float*, cudaStream_t,
                              bool* handled) {
    *handled = false;
    return BSA_OK;
}

bsa_status kvouter_tc(const void*, const void*, const void*, int, int, int, int, int,
                                 const int32_t*, const int32_t*, const int32_t*, const int32_t*,
                                 const int32_t*, int, int, int, int, int, float, void*, float*,
                                 cudaStream_t, bool* handled) {
    *handled = false;
    return BSA_OK;
}

}  // namespace bsa
