// Grouped GEMM over routed experts (tcgen05).  Not built yet: the entry point
// reports Q4_ERR_UNSUPPORTED.
#include "q4_internal.h"

using namespace q4i;

extern "C" q4_status q4_moe_gemm(const uint32_t* Wq, const uint16_t* scales, const uint16_t* biases,
                                 const uint16_t* X, const int32_t* expert_ids, const int32_t* offsets, void* Y,
                                 const q4_moe_desc* desc, q4_stream_t stream) {
    (void)Wq; (void)scales; (void)biases; (void)X; (void)expert_ids; (void)offsets; (void)Y; (void)desc;
    (void)stream;
    clear_error();
    return fail(Q4_ERR_UNSUPPORTED, "q4_moe_gemm is not built in this version");
}
