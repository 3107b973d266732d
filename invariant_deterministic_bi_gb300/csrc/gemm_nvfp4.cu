// gemm_nvfp4.cu -- placeholder until the block-scaled kernel lands.
#include "bi_internal.h"

namespace bi {

void plan_gemm_nvfp4(int64_t M, int64_t N, int64_t K, int sms, bi_plan_t *pl) {
    pl->op = BI_OP_GEMM_NVFP4;
    (void)M; (void)N; (void)K; (void)sms;
}

bi_status launch_gemm_nvfp4(const uint8_t *, const uint8_t *, const uint8_t *, const uint8_t *, float, void *,
                            int64_t, int64_t, int64_t, cudaStream_t) {
    return BI_ERR_UNSUPPORTED;
}

}  // namespace bi
