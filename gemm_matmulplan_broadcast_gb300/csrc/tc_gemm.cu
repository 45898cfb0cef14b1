// GENERAL_TC: tcgen05 tensor-core GEMM for FLOAT16 / BFLOAT16 (placeholder
// until the kernel lands: the plan never selects it while tc_shape_ok is false).
#include "common.cuh"

namespace olc {

bool tc_shape_ok(olc_dtype dt, int64_t N, int64_t K) {
    (void)dt; (void)N; (void)K;
    return false;
}

cudaError_t launch_general_tc(olc_dtype dt, const Problem& p, int sm_count, cudaStream_t s) {
    (void)dt; (void)p; (void)sm_count; (void)s;
    return cudaErrorNotSupported;
}

}  // namespace olc
