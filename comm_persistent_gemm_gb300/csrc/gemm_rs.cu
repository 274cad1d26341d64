// gemm_rs.cu -- GEMM + reduce-scatter as one self-scheduling persistent launch.
#include "engine.cuh"
#include "launch.h"

namespace kosmos {

kosmos_status launch_rs_bf16(const RsLaunch &L, cudaStream_t stream) {
    (void)L; (void)stream;
    return KOSMOS_ERR_UNSUPPORTED;
}

}  // namespace kosmos
