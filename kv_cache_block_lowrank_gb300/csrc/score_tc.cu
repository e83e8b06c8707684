// score_tc.cu -- block scores for prefill chunks on the tcgen05 tensor cores (not built yet).
#include "ptx.cuh"

namespace hss {

bool score_tc_supported(const ScoreArgs& a) {
    (void)a;
    return false;
}

hss_status launch_score_tc(const ScoreArgs& a, cudaStream_t stream) {
    (void)a;
    (void)stream;
    return HSS_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace hss
