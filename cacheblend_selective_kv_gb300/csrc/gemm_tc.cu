// Tensor-core (tcgen05) GEMM path: placeholder until the kernel lands.
#include "cb_common.cuh"

namespace cb {
bool tc_init(Model& m, std::string& err) { (void)m; err = "tensor-core path not built"; return false; }
void tc_destroy(Model& m) { (void)m; }
cudaError_t launch_gemm_tc(const Model&, int, int, int, int, const GemmW&, int, const EpiParams&, cudaStream_t, int*) {
    return cudaErrorNotSupported;
}
}  // namespace cb
