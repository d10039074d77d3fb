// va_tc.cu -- tcgen05 tensor-core split-K partial kernel (K1, TC path).
#include "va_common.cuh"

namespace va {

bool tc_supported(int, int, int) { return false; }
int tc_auto_nsplit(int, int, int, int) { return 1; }
cudaError_t init_partial_tc() { return cudaSuccess; }
cudaError_t launch_partial_tc(const Params&, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace va
