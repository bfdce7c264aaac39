// Launchers of the tensor-memory GEMMs that are not built yet: they report
// "not supported" so the C ABI returns an error instead of launching.
#include "wq_internal.h"

namespace wq {
cudaError_t launch_wo_gemm(const WoArgs& a, int bits, cudaStream_t s) { return launch_wo_skinny(a, bits, s); }
}  // namespace wq
