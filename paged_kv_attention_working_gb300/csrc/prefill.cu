// placeholder until the tensor-core kernel lands
#include "plan.h"
namespace pie {
cudaError_t launch_prefill(const Geometry&, const PlanView& p, int, const void*, const void*, const void*, void*,
                           float*, float*, float*, int*, cudaStream_t) {
  return p.n_pre ? cudaErrorNotSupported : cudaSuccess;
}
}  // namespace pie
