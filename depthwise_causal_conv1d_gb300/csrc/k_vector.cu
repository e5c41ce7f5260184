// Vector kernels without the duplicate check: the update, unchecked and range-checked.
// The family itself is in ccu_vector.cuh.
//
// Update definition: cuDNN page "Causal Conv1d Decode Update", introduction (update
// block).
#include "ccu_vector.cuh"

namespace ccu {

cudaError_t launch_vector_checked(const UpdateParams &p, int act, cudaStream_t stream);

cudaError_t launch_vector(const UpdateParams &p, int act, cudaStream_t stream) {
  if (p.owner != nullptr) return launch_vector_checked(p, act, stream);
  return launch_vector_impl<false>(p, act, stream);
}

}  // namespace ccu
