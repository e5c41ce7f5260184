// Vector kernels with the duplicate check of ccu_conv1d_update_checked_ex (each warp claims
// its row's slot once, after issuing the row's loads; see drop_if_duplicate_warp). A
// translation unit of their own keeps that code out of the unchecked kernels and compiles
// in parallel with them. The family itself is in ccu_vector.cuh.
//
// Duplicate check: cuDNN page "Causal Conv1d Decode Update", "Current native
// implementation", last paragraph (repeated non-padding slots), reported instead of trapped.
#include "ccu_vector.cuh"

namespace ccu {

cudaError_t launch_vector_checked(const UpdateParams &p, int act, cudaStream_t stream) {
  return launch_vector_impl<true>(p, act, stream);
}

}  // namespace ccu
