// Multi-token update, vector kernels for widths 2 and 3 (the family is in ccu_multi.cuh; a
// translation unit of their own compiles in parallel with the width-4 ones).
//
// Widths other than four: cuDNN page "Causal Conv1d Decode Update", "Current native
// implementation" (other semantically valid widths).
#include "ccu_multi.cuh"

namespace ccu {

namespace {

// Widths 2 and 3 with L = W - 1..4 (the short states they are used with; longer states run
// on the scalar kernel).
template <int ACT>
cudaError_t launch_narrow_A(const UpdateParams &p, const MultiParams &m, dim3 grid, dim3 block,
                            cudaStream_t stream) {
  switch (p.W * 16 + p.L) {
    case 3 * 16 + 2: return launch_vec_L<2, 3, ACT>(p, m, grid, block, stream);
    case 3 * 16 + 3: return launch_vec_L<3, 3, ACT>(p, m, grid, block, stream);
    case 3 * 16 + 4: return launch_vec_L<4, 3, ACT>(p, m, grid, block, stream);
    case 2 * 16 + 1: return launch_vec_L<1, 2, ACT>(p, m, grid, block, stream);
    case 2 * 16 + 2: return launch_vec_L<2, 2, ACT>(p, m, grid, block, stream);
    case 2 * 16 + 3: return launch_vec_L<3, 2, ACT>(p, m, grid, block, stream);
    case 2 * 16 + 4: return launch_vec_L<4, 2, ACT>(p, m, grid, block, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_multi_vector_narrow(const UpdateParams &p, const MultiParams &m, int act, dim3 grid,
                                       dim3 block, cudaStream_t stream) {
  return act == 1 ? launch_narrow_A<1>(p, m, grid, block, stream) : launch_narrow_A<0>(p, m, grid, block, stream);
}

}  // namespace ccu
