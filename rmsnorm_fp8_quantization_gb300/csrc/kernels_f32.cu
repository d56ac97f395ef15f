// Kernel instantiations for f32 inputs.
#include "launch.cuh"

namespace gbn {

const KernelTable& kernels_f32() {
  using L = Launch<float>;
  static const KernelTable table = {&L::fwd_occupancy, &L::fwd_launch, &L::stripe_launch,
                                    &L::bwd_occupancy, &L::bwd_launch};
  return table;
}

}  // namespace gbn
