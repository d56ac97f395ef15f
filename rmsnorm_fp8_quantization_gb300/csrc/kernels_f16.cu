// Kernel instantiations for f16 inputs.
#include "launch.cuh"

namespace gbn {

const KernelTable& kernels_f16() {
  using L = Launch<__half>;
  static const KernelTable table = {&L::fwd_occupancy, &L::fwd_launch, &L::stripe_launch,
                                    &L::bwd_occupancy, &L::bwd_launch};
  return table;
}

}  // namespace gbn
