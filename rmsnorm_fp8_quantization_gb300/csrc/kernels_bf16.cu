// Kernel instantiations for bf16 inputs.
#include "launch.cuh"

namespace gbn {

const KernelTable& kernels_bf16() {
  using L = Launch<__nv_bfloat16>;
  static const KernelTable table = {&L::fwd_occupancy, &L::fwd_launch, &L::stripe_launch,
                                    &L::bwd_occupancy, &L::bwd_launch};
  return table;
}

}  // namespace gbn
