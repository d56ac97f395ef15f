// Kernel instantiations for f32 inputs.
#include "launch.cuh"

namespace gbn {

const KernelTable& kernels_f32() {
  using L = Launch<float>;
  static const KernelTable table = {
      &L::fwd_generic_occupancy, &L::fwd_generic_launch, &L::stripe_max_clusters, &L::stripe_launch,
      &L::colwise_occupancy,     &L::colwise_launch,
      &L::bwd_generic_occupancy, &L::bwd_generic_launch, &L::fwd_ring_occupancy,
      &L::fwd_ring_launch,       &L::bwd_ring_occupancy, &L::bwd_ring_launch,
      &L::fwd_cluster_max_clusters, &L::fwd_cluster_launch, &L::bwd_cluster_max_clusters,
      &L::bwd_cluster_launch,       &L::probe_copy_timeout,     &L::read_device_error};
  return table;
}

}  // namespace gbn
