// Kernel instantiations for tile N = 256 on 2 x 2 clusters: A shared along cluster rows, B
// along cluster columns, both by multicast
#include "launch.cuh"

namespace clcg {
cudaError_t launch_n256_c2x2(int sched, const Params& p, int grid_ctas, cudaStream_t stream) {
  return launch_shape<256, 4, false, 2>(sched, p, grid_ctas, stream);
}
cudaError_t max_clusters_n256_c2x2(int* out) { return max_clusters_shape<256, 4, false, 2>(out); }
cudaError_t warm_n256_c2x2(const Params& p0, cudaStream_t s) { return warm_shape<256, 4, false, 2>(p0, s); }
}  // namespace clcg
