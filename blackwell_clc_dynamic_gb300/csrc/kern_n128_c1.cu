// Kernel instantiations for tile N = 128, cluster of 1 CTA(s)
#include "launch.cuh"

namespace clcg {
cudaError_t launch_n128_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream) {
  return launch_shape<128, 1, false>(sched, p, grid_ctas, stream);
}
cudaError_t max_clusters_n128_c1(int* out) { return max_clusters_shape<128, 1, false>(out); }
cudaError_t warm_n128_c1(const Params& p0, cudaStream_t s) { return warm_shape<128, 1, false>(p0, s); }
}  // namespace clcg
