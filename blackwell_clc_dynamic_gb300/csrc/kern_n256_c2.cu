// Kernel instantiations for tile N = 256, cluster of 2 CTA(s), CTA-pair MMA
#include "launch.cuh"

namespace clcg {
cudaError_t launch_n256_c2(int sched, const Params& p, int grid_ctas, cudaStream_t stream) {
  return launch_shape<256, 2, true>(sched, p, grid_ctas, stream);
}
cudaError_t max_clusters_n256_c2(int* out) { return max_clusters_shape<256, 2, true>(out); }
cudaError_t warm_n256_c2(const Params& p0, cudaStream_t s) { return warm_shape<256, 2, true>(p0, s); }
}  // namespace clcg
