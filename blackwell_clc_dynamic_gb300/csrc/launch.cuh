// Host-side launch helpers for the GEMM kernel instantiations (one translation unit per
// tile / cluster shape so the library builds in parallel).
#pragma once
#include <cuda_runtime.h>
#include <string.h>

#include "kernel.cuh"

namespace clcg {

// grid_ctas = clusters x CL; the grid is (grid_ctas / CLY) x CLY with clusters of CLX x CLY.
template <int BN, int CL, bool PAIR, int RN = 1>
cudaError_t launch_shape(int sched, const Params& p, int grid_ctas, cudaStream_t stream) {
  using C = Cfg<BN, CL, PAIR, RN>;
  void (*k)(const Params) = nullptr;
  switch (sched) {
    case SCHED_CLC: k = gemm_kernel<BN, CL, PAIR, SCHED_CLC, RN>; break;
    case SCHED_STATIC: k = gemm_kernel<BN, CL, PAIR, SCHED_STATIC, RN>; break;
    case SCHED_NONPERSISTENT: k = gemm_kernel<BN, CL, PAIR, SCHED_NONPERSISTENT, RN>; break;
    default: return cudaErrorInvalidValue;
  }
  if (grid_ctas % CL != 0) return cudaErrorInvalidValue;
  constexpr int smem = C::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid_ctas / C::CLY), C::CLY, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::CLX;
  attr[0].val.clusterDim.y = C::CLY;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, p);
}

// Launch the three schedule variants of a shape once, over an empty problem (p0.total = 0:
// every role finds no tile and the kernel exits).  Whatever a kernel's first launch costs
// (under CUDA's lazy module loading it loads the code, and that can wait until the device
// is idle) is paid here, not at a later launch that would wait for a kernel holding SMs,
// such as the occupier spinning on a host flag.
template <int BN, int CL, bool PAIR, int RN = 1>
cudaError_t warm_shape(const Params& p0, cudaStream_t s) {
  for (int sched = SCHED_CLC; sched <= SCHED_NONPERSISTENT; ++sched) {
    cudaError_t e = launch_shape<BN, CL, PAIR, RN>(sched, p0, CL, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int BN, int CL, bool PAIR, int RN = 1>
cudaError_t max_clusters_shape(int* out) {
  using C = Cfg<BN, CL, PAIR, RN>;
  void (*k)(const Params) = gemm_kernel<BN, CL, PAIR, SCHED_CLC, RN>;
  constexpr int smem = C::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C::CLX * 1024, C::CLY, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::CLX;
  attr[0].val.clusterDim.y = C::CLY;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, (const void*)k, &cfg);
}

// Defined in the per-shape translation units (c2 = CTA pair; c2mc / c4mc = clusters of 2 /
// 4 CTAs with their own MMAs sharing B by multicast; c2x2 = 2 x 2 clusters sharing A along
// rows and B along columns).
cudaError_t launch_n128_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c1(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2mc(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c4mc(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t launch_n256_c2x2(int sched, const Params& p, int grid_ctas, cudaStream_t stream);
cudaError_t max_clusters_n128_c1(int* out);
cudaError_t max_clusters_n256_c1(int* out);
cudaError_t max_clusters_n256_c2(int* out);
cudaError_t max_clusters_n256_c2mc(int* out);
cudaError_t max_clusters_n256_c4mc(int* out);
cudaError_t max_clusters_n256_c2x2(int* out);
cudaError_t warm_n128_c1(const Params& p0, cudaStream_t s);
cudaError_t warm_n256_c1(const Params& p0, cudaStream_t s);
cudaError_t warm_n256_c2(const Params& p0, cudaStream_t s);
cudaError_t warm_n256_c2mc(const Params& p0, cudaStream_t s);
cudaError_t warm_n256_c4mc(const Params& p0, cudaStream_t s);
cudaError_t warm_n256_c2x2(const Params& p0, cudaStream_t s);

// Shapes whose CTAs share operand tiles by TMA multicast loads: clusters of 2 that run
// their own MMAs (not the CTA pair), clusters of 4 (4 x 1 x 1 and 2 x 2 x 1).  They run only
// in a process that sees one GPU, on memory of that GPU.
inline bool uses_tma_multicast(int cl, bool pair) { return cl == 4 || (cl == 2 && !pair); }

// True when `p` points into device memory of device `dev`: not host (pinned or pageable),
// not managed, not another GPU's memory.  Every tensor map is encoded only over such
// memory.
inline bool on_device(const void* p, int dev) {
  cudaPointerAttributes a;
  memset(&a, 0, sizeof a);
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

// Launch every kernel of the library once over an empty problem on stream `s` (see
// warm_shape) and wait for them; the TMA multicast shapes only if `with_multicast`.
// `err` receives device error words (none are expected).
inline cudaError_t warm_all(int* err, cudaStream_t s, bool with_multicast) {
  Params p0;
  memset(&p0, 0, sizeof p0);
  p0.total = 0;               // no tile: every role exits at once
  p0.hold_scheduler = 1;      // and the CLC scheduler issues nothing
  p0.raster_group = 1;
  p0.err = err;
  p0.timeout_ns = 2000000000LL;
  p0.inject_fail_after = -1;
  cudaError_t (*plain[])(const Params&, cudaStream_t) = {warm_n128_c1, warm_n256_c1, warm_n256_c2};
  cudaError_t (*mcast[])(const Params&, cudaStream_t) = {warm_n256_c2mc, warm_n256_c4mc, warm_n256_c2x2};
  for (auto f : plain) {
    cudaError_t e = f(p0, s);
    if (e != cudaSuccess) return e;
  }
  if (with_multicast) {
    for (auto f : mcast) {
      cudaError_t e = f(p0, s);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaStreamSynchronize(s);
}

// The launch function of a shape (nullptr if unsupported).
inline cudaError_t launch_any(int bn, int cl, bool pair, int sched, const Params& p, int grid, cudaStream_t s,
                              int rn = 1) {
  if (cl == 4 && rn == 2) return launch_n256_c2x2(sched, p, grid, s);
  if (cl == 2 && pair) return launch_n256_c2(sched, p, grid, s);
  if (cl == 2) return launch_n256_c2mc(sched, p, grid, s);
  if (cl == 4) return launch_n256_c4mc(sched, p, grid, s);
  if (bn == 128) return launch_n128_c1(sched, p, grid, s);
  return launch_n256_c1(sched, p, grid, s);
}

inline cudaError_t max_clusters_any(int bn, int cl, bool pair, int* out, int rn = 1) {
  if (cl == 4 && rn == 2) return max_clusters_n256_c2x2(out);
  if (cl == 2 && pair) return max_clusters_n256_c2(out);
  if (cl == 2) return max_clusters_n256_c2mc(out);
  if (cl == 4) return max_clusters_n256_c4mc(out);
  if (bn == 128) return max_clusters_n128_c1(out);
  return max_clusters_n256_c1(out);
}

}  // namespace clcg
