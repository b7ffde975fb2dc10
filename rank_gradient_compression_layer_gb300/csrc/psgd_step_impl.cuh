// Instantiation of the phase kernels for one padded rank (PSGD_RP).
#include "psgd_dispatch.h"
#include "psgd_kernels.cuh"
#if PSGD_RP <= 4
#include "psgd_fused.cuh"
#include "psgd_cluster.cuh"
#endif
#if PSGD_RP >= 16
#include "psgd_mma.cuh"
#endif

#define PSGD_CAT2(a, b) a##b
#define PSGD_CAT(a, b) PSGD_CAT2(a, b)

namespace psgd {
namespace {

constexpr int kRP = PSGD_RP;
constexpr size_t kP3Dyn = p3_dyn_bytes(kRP);

#if PSGD_RP >= 8
// r >= 8: the register-tiled kernels
constexpr size_t kP1TDyn = (size_t)(2 * kRP * kP1TRow + Cfg<kRP>::R1 * kRP) * sizeof(float);
#endif

// A phase kernel launched as a programmatic dependent of the kernel before it
// in the stream (the kernels wait for it in pdl_enter before reading anything
// a kernel of the step writes; only the later phases' tile and layer tables,
// written before the step, are read earlier).
cudaError_t launch_dependent(void (*kernel)(StepArgs), int tiles, int threads, size_t smem, cudaStream_t s,
                             const StepArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

cudaError_t launch(int phase, const StepArgs& a, int tiles, cudaStream_t s) {
  if (tiles <= 0) return cudaSuccess;
  switch (phase) {
    case kProject: {
#if PSGD_RP >= 16
      if (!a.unbiased) return launch_dependent(p1m_kernel<kRP>, tiles, kMThreads, MmaCfg<kRP>::SMEM, s, a);
#endif
#if PSGD_RP >= 8
      return launch_dependent(p1t_kernel<kRP>, tiles, kTThreads, kP1TDyn, s, a);
#else
      const int warps = a.W < Cfg<kRP>::P1_WARPS ? a.W : Cfg<kRP>::P1_WARPS;
      return launch_dependent(p1_kernel<kRP>, tiles, 32 * warps, 0, s, a);
#endif
    }
    case kOrthonormalise: {
      cudaError_t e = launch_dependent(ph_kernel<kRP>, tiles, kPhThreads, 0, s, a);
#if PSGD_RP >= 8
      // the second pass's Phat rows, once per row (r <= 4: in the back-project)
      if (e == cudaSuccess) e = launch_dependent(pf_kernel<kRP>, tiles, ph_rows(kRP), 0, s, a);
#endif
      return e;
    }
    case kBackProject:
      return launch_dependent(p3_kernel<kRP>, tiles, kP3Threads, kP3Dyn, s, a);
    case kDecompress:
#if PSGD_RP >= 8
      return launch_dependent(ut_kernel<kRP>, tiles, kSeg * 4, 0, s, a);
#else
      return launch_dependent(u_kernel<kRP>, tiles, kUThreads, 0, s, a);
#endif
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_error(float* E, const float* B, const float* Phat, const float* Qw, int n, int m, int ld,
                         cudaStream_t s) {
  const int64_t total = (int64_t)n * m;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  error_kernel<kRP><<<(int)blocks, 256, 0, s>>>(E, B, Phat, Qw, n, m, ld);
  return cudaGetLastError();
}

cudaError_t prepare() {
  cudaError_t e = cudaFuncSetAttribute(p3_kernel<kRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kP3Dyn);
#if PSGD_RP >= 8
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(p1t_kernel<kRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kP1TDyn);
#endif
#if PSGD_RP >= 16
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(p1m_kernel<kRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MmaCfg<kRP>::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(p3m_kernel<kRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BmmaCfg<kRP>::SMEM);
#endif
#if PSGD_RP <= 4
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(p1c_kernel<kRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kYSmemMax);
#endif
  return e;
}

cudaError_t occupancy(int phase, int W, int* ctas) {
  switch (phase) {
#if PSGD_RP >= 8
    case kProject:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, p1t_kernel<kRP>, kTThreads, kP1TDyn);
    case kBackProject:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, p3_kernel<kRP>, kP3Threads, kP3Dyn);
    case kDecompress:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, ut_kernel<kRP>, kSeg * 4, 0);
#else
    case kProject: {
      const int warps = W < Cfg<kRP>::P1_WARPS ? W : Cfg<kRP>::P1_WARPS;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, p1_kernel<kRP>, 32 * warps, 0);
    }
    case kBackProject:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, p3_kernel<kRP>, kP3Threads, kP3Dyn);
    case kDecompress:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, u_kernel<kRP>, kUThreads, 0);
#endif
    default:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, ph_kernel<kRP>, kPhThreads, 0);
  }
}

#if PSGD_RP >= 16
cudaError_t launch_bmma(const StepArgs& a, int tiles, cudaStream_t s) {
  if (tiles <= 0) return cudaSuccess;
  return launch_dependent(p3m_kernel<kRP>, tiles, kBThreads, BmmaCfg<kRP>::SMEM, s, a);
}
#endif

cudaError_t launch_gram(const StepArgs& a, int tiles, cudaStream_t s) {
  if (tiles <= 0) return cudaSuccess;
  return launch_dependent(gram_kernel<kRP>, tiles, kGramThreads, 0, s, a);
}

#if PSGD_RP <= 4
cudaError_t launch_fused(const StepArgs& a, int ctas, cudaStream_t s) {
  if (ctas <= 0) return cudaSuccess;
  return launch_dependent(fused_step_kernel<kRP>, ctas, kFThreads, 0, s, a);
}

cudaError_t occupancy_fused(int* ctas) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, fused_step_kernel<kRP>, kFThreads, 0);
}

// The one-pass project: `clusters` clusters of `cs` CTAs, each with `smem`
// bytes of dynamic shared memory, launched as a programmatic dependent like
// the phase kernels.
cudaLaunchConfig_t cluster_config(int clusters, int cs, size_t smem, cudaStream_t s, cudaLaunchAttribute (&attr)[2],
                                  bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * cs));
  cfg.blockDim = dim3((unsigned)kYThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

cudaError_t launch_cluster(const StepArgs& a, int clusters, int cs, size_t smem, cudaStream_t s) {
  if (clusters <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = cluster_config(clusters, cs, smem, s, attr, true);
  return cudaLaunchKernelEx(&cfg, p1c_kernel<kRP>, a);
}

// Clusters of cs CTAs of the one-pass project that fit on the GPU at once.
cudaError_t occupancy_cluster(int cs, size_t smem, int* clusters) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = cluster_config(1, cs, smem, nullptr, attr, false);
  return cudaOccupancyMaxActiveClusters(clusters, p1c_kernel<kRP>, &cfg);
}
#endif

}  // namespace

extern const KernelSet PSGD_CAT(kKernelsR, PSGD_RP) = {
    kRP, launch, launch_error, prepare, occupancy, Cfg<kRP>::R1, Cfg<kRP>::RU, Cfg<kRP>::RSB,
#if PSGD_RP <= 4
    launch_fused, occupancy_fused,
#else
    nullptr, nullptr,
#endif
    launch_gram,
#if PSGD_RP >= 16
    kMRows, kMCols,
#else
    0, 0,
#endif
#if PSGD_RP <= 4
    launch_cluster, occupancy_cluster,
#else
    nullptr, nullptr,
#endif
#if PSGD_RP >= 16
    launch_bmma, kBRows
#else
    nullptr, 0
#endif
};

}  // namespace psgd
