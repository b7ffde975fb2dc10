// Instantiation of the step kernels for one padded rank (PSGD_RP).
#include "psgd_dispatch.h"
#include "psgd_kernels.cuh"

#define PSGD_CAT2(a, b) a##b
#define PSGD_CAT(a, b) PSGD_CAT2(a, b)

namespace psgd {
namespace {

constexpr int kRP = PSGD_RP;

cudaError_t launch_step(const StepArgs& a, int grid, size_t smem, cudaStream_t s) {
  step_kernel<kRP><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
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

size_t smem_bytes() { return step_smem_bytes<kRP>(); }

cudaError_t prepare(size_t smem, int* ctas_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(step_kernel<kRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, step_kernel<kRP>, kThreads, smem);
}

}  // namespace

extern const KernelSet PSGD_CAT(kKernelsR, PSGD_RP) = {kRP,          launch_step,   launch_error, smem_bytes,
                                                       Cfg<kRP>::R1, Cfg<kRP>::NF4, Cfg<kRP>::RSU,
                                                       Cfg<kRP>::GSU, prepare};

}  // namespace psgd
