// Per-rank kernel entry points.  Each psgd_step_rN.cu instantiates the step
// kernels for one padded rank N and exports them through a KernelSet.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "psgd_internal.h"

namespace psgd {

struct KernelSet {
  int rp;
  // persistent step kernel: grid CTAs of kThreads threads (every warp works alone)
  cudaError_t (*step)(const StepArgs& a, int grid, size_t smem, cudaStream_t s);
  // E = B - Phat Q_w^T of one layer, dense n x m
  cudaError_t (*error)(float* E, const float* B, const float* Phat, const float* Qw, int n, int m, int ld,
                       cudaStream_t s);
  // dynamic shared memory of the step kernel
  size_t (*smem_bytes)();
  // P1 rows and float4 columns per item; U rows and segments per item
  int rs1, nf4, rsu, gsu;
  // raise the kernel's dynamic shared memory limit; resident CTAs per SM
  cudaError_t (*prepare)(size_t smem, int* ctas_per_sm);
};

extern const KernelSet kKernelsR1, kKernelsR2, kKernelsR4, kKernelsR8, kKernelsR16, kKernelsR32;

}  // namespace psgd
