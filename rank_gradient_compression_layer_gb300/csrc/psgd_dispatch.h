// Per-rank kernel entry points.  Each psgd_step_rN.cu instantiates the phase
// kernels for one padded rank N and exports them through a KernelSet.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "psgd_internal.h"

namespace psgd {

enum Phase : int { kProject = 0, kOrthonormalise = 1, kBackProject = 2, kDecompress = 3, kPhases = 4 };

struct KernelSet {
  int rp;
  // one phase kernel over `tiles` tiles (a.tiles must point at that phase's tiles)
  cudaError_t (*launch)(int phase, const StepArgs& a, int tiles, cudaStream_t s);
  // E = B - Phat Q_w^T of one layer, dense n x m
  cudaError_t (*error)(float* E, const float* B, const float* Phat, const float* Qw, int n, int m, int ld,
                       cudaStream_t s);
  // one-time set-up (shared memory limits)
  cudaError_t (*prepare)();
  // resident CTAs per SM of a phase kernel for W workers
  cudaError_t (*occupancy)(int phase, int W, int* ctas_per_sm);
  // tile geometry: most project rows per tile, most decompress rows per tile,
  // rows per project pass
  int r1, ru, rsb;
  // the fused step (padded ranks <= 4; null above): one launch of `ctas` CTAs
  // over a.n_items queue items, and its resident CTAs per SM
  cudaError_t (*launch_fused)(const StepArgs& a, int ctas, cudaStream_t s);
  cudaError_t (*occupancy_fused)(int* ctas_per_sm);
  // split step: the Gram factor of an all-reduced P over `tiles` row blocks
  cudaError_t (*launch_gram)(const StepArgs& a, int tiles, cudaStream_t s);
  // the project phase runs on the tensor cores (padded ranks 16, 32; not the
  // unbiased variant): its tiles have mma_rows rows and mma_cols columns
  int mma_rows, mma_cols;
  // the one-pass project (padded ranks <= 4; null above): `clusters`
  // clusters of `cs` CTAs with `smem` bytes of dynamic shared memory each
  // over a.tiles, and the clusters of that shape resident at once
  cudaError_t (*launch_cluster)(const StepArgs& a, int clusters, int cs, size_t smem, cudaStream_t s);
  cudaError_t (*occupancy_cluster)(int cs, size_t smem, int* clusters);
  // the back-project on the tensor cores (padded ranks 16, 32; null below):
  // tiles of bmma_rows-row chunks over (row tile, segment) with every worker
  cudaError_t (*launch_bmma)(const StepArgs& a, int tiles, cudaStream_t s);
  int bmma_rows;
};

extern const KernelSet kKernelsR1, kKernelsR2, kKernelsR4, kKernelsR8, kKernelsR16, kKernelsR32;

}  // namespace psgd
