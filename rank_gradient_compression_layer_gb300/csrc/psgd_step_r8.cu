// Step kernels for padded rank 8.
#define PSGD_RP 8
#include "psgd_step_impl.cuh"
