// Step kernels for padded rank 1.
#define PSGD_RP 1
#include "psgd_step_impl.cuh"
