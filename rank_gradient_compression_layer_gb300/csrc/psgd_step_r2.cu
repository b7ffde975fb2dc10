// Step kernels for padded rank 2.
#define PSGD_RP 2
#include "psgd_step_impl.cuh"
