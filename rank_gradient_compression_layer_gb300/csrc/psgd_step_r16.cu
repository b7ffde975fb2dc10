// Step kernels for padded rank 16.
#define PSGD_RP 16
#include "psgd_step_impl.cuh"
