// Step kernels for padded rank 4.
#define PSGD_RP 4
#include "psgd_step_impl.cuh"
