// Step kernels for padded rank 32.
#define PSGD_RP 32
#include "psgd_step_impl.cuh"
