// Forward kernels instantiated for f32 I/O.
#include "dispatch.cuh"
NF_INSTANTIATE_FWD(float, f32)
