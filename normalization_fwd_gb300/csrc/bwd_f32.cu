// Backward kernels instantiated for f32 I/O.
#include "dispatch.cuh"
NF_INSTANTIATE_BWD(float, f32)
