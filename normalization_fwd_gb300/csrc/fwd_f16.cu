// Forward kernels instantiated for f16 I/O.
#include "dispatch.cuh"
NF_INSTANTIATE_FWD(nf::f16, f16)
