// Forward kernels instantiated for bf16 I/O.
#include "dispatch.cuh"
NF_INSTANTIATE_FWD(nf::bf16, bf16)
