// Backward kernels instantiated for bf16 I/O.
#include "dispatch.cuh"
NF_INSTANTIATE_BWD(nf::bf16, bf16)
