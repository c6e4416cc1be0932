// Decode kernels: PAGED layout, bf16 cache (tensor cores).
#include "decode_inst.cuh"
KVC_INST_MMA_ALL_D(true, false)
