// Decode kernels: PAGED layout, INT8 cache (tensor cores).
#include "decode_inst.cuh"
KVC_INST_MMA_Q8(true, false)
