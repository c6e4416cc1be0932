// Decode kernels: PAGED layout, f32 cache.
#include "decode_inst.cuh"
KVC_INST_ALL_D(float, true, false)
