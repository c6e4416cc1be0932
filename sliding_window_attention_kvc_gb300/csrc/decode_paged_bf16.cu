// Decode kernels: PAGED layout, bf16 cache.
#include "decode_inst.cuh"
KVC_INST_ALL_D(__nv_bfloat16, true, false)
