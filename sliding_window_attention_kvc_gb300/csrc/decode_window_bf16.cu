// Decode kernels: RING / SINK_RING layouts, bf16 cache.
#include "decode_inst.cuh"
KVC_INST_ALL_D(__nv_bfloat16, false, false)
KVC_INST_ALL_D(__nv_bfloat16, false, true)
