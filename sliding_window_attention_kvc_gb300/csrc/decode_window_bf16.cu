// Decode kernels: RING / SINK_RING layouts, bf16 cache (tensor cores).
#include "decode_inst.cuh"
KVC_INST_MMA_ALL_D(false, false)
KVC_INST_MMA_ALL_D(false, true)
