// Decode kernels: RING / SINK_RING layouts, f32 cache.
#include "decode_inst.cuh"
KVC_INST_ALL_D(float, false, false)
KVC_INST_ALL_D(float, false, true)
