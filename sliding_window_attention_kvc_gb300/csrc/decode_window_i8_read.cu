// Decode kernels: RING / SINK_RING layouts, INT8 cache with read-time RoPE
// (tensor cores).
#include "decode_inst.cuh"
KVC_INST_MMA_Q8(false, true)
