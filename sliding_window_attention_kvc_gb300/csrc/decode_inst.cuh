// Explicit instantiation of the decode launchers; included by the decode_*.cu
// translation units so the heavy template code compiles in parallel.
#pragma once
#include "kvc_decode_mma.cuh"

// fp32 caches: CUDA-core kernel (kvc_decode.cuh)
#define KVC_INST(E, D, GH, PG, RD) \
    template cudaError_t kvc::launch_decode_t<E, D, GH, PG, RD>(const kvc::DecodeParams&, dim3, cudaStream_t);

#define KVC_INST_ALL_D(E, PG, RD)   \
    KVC_INST(E, 64, 1, PG, RD)      \
    KVC_INST(E, 64, 2, PG, RD)      \
    KVC_INST(E, 64, 4, PG, RD)      \
    KVC_INST(E, 128, 1, PG, RD)     \
    KVC_INST(E, 128, 2, PG, RD)     \
    KVC_INST(E, 128, 4, PG, RD)     \
    KVC_INST(E, 256, 1, PG, RD)     \
    KVC_INST(E, 256, 2, PG, RD)     \
    KVC_INST(E, 256, 4, PG, RD)

// bf16 and INT8 caches: tensor-core kernel (kvc_decode_mma.cuh)
#define KVC_INST_MMA(D, GH, PG, RD, Q8)                                                               \
    template cudaError_t kvc::launch_decode_mma_t<D, GH, PG, RD, Q8>(const kvc::DecodeParams&,          \
                                                                     const kvc::KvTensorMaps&, dim3,     \
                                                                     cudaStream_t);

#define KVC_INST_MMA_ALL_D(PG, RD)        \
    KVC_INST_MMA(64, 1, PG, RD, false)    \
    KVC_INST_MMA(64, 2, PG, RD, false)    \
    KVC_INST_MMA(64, 4, PG, RD, false)    \
    KVC_INST_MMA(128, 1, PG, RD, false)   \
    KVC_INST_MMA(128, 2, PG, RD, false)   \
    KVC_INST_MMA(128, 4, PG, RD, false)   \
    KVC_INST_MMA(256, 1, PG, RD, false)   \
    KVC_INST_MMA(256, 2, PG, RD, false)   \
    KVC_INST_MMA(256, 4, PG, RD, false)

// INT8: head_dim 128 and 256; read-time RoPE on window caches only
#define KVC_INST_MMA_Q8(PG, RD)        \
    KVC_INST_MMA(128, 1, PG, RD, true) \
    KVC_INST_MMA(128, 2, PG, RD, true) \
    KVC_INST_MMA(128, 4, PG, RD, true) \
    KVC_INST_MMA(256, 1, PG, RD, true) \
    KVC_INST_MMA(256, 2, PG, RD, true) \
    KVC_INST_MMA(256, 4, PG, RD, true)
