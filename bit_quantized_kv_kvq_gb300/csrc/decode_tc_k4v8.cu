// Tensor-core decode kernels: 4-bit keys, 8-bit values.
#define KVQ_TC_KB 4
#define KVQ_TC_VB 8
#include "decode_tc_dispatch.cuh"
