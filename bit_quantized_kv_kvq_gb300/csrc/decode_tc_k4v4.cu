// Tensor-core decode kernels: 4-bit keys, 4-bit values.
#define KVQ_TC_KB 4
#define KVQ_TC_VB 4
#include "decode_tc_dispatch.cuh"
