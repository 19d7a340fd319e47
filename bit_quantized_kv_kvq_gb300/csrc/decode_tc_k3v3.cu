// Tensor-core decode kernels: 3-bit keys, 3-bit values.
#define KVQ_TC_KB 3
#define KVQ_TC_VB 3
#include "decode_tc_dispatch.cuh"
