// Prefill kernels without outliers, values with 3-bit codes.
#define KVQ_PF_VB 3
#define KVQ_PF_VSYM 0
#include "prefill_fast_dispatch.cuh"
