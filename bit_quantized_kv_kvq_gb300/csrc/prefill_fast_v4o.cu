// Prefill kernels with the outlier split, values with 4-bit codes.
#define KVQ_PF_VB 4
#define KVQ_PF_VSYM 0
#define KVQ_PF_OUTL 1
#include "prefill_fast_dispatch.cuh"
