// Prefill kernels with the outlier split, values with 8-bit codes.
#define KVQ_PF_VB 8
#define KVQ_PF_VSYM 0
#define KVQ_PF_OUTL 1
#include "prefill_fast_dispatch.cuh"
