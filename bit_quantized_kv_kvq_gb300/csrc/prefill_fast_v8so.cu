// Prefill kernels with the outlier split, values with 8-bit codes (symmetric).
#define KVQ_PF_VB 8
#define KVQ_PF_VSYM 1
#define KVQ_PF_OUTL 1
#include "prefill_fast_dispatch.cuh"
