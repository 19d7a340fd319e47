// Prefill kernels without outliers, values with 8-bit codes (symmetric).
#define KVQ_PF_VB 8
#define KVQ_PF_VSYM 1
#include "prefill_fast_dispatch.cuh"
