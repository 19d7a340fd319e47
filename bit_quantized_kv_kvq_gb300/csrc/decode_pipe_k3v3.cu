#define KVQ_PIPE_KB 3
#define KVQ_PIPE_VB 3
#include "decode_pipe_launch.cuh"
