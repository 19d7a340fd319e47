#define KVQ_PIPE_KB 8
#define KVQ_PIPE_VB 4
#include "decode_pipe_launch.cuh"
