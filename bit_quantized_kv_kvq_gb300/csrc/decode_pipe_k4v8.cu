#define KVQ_PIPE_KB 4
#define KVQ_PIPE_VB 8
#include "decode_pipe_launch.cuh"
