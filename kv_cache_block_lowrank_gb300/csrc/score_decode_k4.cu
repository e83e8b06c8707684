// score_decode_k4.cu -- the decode scorer's kernels for r = 64 (KSTEPS = 4), in a translation
// unit of their own so that the build compiles the four r cases in parallel.
#include "score_decode_kernel.cuh"

HSS_DECODE_INSTANCES(, 4)
