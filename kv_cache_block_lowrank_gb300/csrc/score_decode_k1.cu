// score_decode_k1.cu -- the decode scorer's kernels for r = 16 (KSTEPS = 1), in a translation
// unit of their own so that the build compiles the four r cases in parallel.
#include "score_decode_kernel.cuh"

HSS_DECODE_INSTANCES(, 1)
