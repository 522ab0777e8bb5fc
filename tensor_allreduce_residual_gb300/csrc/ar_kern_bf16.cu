// ar_kern_bf16.cu -- kernels and launchers for __nv_bfloat16 elements (one translation
// unit per element type so the three compile in parallel).
#include "ar_launch.cuh"

AR_INSTANTIATE_LAUNCHERS(__nv_bfloat16)
