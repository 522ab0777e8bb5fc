// ar_kern_f16.cu -- kernels and launchers for __half elements (one translation
// unit per element type so the three compile in parallel).
#include "ar_launch.cuh"

AR_INSTANTIATE_LAUNCHERS(__half)
