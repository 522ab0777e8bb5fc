// ar_kern_f32.cu -- kernels and launchers for float elements (one translation
// unit per element type so the three compile in parallel).
#include "ar_launch.cuh"

AR_INSTANTIATE_LAUNCHERS(float)
