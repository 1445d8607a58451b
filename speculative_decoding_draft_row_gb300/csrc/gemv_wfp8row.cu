// gemv_wfp8row.cu - the head GEMV kernels for FP8 weights with a row scale.
#include "gemv_kernel.cuh"

TFD_GEMV_INSTANTIATE(TFD_W_FP8_ROW)
