// gemv_wbf16.cu - the head GEMV kernels for bf16 weights.
#include "gemv_kernel.cuh"

TFD_GEMV_INSTANTIATE(TFD_W_BF16)
