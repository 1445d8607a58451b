// gemv_wfp8blk.cu - the head GEMV kernels for FP8 weights with 32x32 block scales (plain and
// interleaved codes).
#include "gemv_kernel.cuh"

TFD_GEMV_INSTANTIATE(TFD_W_FP8_BLOCK32)
TFD_GEMV_INSTANTIATE(TFD_W_FP8_BLOCK32_IL)
