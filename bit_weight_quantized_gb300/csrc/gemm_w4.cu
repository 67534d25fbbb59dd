// gemm_w4.cu -- the tiled kernel for 4-bit weights (one width per file so
// that the widths compile in parallel).
#include "gemm.cuh"

QMM_GEMM_WIDTH(4)
