// gemm_w7.cu -- the tiled kernel for 7-bit weights (one width per file so
// that the widths compile in parallel).
#include "gemm.cuh"

QMM_GEMM_WIDTH(7)
