// gemm_w6.cu -- the tiled kernel for 6-bit weights (one width per file so
// that the widths compile in parallel).
#include "gemm.cuh"

QMM_GEMM_WIDTH(6)
