// The grouped expert GEMM of ffn_mma_kernel.cuh for the FP4-activation
// variant (activations as packed E2M1 per 32 with UE8M0 scales, kind::mxf4),
// in a translation unit of its own so that it compiles beside the FP8 one.
#define MOE_FFN_MMA_INSTANTIATE launch_ffn_mma_fp4
#define MOE_FFN_MMA_A4 1
#include "ffn_mma_kernel.cuh"
