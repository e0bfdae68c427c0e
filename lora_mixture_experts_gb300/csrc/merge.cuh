// Host-visible declaration of the merged-weight kernel (merge.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace moelora {

// Wm[e] = W[e] + B[e] A[e] for e < E: W, Wm [E][rows][cols], B [E][rows][r],
// A [E][r][cols] (bf16; fp32 accumulation, one rounding).
cudaError_t launch_merge(const __nv_bfloat16* W, const __nv_bfloat16* B, const __nv_bfloat16* A,
                         __nv_bfloat16* Wm, int E, int rows, int cols, int r, cudaStream_t stream);

}  // namespace moelora
