// Host-visible declaration of the merged-weight kernel (merge.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace moelora {

// Wm[e] = W[e] + B[e] A[e] for e < E: W, Wm [E][rows][cols], B [E][rows][r],
// A [E][r][cols] (bf16; fp32 accumulation on the tensor cores, one
// rounding).  r is a multiple of 16 up to 128.  Tensor maps (bf16, 3D
// (inner, rows, E)): map_w / map_wm over W / Wm with 64 x 128 boxes and the
// 128-byte swizzle; map_b over B with lw x 128 boxes, lw the largest of 64,
// 32, 16 dividing r, and the (lw * 2)-byte swizzle.
cudaError_t launch_merge(const CUtensorMap& map_w, const CUtensorMap& map_wm, const CUtensorMap& map_b,
                         const __nv_bfloat16* A, int E, int rows, int cols, int r, int num_sms,
                         cudaStream_t stream);

}  // namespace moelora
