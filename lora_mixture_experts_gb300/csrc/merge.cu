// Merged-weight fast path: W' = W + B A for one adapter, every expert, both
// projections (the hybrid-attention decoder page merges its LoRA into the
// base weights once, with merge_and_unload, so serving pays no LoRA cost).
// Stored layouts: W [rows][cols], B [rows][r], A [r][cols]; W' rows x cols.
// Memory-bound (read W, write W'): a CTA owns 32 rows x 256 columns, keeps
// the 32 x r slice of B and the r x 256 slice of A in shared memory and
// accumulates the r products of each output in fp32, one bf16 rounding.
#include "common.cuh"
#include "merge.cuh"

namespace moelora {
namespace {

constexpr int kMergeRows = 32;
constexpr int kMergeCols = 256;
constexpr int kMergeThreads = 256;   // thread = 1 row x 32 consecutive columns

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(
    const __nv_bfloat16* __restrict__ W, const __nv_bfloat16* __restrict__ B,
    const __nv_bfloat16* __restrict__ A, __nv_bfloat16* __restrict__ Wm, int rows, int cols, int r,
    long long w_stride, long long b_stride, long long a_stride) {
  // blockIdx.z = expert; w/b/a_stride = elements between experts
  extern __shared__ float sm[];
  float* sa = sm;                          // [r][kMergeCols]
  float* sb = sm + r * kMergeCols;         // [kMergeRows][r]
  const int e = blockIdx.z;
  const int row0 = blockIdx.y * kMergeRows;
  const int col0 = blockIdx.x * kMergeCols;
  const __nv_bfloat16* We = W + e * w_stride;
  const __nv_bfloat16* Be = B + e * b_stride;
  const __nv_bfloat16* Ae = A + e * a_stride;
  __nv_bfloat16* Wme = Wm + e * w_stride;
  for (int i = threadIdx.x; i < r * kMergeCols; i += kMergeThreads) {
    const int q = i / kMergeCols, c = col0 + i % kMergeCols;
    sa[i] = c < cols ? __bfloat162float(Ae[static_cast<size_t>(q) * cols + c]) : 0.0f;
  }
  for (int i = threadIdx.x; i < kMergeRows * r; i += kMergeThreads) {
    const int rr = row0 + i / r, q = i % r;
    sb[i] = rr < rows ? __bfloat162float(Be[static_cast<size_t>(rr) * r + q]) : 0.0f;
  }
  __syncthreads();
  const int lr = threadIdx.x / 8;                 // row of this thread in the tile
  const int lc = (threadIdx.x % 8) * 32;          // first of its 32 columns
  const int row = row0 + lr;
  if (row >= rows) return;
  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
  for (int q = 0; q < r; ++q) {
    const float b = sb[lr * r + q];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = fmaf(b, sa[q * kMergeCols + lc + j], acc[j]);
  }
  const size_t base = static_cast<size_t>(row) * cols + col0 + lc;
  for (int j = 0; j < 32; ++j) {
    const int c = col0 + lc + j;
    if (c < cols) Wme[base + j] = __float2bfloat16_rn(__bfloat162float(We[base + j]) + acc[j]);
  }
}

}  // namespace

cudaError_t launch_merge(const __nv_bfloat16* W, const __nv_bfloat16* B, const __nv_bfloat16* A,
                         __nv_bfloat16* Wm, int E, int rows, int cols, int r, cudaStream_t stream) {
  const dim3 grid((cols + kMergeCols - 1) / kMergeCols, (rows + kMergeRows - 1) / kMergeRows, E);
  const size_t smem = static_cast<size_t>(r) * (kMergeCols + kMergeRows) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  merge_kernel<<<grid, kMergeThreads, smem, stream>>>(
      W, B, A, Wm, rows, cols, r, static_cast<long long>(rows) * cols,
      static_cast<long long>(rows) * r, static_cast<long long>(r) * cols);
  return cudaGetLastError();
}

}  // namespace moelora
