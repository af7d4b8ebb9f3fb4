// Set-up helper: the Gram matrix X^T X of one head's keys (or values), whose
// eigenvectors give the rotation R ("MosaicKV：...阅读笔记", Eq. (4), (6)-(8):
// K^T K = V diag(sigma^2) V^T, R = V^T).  The eigensolve itself runs on the
// host, as on the pages; this kernel only forms the d x d product on the GPU
// so that long contexts need not be copied to the host.
#include "mk_internal.cuh"

namespace mk {

// 256 threads; each owns an 8x8 sub-block of the 128x128 result and walks a
// grid-strided range of 64-row chunks staged in shared memory.
__global__ void __launch_bounds__(256) k_gram(const uint16_t* __restrict__ x, int64_t n_rows, int64_t row_stride,
                                              float* __restrict__ gram) {
  __shared__ __align__(16) float xs[64][D + 4];
  const int tid = threadIdx.x;
  const int bi = tid >> 4, bj = tid & 15;
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;
  for (int64_t r0 = (int64_t)blockIdx.x * 64; r0 < n_rows; r0 += (int64_t)gridDim.x * 64) {
    const int nr = (int)min((int64_t)64, n_rows - r0);
    __syncthreads();
    for (int i = tid; i < 64 * D; i += blockDim.x) {
      const int rr = i / D, c = i % D;
      xs[rr][c] = rr < nr ? bf2f(x[(r0 + rr) * row_stride + c]) : 0.0f;
    }
    __syncthreads();
    for (int rr = 0; rr < 64; ++rr) {
      float a[8], b[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        a[k] = xs[rr][8 * bi + k];
        b[k] = xs[rr][8 * bj + k];
      }
#pragma unroll
      for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[p][q] = fmaf(a[p], b[q], acc[p][q]);
    }
  }
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int q = 0; q < 8; ++q) atomicAdd(&gram[(8 * bi + p) * D + 8 * bj + q], acc[p][q]);
}

cudaError_t launch_gram(const uint16_t* x, int64_t n_rows, int64_t row_stride, float* gram, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(gram, 0, sizeof(float) * D * D, s);
  if (e != cudaSuccess) return e;
  int64_t chunks = (n_rows + 63) / 64;
  int grid = (int)(chunks < 304 ? chunks : 304);
  if (grid < 1) grid = 1;
  k_gram<<<grid, 256, 0, s>>>(x, n_rows, row_stride, gram);
  return cudaGetLastError();
}

}  // namespace mk
