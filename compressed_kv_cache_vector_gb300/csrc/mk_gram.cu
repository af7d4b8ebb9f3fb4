// Set-up helper: the Gram matrix X^T X of one head's keys (or values), whose
// eigenvectors give the rotation R ("MosaicKV：...阅读笔记", Eq. (4), (6)-(8):
// K^T K = V diag(sigma^2) V^T, R = V^T).  The eigensolve itself runs on the
// host, as on the pages; this kernel only forms the d x d product on the GPU
// so that long contexts need not be copied to the host.
//
// Tensor cores: chunks of 64 rows are staged in shared memory (cp.async,
// double-buffered); warp w accumulates rows [16w, 16w+16) of X^T X over all
// 128 columns with mma.sync m16n8k16 (bf16 products are exact, fp32
// accumulation); each CTA adds its partial to the output with atomics.
#include "mk_internal.cuh"

namespace mk {

namespace {
constexpr int kChunk = 64;
constexpr int kGRow = D + 8;  // padded bf16 row (272 bytes)

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
}  // namespace

__global__ void __launch_bounds__(256) k_gram(const uint16_t* __restrict__ x, int64_t n_rows, int64_t row_stride,
                                              float* __restrict__ gram) {
  __shared__ __align__(16) uint16_t xs[2][kChunk][kGRow];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
  const int64_t n_chunks = (n_rows + kChunk - 1) / kChunk;
  auto stage = [&](int64_t ch, int buf) {
    const int64_t r0 = ch * kChunk;
    for (int i = tid; i < kChunk * 16; i += blockDim.x) {
      const int rr = i >> 4, prt = i & 15;
      uint16_t* dst = &xs[buf][rr][prt * 8];
      if (r0 + rr < n_rows) cp_async16(dst, x + (r0 + rr) * row_stride + prt * 8);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
  };
  float acc[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[nt][k] = 0.0f;

  int64_t ch = blockIdx.x;
  int buf = 0;
  if (ch < n_chunks) stage(ch, 0);
  cp_async_commit();
  for (; ch < n_chunks; ch += gridDim.x) {
    if (ch + gridDim.x < n_chunks) stage(ch + gridDim.x, buf ^ 1);
    cp_async_commit();
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    __syncthreads();
#pragma unroll
    for (int kc = 0; kc < kChunk / 16; ++kc) {
      // A = X^T[i][r] for i in [16 warp, +16), r in this 16-row slice:
      // transposed 8x8 blocks of X (rows r, columns i).
      uint32_t a[4];
      ldsm_x4_t(a, &xs[buf][kc * 16 + ri + (mi >> 1) * 8][warp * 16 + (mi & 1) * 8]);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        // B = X[r][j] for two 8-column tiles: transposed 8x8 blocks.
        uint32_t b[4];
        ldsm_x4_t(b, &xs[buf][kc * 16 + ri + (mi & 1) * 8][np * 16 + (mi >> 1) * 8]);
        mma_bf16(acc[2 * np], a, b[0], b[1]);
        mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
      }
    }
    __syncthreads();
    buf ^= 1;
  }
  cp_async_wait_all();
  // acc[nt]: rows i = 16 warp + g (+8), columns j = 8 nt + 2 tig (+1).
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int i = warp * 16 + g, j = nt * 8 + 2 * tig;
    atomicAdd(&gram[i * D + j], acc[nt][0]);
    atomicAdd(&gram[i * D + j + 1], acc[nt][1]);
    atomicAdd(&gram[(i + 8) * D + j], acc[nt][2]);
    atomicAdd(&gram[(i + 8) * D + j + 1], acc[nt][3]);
  }
}

cudaError_t launch_gram(const uint16_t* x, int64_t n_rows, int64_t row_stride, float* gram, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(gram, 0, sizeof(float) * D * D, s);
  if (e != cudaSuccess) return e;
  const int64_t chunks = (n_rows + kChunk - 1) / kChunk;
  int grid = (int)(chunks < 152 ? chunks : 152);
  if (grid < 1) grid = 1;
  k_gram<<<grid, 256, 0, s>>>(x, n_rows, row_stride, gram);
  return cudaGetLastError();
}

}  // namespace mk
