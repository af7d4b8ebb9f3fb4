// Block selection: rotate the query (q' = q R_k^T), score every middle block
// from its per-channel min/max keys, keep the top-k blocks.
//
// Method: "MosaicKV：...阅读笔记" (zhongzhuzhou.org), Eq. (12) (block score
// from the compressed keys, with q' the rotated query) and the description
// of Quest's per-block min/max bound; "MosaicKV: Serving Long-Context LLM
// with Dynamic Two-D KV Cache Compression" (paperlayer.ai), sec. 4.2 stage 2
// (top-k token blocks before each decode attention layer) and sec. 5.3
// (inverse rotation merged into the query).
#include "mk_internal.cuh"

namespace mk {

__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) == 0) b = 0;  // -0 and +0 are the same score
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// grid (chunks, n_seqs * n_kv); 256 threads.
template <int G>
__global__ void __launch_bounds__(256) k_score(Layout L, int layer, CallSeqs cs, const uint16_t* __restrict__ q,
                                               float* __restrict__ scores_out) {
  const int ci = blockIdx.y / L.n_kv, kvh = blockIdx.y - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = unit_index(L, layer, seq, kvh);
  __shared__ float qs[G][D];
  __shared__ __align__(16) float qr[D][G];
  __shared__ int s_abort, s_T;
  if (tid == 0) {
    s_abort = has_error(L);
    s_T = L.desc[u].T;
  }
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    qs[h][c] = bf2f(q[((int64_t)ci * L.n_kv * G + (int64_t)kvh * G + h) * D + c]);
  }
  __syncthreads();
  if (s_abort) return;
  const char* base = unit_base(L, u);
  extern __shared__ __align__(16) float Rs[];   // R_k^T [128][128]
  {
    const float4* src = reinterpret_cast<const float4*>(base + L.off_rkt);
    for (int i = tid; i < D * D / 4; i += blockDim.x) cp_async16(reinterpret_cast<float4*>(Rs) + i, src + i);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
  }
  if (tid < D) {
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.0f;
    for (int j = 0; j < D; ++j) {
      const float rr = Rs[j * D + tid];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = fmaf(qs[h][j], rr, acc[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      qr[tid][h] = acc[h];
      if (blockIdx.x == 0) L.qrot[(((int64_t)seq * L.n_kv + kvh) * G + h) * D + tid] = acc[h];
    }
  }
  __syncthreads();
  float qreg[4][G];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int h = 0; h < G; ++h) qreg[i][h] = qr[4 * lane + i][h];

  const int nblk = n_mid_blocks(L, s_T);
  const uint16_t* meta = reinterpret_cast<const uint16_t*>(base + L.off_meta);
  float* sc = L.scores + ((int64_t)seq * L.n_kv + kvh) * L.nblk_cap;
  float* so = scores_out ? scores_out + ((int64_t)ci * L.n_kv + kvh) * L.nblk_cap : nullptr;
  const float inv_sqrt_d = 0.08838834764831845f;
  for (int b = blockIdx.x * 8 + warp; b < nblk; b += gridDim.x * 8) {
    const uint2 mn4 = __ldg(reinterpret_cast<const uint2*>(meta + (int64_t)b * 2 * D) + lane);
    const uint2 mx4 = __ldg(reinterpret_cast<const uint2*>(meta + (int64_t)b * 2 * D + D) + lane);
    const float mn[4] = {bf2f(mn4.x & 0xffff), bf2f(mn4.x >> 16), bf2f(mn4.y & 0xffff), bf2f(mn4.y >> 16)};
    const float mx[4] = {bf2f(mx4.x & 0xffff), bf2f(mx4.x >> 16), bf2f(mx4.y & 0xffff), bf2f(mx4.y >> 16)};
    float best = -INFINITY;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) s = fmaf(qreg[i][h], qreg[i][h] >= 0.0f ? mx[i] : mn[i], s);
      s = warp_sum(s);
      best = fmaxf(best, s);
    }
    best *= inv_sqrt_d;
    if (lane == 0) {
      sc[b] = best;
      if (so) so[b] = best;
    }
  }
}

// Block-wide exclusive scan of 0/1 flags over 1024 threads; returns the
// prefix and writes the total to *total.
__device__ __forceinline__ int block_flag_scan(bool f, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(FULL, f);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    const int v = warp_tot[lane];
    const int ex = warp_excl_scan(v, lane);
    warp_tot[lane] = ex;
    if (lane == 31) warp_tot[32] = ex + v;
  }
  __syncthreads();
  *total = warp_tot[32];
  return warp_tot[warp] + in_warp;
}

// One CTA (1024 threads) per (sequence, kv head): k largest scores among the
// scored segments' blocks, ties to the lower id, written in ascending order.
__global__ void __launch_bounds__(1024) k_topk(Layout L, int layer, CallSeqs cs, int32_t* __restrict__ ids,
                                               int32_t* __restrict__ n_sel) {
  const int ci = blockIdx.x / L.n_kv, kvh = blockIdx.x - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = unit_index(L, layer, seq, kvh);
  __shared__ UnitDesc ud;
  __shared__ unsigned hist[256];
  __shared__ int warp_tot[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining, s_abort;
  if (tid == 0) {
    ud = L.desc[u];
    s_abort = has_error(L);
  }
  __syncthreads();
  if (s_abort) return;
  const int nblk = n_mid_blocks(L, ud.T);
  const int n_cand = n_scored_blocks(ud, nblk);
  const int k = n_select(L, n_cand);
  const float* sc = L.scores + ((int64_t)seq * L.n_kv + kvh) * L.nblk_cap;
  int32_t* out = ids + ((int64_t)ci * L.n_kv + kvh) * L.k_max;

  uint32_t prefix = 0, mask = 0;
  int need = 0;
  const bool all = k >= n_cand;
  if (!all) {
    if (tid == 0) s_remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      for (int b = tid; b < nblk; b += blockDim.x) {
        if (ud.always[seg_of_block(ud, b)]) continue;
        const uint32_t key = ordered_key(sc[b]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        const int rem = s_remaining;
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) cnt += (int)hist[255 - (8 * lane + i)];
        const int ex = warp_excl_scan(cnt, lane);
        const unsigned hit = __ballot_sync(FULL, ex + cnt >= rem);
        const int src = __ffs(hit) - 1;
        if (lane == src) {
          int acc = ex;
          for (int i = 0; i < 8; ++i) {
            const int dgt = 255 - (8 * lane + i);
            const int hcount = (int)hist[dgt];
            if (acc + hcount >= rem) {
              s_prefix = (uint32_t)dgt;
              s_remaining = rem - acc;
              break;
            }
            acc += hcount;
          }
        }
      }
      __syncthreads();
      prefix |= s_prefix << shift;
      mask |= 255u << shift;
      __syncthreads();
    }
    need = s_remaining;
  }

  int run_sel = 0, run_tie = 0;
  for (int b0 = 0; b0 < nblk; b0 += blockDim.x) {
    const int b = b0 + tid;
    bool cand = false;
    uint32_t key = 0;
    if (b < nblk) {
      cand = !ud.always[seg_of_block(ud, b)];
      if (cand && !all) key = ordered_key(sc[b]);
    }
    const bool is_eq = cand && !all && key == prefix;
    int tie_tot;
    const int tie_ex = block_flag_scan(is_eq, warp_tot, &tie_tot) + run_tie;
    const bool sel = cand && (all || key > prefix || (is_eq && tie_ex < need));
    int sel_tot;
    const int pos = block_flag_scan(sel, warp_tot, &sel_tot) + run_sel;
    if (sel && pos < L.k_max) out[pos] = b;
    run_tie += tie_tot;
    run_sel += sel_tot;
  }
  if (tid == 0) n_sel[(int64_t)ci * L.n_kv + kvh] = k;
}

cudaError_t launch_block_select(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* q,
                                int32_t* ids, int32_t* n_sel, float* scores_out, int max_nblk,
                                cudaStream_t s) {
  const int units = cs.n * L.n_kv;
  int chunks = (2 * 152 + units - 1) / units;
  const int max_chunks = (max_nblk + 7) / 8;
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  dim3 grid(chunks, units);
  const int smem = D * D * (int)sizeof(float);
#define MK_SCORE_CASE(GG)                                                                                  \
  case GG: {                                                                                               \
    static bool set = false;                                                                               \
    if (!set) {                                                                                            \
      cudaError_t e = cudaFuncSetAttribute(k_score<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); \
      if (e != cudaSuccess) return e;                                                                      \
      set = true;                                                                                          \
    }                                                                                                      \
    k_score<GG><<<grid, 256, smem, s>>>(L, layer, cs, q, scores_out);                                      \
    break;                                                                                                 \
  }
  switch (L.G) {
    MK_SCORE_CASE(1)
    MK_SCORE_CASE(2)
    MK_SCORE_CASE(4)
    MK_SCORE_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef MK_SCORE_CASE
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_topk<<<units, 1024, 0, s>>>(L, layer, cs, ids, n_sel);
  return cudaGetLastError();
}

}  // namespace mk
