// Block selection: rotate the query (q' = q R_k^T), score every middle block
// from its per-channel min/max keys, keep the top-k blocks.
//
// Method: "MosaicKV：...阅读笔记" (zhongzhuzhou.org), Eq. (12) (block score
// from the compressed keys with the rotated query q') and the description
// of Quest's per-block min/max bound; "MosaicKV: Serving Long-Context LLM
// with Dynamic Two-D KV Cache Compression" (paperlayer.ai), sec. 4.2 stage 2
// (top-k token blocks before each decode attention layer) and sec. 5.3
// (inverse rotation merged into the query).
//
// GB300 structure: one kernel, P CTAs per (sequence, kv head).
//  * Each CTA stages R_k^T (cp.async) and forms q' for the group's heads.
//  * Scoring is a dense contraction: for block b and head h,
//      sum_j max(q'_hj mn_bj, q'_hj mx_bj) = [mn_b | mx_b] . [min(q'_h,0) | max(q'_h,0)]
//    over K = 256.  Meta tiles of 16 blocks are staged with cp.async and
//    multiplied on the tensor cores (mma.sync m16n8k16).  The fp32 operand is
//    split exactly into three bf16 parts (24 = 3 x 8 significant bits) and the
//    meta values are bf16, so every product is exact and the accumulation is
//    fp32: the scores keep fp32 accuracy.
//  * The last CTA of each (sequence, kv head) to finish (atomic counter, no
//    waiting) runs the radix top-k over the unit's scores in shared memory.
#include <algorithm>

#include "mk_internal.cuh"

namespace mk {

namespace {
constexpr int kSelWarps = 8;
constexpr int kMT = 16;                       // blocks per MMA tile
constexpr int kMetaRow = 2 * D + 8;           // padded bf16 row (528 bytes): ldmatrix conflict-free
constexpr int kMetaTile = kMT * kMetaRow * 2; // bytes per staged tile
constexpr int kSelSmem = kSelWarps * 2 * kMetaTile;  // double-buffered tiles (also holds R_k^T and keys)
static_assert(kSelSmem >= D * D * 4, "R_k^T staging fits in the tile area");

__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) == 0) b = 0;  // -0 and +0 are the same score
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
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
// Exact three-way split of an fp32 value into bf16 parts (x = p0 + p1 + p2
// for normal x: each part takes the next 8 significant bits).
__device__ __forceinline__ void split3(float x, uint16_t (&p)[3]) {
  float r = x;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const __nv_bfloat16 h = __float2bfloat16_rz(r);
    p[i] = __bfloat16_as_ushort(h);
    r -= __bfloat162float(h);
  }
}

// Ties (keys equal to the threshold) held by warps 0..w-1.
__device__ __forceinline__ int tie_before(const int* warp_tot, int w) {
  int t = 0;
  for (int i = 0; i < w; ++i) t += warp_tot[8 + i];
  return t;
}

}  // namespace

// grid: P CTAs per (sequence, kv head) of the call; 256 threads.
template <int G>
__global__ void __launch_bounds__(256, 1) k_select(Layout L, int layer, CallSeqs cs, int P,
                                                   const uint16_t* __restrict__ q, int32_t* __restrict__ ids,
                                                   int32_t* __restrict__ n_sel, float* __restrict__ scores_out) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float qs[G][D];
  __shared__ float qr[2][G][D];
  __shared__ UnitDesc ud;
  __shared__ unsigned hist[256];
  __shared__ int warp_tot[33];
  __shared__ int s_rem, s_abort, s_last;
  __shared__ uint32_t s_lo, s_hi;

  const int unit_call = blockIdx.x / P, part = blockIdx.x - unit_call * P;
  const int ci = unit_call / L.n_kv, kvh = unit_call - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t u = unit_index(L, layer, seq, kvh);
  const int64_t slot = (int64_t)seq * L.n_kv + kvh;
  for (int i = tid; i < G * D; i += blockDim.x)
    qs[i / D][i % D] = bf2f(q[((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D + i]);
  const char* base = unit_base(L, u);
  {
    const float4* src = reinterpret_cast<const float4*>(base + L.off_rkt);
    for (int i = tid; i < D * D / 4; i += blockDim.x) cp_async16(reinterpret_cast<float4*>(smem) + i, src + i);
    cp_async_commit();
    cp_async_wait_all();
  }
  __syncthreads();

  // q'_h[c] = sum_j q_h[j] R_k[c][j]: thread (c, half of j), halves added.
  {
    const float* Rs = reinterpret_cast<const float*>(smem);
    const int c = tid & (D - 1), half = tid >> 7;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.0f;
    for (int j = half * 64; j < half * 64 + 64; ++j) {
      const float rr = Rs[j * D + c];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = fmaf(qs[h][j], rr, acc[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) qr[half][h][c] = acc[h];
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    const float v = qr[0][h][c] + qr[1][h][c];
    qr[0][h][c] = v;
  }
  __syncthreads();

  // B fragments of [min(q',0) | max(q',0)] (k = 0..255, n = head), 3 exact parts.
  uint32_t bq[3][16][2];
#pragma unroll
  for (int kc = 0; kc < 16; ++kc)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint16_t e0[3] = {0, 0, 0}, e1[3] = {0, 0, 0};
      if (g < G) {
        const int k = kc * 16 + hf * 8 + 2 * tig;
        const float x0 = k < D ? fminf(qr[0][g][k], 0.0f) : fmaxf(qr[0][g][k - D], 0.0f);
        const float x1 = (k + 1) < D ? fminf(qr[0][g][k + 1], 0.0f) : fmaxf(qr[0][g][k + 1 - D], 0.0f);
        split3(x0, e0);
        split3(x1, e1);
      }
#pragma unroll
      for (int s = 0; s < 3; ++s) bq[s][kc][hf] = (uint32_t)e0[s] | ((uint32_t)e1[s] << 16);
    }
  // Everything above used only q and R_k.  From here on the kernel reads
  // what the append kernel wrote (lengths, block keys).
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    s_abort = has_error(L);
    ud = L.desc[u];
  }
  if (part == 0)
    for (int i = tid; i < G * D; i += blockDim.x) L.qrot[slot * G * D + i] = qr[0][i / D][i % D];
  __syncthreads();  // also: the R_k^T area becomes the tile stages
  if (s_abort) return;

  const int nblk = n_mid_blocks(L, ud.T);
  const int ntiles = (nblk + kMT - 1) / kMT;
  const int tper = (ntiles + P - 1) / P;
  const int t0 = part * tper, t1 = min(ntiles, t0 + tper);
  const uint16_t* meta = reinterpret_cast<const uint16_t*>(base + L.off_meta);
  float* sc = L.scores + slot * L.scores_stride;
  float* so = scores_out ? scores_out + ((int64_t)ci * L.n_kv + kvh) * L.nblk_cap : nullptr;
  unsigned char* stg = smem + (size_t)warp * 2 * kMetaTile;
  auto issue = [&](int t, unsigned char* dst) {
    if (t >= t1) return;
    for (int i = lane; i < kMT * 32; i += 32) {
      const int row = i >> 5, prt = i & 31;
      const int b = t * kMT + row;
      if (b < nblk) cp_async16(dst + row * kMetaRow * 2 + prt * 16, meta + (int64_t)b * 2 * D + prt * 8);
    }
  };
  const float inv_sqrt_d = 0.08838834764831845f;
  int st = 0;
  int t = t0 + warp;
  issue(t, stg);
  cp_async_commit();
  for (; t < t1; t += kSelWarps) {
    issue(t + kSelWarps, stg + (size_t)(st ^ 1) * kMetaTile);
    cp_async_commit();
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    __syncwarp();
    const uint16_t* tile = reinterpret_cast<const uint16_t*>(stg + (size_t)st * kMetaTile);
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int mi = lane >> 3, ri = lane & 7;
    const uint16_t* arow = tile + (ri + (mi & 1) * 8) * kMetaRow + (mi >> 1) * 8;
#pragma unroll
    for (int kc = 0; kc < 16; ++kc) {
      uint32_t a[4];
      ldsm_x4(a, arow + kc * 16);
      mma_bf16(s, a, bq[0][kc][0], bq[0][kc][1]);
      mma_bf16(s, a, bq[1][kc][0], bq[1][kc][1]);
      mma_bf16(s, a, bq[2][kc][0], bq[2][kc][1]);
    }
    // rows: blocks g, g+8; columns: heads 2tig, 2tig+1 -> max over the group's heads
    const bool h0 = 2 * tig < G, h1 = 2 * tig + 1 < G;
    float b_lo = fmaxf(h0 ? s[0] : -INFINITY, h1 ? s[1] : -INFINITY);
    float b_hi = fmaxf(h0 ? s[2] : -INFINITY, h1 ? s[3] : -INFINITY);
    b_lo = fmaxf(b_lo, __shfl_xor_sync(FULL, b_lo, 1));
    b_hi = fmaxf(b_hi, __shfl_xor_sync(FULL, b_hi, 1));
    b_lo = fmaxf(b_lo, __shfl_xor_sync(FULL, b_lo, 2));
    b_hi = fmaxf(b_hi, __shfl_xor_sync(FULL, b_hi, 2));
    if (tig == 0) {
      const int b0 = t * kMT + g, b1 = b0 + 8;
      if (b0 < nblk) {
        sc[b0] = b_lo * inv_sqrt_d;
        if (so) so[b0] = b_lo * inv_sqrt_d;
      }
      if (b1 < nblk) {
        sc[b1] = b_hi * inv_sqrt_d;
        if (so) so[b1] = b_hi * inv_sqrt_d;
      }
    }
    __syncwarp();
    st ^= 1;
  }
  cp_async_wait_all();

  // ---- the last CTA of this (sequence, kv head) selects the top-k ---------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&L.counters[L.max_seqs * L.n_kv + slot], 1);
    s_last = (prev == P - 1);
    if (prev == P - 1) L.counters[L.max_seqs * L.n_kv + slot] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int n_cand = n_scored_blocks(ud, nblk);
  const int k = n_select(L, n_cand);
  int32_t* out = ids + ((int64_t)ci * L.n_kv + kvh) * L.k_max;
  const bool all = k >= n_cand;
  const int nth = blockDim.x, nw = nth >> 5;
  // Keys in shared memory: one cp.async burst of the unit's scores, then
  // converted in place (0 marks a block that is not a candidate: an
  // always-attended segment; real scores never map to 0, and k <= #candidates
  // keeps the top k away from it).
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  const bool in_smem = (size_t)nblk * 4 <= (size_t)kSelSmem;
  if (in_smem) {
    for (int i = tid; i < (nblk + 3) / 4; i += nth) cp_async16(keys + 4 * i, sc + 4 * i);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    for (int b = tid; b < nblk; b += nth) {
      const float f = __uint_as_float(keys[b]);
      keys[b] = ud.always[seg_of_block(ud, b)] ? 0u : ordered_key(f);
    }
    __syncthreads();
  }
  auto key_of = [&](int b) -> uint32_t {
    if (in_smem) return keys[b];
    return ud.always[seg_of_block(ud, b)] ? 0u : ordered_key(__ldcg(sc + b));
  };

  // Threshold search: the k-th largest candidate key lies in [lo, hi]; each
  // pass counts the keys of that range in <= 256 bins of power-of-two width
  // (spread over the data's own range, so few threads share a bin) and keeps
  // the bin holding the k-th key, until the range is a single key value.
  uint32_t prefix = 0;  // the threshold key once the search ends
  int need = 0;         // how many keys equal to it are taken (lowest ids first)
  if (!all) {
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int b = tid; b < nblk; b += nth) {
      const uint32_t key = key_of(b);
      if (key != 0u) {
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
    }
    kmin = __reduce_min_sync(FULL, kmin);
    kmax = __reduce_max_sync(FULL, kmax);
    if (lane == 0) {
      hist[warp] = kmin;
      hist[32 + warp] = kmax;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t a = 0xffffffffu, b = 0u;
      for (int w = 0; w < nw; ++w) {
        a = min(a, hist[w]);
        b = max(b, hist[32 + w]);
      }
      s_lo = a;
      s_hi = b;
      s_rem = k;
    }
    __syncthreads();
    for (int pass = 0; pass < 40; ++pass) {
      const uint32_t lo = s_lo, hi = s_hi;
      if (lo == hi) break;
      const uint32_t span = hi - lo;  // >= 1
      const int sh = max(0, 32 - __clz(span) - 8);  // bins of width 2^sh: (span >> sh) < 256
      for (int i = tid; i < 256; i += nth) hist[i] = 0;
      __syncthreads();
      for (int b = tid; b < nblk; b += nth) {
        const uint32_t key = key_of(b);
        if (key != 0u && key >= lo && key <= hi) atomicAdd(&hist[(key - lo) >> sh], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        const int rem = s_rem;
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) cnt += (int)hist[255 - (8 * lane + i)];
        const int ex = warp_excl_scan(cnt, lane);
        const unsigned hit = __ballot_sync(FULL, ex + cnt >= rem);
        const int src = __ffs(hit) - 1;
        if (lane == src) {
          int acc = ex;
          for (int i = 0; i < 8; ++i) {
            const int bin = 255 - (8 * lane + i);
            const int hc = (int)hist[bin];
            if (acc + hc >= rem) {
              const uint32_t blo = lo + ((uint32_t)bin << sh);
              const uint64_t bhi = (uint64_t)blo + ((1ull << sh) - 1ull);
              s_lo = blo;
              s_hi = bhi < (uint64_t)hi ? (uint32_t)bhi : hi;
              s_rem = rem - acc;
              break;
            }
            acc += hc;
          }
        }
      }
      __syncthreads();
    }
    prefix = s_lo;
    need = s_rem;
  }

  // Ordered compaction: warp w owns blocks [w*RW, (w+1)*RW), walked 32 at a
  // time with ballots; one block-wide scan gives each warp its offsets.
  const int RW = ((nblk + nw - 1) / nw + 31) & ~31;
  const int wb0 = warp * RW, wb1 = min(nblk, wb0 + RW);
  int w_gt = 0, w_eq = 0;
  for (int b0 = wb0; b0 < wb1; b0 += 32) {
    const int b = b0 + lane;
    const uint32_t key = b < wb1 ? key_of(b) : 0u;
    w_gt += __popc(__ballot_sync(FULL, key != 0u && (all || key > prefix)));
    w_eq += __popc(__ballot_sync(FULL, key != 0u && !all && key == prefix));
  }
  if (lane == 0) {
    warp_tot[warp] = w_gt;
    warp_tot[8 + warp] = w_eq;
  }
  __syncthreads();
  int sel_off = 0, tie_off = 0;
  for (int w = 0; w < warp; ++w) tie_off += warp_tot[8 + w];
  for (int w = 0; w < warp; ++w) sel_off += warp_tot[w] + max(0, min(warp_tot[8 + w], need - tie_before(warp_tot, w)));
  for (int b0 = wb0; b0 < wb1; b0 += 32) {
    const int b = b0 + lane;
    const uint32_t key = b < wb1 ? key_of(b) : 0u;
    const unsigned gt = __ballot_sync(FULL, key != 0u && (all || key > prefix));
    const unsigned eq = __ballot_sync(FULL, key != 0u && !all && key == prefix);
    const unsigned lt_mask = (1u << lane) - 1u;
    const int tie_rank = tie_off + __popc(eq & lt_mask);
    const bool take_tie = ((eq >> lane) & 1u) && tie_rank < need;
    const unsigned tk = __ballot_sync(FULL, take_tie);
    const unsigned sel = gt | tk;
    if ((sel >> lane) & 1u) {
      const int pos = sel_off + __popc(sel & lt_mask);
      if (pos < L.k_max) out[pos] = b;
    }
    sel_off += __popc(sel);
    tie_off += __popc(eq);
  }
  if (tid == 0) n_sel[(int64_t)ci * L.n_kv + kvh] = k;
}

cudaError_t launch_block_select(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* q,
                                int32_t* ids, int32_t* n_sel, float* scores_out, int max_nblk,
                                cudaStream_t s) {
  const int units = cs.n * L.n_kv;
  const int tiles = (max_nblk + kMT - 1) / kMT;
  int P = std::max(1, 152 / units);
  P = std::min(P, std::max(1, (tiles + kSelWarps - 1) / kSelWarps));
  const dim3 grid(units * P);
#define MK_SEL_CASE(GG)                                                                                      \
  case GG: {                                                                                                 \
    static bool set = false;                                                                                 \
    if (!set) {                                                                                              \
      cudaError_t e = cudaFuncSetAttribute(k_select<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelSmem); \
      if (e != cudaSuccess) return e;                                                                        \
      set = true;                                                                                            \
    }                                                                                                        \
    return launch_pdl(k_select<GG>, grid, dim3(256), kSelSmem, s, 0, L, layer, cs, P, q, ids, n_sel,        \
                      scores_out);                                                                           \
  }
  switch (L.G) {
    MK_SEL_CASE(1)
    MK_SEL_CASE(2)
    MK_SEL_CASE(4)
    MK_SEL_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef MK_SEL_CASE
  return cudaGetLastError();
}

}  // namespace mk
