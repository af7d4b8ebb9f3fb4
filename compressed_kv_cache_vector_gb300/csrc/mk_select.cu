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
//  * Each score is written as an order-preserving 32-bit key (0 for blocks of
//    always-attended segments, which are not candidates) and counted in a
//    4096-bin histogram of the keys' top 12 bits, kept in shared memory and
//    added to the unit's histogram in global memory when the CTA is done.
//  * The last CTA of each (sequence, kv head) to finish (atomic counter, no
//    waiting) selects the top k.  It stages the histogram and all keys with
//    one bulk copy each (a single SM moves them far faster that way than with
//    16-byte requests); the histogram gives the coarse bin of the k-th
//    largest key, two 1024-bin passes over the keys inside it give the exact
//    threshold, and the ids are written in ascending order from per-thread
//    bit masks and one block scan.  Every loop does the same work on every
//    thread (no per-key serial chains), because a single CTA of 8 warps runs
//    it and its time is latency, not bandwidth.
#include <algorithm>

#include "mk_append_body.cuh"

namespace mk {

namespace {
constexpr int kSelWarps = 8;
constexpr int kMT = 16;                       // blocks per MMA tile
constexpr int kMetaRow = 2 * D + 8;           // padded bf16 row (528 bytes): ldmatrix conflict-free
constexpr int kMetaTile = kMT * kMetaRow * 2; // bytes per staged tile
constexpr int kSelSmem = kSelWarps * 2 * kMetaTile;  // double-buffered tiles (also holds R_k^T)
constexpr int kSelSmemMax = 192 * 1024;              // dynamic shared memory cap (top-k key staging)
constexpr int kFineBins = 1024;
static_assert(kSelSmem >= 2 * D * D * 4 + 2 * D * 4 + 2 * D * 2, "R_k^T, R_v^T and the append scratch fit in the tile area");

// Top-k plan for nblk keys: each thread owns CPT 16-byte chunks (4 keys),
// CPT a multiple of 8; the keys are staged in shared memory when they fit
// beside the two per-thread mask arrays (else read from global memory).
__host__ __device__ inline int topk_cpt(int nblk) {
  const int nch = (nblk + 3) >> 2;
  return ((nch + 255) / 256 + 7) & ~7;
}
__host__ __device__ inline int64_t topk_mask_bytes(int cpt) { return (int64_t)256 * cpt; }

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

// Exclusive prefix sums of two per-thread counts over the CTA (256 threads).
__device__ __forceinline__ int2 block_excl_scan2(int a, int b, int2* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int xa = a, xb = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(FULL, xa, o), yb = __shfl_up_sync(FULL, xb, o);
    if (lane >= o) {
      xa += ya;
      xb += yb;
    }
  }
  if (lane == 31) wsum[warp] = make_int2(xa, xb);
  __syncthreads();
  int pa = 0, pb = 0;
  for (int w = 0; w < warp; ++w) {
    pa += wsum[w].x;
    pb += wsum[w].y;
  }
  __syncthreads();
  return make_int2(pa + xa - a, pb + xb - b);
}

// Histogram h of NB bins, bin index increasing with the key: find the bin
// holding the rem-th largest key.  Thread t reads the t-th slice of NB/256
// bins from the top; the thread whose slice holds it writes the bin and the
// rank of the key inside the bin.  Ends with a barrier.
template <int NB>
__device__ __forceinline__ void find_bin(const uint32_t* h, int rem, int2* wsum, int* s_bin, int* s_rem) {
  constexpr int PER = NB / 256;
  static_assert(PER % 4 == 0, "slices of whole 16-byte words");
  const int t = threadIdx.x;
  const uint4* hv = reinterpret_cast<const uint4*>(h + NB - PER * (t + 1));
  uint32_t v[PER];
#pragma unroll
  for (int i = 0; i < PER / 4; ++i) {
    const uint4 x = hv[i];
    v[4 * i] = x.x;
    v[4 * i + 1] = x.y;
    v[4 * i + 2] = x.z;
    v[4 * i + 3] = x.w;
  }
  int c = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) c += (int)v[i];
  const int ex = block_excl_scan2(c, 0, wsum).x;
  if (ex < rem && ex + c >= rem) {
    int acc = ex;
#pragma unroll
    for (int i = PER - 1; i >= 0; --i) {
      const int hb = (int)v[i];
      if (acc < rem && acc + hb >= rem) {
        *s_bin = NB - PER * (t + 1) + i;
        *s_rem = rem - acc;
      }
      acc += hb;
    }
  }
  __syncthreads();
}

// Top-k over the staged keys for nch <= 256 * kRoundsMax chunks of 4 keys:
// thread tid takes chunks j * 256 + tid (round j), so the block's key order
// is (j, tid) and every load of a round is conflict free.  The code runs once
// per launch on its SM, where each instruction not yet in the instruction
// cache costs a fetch, so every pass is a short loop.  sc: 1024 words of
// shared scratch.
//  * Threshold: the coarse bin of the histogram brackets it; counting passes
//    (interpolated in count space, with a bisection step whenever one shrank
//    the bracket by less than half) narrow the bracket until it holds at most
//    256 keys, which are then ranked exactly.
//  * Output: per round, a block's key above the threshold goes to position
//    (keys above it before it) + min(ties before it, need); a tie is taken
//    when fewer than `need` ties precede it.  The counts before a key come
//    from per-round per-warp totals and a warp scan of packed counts.
constexpr int kRoundsMax = 16;
constexpr int SC_CNT = 0, SC_G = 16, SC_GN = 276, SC_THR = 277, SC_WT = 280, SC_BT = 280 + 8 * kRoundsMax;  // SC_G: 256 keys + 4 pad
static_assert(SC_BT + 8 * kRoundsMax <= 1024, "scratch");
__device__ void topk_loop(const uint4* ks, int nch, int nblk, int k, bool all, const uint32_t* hc, uint32_t* sc,
                          int2* wsum, int* s_bin, int* s_rem, int32_t* out, int k_max) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rounds = (nch + 255) >> 8;
  // This thread's chunk of round j, keys past nblk zero.
  auto chunk = [&](int j) -> uint4 {
    const int c = j * 256 + tid;
    uint4 v = c < nch ? ks[c] : make_uint4(0, 0, 0, 0);
    if (4 * c + 1 >= nblk) v.y = 0u;
    if (4 * c + 2 >= nblk) v.z = 0u;
    if (4 * c + 3 >= nblk) v.w = 0u;
    return v;
  };
  int par = 0;
  // Block-wide number of keys >= x (one barrier; the two count slots alternate).
  auto cge = [&](uint64_t x) -> int {
    int c = 0;
    if (x <= 0xffffffffull) {
      const uint32_t xx = (uint32_t)x;
#pragma unroll 4
      for (int j = 0; j < rounds; ++j) {
        const uint4 v = chunk(j);
        c += (v.x >= xx) + (v.y >= xx) + (v.z >= xx) + (v.w >= xx);
      }
    }
    c = (int)__reduce_add_sync(FULL, (unsigned)c);
    if (lane == 0) sc[SC_CNT + par * 8 + warp] = (uint32_t)c;
    __syncthreads();
    const uint4 c0 = *reinterpret_cast<const uint4*>(sc + SC_CNT + par * 8);
    const uint4 c1 = *reinterpret_cast<const uint4*>(sc + SC_CNT + par * 8 + 4);
    par ^= 1;
    return (int)((c0.x + c0.y) + (c0.z + c0.w) + (c1.x + c1.y) + (c1.z + c1.w));
  };

  uint32_t thr = 1u;  // every candidate (key >= 1) when all are taken
  int need = 0;
  if (!all) {
    find_bin<kKeyBins>(hc, k, wsum, s_bin, s_rem);
    const uint64_t b = (uint64_t)*s_bin;
    uint64_t lo = b << 20 ? b << 20 : 1ull, hi = (b << 20) | 0xfffffull;
    int c_hi = k - *s_rem;             // keys above hi
    int c_lo = c_hi + (int)hc[b];      // keys >= lo
    bool bisect = false;
    while (lo < hi && c_lo - c_hi > 64) {
      uint64_t x;
      if (bisect) {
        x = lo + (hi - lo + 1) / 2;
      } else {
        // cge falls from c_lo at lo to c_hi at hi + 1; aim where it crosses k
        // (fp32: the step only needs to be roughly right).
        const float f = __fdividef((float)(k - c_hi), (float)(c_lo - c_hi));
        const uint64_t d = (uint64_t)(f * (float)(hi + 1 - lo));
        x = hi + 1 - d;
        x = x < lo + 1 ? lo + 1 : (x > hi ? hi : x);
      }
      const uint64_t w0 = hi - lo;
      const int c = cge(x);
      if (c >= k) {
        lo = x;
        c_lo = c;
      } else {
        hi = x - 1;
        c_hi = c;
      }
      bisect = !bisect && (hi - lo) > w0 / 2;
    }
    if (lo < hi) {
      // At most 64 keys lie in [lo, hi]: gather and rank them.
      if (tid == 0) sc[SC_GN] = 0u;
      __syncthreads();
#pragma unroll 1
      for (int j = 0; j < rounds; ++j) {
        const uint4 v = chunk(j);
        const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const bool in = e[q] >= lo && e[q] <= hi;
          const unsigned bal = __ballot_sync(FULL, in);
          if (bal) {
            unsigned pos = 0u;
            if (lane == 0) pos = atomicAdd(&sc[SC_GN], (unsigned)__popc(bal));
            pos = __shfl_sync(FULL, pos, 0) + (unsigned)__popc(bal & ((1u << lane) - 1u));
            if (in) sc[SC_G + pos] = e[q];
          }
        }
      }
      __syncthreads();
      const int m = (int)sc[SC_GN];
      if (tid < 3) sc[SC_G + m + tid] = 0u;  // pad to whole 16-byte words (0 is never a candidate key)
      __syncthreads();
      const int want = k - c_hi;  // rank of the threshold among them (1 = largest)
      if (tid < m) {
        const uint32_t key = sc[SC_G + tid];
        int gt = 0, eq = 0;
#pragma unroll 2
        for (int i = 0; i < m; i += 4) {
          const uint4 o = *reinterpret_cast<const uint4*>(sc + SC_G + i);
          gt += (o.x > key) + (o.y > key) + (o.z > key) + (o.w > key);
          eq += (o.x == key) + (o.y == key) + (o.z == key) + (o.w == key);
        }
        if (gt < want && gt + eq >= want) sc[SC_THR] = key;
      }
      __syncthreads();
      lo = sc[SC_THR];
    }
    thr = (uint32_t)lo;
    need = k - cge((uint64_t)thr + 1);  // ties to take
  }

  // Keys above thr (all candidates when every one is taken) and ties of one
  // chunk, as 4-bit masks.
  auto masks = [&](int j, uint32_t& gm, uint32_t& em) {
    const uint4 v = chunk(j);
    const uint32_t e[4] = {v.x, v.y, v.z, v.w};
    gm = 0u;
    em = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      gm |= (all ? e[q] != 0u : e[q] > thr) ? 1u << q : 0u;
      em |= (!all && e[q] == thr) ? 1u << q : 0u;
    }
  };
  // Per round: warp totals of (above, ties), packed as above | ties << 16.
#pragma unroll 4
  for (int j = 0; j < rounds; ++j) {
    uint32_t gm, em;
    masks(j, gm, em);
    const unsigned t = __reduce_add_sync(FULL, (unsigned)__popc(gm) | ((unsigned)__popc(em) << 16));
    if (lane == 0) sc[SC_WT + j * 8 + warp] = t;
  }
  __syncthreads();
  // Base of (round j, warp w) = exclusive scan of the totals in (j, w) order
  // (at most 128 of them: threads 0-127, warp scans, then earlier warps' sums).
  uint32_t wv = 0u, winc = 0u;
  if (warp < 4) {
    wv = tid < rounds * 8 ? sc[SC_WT + tid] : 0u;
    winc = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, winc, o);
      if (lane >= o) winc += y;
    }
    if (lane == 31) sc[SC_CNT + warp] = winc;  // the count slots are free now
  }
  __syncthreads();
  if (tid < rounds * 8) {
    uint32_t add = 0u;
#pragma unroll 1
    for (int w = 0; w < warp; ++w) add += sc[SC_CNT + w];
    sc[SC_BT + tid] = add + winc - wv;
  }
  __syncthreads();
#pragma unroll 1
  for (int j = 0; j < rounds; ++j) {
    uint32_t gm, em;
    masks(j, gm, em);
    const uint32_t own = (uint32_t)__popc(gm) | ((uint32_t)__popc(em) << 16);
    uint32_t inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += y;
    }
    const uint32_t before = sc[SC_BT + j * 8 + warp] + inc - own;
    const int g_before = (int)(before & 0xffffu), e_before = (int)(before >> 16);
    // ties this chunk takes: those still below `need`
    const int take_eq = max(0, min(__popc(em), need - e_before));
    uint32_t tm = em;
    while (__popc(tm) > take_eq) tm &= ~(1u << (31 - __clz(tm)));  // keep the lowest ids
    const uint32_t take = gm | tm;
    const int p0 = g_before + min(e_before, need);
    const int c = j * 256 + tid;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int p = p0 + __popc(take & ((1u << q) - 1u));
      if (((take >> q) & 1u) && p < k_max) out[p] = 4 * c + q;
    }
  }
}

}  // namespace

// grid: P CTAs per (sequence, kv head) of the call; 256 threads.
// With APPEND, the kernel first appends one new token per sequence (the
// decode step's append, fused): CTA 0 of each unit evicts the window token
// that leaves the window, rotates and stores the new one, and scores the
// unit's last tiles afterwards (the evicted token lands in the last block);
// the last CTA of the unit advances the device length.  kin/vin:
// [n_seqs][n_kv][128] bf16.
template <int G, bool APPEND>
__global__ void __launch_bounds__(256, 1) k_select(Layout L, int layer, CallSeqs cs, int P,
                                                   const uint16_t* __restrict__ q, int32_t* __restrict__ ids,
                                                   int32_t* __restrict__ n_sel, float* __restrict__ scores_out,
                                                   int dyn_bytes, const uint16_t* __restrict__ kin,
                                                   const uint16_t* __restrict__ vin) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float qs[G][D];
  __shared__ float qr[2][G][D];
  __shared__ UnitDesc ud;
  __shared__ __align__(16) uint32_t hc[kKeyBins];   // coarse key histogram
  __shared__ __align__(16) uint32_t hf[kFineBins];  // fine histogram of the threshold search
  __shared__ int2 wsum[kSelWarps];
  __shared__ int s_abort, s_last, s_bin, s_rem;
  __shared__ uint64_t s_bar;  // top-k staging barrier

  const int unit_call = blockIdx.x / P, part = blockIdx.x - unit_call * P;
  const int ci = unit_call / L.n_kv, kvh = unit_call - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t u = unit_index(L, layer, seq, kvh);
  const int64_t slot = (int64_t)seq * L.n_kv + kvh;
  for (int i = tid; i < G * D; i += blockDim.x)
    qs[i / D][i % D] = bf2f(q[((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D + i]);
  for (int i = tid; i < kKeyBins / 4; i += blockDim.x) reinterpret_cast<uint4*>(hc)[i] = make_uint4(0, 0, 0, 0);
  const char* base = unit_base(L, u);
  {
    // R_k^T (and, for the appending CTA, R_v^T right after it in the unit).
    const int nmat = (APPEND && part == 0) ? 2 : 1;
    const float4* src = reinterpret_cast<const float4*>(base + L.off_rkt);
    for (int i = tid; i < nmat * D * D / 4; i += blockDim.x) cp_async16(reinterpret_cast<float4*>(smem) + i, src + i);
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
    for (int hf2 = 0; hf2 < 2; ++hf2) {
      uint16_t e0[3] = {0, 0, 0}, e1[3] = {0, 0, 0};
      if (g < G) {
        const int k = kc * 16 + hf2 * 8 + 2 * tig;
        const float x0 = k < D ? fminf(qr[0][g][k], 0.0f) : fmaxf(qr[0][g][k - D], 0.0f);
        const float x1 = (k + 1) < D ? fminf(qr[0][g][k + 1], 0.0f) : fmaxf(qr[0][g][k + 1 - D], 0.0f);
        split3(x0, e0);
        split3(x1, e1);
      }
#pragma unroll
      for (int s = 0; s < 3; ++s) bq[s][kc][hf2] = (uint32_t)e0[s] | ((uint32_t)e1[s] << 16);
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

  int T_cur = ud.T;
  if (APPEND) {
    const int n = cs.n_new[ci];
    if (T_cur + n > L.cap_tokens) {
      if (part == 0 && tid == 0) set_error(L, ERR_CAPACITY, (int32_t)u, T_cur + n);
      return;
    }
    if (part == 0) {
      const int64_t in_stride = (int64_t)L.n_kv * D;
      const int64_t row0 = (int64_t)cs.row_off[ci] * in_stride + (int64_t)kvh * D;
      float* xs = reinterpret_cast<float*>(smem + 2 * D * D * 4);
      uint16_t* rot = reinterpret_cast<uint16_t*>(xs + n * 2 * D);
      append_small_body(L, ud, const_cast<char*>(base), T_cur, n, n, kin + row0, vin + row0, in_stride,
                        reinterpret_cast<const float*>(smem), xs, rot);
      __threadfence();  // the updated block min/max before this CTA's own tiles are read
    }
    T_cur += n;
  }
  const int nblk = n_mid_blocks(L, T_cur);
  const int ntiles = (nblk + kMT - 1) / kMT;
  const int tper = (ntiles + P - 1) / P;
  // With APPEND, CTA 0 takes the last tiles (after its own append).
  const int t1 = APPEND ? max(0, ntiles - part * tper) : min(ntiles, part * tper + tper);
  const int t0 = APPEND ? max(0, t1 - tper) : part * tper;
  const uint16_t* meta = reinterpret_cast<const uint16_t*>(base + L.off_meta);
  uint32_t* kw = L.keys + slot * L.keys_stride;
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
  // Write block b's score: the user's fp32 copy, the key, the histogram count.
  auto emit = [&](int b, float sc) {
    if (so) so[b] = sc;
    const uint32_t key = ud.always[seg_of_block(ud, b)] ? 0u : ordered_key(sc);
    kw[b] = key;
    if (key) atomicAdd(&hc[key >> 20], 1u);
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
      if (b0 < nblk) emit(b0, b_lo * inv_sqrt_d);
      if (b1 < nblk) emit(b1, b_hi * inv_sqrt_d);
    }
    __syncwarp();
    st ^= 1;
  }
  cp_async_wait_all();
  __syncthreads();
  // Add this CTA's histogram to the unit's.
  uint32_t* gh = L.khist + slot * kKeyBins;
  for (int i = tid; i < kKeyBins / 4; i += blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(hc)[i];
    if (v.x) atomicAdd(gh + 4 * i, v.x);
    if (v.y) atomicAdd(gh + 4 * i + 1, v.y);
    if (v.z) atomicAdd(gh + 4 * i + 2, v.z);
    if (v.w) atomicAdd(gh + 4 * i + 3, v.w);
  }

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
  if (APPEND && tid == 0) L.desc[u].T = T_cur;  // every CTA of the unit has read the old length
  __threadfence();

  const int n_cand = n_scored_blocks(ud, nblk);
  const int k = n_select(L, n_cand);
  int32_t* out = ids + ((int64_t)ci * L.n_kv + kvh) * L.k_max;
  const bool all = k >= n_cand;  // every candidate is taken
  const int nch = (nblk + 3) >> 2;
  const int CPT = topk_cpt(nblk), NG = CPT >> 3;
  const int64_t kbytes = (int64_t)nch * 16;
  const bool staged = kbytes + topk_mask_bytes(CPT) <= (int64_t)dyn_bytes;
  uint4* ks = reinterpret_cast<uint4*>(smem);
  uint32_t* m_gt = reinterpret_cast<uint32_t*>(smem + (staged ? kbytes : 0));
  uint32_t* m_eq = m_gt + NG * 256;

  // The unit's coarse histogram and its keys, one bulk copy each (the scoring
  // CTAs' writes were acquired through the counter).
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    mbar_init_fence();
    fence_proxy_async_all();
    mbar_expect_tx(&s_bar, (unsigned)(kKeyBins * 4 + (staged ? kbytes : 0)));
    bulk_g2s(hc, gh, kKeyBins * 4, &s_bar);
    if (staged) bulk_g2s(ks, kw, (unsigned)kbytes, &s_bar);
  }
  __syncthreads();
  if (!mbar_wait(&s_bar, 0)) {
    if (tid == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, -2, (int32_t)MK_ETIMEOUT);
    (void)mbar_wait(&s_bar, 0);
    return;
  }
  for (int i = tid; i < kKeyBins / 4; i += blockDim.x) reinterpret_cast<uint4*>(gh)[i] = make_uint4(0, 0, 0, 0);
  if (staged && nch <= 256 * kRoundsMax) {
    topk_loop(ks, nch, nblk, k, all, hc, hf, wsum, &s_bin, &s_rem, out, L.k_max);
    if (tid == 0) n_sel[(int64_t)ci * L.n_kv + kvh] = k;
    return;
  }
  // Larger block counts: thread tid owns chunks tid * CPT .. + CPT - 1 (4 keys each, keys past
  // nblk read as 0).  Within each group of 8 chunks it visits chunk
  // jj ^ (tid & 7) at step jj, so the 8 threads of a quarter warp read 8
  // different 16-byte bank groups.
  auto chunk = [&](int lc) -> uint4 {
    const int c = tid * CPT + lc;
    if (c >= nch) return make_uint4(0, 0, 0, 0);
    uint4 v = staged ? ks[c] : __ldcg(reinterpret_cast<const uint4*>(kw) + c);
    const int e0 = 4 * c;
    if (e0 + 1 >= nblk) v.y = 0u;
    if (e0 + 2 >= nblk) v.z = 0u;
    if (e0 + 3 >= nblk) v.w = 0u;
    return v;
  };

  // Threshold: the coarse bin of the k-th largest key, then two passes of
  // kFineBins bins over the keys inside it (the bin spans 2^20 key values).
  uint32_t thr = 0;
  int need = 0;
  if (!all) {
    find_bin<kKeyBins>(hc, k, wsum, &s_bin, &s_rem);
    uint32_t lo = max(1u, (uint32_t)s_bin << 20), hi = ((uint32_t)s_bin << 20) | 0xfffffu;
    int rem = s_rem;
    for (int pass = 0; pass < 2 && lo != hi; ++pass) {
      const int sh = max(0, 32 - __clz(hi - lo) - 10);  // (hi - lo) >> sh < kFineBins
      for (int i = tid; i < kFineBins; i += blockDim.x) hf[i] = 0;
      __syncthreads();
      for (int gi = 0; gi < NG; ++gi) {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const uint4 v = chunk(gi * 8 + (jj ^ (tid & 7)));
          const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (e[q] - lo <= hi - lo) atomicAdd(&hf[(e[q] - lo) >> sh], 1u);
        }
      }
      __syncthreads();
      find_bin<kFineBins>(hf, rem, wsum, &s_bin, &s_rem);
      const uint32_t nlo = lo + ((uint32_t)s_bin << sh);
      const uint64_t nhi = (uint64_t)nlo + ((1ull << sh) - 1ull);
      hi = nhi < (uint64_t)hi ? (uint32_t)nhi : hi;
      lo = nlo;
      rem = s_rem;
    }
    thr = lo;
    need = rem;  // keys equal to thr that are taken, lowest block ids first
  }

  // Per 32 keys: masks of the keys above thr (all candidates when every one
  // is taken) and of the ties.
  int n_gt = 0, n_eq = 0;
  for (int gi = 0; gi < NG; ++gi) {
    uint32_t gm = 0, em = 0;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int lj = jj ^ (tid & 7);
      const uint4 v = chunk(gi * 8 + lj);
      const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t bit = 1u << (lj * 4 + q);
        if (all ? e[q] != 0u : e[q] > thr) gm |= bit;
        else if (!all && e[q] == thr) em |= bit;
      }
    }
    m_gt[gi * 256 + tid] = gm;
    m_eq[gi * 256 + tid] = em;
    n_gt += __popc(gm);
    n_eq += __popc(em);
  }
  const int2 ex = block_excl_scan2(n_gt, n_eq, wsum);

  // Ordered output: thread tid's ids follow those of threads 0..tid-1.
  int take_eq = all ? 0 : max(0, min(n_eq, need - ex.y));
  int pos = ex.x + min(ex.y, need);
  const int kbase = tid * CPT * 4;
  for (int gi = 0; gi < NG; ++gi) {
    uint32_t sel = m_gt[gi * 256 + tid];
    uint32_t em = m_eq[gi * 256 + tid];
    while (take_eq > 0 && em) {
      sel |= em & (0u - em);
      em &= em - 1;
      --take_eq;
    }
    if (sel) {
#pragma unroll
      for (int bb = 0; bb < 32; ++bb) {
        const int p = pos + __popc(sel & ((1u << bb) - 1u));
        if (((sel >> bb) & 1u) && p < L.k_max) out[p] = kbase + gi * 32 + bb;
      }
    }
    pos += __popc(sel);
  }
  if (tid == 0) n_sel[(int64_t)ci * L.n_kv + kvh] = k;
}

bool select_plan_ok(const Layout& L) {
  // Without staged keys the selection still needs its two mask arrays.
  return topk_mask_bytes(topk_cpt(std::max(1, L.nblk_cap))) <= (int64_t)kSelSmem;
}

cudaError_t launch_block_select(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* q,
                                int32_t* ids, int32_t* n_sel, float* scores_out, int max_nblk,
                                cudaStream_t s, const uint16_t* kin, const uint16_t* vin) {
  const int units = cs.n * L.n_kv;
  const int tiles = (max_nblk + kMT - 1) / kMT;
  int P = std::max(1, 152 / units);
  P = std::min(P, std::max(1, (tiles + kSelWarps - 1) / kSelWarps));
  const dim3 grid(units * P);
  // Dynamic shared memory: the meta tile stages, or the top-k's keys and
  // masks for the context's largest block count, whichever is larger (the
  // tile stages also hold R_k^T and R_v^T plus the append scratch).
  const int cpt = topk_cpt(L.nblk_cap);
  const int64_t want = (int64_t)16 * ((L.nblk_cap + 3) / 4) + topk_mask_bytes(cpt);
  const int dyn = (int)std::max<int64_t>(kSelSmem, std::min<int64_t>(kSelSmemMax, want));
  const bool append = kin != nullptr;
#define MK_SEL_CASE(GG)                                                                                       \
  case GG: {                                                                                                  \
    static int set[2] = {0, 0};                                                                               \
    auto kern = append ? k_select<GG, true> : k_select<GG, false>;                                             \
    if (set[append] < dyn) {                                                                                  \
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);           \
      if (e != cudaSuccess) return e;                                                                         \
      set[append] = dyn;                                                                                      \
    }                                                                                                         \
    return launch_pdl(kern, grid, dim3(256), dyn, s, 0, L, layer, cs, P, q, ids, n_sel, scores_out, dyn, kin, \
                      vin);                                                                                   \
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
