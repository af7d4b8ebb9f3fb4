// Append + compress: rotate new K/V vectors into the head's basis, keep sink
// and window tokens dense, and compress each token that leaves the window
// into its middle block's packed page (per-vector top-r) while updating the
// block's min/max keys.
//
// Method: "MosaicKV：...阅读笔记" (zhongzhuzhou.org), Eq. (7)/(8) for the
// rotation of each new token, Eq. (9) and Algorithm 1 for the per-vector
// top-r selection; "MosaicKV: Serving Long-Context LLM with Dynamic Two-D KV
// Cache Compression" (paperlayer.ai), sec. 4.2 stage 1 and sec. 5.1 (packed
// contiguous storage) and sec. 5.2 (prefill encoding of K, V and block keys).
#include "mk_append_body.cuh"

namespace mk {

__global__ void k_init_desc(Layout L, int layer, int seq, UnitDesc d) {
  const int kvh = threadIdx.x;
  if (kvh < L.n_kv) L.desc[unit_index(L, layer, seq, kvh)] = d;
}

// Decode-path append: one CTA per (sequence, kv head).  Evicts the tokens
// that leave the window into the middle, then rotates and stores the (few)
// new tokens.  Reads and advances the device-resident length, so a captured
// CUDA graph of it stays valid across replays.
__global__ void __launch_bounds__(256) k_append_small(Layout L, int layer, CallSeqs cs,
                                                      const uint16_t* __restrict__ kin,
                                                      const uint16_t* __restrict__ vin, int evict_only) {
  const int ci = blockIdx.x / L.n_kv;
  const int kvh = blockIdx.x - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int n = cs.n_new[ci];
  const int tid = threadIdx.x;
  const int64_t u = unit_index(L, layer, seq, kvh);
  __shared__ UnitDesc ud;
  __shared__ float xs[kSmallAppend][2][D];
  __shared__ __align__(16) uint16_t rot[kSmallAppend][2][D];
  __shared__ int s_abort;
  char* base = unit_base(L, u);
  // Stage R_k^T and R_v^T (contiguous in the unit, written only by
  // mk_set_rotation) while the previous kernel finishes and the eviction runs.
  extern __shared__ __align__(16) float Rs[];   // [2][128*128] when rotating
  if (!evict_only && n > 0 && n <= kSmallAppend) {
    const float4* src = reinterpret_cast<const float4*>(base + L.off_rkt);
    for (int i = tid; i < 2 * D * D / 4; i += blockDim.x) cp_async16(reinterpret_cast<float4*>(Rs) + i, src + i);
    cp_async_commit();
  }
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    s_abort = has_error(L);
    ud = L.desc[u];
  }
  __syncthreads();
  const int T_old = ud.T;
  const int T_new = T_old + n;
  if (s_abort || T_new > L.cap_tokens || (!evict_only && n > kSmallAppend)) {
    if (!s_abort && tid == 0) set_error(L, ERR_CAPACITY, (int32_t)u, T_new);
    cp_async_wait_all();
    return;
  }
  if (evict_only) {
    // Evictions only (the bulk path rotates the new tokens).
    append_small_body(L, ud, base, T_old, n, 0, kin, vin, 0, nullptr, nullptr, nullptr);
    if (tid == 0) L.desc[u].T = T_new;
    cp_async_wait_all();
    return;
  }
  const int64_t in_stride = (int64_t)L.n_kv * D;
  const int64_t row0 = (int64_t)cs.row_off[ci] * in_stride + (int64_t)kvh * D;
  append_small_body(L, ud, base, T_old, n, n, kin + row0, vin + row0, in_stride, Rs, &xs[0][0][0], &rot[0][0][0]);
  if (tid == 0) L.desc[u].T = T_new;
}

// Bulk append of new tokens (prefill): tiles of up to 128 positions aligned so
// that every middle block sits in one tile, one CTA per (tile, kv head).
// The rotation of the tile is a dense GEMM on the 5th-generation tensor
// cores: D[128 tok x 128 ch] = X[128 x 128] R^T with X the tile's bf16 keys
// (values) and R split exactly into three bf16 parts (pre-split in the unit
// at mk_set_rotation), 24 tcgen05.mma (3 parts x 8 k-steps of 16) per
// tensor accumulating in fp32 in tensor memory.  Every product is exact and
// the sum is fp32, as in the per-token path.  The epilogue rounds the
// accumulators to bf16 rows in shared memory, where one warp per token does
// the top-r selection and packing, and the block min/max follow.
namespace {
constexpr int kRotRow = D + 8;                                  // padded bf16 row of the rotated tile
constexpr int kBulkXBytes = kTileTokens * D * 2;                // 32 KB tensor-core A tile
constexpr int kBulkRBytes = 3 * D * D * 2;                      // 96 KB: the three parts of R
constexpr int kBulkRotBytes = 2 * kTileTokens * kRotRow * 2;    // rotated K and V rows
constexpr int kBulkSmem = kBulkXBytes + kBulkRBytes + kBulkRotBytes + kTileTokens * 32;
constexpr uint32_t kBulkIdesc = umma_idesc_bf16(128, 128);
}  // namespace

__global__ void __launch_bounds__(256) k_append_bulk(Layout L, int layer, CallSeqs cs,
                                                     const uint16_t* __restrict__ kin,
                                                     const uint16_t* __restrict__ vin) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* Xs = smem;                                     // A: tile rows, K-major core matrices
  unsigned char* Rp = smem + kBulkXBytes;                       // B: three parts of R
  uint16_t* rot = reinterpret_cast<uint16_t*>(Rp + kBulkRBytes);  // [2][128][kRotRow]
  uint8_t* keepk = reinterpret_cast<uint8_t*>(rot + 2 * kTileTokens * kRotRow);  // [128][32] nibbles
  __shared__ UnitDesc ud;
  __shared__ int s_ci, s_abort, s_fail;
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t bar_copy, bar_mma;

  const int tile = blockIdx.x, kvh = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    int lo = 0, hi = cs.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cs.tile_off[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    s_ci = lo;
    s_abort = has_error(L);
    s_fail = 0;
    ud = L.desc[unit_index(L, layer, cs.seq[lo], kvh)];
    mbar_init(&bar_copy, 1);
    mbar_init(&bar_mma, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (s_abort) return;
  const int ci = s_ci;
  const int seq = cs.seq[ci];
  const int64_t u = unit_index(L, layer, seq, kvh);
  const int T_old = cs.T_old[ci], T_new = T_old + cs.n_new[ci];
  const int S = L.S, W = L.W, B = L.B;
  const int j = tile - cs.tile_off[ci];
  const int f = tile_first_boundary(T_old, S);
  const int lo = j == 0 ? T_old : f + (j - 1) * kTileTokens;
  const int hi = min(T_new, j == 0 ? f : lo + kTileTokens);
  const int nt = hi - lo;
  if (nt <= 0) return;
  char* base = unit_base(L, u);
  const int64_t in_stride = (int64_t)L.n_kv * D;
  const int64_t row0 = cs.row_off[ci] + (lo - T_old);

  if (warp == 0) tmem_alloc(&s_tmem, 256);  // K accumulators in columns 0-127, V in 128-255
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = s_tmem;

  for (int w = 0; w < 2; ++w) {
    // R parts: one bulk copy (contiguous, already in operand layout).
    if (tid == 0) {
      fence_proxy_async();
      mbar_expect_tx(&bar_copy, kBulkRBytes);
      bulk_g2s(Rp, base + (w == 0 ? L.off_rkp : L.off_rvp), kBulkRBytes, &bar_copy);
    }
    // X: the tile's rows, 16 bytes (8 channels) per load, into core matrices;
    // rows past the tile's tokens are zero.
    const uint16_t* src = (w == 0 ? kin : vin) + (int64_t)kvh * D;
    for (int i = tid; i < kTileTokens * (D / 8); i += blockDim.x) {
      const int t = i >> 4, c8 = i & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < nt) v = *reinterpret_cast<const uint4*>(src + (row0 + t) * in_stride + c8 * 8);
      *reinterpret_cast<uint4*>(Xs + umma_kmajor_offset(t, c8 * 8)) = v;
    }
    fence_proxy_async();
    __syncthreads();
    if (!mbar_wait(&bar_copy, (unsigned)w)) {
      if (tid == 0) s_fail = 1;
    }
    __syncthreads();
    if (s_fail) break;
    if (tid == 0) {
      tmem_fence_after_sync();
      for (int p = 0; p < 3; ++p)
        for (int kk = 0; kk < D / 16; ++kk)
          umma_bf16(tmem + (uint32_t)(w * 128), umma_desc(Xs + kk * 256, 128, 2048),
                    umma_desc(Rp + p * D * D * 2 + kk * 256, 128, 2048), kBulkIdesc, p > 0 || kk > 0);
      umma_commit(&bar_mma);
    }
    // The next tensor's X and R overwrite the operands: wait for the MMAs.
    if (!mbar_wait(&bar_mma, (unsigned)w)) {
      if (tid == 0) s_fail = 1;
    }
    tmem_fence_after_sync();
    __syncthreads();
    if (s_fail) break;
  }
  if (s_fail) {
    // A copy or the MMAs did not complete in time: report it, give the
    // hardware another bounded wait, free the tensor memory and stop.
    if (tid == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, -3, (int32_t)MK_ETIMEOUT);
    (void)mbar_wait(&bar_copy, 0);
    (void)mbar_wait(&bar_mma, 0);
    tmem_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
    return;
  }

  // Epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (tokens), columns of
  // half w / 4, rounds to bf16 and stores the rows.
  {
    const int q = warp & 3, h = warp >> 2;
    const int t = 32 * q + lane;
    for (int w = 0; w < 2; ++w)
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        const int col = h * 64 + c * 32;
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(w * 128 + col), v);
        uint4* dst = reinterpret_cast<uint4*>(rot + ((size_t)w * kTileTokens + t) * kRotRow + col);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = (uint32_t)f2bf(__uint_as_float(v[8 * g + 2 * e])) |
                    ((uint32_t)f2bf(__uint_as_float(v[8 * g + 2 * e + 1])) << 16);
          dst[g] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);

  uint16_t* sink_k = reinterpret_cast<uint16_t*>(base + L.off_sink_k);
  uint16_t* sink_v = reinterpret_cast<uint16_t*>(base + L.off_sink_v);
  uint16_t* win_k = reinterpret_cast<uint16_t*>(base + L.off_win_k);
  uint16_t* win_v = reinterpret_cast<uint16_t*>(base + L.off_win_v);
  // One token: dense (sink or window) or compressed.
  auto one_token = [&](int t) {
    const int p = lo + t;
    const uint16_t* rk = rot + (size_t)t * kRotRow;
    const uint16_t* rv = rot + (size_t)(kTileTokens + t) * kRotRow;
    if (p < S || p >= T_new - W) {
      uint16_t* dk = p < S ? sink_k + (int64_t)p * D : win_k + (int64_t)((p - S) % W) * D;
      uint16_t* dv = p < S ? sink_v + (int64_t)p * D : win_v + (int64_t)((p - S) % W) * D;
      reinterpret_cast<uint2*>(dk)[lane] = reinterpret_cast<const uint2*>(rk)[lane];
      reinterpret_cast<uint2*>(dv)[lane] = reinterpret_cast<const uint2*>(rv)[lane];
    } else {
      keepk[t * 32 + lane] = (uint8_t)compress_kv(L, ud, base, p, rk, rv, lane);
    }
  };
  // Warp w takes tokens w, w + 8, ...; two middle tokens at a time share their
  // top-r searches' reductions (four searches per chain).
  const auto middle = [&](int t) { const int p = lo + t; return p >= S && p < T_new - W; };
  for (int t = warp; t < nt; t += 16) {
    const int t2 = t + 8;
    if (t2 < nt && middle(t) && middle(t2)) {
      unsigned ka, kb;
      compress_kv2(L, ud, base, lo + t, lo + t2, rot + (size_t)t * kRotRow, rot + (size_t)(kTileTokens + t) * kRotRow,
                   rot + (size_t)t2 * kRotRow, rot + (size_t)(kTileTokens + t2) * kRotRow, lane, ka, kb);
      keepk[t * 32 + lane] = (uint8_t)ka;
      keepk[t2 * 32 + lane] = (uint8_t)kb;
    } else {
      one_token(t);
      if (t2 < nt) one_token(t2);
    }
  }
  __syncthreads();

  // Block min/max over the zero-filled compressed keys of this tile's middle tokens.
  const int mlo = max(lo, S), mhi = min(hi, T_new - W);
  if (mlo < mhi && tid < D) {
    const int c = tid;
    uint16_t* meta = reinterpret_cast<uint16_t*>(base + L.off_meta);
    const int b0 = (mlo - S) / B, b1 = (mhi - 1 - S) / B;
    for (int b = b0; b <= b1; ++b) {
      const int blo = S + b * B;
      const int st = max(blo, mlo), en = min(blo + B, mhi);
      float mn = 0.f, mx = 0.f;
      bool have = st > blo;
      if (have) {
        mn = bf2f(meta[(int64_t)b * 2 * D + c]);
        mx = bf2f(meta[(int64_t)b * 2 * D + D + c]);
      }
      for (int p = st; p < en; ++p) {
        const int t = p - lo;
        const bool kept = (keepk[t * 32 + (c >> 2)] >> (c & 3)) & 1;
        const float kt = kept ? bf2f(rot[(size_t)t * kRotRow + c]) : 0.0f;
        if (!have) { mn = kt; mx = kt; have = true; }
        else { mn = fminf(mn, kt); mx = fmaxf(mx, kt); }
      }
      meta[(int64_t)b * 2 * D + c] = f2bf(mn);
      meta[(int64_t)b * 2 * D + D + c] = f2bf(mx);
      if (L.meta_c > 0) {  // the rows for the compressed keys, over the (now free) A tile
        uint16_t* bm = reinterpret_cast<uint16_t*>(Xs) + (b - b0) * 2 * D;
        bm[c] = f2bf(mn);
        bm[D + c] = f2bf(mx);
      }
    }
  }
  if (L.meta_c > 0 && mlo < mhi) {
    __syncthreads();
    const int b0 = (mlo - S) / B, b1 = (mhi - 1 - S) / B;
    for (int b = b0 + warp; b <= b1; b += 8) {
      const uint16_t* bm = reinterpret_cast<const uint16_t*>(Xs) + (b - b0) * 2 * D;
      uint16_t mn[4], mx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mn[i] = bm[4 * lane + i];
        mx[i] = bm[D + 4 * lane + i];
      }
      compress_key_row(L, base, b, mn, mx, lane);
    }
  }
}

// A segment's channel count and truncation after a swap of its pages
// (double-buffered re-compression); the flags keep the always bit.
__global__ void k_set_segment(Layout L, int64_t u, int seg, int r, int keep) {
  if (threadIdx.x == 0) {
    L.desc[u].r[seg] = r;
    L.desc[u].sflags[seg] = (L.desc[u].sflags[seg] & 1) | (keep << 8);
  }
}

cudaError_t launch_set_segment(const Layout& L, int64_t u, int seg, int r, int keep, cudaStream_t s) {
  k_set_segment<<<1, 32, 0, s>>>(L, u, seg, r, keep);
  return cudaGetLastError();
}

cudaError_t launch_init_desc(const Layout& L, int layer, int seq, const UnitDesc& d, cudaStream_t s) {
  k_init_desc<<<1, 32 * ((L.n_kv + 31) / 32), 0, s>>>(L, layer, seq, d);
  return cudaGetLastError();
}

cudaError_t launch_append_small(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* k,
                                const uint16_t* v, int evict_only, cudaStream_t s) {
  const size_t smem = evict_only ? 0 : (size_t)2 * D * D * sizeof(float);
  cudaError_t e = kernel_smem_attr((const void*)k_append_small, 2 * D * D * (int)sizeof(float), 256, nullptr,
                                   nullptr);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_append_small, dim3(cs.n * L.n_kv), dim3(256), smem, s, 0, L, layer, cs, k, v, evict_only);
}

cudaError_t launch_append_bulk(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* k,
                               const uint16_t* v, int total_tiles, cudaStream_t s) {
  cudaError_t e = kernel_smem_attr((const void*)k_append_bulk, kBulkSmem, 256, nullptr, nullptr);
  if (e != cudaSuccess) return e;
  dim3 grid(total_tiles, L.n_kv);
  k_append_bulk<<<grid, 256, kBulkSmem, s>>>(L, layer, cs, k, v);
  return cudaGetLastError();
}

}  // namespace mk
