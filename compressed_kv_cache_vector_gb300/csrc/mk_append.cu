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
// that every middle block sits in one tile.  A work item is one tensor (keys
// or values) of one tile of one kv head; the kernel is persistent: each CTA
// takes a contiguous run of items ordered by (tensor, kv head, tile), so it
// loads that head's rotation once and streams its tiles.
//  * The rotation of a tile is a dense GEMM on the 5th-generation tensor
//    cores: D[128 tok x 128 ch] = X[128 x 128] R^T with X the tile's bf16 rows
//    and R split exactly into three bf16 parts (pre-split in the unit at
//    mk_set_rotation, one 96 KB bulk copy), 24 tcgen05.mma (3 parts x 8
//    k-steps of 16) accumulating in fp32 in tensor memory.  Every product is
//    exact and the sum is fp32, as in the per-token path.
//  * Pipeline: the next item's rows arrive by 16-byte cp.async copies into
//    the other operand buffer while the current item is compressed; its MMAs
//    are issued as soon as the current accumulators have been read out.
//  * The epilogue rounds the accumulators to bf16 rows in shared memory.
//    Each token is then compressed by a pair of threads (64 channels each)
//    without warp-wide reductions: the r-th largest magnitude is found
//    bitwise from the top, every step counting the 64 magnitudes >= the
//    candidate two at a time in 32-bit words (guard-bit subtraction), and the
//    pair adding its two counts with one shuffle.  So 16 tokens proceed
//    independently in each warp.  Key items then fold the block min/max.
namespace {
constexpr int kRotRow = D + 8;                                  // padded bf16 row of the rotated tile
constexpr int kBulkXBytes = kTileTokens * D * 2;                // 32 KB tensor-core A tile
constexpr int kBulkRBytes = 3 * D * D * 2;                      // 96 KB: the three parts of R
constexpr int kBulkRotBytes = kTileTokens * kRotRow * 2;        // one tensor's rotated rows
constexpr int kBulkKeepBytes = kTileTokens * 16;                // keep bits of the key rows
constexpr int kBulkMetaBytes = (kTileTokens / 16) * 2 * D * 2;  // block min/max rows for the compressed keys
constexpr int kStageR = 68;                                     // packed rows staged for r <= 68
constexpr int kBulkStageBytes = kTileTokens * kStageR * 3;      // values (bf16) then indices (u8)
constexpr int kBulkSmem =
    kBulkRBytes + 2 * kBulkXBytes + kBulkRotBytes + kBulkKeepBytes + kBulkMetaBytes + kBulkStageBytes;
static_assert(kBulkSmem + 1024 <= 227 * 1024, "bulk append shared memory");
constexpr uint32_t kBulkIdesc = umma_idesc_bf16(128, 128);

// One work item: tensor (0 keys, 1 values), kv head, call sequence, and the
// tile's positions [lo, hi) with its first input row.
struct BulkItem {
  int w, kvh, ci, lo, hi;
  int64_t row0;
};
__device__ __forceinline__ BulkItem bulk_item(const Layout& L, const CallSeqs& cs, int total_tiles, int it) {
  BulkItem b;
  const int per_w = L.n_kv * total_tiles;
  b.w = it / per_w;
  const int rem = it - b.w * per_w;
  b.kvh = rem / total_tiles;
  const int tile = rem - b.kvh * total_tiles;
  int lo = 0, hi = cs.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cs.tile_off[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  b.ci = lo;
  const int T_old = cs.T_old[lo], T_new = T_old + cs.n_new[lo];
  const int j = tile - cs.tile_off[lo];
  const int f = tile_first_boundary(T_old, L.S);
  b.lo = j == 0 ? T_old : f + (j - 1) * kTileTokens;
  b.hi = min(T_new, j == 0 ? f : b.lo + kTileTokens);
  b.row0 = cs.row_off[lo] + (b.lo - T_old);
  return b;
}
}  // namespace

// Grouped bitmap ([S] sec. 5.1): the energies of the 64 / GG groups of g
// adjacent channels in one thread's half row (channels 64 h ..), the fp32 sum
// of squares in channel order, as key bits (non-negative floats order as
// their bit patterns); groups from kp on count 0, slots past 64 / GG are 0.
template <int GG>
__device__ __forceinline__ void group_keys(const uint4* row4, int h, int kp, bool live, uint32_t kw[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) kw[j] = 0u;
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 x = live ? row4[j] : make_uint4(0, 0, 0, 0);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = 8 * j + e;  // channel within the half
      const float v = __uint_as_float((e & 1 ? xs[e >> 1] >> 16 : xs[e >> 1] & 0xffffu) << 16);
      const float sq = __fmul_rn(v, v);
      acc = c % GG == 0 ? sq : __fadd_rn(acc, sq);
      if (c % GG == GG - 1) kw[c / GG] = 64 * h + c - (GG - 1) < kp ? __float_as_uint(acc) : 0u;
    }
  }
}
// Channel keep bits of a half row from its kept groups (bit j: group j).
template <int GG>
__device__ __forceinline__ uint64_t spread_groups(uint64_t kg) {
  uint64_t out = 0ull;
#pragma unroll
  for (int j = 0; j < 64 / GG; ++j)
    if (kg >> j & 1ull) out |= ((GG == 64 ? ~0ull : (1ull << GG) - 1ull)) << (GG * j);
  return out;
}

// BM: bitmap pages (element group per segment); the uint8-index and uncompressed
// formats take BM = false, without the grouped search.
template <bool BM>
__global__ void __launch_bounds__(256, 1) k_append_bulk(Layout L, int layer, CallSeqs cs,
                                                     const uint16_t* __restrict__ kin,
                                                     const uint16_t* __restrict__ vin, int total_tiles,
                                                     int items_per_cta) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* Rp = smem;                                                  // B: three parts of R
  unsigned char* Xb = smem + kBulkRBytes;                                    // A: two tile buffers
  uint16_t* rot = reinterpret_cast<uint16_t*>(Xb + 2 * kBulkXBytes);        // [128][kRotRow]
  uint32_t* keepw = reinterpret_cast<uint32_t*>(rot + kTileTokens * kRotRow);  // [128][4] keep bits
  uint16_t* bm = reinterpret_cast<uint16_t*>(keepw) + kBulkKeepBytes / 2;         // [8][2][128]
  uint16_t* stv = bm + kBulkMetaBytes / 2;                                        // [128][kStageR] packed values
  uint8_t* sti = reinterpret_cast<uint8_t*>(stv + kTileTokens * kStageR);         // [128][kStageR] packed indices
  __shared__ __align__(16) UnitDesc ud;
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t bar_r, bar_mma;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_items = 2 * L.n_kv * total_tiles;
  const int it0 = blockIdx.x * items_per_cta;
  const int it1 = min(n_items, it0 + items_per_cta);
  if (it0 >= it1) return;  // whole CTA, before any barrier
  if (tid == 0) {
    s_abort = has_error(L);
    mbar_init(&bar_r, 1);
    mbar_init(&bar_mma, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&s_tmem, 128);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int S = L.S, W = L.W, B = L.B;
  const int64_t in_stride = (int64_t)L.n_kv * D;

  // The tile's rows of item b into operand buffer xb by 16-byte cp.async,
  // in the tensor cores' K-major core-matrix layout; rows past its tokens zero.
  auto load_x = [&](const BulkItem& b, unsigned char* xb) {
    const uint16_t* src = (b.w == 0 ? kin : vin) + (int64_t)b.kvh * D;
    const int nt = b.hi - b.lo;
    for (int i = tid; i < kTileTokens * (D / 8); i += blockDim.x) {
      const int t = i >> 4, c8 = i & 15;
      unsigned char* dst = xb + umma_kmajor_offset(t, c8 * 8);
      if (t < nt)
        cp_async16(dst, src + (b.row0 + t) * in_stride + c8 * 8);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  };
  // R parts of item b's tensor and head into Rp (no MMA may be reading Rp).
  unsigned r_phase = 0, mma_phase = 0;
  bool r_pending = false, mma_pending = false;
  auto r_key = [&](const BulkItem& b) { return (b.w * MK_MAX_CALL_SEQS + b.ci) * L.n_kv + b.kvh; };
  auto load_r = [&](const BulkItem& b) -> bool {
    if (tid == 0) {
      const char* ub = unit_base(L, unit_index(L, layer, cs.seq[b.ci], b.kvh));
      fence_proxy_async();
      mbar_expect_tx(&bar_r, kBulkRBytes);
      bulk_g2s(Rp, ub + (b.w == 0 ? L.off_rkp : L.off_rvp), kBulkRBytes, &bar_r);
    }
    r_pending = true;
    const bool ok = __syncthreads_and(mbar_wait(&bar_r, r_phase) ? 1 : 0) != 0;
    if (ok) {
      r_phase ^= 1u;
      r_pending = false;
    }
    return ok;
  };
  // 24 MMAs of one tile (tid 0), committed to bar_mma.
  auto issue_mma = [&](const unsigned char* xb) {
    if (tid == 0) {
      tmem_fence_after_sync();
      for (int p = 0; p < 3; ++p)
        for (int kk = 0; kk < D / 16; ++kk)
          umma_bf16(tmem, umma_desc(xb + kk * 256, 128, 2048), umma_desc(Rp + p * D * D * 2 + kk * 256, 128, 2048),
                    kBulkIdesc, p > 0 || kk > 0);
      umma_commit(&bar_mma);
    }
    mma_pending = true;
  };

  const bool aborted = s_abort != 0;  // an earlier kernel set the error word: do nothing
  bool ok = !aborted;
  BulkItem cur = bulk_item(L, cs, total_tiles, it0), nxt = cur;
  int rk = -1, xbuf = 0;
  if (ok) {
    load_x(cur, Xb);
    ok = load_r(cur);
    rk = r_key(cur);
  }
  if (ok) {
    cp_async_wait_all();
    fence_proxy_async();  // rows written by this thread, read by the tensor cores
    __syncthreads();
    issue_mma(Xb);
    if (it0 + 1 < it1) {
      nxt = bulk_item(L, cs, total_tiles, it0 + 1);
      load_x(nxt, Xb + kBulkXBytes);
    }
  }
  for (int it = it0; ok && it < it1; ++it) {
    const bool have_next = it + 1 < it1;
    // Accumulators of `cur` are complete.
    ok = __syncthreads_and(mbar_wait(&bar_mma, mma_phase) ? 1 : 0) != 0;
    if (!ok) break;
    mma_phase ^= 1u;
    mma_pending = false;
    tmem_fence_after_sync();
    const int seq = cs.seq[cur.ci];
    const int64_t u = unit_index(L, layer, seq, cur.kvh);
    if (tid == 0) ud = L.desc[u];
    // Epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (tokens), columns
    // of half w / 4, rounds to bf16 and stores the rows.
    {
      const int q = warp & 3, h = warp >> 2;
      const int t = 32 * q + lane;
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        const int col = h * 64 + c * 32;
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col, v);
        uint4* dst = reinterpret_cast<uint4*>(rot + (size_t)t * kRotRow + col);
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
    cp_async_wait_all();  // the next item's rows
    fence_proxy_async();
    __syncthreads();      // rows of `cur` complete; TMEM read out; next rows visible
    if (have_next) {
      if (r_key(nxt) != rk) {  // another tensor, head or sequence: its rotation (the last MMA is done)
        ok = load_r(nxt);
        rk = r_key(nxt);
        if (!ok) break;
      }
      issue_mma(Xb + (xbuf ^ 1) * kBulkXBytes);
    }
    BulkItem nn = nxt;
    if (it + 2 < it1) {  // the item after next, into the buffer `cur` used (its MMAs are done)
      nn = bulk_item(L, cs, total_tiles, it + 2);
      load_x(nn, Xb + xbuf * kBulkXBytes);
    }

    // Compress `cur`: the thread pair (2t, 2t + 1) takes token t, each
    // thread 64 channels (h = tid & 1: channels 64h .. 64h + 63).
    char* base = unit_base(L, u);
    const int T_new = cs.T_old[cur.ci] + cs.n_new[cur.ci];
    const int nt = cur.hi - cur.lo, lo = cur.lo, is_v = cur.w;
    const int mlo = max(lo, S), mhi = min(cur.hi, T_new - W);  // this tile's middle tokens
    const int b0 = (mlo - S) / B, b1 = mlo < mhi ? (mhi - 1 - S) / B : b0 - 1;
    {
      const int t = tid >> 1, h = tid & 1;
      const int p = lo + t;
      const bool in = t < nt;
      const bool live = in && p >= S && p < T_new - W &&
                        in_bounds(L, (p - S) / B < L.nblk_cap && p - S - b0 * B < kTileTokens, SITE_PREFILL_PAGE, p);
      const uint16_t* row = rot + (size_t)t * kRotRow + 64 * h;
      const uint4* row4 = reinterpret_cast<const uint4*>(row);
      if (in && !live) {  // sink or window: the rotated row, dense
        uint16_t* d = reinterpret_cast<uint16_t*>(base + (is_v ? L.off_sink_v : L.off_sink_k));
        if (p >= S) d = reinterpret_cast<uint16_t*>(base + (is_v ? L.off_win_v : L.off_win_k)) + (int64_t)((p - S) % W) * D;
        else d += (int64_t)p * D;
#pragma unroll
        for (int j = 0; j < 8; ++j) reinterpret_cast<uint4*>(d + 64 * h)[j] = row4[j];
      }
      const int m = live ? p - S : 0;
      const int b = m / B, tt = m - b * B;
      const int sg = seg_of_block(ud, b);
      const int r = live ? ud.r[sg] : 0, kp = seg_keep(ud, sg);
      uint32_t keep_lo = 0u, keep_hi = 0u;  // keep bits of channels 64h + 0..31 and 64h + 32..63
      if (L.dense_pages) {
        if (live) {
          uint4* d = reinterpret_cast<uint4*>(base + L.off_pages + (int64_t)b * L.page_stride +
                                              ((int64_t)(is_v * B + tt) * D + 64 * h) * 2);
#pragma unroll
          for (int j = 0; j < 8; ++j) d[j] = row4[j];
          keep_lo = keep_hi = ~0u;
        }
      } else {
        keep_lo = 0u;
        uint32_t kw[32];
        uint64_t gt = 0ull, eq = 0ull;
        const int gg = BM ? seg_group(ud, sg) : 0;
        // Threads of a pair hold the same token, so they take the same
        // branch below; with bitmap pages the warp's tokens may span two
        // segments of different group sizes, so the pair's shuffles name the
        // pair only.
        const unsigned pmask = BM ? 3u << (lane & 30) : FULL;
        int kneed = r;  // units to keep: channels, or groups of gg channels
        if (gg <= 1) {
          // 15-bit magnitudes, two per word, each under a guard bit: for a
          // candidate c, bit 15 (31) of (word - c | c << 16) is set exactly
          // when the low (high) magnitude is >= c.  Truncated channels count 0.
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 x = live ? row4[j] : make_uint4(0, 0, 0, 0);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c0 = 64 * h + 8 * j + 2 * e;
              uint32_t w = xs[e] & 0x7fff7fffu;
              if (c0 >= kp) w &= 0xffff0000u;
              if (c0 + 1 >= kp) w &= 0x0000ffffu;
              kw[4 * j + e] = w | 0x80008000u;
            }
          }
          // The r-th largest magnitude thr: the largest value with at least r
          // magnitudes >= it (bitwise from the top; the pair adds its counts).
          // The flags of 16 words (32 magnitudes) are gathered into one word
          // (word j's two flags shifted right by j) and counted by one popc.
          uint32_t thr = 0u;
#pragma unroll 1
          for (int bit = 14; bit >= 0; --bit) {
            const uint32_t cand = thr | (1u << bit);
            const uint32_t cc = cand | (cand << 16);
            int n = 0;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              uint32_t f = 0u;
#pragma unroll
              for (int j = 0; j < 16; ++j) f |= ((kw[16 * g + j] - cc) & 0x80008000u) >> j;
              n += __popc(f);
            }
            n += __shfl_xor_sync(pmask, n, 1);
            if (n >= r) thr = cand;
          }
          // Above thr: kept.  Equal to thr: the lowest channels, as many as the
          // r - #above still needed (the lower half's ties come first).
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const uint32_t lo16 = kw[j] & 0x7fffu, hi16 = (kw[j] >> 16) & 0x7fffu;
            gt |= (uint64_t)(lo16 > thr) << (2 * j) | (uint64_t)(hi16 > thr) << (2 * j + 1);
            eq |= (uint64_t)(lo16 == thr) << (2 * j) | (uint64_t)(hi16 == thr) << (2 * j + 1);
          }
        } else {
          // Grouped bitmap: the r / gg groups of largest energy, ties to the
          // lower group.  31-bit keys, one per group (ng = 64 / gg of them
          // per thread, the rest 0): the (r / gg)-th largest energy by a
          // bitwise search, each step gathering the sign bits of key - cand
          // (set when key < cand) into one word.
          if (gg == 2) group_keys<2>(row4, h, kp, live, kw);
          else if (gg == 4) group_keys<4>(row4, h, kp, live, kw);
          else group_keys<8>(row4, h, kp, live, kw);
          kneed = r / max(gg, 1);  // (gg >= 2 here; the bound keeps dead code of the uint8 instance clean)
          const int ng = 64 / max(gg, 1);
          uint32_t thr = 0u;
#pragma unroll 1
          for (int bit = 30; bit >= 0; --bit) {
            const uint32_t cand = thr | (1u << bit);
            uint32_t f = 0u;
#pragma unroll
            for (int j = 0; j < 32; ++j) f |= ((kw[j] - cand) >> 31) << j;
            int n = 32 - __popc(f);  // zero slots never reach cand >= 1
            n += __shfl_xor_sync(pmask, n, 1);
            if (n >= kneed) thr = cand;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            gt |= (uint64_t)(kw[j] > thr) << j;
            eq |= (uint64_t)(kw[j] == thr && j < ng) << j;
          }
        }
        const int n_gt = __popcll(gt), n_eq = __popcll(eq);
        const int pair_gt = n_gt + __shfl_xor_sync(FULL, n_gt, 1);
        const int eq_lower = __shfl_xor_sync(FULL, n_eq, 1);
        const int need = kneed - pair_gt - (h ? eq_lower : 0);
        int take = need < 0 ? 0 : (need > n_eq ? n_eq : need);
        while (__popcll(eq) > take) eq &= ~(1ull << (63 - __clzll(eq)));  // keep the lowest channels
        uint64_t keepg = gt | eq;  // channels, or groups of this half
        if (!live) keepg = 0ull;
        uint64_t keep = gg == 2 ? spread_groups<2>(keepg) : gg == 4 ? spread_groups<4>(keepg)
                      : gg == 8 ? spread_groups<8>(keepg) : keepg;
        keep_lo = (uint32_t)keep;
        keep_hi = (uint32_t)(keep >> 32);
        // Packed row, in channel order: thread 0 of the pair writes ranks
        // 0 .. r2 - 1 from the lowest channel up, thread 1 ranks r - 1 down to
        // r2 from the highest, so both do the same work.  Staged rows (r <=
        // kStageR) go to the block's run in shared memory, [tt][r], written
        // out below; else straight into the page.
        const uint32_t o_lo = __shfl_xor_sync(FULL, keep_lo, 1), o_hi = __shfl_xor_sync(FULL, keep_hi, 1);
        if (live) {
          const uint64_t mine = (uint64_t)keep_lo | ((uint64_t)keep_hi << 32);
          const uint64_t other = (uint64_t)o_lo | ((uint64_t)o_hi << 32);
          const uint64_t m0 = h ? other : mine, m1 = h ? mine : other;  // channels 0-63, 64-127
          const bool staged = r <= kStageR;
          char* page = base + L.off_pages + (int64_t)b * L.page_stride;
          const int pb = BM ? 16 / gg : r, Br = B * r, Bp = B * pb;  // page: [2Br][Bp][2Br][Bp]
          uint16_t* val = staged ? stv + (b - b0) * B * kStageR + tt * r
                                 : reinterpret_cast<uint16_t*>(page + (is_v ? 2 * Br + Bp : 0)) + tt * r;
          uint8_t* idx = staged ? sti + (b - b0) * B * kStageR + tt * pb
                                : reinterpret_cast<uint8_t*>(page + (is_v ? 4 * Br + Bp : 2 * Br)) + tt * pb;
          if (gg) {
            // Bitmap ([S] sec. 5.1): this half's 64 / gg bits at byte 8 h / gg.
            uint8_t* d = idx + h * (8 / max(gg, 1));
            if (gg == 1) {
              reinterpret_cast<uint32_t*>(d)[0] = keep_lo;
              reinterpret_cast<uint32_t*>(d)[1] = keep_hi;
            } else if (gg == 2) {
              *reinterpret_cast<uint32_t*>(d) = (uint32_t)keepg;
            } else if (gg == 4) {
              *reinterpret_cast<uint16_t*>(d) = (uint16_t)keepg;
            } else {
              *d = (uint8_t)keepg;
            }
          }
          const uint16_t* rowf = rot + (size_t)t * kRotRow;
          const int r2 = (r + 1) >> 1;
          if (h == 0) {
            uint64_t mm = m0;
            int cb = 0;
            for (int k = 0; k < r2; ++k) {
              if (mm == 0ull) {
                mm = m1;
                cb = 64;
              }
              const int c = cb + __ffsll((long long)mm) - 1;
              mm &= mm - 1ull;
              val[k] = rowf[c];
              if (!gg) idx[k] = (uint8_t)c;
            }
          } else {
            uint64_t mm = m1;
            int cb = 64;
            for (int k = r - 1; k >= r2; --k) {
              if (mm == 0ull) {
                mm = m0;
                cb = 0;
              }
              const int bit = 63 - __clzll((long long)mm);
              mm &= ~(1ull << bit);
              val[k] = rowf[cb + bit];
              if (!gg) idx[k] = (uint8_t)(cb + bit);
            }
          }
        }
      }
      if (!is_v && in) {
        keepw[t * 4 + 2 * h] = keep_lo;
        keepw[t * 4 + 2 * h + 1] = keep_hi;
      }
    }
    // Write the staged packed rows out, block by block: a block's new tokens
    // [st, en) own one contiguous run of values (and of indices) in the page
    // and in the staging area.  Whole blocks go out by bulk copies (16-byte
    // aligned runs of B r values and B r indices); partial ones by
    // consecutive threads.
    fence_proxy_async();  // the staged rows are read by the bulk copies
    __syncthreads();
    if (!L.dense_pages)
      for (int b = b0; b <= b1; ++b) {
        const int r = ud.r[seg_of_block(ud, b)];
        if (r > kStageR) continue;  // written directly above
        if (!in_bounds(L, b < L.nblk_cap, SITE_PREFILL_OUT, b)) continue;
        const int blo = S + b * B;
        const int st = max(blo, mlo), en = min(blo + B, mhi);
        char* page = base + L.off_pages + (int64_t)b * L.page_stride;
        const int pb = BM ? 16 / seg_group(ud, seg_of_block(ud, b)) : r, Br = B * r, Bp = B * pb;  // [2Br][Bp][2Br][Bp]
        uint16_t* val = reinterpret_cast<uint16_t*>(page + (is_v ? 2 * Br + Bp : 0)) + (st - blo) * r;
        uint8_t* idx = reinterpret_cast<uint8_t*>(page + (is_v ? 4 * Br + Bp : 2 * Br)) + (st - blo) * pb;
        const uint16_t* sv = stv + (b - b0) * B * kStageR + (st - blo) * r;
        const uint8_t* si = sti + (b - b0) * B * kStageR + (st - blo) * pb;
        const int n = (en - st) * r;
        if (st == blo && en == blo + B) {
          if (tid == 0) {
            bulk_s2g(val, sv, (unsigned)(2 * Br));
            bulk_s2g(idx, si, (unsigned)Bp);
          }
        } else if (!BM) {
          for (int i = tid; i < n; i += blockDim.x) {
            val[i] = sv[i];
            idx[i] = si[i];
          }
        } else {
          for (int i = tid; i < n; i += blockDim.x) val[i] = sv[i];
          for (int i = tid; i < (en - st) * pb; i += blockDim.x) idx[i] = si[i];
        }
      }
    if (tid == 0) {
      bulk_commit();
      bulk_wait_read();  // the staging area is reused next (block min/max, next item)
    }
    __syncthreads();
    if (!is_v) {
      // Block min/max over the zero-filled compressed keys of this tile's middle tokens.
      // Four threads per channel pair, each over a quarter of a block's new
      // tokens, with bf16x2 min/max (exact) on the zero-filled rows; the
      // quarters meet in the staging area, free once the packed rows are out.
      uint32_t* pm = reinterpret_cast<uint32_t*>(stv);  // [block][quarter][min | max][64 pairs]
      {
        const int cp = tid & 63, qq = tid >> 6;
        const int sh = (2 * cp) & 31;
        const uint32_t* rot2 = reinterpret_cast<const uint32_t*>(rot);
        for (int b = b0; b <= b1; ++b) {
          const int blo = S + b * B;
          const int st = max(blo, mlo), en = min(blo + B, mhi);
          const int len = en - st;
          const int a0 = st + (len * qq) / 4, a1 = st + (len * (qq + 1)) / 4;
          __nv_bfloat162 mn[2], mx[2];
          mn[0] = mn[1] = __halves2bfloat162(__ushort_as_bfloat16(0x7f80), __ushort_as_bfloat16(0x7f80));
          mx[0] = mx[1] = __halves2bfloat162(__ushort_as_bfloat16(0xff80), __ushort_as_bfloat16(0xff80));
          int q = a0;
          for (; q + 1 < a1; q += 2)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int t = q + e - lo;
              const uint32_t kb = keepw[t * 4 + (cp >> 4)] >> sh;
              const uint32_t v = rot2[(size_t)t * (kRotRow / 2) + cp] &
                                 ((kb & 1u ? 0x0000ffffu : 0u) | (kb & 2u ? 0xffff0000u : 0u));
              const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&v);
              mn[e] = __hmin2(mn[e], x);
              mx[e] = __hmax2(mx[e], x);
            }
          if (q < a1) {
            const int t = q - lo;
            const uint32_t kb = keepw[t * 4 + (cp >> 4)] >> sh;
            const uint32_t v = rot2[(size_t)t * (kRotRow / 2) + cp] &
                               ((kb & 1u ? 0x0000ffffu : 0u) | (kb & 2u ? 0xffff0000u : 0u));
            const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&v);
            mn[0] = __hmin2(mn[0], x);
            mx[0] = __hmax2(mx[0], x);
          }
          const __nv_bfloat162 m0 = __hmin2(mn[0], mn[1]), m1 = __hmax2(mx[0], mx[1]);
          uint32_t* dst = pm + ((b - b0) * 4 + qq) * 128;
          dst[cp] = *reinterpret_cast<const uint32_t*>(&m0);
          dst[64 + cp] = *reinterpret_cast<const uint32_t*>(&m1);
        }
      }
      __syncthreads();
      if (tid < 64) {
        const int cp = tid;
        uint32_t* meta2 = reinterpret_cast<uint32_t*>(base + L.off_meta);
        for (int b = b0; b <= b1; ++b) {
          if (!in_bounds(L, b < L.nblk_cap, SITE_PREFILL_META, b)) continue;
          const int blo = S + b * B;
          const uint32_t* src = pm + (b - b0) * 4 * 128;
          uint32_t u = src[cp], w = src[64 + cp];
          __nv_bfloat162 mn = *reinterpret_cast<const __nv_bfloat162*>(&u);
          __nv_bfloat162 mx = *reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
          for (int k = 1; k < 4; ++k) {
            u = src[k * 128 + cp];
            w = src[k * 128 + 64 + cp];
            mn = __hmin2(mn, *reinterpret_cast<const __nv_bfloat162*>(&u));
            mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&w));
          }
          if (max(blo, mlo) > blo) {  // the block held tokens before this tile
            u = meta2[(int64_t)b * D + cp];
            w = meta2[(int64_t)b * D + 64 + cp];
            mn = __hmin2(mn, *reinterpret_cast<const __nv_bfloat162*>(&u));
            mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&w));
          }
          const uint32_t mnu = *reinterpret_cast<const uint32_t*>(&mn), mxu = *reinterpret_cast<const uint32_t*>(&mx);
          meta2[(int64_t)b * D + cp] = mnu;
          meta2[(int64_t)b * D + 64 + cp] = mxu;
          if (L.meta_c > 0) {  // the rows for the compressed keys
            uint32_t* row = reinterpret_cast<uint32_t*>(bm + (b - b0) * 2 * D);
            row[cp] = mnu;
            row[64 + cp] = mxu;
          }
        }
      }
      if (L.meta_c > 0 && mlo < mhi) {
        __syncthreads();
        for (int b = b0 + warp; b <= b1; b += 8) {
          const uint16_t* row = bm + (b - b0) * 2 * D;
          uint16_t mn[4], mx[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            mn[i] = row[4 * lane + i];
            mx[i] = row[D + 4 * lane + i];
          }
          compress_key_row(L, base, b, mn, mx, lane);
        }
      }
    }
    __syncthreads();  // rot, keepw and ud are free for the next item
    cur = nxt;
    nxt = nn;
    xbuf ^= 1;
  }
  if (!ok && !aborted) {
    // A copy or the MMAs did not complete in time: report it, give the
    // hardware another bounded wait, then free the tensor memory.
    if (tid == 0) set_error(L, ERR_COPY_WAIT, -1, -3, (int32_t)MK_ETIMEOUT);
    if (mma_pending) (void)mbar_wait(&bar_mma, mma_phase);
    if (r_pending) (void)mbar_wait(&bar_r, r_phase);
  }
  cp_async_wait_all();
  if (tid == 0) bulk_wait_all();  // the pages' bulk stores are complete before the kernel ends
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// A segment's channel count, truncation and rotation flag after a swap of its
// pages (double-buffered re-compression); the flags keep the always bit.
__global__ void k_set_segment(Layout L, int64_t u, int seg, int r, int keep, int own) {
  if (threadIdx.x == 0) {
    L.desc[u].r[seg] = r;
    L.desc[u].sflags[seg] = (L.desc[u].sflags[seg] & 0x31) | (own ? 2 : 0) | (keep << 8);  // keeps always and g
  }
}

cudaError_t launch_set_segment(const Layout& L, int64_t u, int seg, int r, int keep, int own, cudaStream_t s) {
  k_set_segment<<<1, 32, 0, s>>>(L, u, seg, r, keep, own);
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
  int sms = 0;
  const auto kern = L.bm_g ? k_append_bulk<true> : k_append_bulk<false>;
  cudaError_t e = kernel_smem_attr((const void*)kern, kBulkSmem, 256, nullptr, &sms);
  if (e != cudaSuccess) return e;
  // Persistent: at most one CTA per SM, each with an equal run of items.
  const int items = 2 * L.n_kv * total_tiles;
  const int grid0 = std::max(1, std::min(items, std::max(sms, 1)));
  const int per = (items + grid0 - 1) / grid0;
  const int grid = (items + per - 1) / per;
  kern<<<grid, 256, kBulkSmem, s>>>(L, layer, cs, k, v, total_tiles, per);
  return cudaGetLastError();
}

}  // namespace mk
