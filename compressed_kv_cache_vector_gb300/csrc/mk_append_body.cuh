// Per-vector compression and the decode-path append body, shared by the
// append kernels and the fused append + block-selection kernel.
//
// Method: "MosaicKV：...阅读笔记" (zhongzhuzhou.org), Eq. (7)/(8) (rotation of
// each new token), Eq. (9) and Algorithm 1 (per-vector top-r); "MosaicKV:
// Serving Long-Context LLM with Dynamic Two-D KV Cache Compression"
// (paperlayer.ai), sec. 4.2 stage 1 and sec. 5.1 (packed contiguous storage).
#pragma once

#include "mk_internal.cuh"

namespace mk {

// Uncompressed pages (the Quest comparator): token slot t of block b holds
// the whole rotated key row at [t] and value row at [B + t] of 128 bf16 words.
// A lane stores its four channels (4*lane .. 4*lane+3).
__device__ __forceinline__ void store_dense_row(const Layout& L, char* base, int b, int t, int is_v,
                                                uint2 four, int lane) {
  uint16_t* row = reinterpret_cast<uint16_t*>(base + L.off_pages + (int64_t)b * L.page_stride) +
                  (int64_t)(is_v * L.B + t) * D;
  reinterpret_cast<uint2*>(row)[lane] = four;
}

// Per-vector top-r of 128 bf16 magnitudes held 4 per lane (channels
// 4*lane .. 4*lane+3).  Keeps the r largest magnitudes, ties to the lower
// channel.  Returns this lane's keep bits; rank0 receives the packed position
// (ascending channel order) of the lane's first kept channel.
//
// The r-th largest magnitude t is found by a bitwise search from the most
// significant bit (the largest t with #{m >= t} >= r); all m > t are kept and
// the r - #{m > t} lowest channels with m == t.
__device__ __forceinline__ unsigned warp_topr(const uint32_t m[4], int r, int lane, int& rank0) {
  uint32_t t = 0;
#pragma unroll
  for (int bit = 14; bit >= 0; --bit) {
    const uint32_t cand = t | (1u << bit);
    const unsigned c = (unsigned)(m[0] >= cand) + (unsigned)(m[1] >= cand) +
                       (unsigned)(m[2] >= cand) + (unsigned)(m[3] >= cand);
    if ((int)__reduce_add_sync(FULL, c) >= r) t = cand;
  }
  const unsigned gt = (unsigned)(m[0] > t) + (unsigned)(m[1] > t) + (unsigned)(m[2] > t) + (unsigned)(m[3] > t);
  const unsigned eq = (unsigned)(m[0] == t) + (unsigned)(m[1] == t) + (unsigned)(m[2] == t) + (unsigned)(m[3] == t);
  const int need = r - (int)__reduce_add_sync(FULL, gt);
  int run = warp_excl_scan((int)eq, lane);
  unsigned keep = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (m[i] > t) {
      keep |= 1u << i;
    } else if (m[i] == t) {
      if (run < need) keep |= 1u << i;
      ++run;
    }
  }
  rank0 = warp_excl_scan(__popc(keep), lane);
  return keep;
}

// Channel-compressed key of block b ([S] sec. 5.2: the per-block keys are
// channel-compressed like the vectors): from the block's min/max row (four
// channels per lane, 4*lane .. 4*lane+3), keep the L.meta_c channels with the
// largest bound magnitude max(|min|, |max|), ties to the lower channel, and
// store them in ascending channel order as [min x m][max x m][channel x m].
// Called by one full warp.
__device__ __forceinline__ void compress_key_row(const Layout& L, char* base, int b, const uint16_t mn[4],
                                                 const uint16_t mx[4], int lane) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = max((uint32_t)(mn[i] & 0x7fffu), (uint32_t)(mx[i] & 0x7fffu));
  int rank;
  const unsigned kb = warp_topr(w, L.meta_c, lane, rank);
  char* row = base + L.off_cmeta + (int64_t)b * L.cmeta_row;
  uint16_t* cmn = reinterpret_cast<uint16_t*>(row);
  uint16_t* cmx = cmn + L.meta_c;
  uint8_t* cch = reinterpret_cast<uint8_t*>(cmx + L.meta_c);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (kb >> i & 1u) {
      cmn[rank] = mn[i];
      cmx[rank] = mx[i];
      cch[rank] = (uint8_t)(4 * lane + i);
      ++rank;
    }
  }
}

// Compresses one rotated vector (128 bf16 words at `row`) of middle position
// `pos` into its page; for a key also folds it into the block's min/max.
// Called by one full warp.  Returns this lane's keep bits.
__device__ __forceinline__ unsigned compress_vec(const Layout& L, const UnitDesc& ud, char* base, int pos,
                                                 const uint16_t* row, int is_v, int lane,
                                                 bool update_meta, uint2* meta_out = nullptr) {
  const int m = pos - L.S;
  const int b = m / L.B;
  const int t = m - b * L.B;
  const int sg = seg_of_block(ud, b);
  const int r = ud.r[sg], keep = seg_keep(ud, sg);
  char* page = base + L.off_pages + (int64_t)b * L.page_stride;
  const int Br = L.B * r;
  uint16_t* val = reinterpret_cast<uint16_t*>(page + (is_v ? 3 * Br : 0));
  uint8_t* idx = reinterpret_cast<uint8_t*>(page + (is_v ? 5 * Br : 2 * Br));
  const uint2 raw = *reinterpret_cast<const uint2*>(row + 4 * lane);
  // The block's min/max are loaded with the row, ahead of the search.
  uint16_t* meta = reinterpret_cast<uint16_t*>(base + L.off_meta) + (int64_t)b * 2 * D;
  uint2 omn = make_uint2(0, 0), omx = make_uint2(0, 0);
  if (update_meta && t != 0) {
    omn = *reinterpret_cast<const uint2*>(meta + 4 * lane);
    omx = *reinterpret_cast<const uint2*>(meta + D + 4 * lane);
  }
  uint16_t v[4] = {(uint16_t)(raw.x & 0xffff), (uint16_t)(raw.x >> 16), (uint16_t)(raw.y & 0xffff),
                   (uint16_t)(raw.y >> 16)};
  // Channels from `keep` on are truncated: magnitude 0, and with r <= keep
  // the ties at 0 go to lower channels, so they are never taken.
  uint32_t mag[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) mag[i] = 4 * lane + i < keep ? v[i] & 0x7fffu : 0u;
  int rank;
  unsigned kbits = 0xfu;
  if (L.dense_pages) {
    store_dense_row(L, base, b, t, is_v, raw, lane);
  } else {
    kbits = warp_topr(mag, r, lane, rank);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (kbits >> i & 1u) {
        val[t * r + rank] = v[i];
        idx[t * r + rank] = (uint8_t)(4 * lane + i);
        ++rank;
      }
    }
  }
  if (update_meta) {
    const uint16_t pmn[4] = {(uint16_t)(omn.x & 0xffff), (uint16_t)(omn.x >> 16), (uint16_t)(omn.y & 0xffff),
                             (uint16_t)(omn.y >> 16)};
    const uint16_t pmx[4] = {(uint16_t)(omx.x & 0xffff), (uint16_t)(omx.x >> 16), (uint16_t)(omx.y & 0xffff),
                             (uint16_t)(omx.y >> 16)};
    uint16_t nmn[4], nmx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float kt = (kbits >> i & 1u) ? bf2f(v[i]) : 0.0f;
      float lo = kt, hi = kt;
      if (t != 0) {
        lo = fminf(bf2f(pmn[i]), kt);
        hi = fmaxf(bf2f(pmx[i]), kt);
      }
      nmn[i] = f2bf(lo);
      nmx[i] = f2bf(hi);
    }
    *reinterpret_cast<uint2*>(meta + 4 * lane) =
        make_uint2((uint32_t)nmn[0] | ((uint32_t)nmn[1] << 16), (uint32_t)nmn[2] | ((uint32_t)nmn[3] << 16));
    *reinterpret_cast<uint2*>(meta + D + 4 * lane) =
        make_uint2((uint32_t)nmx[0] | ((uint32_t)nmx[1] << 16), (uint32_t)nmx[2] | ((uint32_t)nmx[3] << 16));
    if (meta_out) {  // this lane's four channels of the new min and max rows
      meta_out[0] =
          make_uint2((uint32_t)nmn[0] | ((uint32_t)nmn[1] << 16), (uint32_t)nmn[2] | ((uint32_t)nmn[3] << 16));
      meta_out[1] =
          make_uint2((uint32_t)nmx[0] | ((uint32_t)nmx[1] << 16), (uint32_t)nmx[2] | ((uint32_t)nmx[3] << 16));
    }
    if (L.meta_c > 0) compress_key_row(L, base, b, nmn, nmx, lane);
  }
  return kbits;
}

// The same for a token's key and value at once (same r): both searches share
// each warp reduction (counts packed as key | value << 16), which halves the
// dependent reductions per vector.
__device__ __forceinline__ void warp_topr2(const uint32_t mk[4], const uint32_t mv[4], int r, int lane,
                                           unsigned& keep_k, unsigned& keep_v, int& rank_k, int& rank_v) {
  uint32_t tk = 0, tv = 0;
#pragma unroll
  for (int bit = 14; bit >= 0; --bit) {
    const uint32_t ck = tk | (1u << bit), cv = tv | (1u << bit);
    const unsigned c = ((unsigned)(mk[0] >= ck) + (unsigned)(mk[1] >= ck) + (unsigned)(mk[2] >= ck) +
                        (unsigned)(mk[3] >= ck)) |
                       (((unsigned)(mv[0] >= cv) + (unsigned)(mv[1] >= cv) + (unsigned)(mv[2] >= cv) +
                         (unsigned)(mv[3] >= cv))
                        << 16);
    const unsigned sum = __reduce_add_sync(FULL, c);
    if ((int)(sum & 0xffffu) >= r) tk = ck;
    if ((int)(sum >> 16) >= r) tv = cv;
  }
  unsigned gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    gt += (unsigned)(mk[i] > tk) | ((unsigned)(mv[i] > tv) << 16);
    eq += (unsigned)(mk[i] == tk) | ((unsigned)(mv[i] == tv) << 16);
  }
  const unsigned gsum = __reduce_add_sync(FULL, gt);
  const int need_k = r - (int)(gsum & 0xffffu), need_v = r - (int)(gsum >> 16);
  const int run0 = warp_excl_scan((int)eq, lane);
  int run_k = run0 & 0xffff, run_v = run0 >> 16;
  keep_k = 0;
  keep_v = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (mk[i] > tk) {
      keep_k |= 1u << i;
    } else if (mk[i] == tk) {
      if (run_k < need_k) keep_k |= 1u << i;
      ++run_k;
    }
    if (mv[i] > tv) {
      keep_v |= 1u << i;
    } else if (mv[i] == tv) {
      if (run_v < need_v) keep_v |= 1u << i;
      ++run_v;
    }
  }
  const int rk0 = warp_excl_scan(__popc(keep_k) | (__popc(keep_v) << 16), lane);
  rank_k = rk0 & 0xffff;
  rank_v = rk0 >> 16;
}

// Compresses a token's rotated key and value (128 bf16 words each at rk, rv)
// of middle position `pos` into its page (no block min/max: the caller
// folds those).  Called by one full warp.  Returns the key's keep bits.
__device__ __forceinline__ unsigned compress_kv(const Layout& L, const UnitDesc& ud, char* base, int pos,
                                                const uint16_t* rk, const uint16_t* rv, int lane) {
  const int m = pos - L.S;
  const int b = m / L.B;
  const int t = m - b * L.B;
  const int sg = seg_of_block(ud, b);
  const int r = ud.r[sg], keep = seg_keep(ud, sg);
  char* page = base + L.off_pages + (int64_t)b * L.page_stride;
  const int Br = L.B * r;
  const uint2 rawk = *reinterpret_cast<const uint2*>(rk + 4 * lane);
  const uint2 rawv = *reinterpret_cast<const uint2*>(rv + 4 * lane);
  const uint16_t vk[4] = {(uint16_t)(rawk.x & 0xffff), (uint16_t)(rawk.x >> 16), (uint16_t)(rawk.y & 0xffff),
                          (uint16_t)(rawk.y >> 16)};
  const uint16_t vv[4] = {(uint16_t)(rawv.x & 0xffff), (uint16_t)(rawv.x >> 16), (uint16_t)(rawv.y & 0xffff),
                          (uint16_t)(rawv.y >> 16)};
  uint32_t mk[4], mv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // channels from `keep` on are truncated (see compress_vec)
    const bool live = 4 * lane + i < keep;
    mk[i] = live ? vk[i] & 0x7fffu : 0u;
    mv[i] = live ? vv[i] & 0x7fffu : 0u;
  }
  if (L.dense_pages) {
    store_dense_row(L, base, b, t, 0, rawk, lane);
    store_dense_row(L, base, b, t, 1, rawv, lane);
    return 0xfu;
  }
  unsigned keep_k, keep_v;
  int rank_k, rank_v;
  warp_topr2(mk, mv, r, lane, keep_k, keep_v, rank_k, rank_v);
  uint16_t* valk = reinterpret_cast<uint16_t*>(page);
  uint8_t* idxk = reinterpret_cast<uint8_t*>(page + 2 * Br);
  uint16_t* valv = reinterpret_cast<uint16_t*>(page + 3 * Br);
  uint8_t* idxv = reinterpret_cast<uint8_t*>(page + 5 * Br);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (keep_k >> i & 1u) {
      valk[t * r + rank_k] = vk[i];
      idxk[t * r + rank_k] = (uint8_t)(4 * lane + i);
      ++rank_k;
    }
    if (keep_v >> i & 1u) {
      valv[t * r + rank_v] = vv[i];
      idxv[t * r + rank_v] = (uint8_t)(4 * lane + i);
      ++rank_v;
    }
  }
  return keep_k;
}

// Four such searches at once (two tokens' keys and values, each with its own
// r <= 128): every warp reduction carries four 8-bit counts (a lane adds at
// most 4 to each, so no field overflows into the next).
__device__ __forceinline__ void warp_topr4(const uint32_t m[4][4], const int r[4], int lane, unsigned keep[4],
                                           int rank[4]) {
  uint32_t t[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int bit = 14; bit >= 0; --bit) {
    unsigned c = 0;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint32_t cand = t[v] | (1u << bit);
      const unsigned n = (unsigned)(m[v][0] >= cand) + (unsigned)(m[v][1] >= cand) + (unsigned)(m[v][2] >= cand) +
                         (unsigned)(m[v][3] >= cand);
      c |= n << (8 * v);
    }
    const unsigned sum = __reduce_add_sync(FULL, c);
#pragma unroll
    for (int v = 0; v < 4; ++v)
      if ((int)((sum >> (8 * v)) & 0xffu) >= r[v]) t[v] |= 1u << bit;
  }
  unsigned gt = 0, eq = 0;
#pragma unroll
  for (int v = 0; v < 4; ++v)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      gt += (unsigned)(m[v][i] > t[v]) << (8 * v);
      eq += (unsigned)(m[v][i] == t[v]) << (8 * v);
    }
  const unsigned gsum = __reduce_add_sync(FULL, gt);
  const unsigned run0 = (unsigned)warp_excl_scan((int)eq, lane);
  unsigned pc = 0;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int need = r[v] - (int)((gsum >> (8 * v)) & 0xffu);
    int run = (int)((run0 >> (8 * v)) & 0xffu);
    unsigned k = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (m[v][i] > t[v]) {
        k |= 1u << i;
      } else if (m[v][i] == t[v]) {
        if (run < need) k |= 1u << i;
        ++run;
      }
    }
    keep[v] = k;
    pc |= (unsigned)__popc(k) << (8 * v);
  }
  const unsigned rk0 = (unsigned)warp_excl_scan((int)pc, lane);
#pragma unroll
  for (int v = 0; v < 4; ++v) rank[v] = (int)((rk0 >> (8 * v)) & 0xffu);
}

// compress_kv for two middle tokens at once (positions pa, pb; rotated rows
// at rka/rva and rkb/rvb): their four top-r searches share each reduction.
// Returns each token's key keep bits.
__device__ __forceinline__ void compress_kv2(const Layout& L, const UnitDesc& ud, char* base, int pa, int pb,
                                             const uint16_t* rka, const uint16_t* rva, const uint16_t* rkb,
                                             const uint16_t* rvb, int lane, unsigned& keep_a, unsigned& keep_b) {
  const int pos[2] = {pa, pb};
  const uint16_t* rows[4] = {rka, rva, rkb, rvb};
  int rr[4], kp[2], bb[2], tt[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const int m = pos[w] - L.S;
    bb[w] = m / L.B;
    tt[w] = m - bb[w] * L.B;
    const int sg = seg_of_block(ud, bb[w]);
    rr[2 * w] = rr[2 * w + 1] = ud.r[sg];
    kp[w] = seg_keep(ud, sg);
  }
  uint16_t vals[4][4];
  uint32_t mag[4][4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint2 raw = *reinterpret_cast<const uint2*>(rows[v] + 4 * lane);
    vals[v][0] = (uint16_t)(raw.x & 0xffff);
    vals[v][1] = (uint16_t)(raw.x >> 16);
    vals[v][2] = (uint16_t)(raw.y & 0xffff);
    vals[v][3] = (uint16_t)(raw.y >> 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) mag[v][i] = 4 * lane + i < kp[v >> 1] ? vals[v][i] & 0x7fffu : 0u;  // truncated: 0
  }
  if (L.dense_pages) {
#pragma unroll
    for (int v = 0; v < 4; ++v)
      store_dense_row(L, base, bb[v >> 1], tt[v >> 1], v & 1,
                      make_uint2((uint32_t)vals[v][0] | ((uint32_t)vals[v][1] << 16),
                                 (uint32_t)vals[v][2] | ((uint32_t)vals[v][3] << 16)),
                      lane);
    keep_a = keep_b = 0xfu;
    return;
  }
  unsigned keep[4];
  int rank[4];
  warp_topr4(mag, rr, lane, keep, rank);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int w = v >> 1, isv = v & 1, r = rr[v];
    char* page = base + L.off_pages + (int64_t)bb[w] * L.page_stride;
    const int Br = L.B * r;
    uint16_t* val = reinterpret_cast<uint16_t*>(page + (isv ? 3 * Br : 0));
    uint8_t* idx = reinterpret_cast<uint8_t*>(page + (isv ? 5 * Br : 2 * Br));
    int rk = rank[v];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (keep[v] >> i & 1u) {
        val[tt[w] * r + rk] = vals[v][i];
        idx[tt[w] * r + rk] = (uint8_t)(4 * lane + i);
        ++rk;
      }
    }
  }
  keep_a = keep[0];
  keep_b = keep[2];
}

// Decode-path append of n new tokens to one (sequence, kv head) by one CTA of
// 256 threads: evicts the window tokens that leave it into the middle
// (select, pack, block min/max), then rotates the first n_rot (0 or n, at
// most kSmallAppend) new tokens (k' = k R_k^T, v' = v R_v^T with
// Rs = [R_k^T | R_v^T] in shared memory, possibly still arriving by
// cp.async) and stores them.  kin/vin point at the unit's first new row;
// xs: n_rot*2*128 floats and rot: n_rot*2*128 bf16 of shared scratch.
// Leaves the device length to the caller.  Ends with a barrier.
__device__ __forceinline__ void append_small_body(const Layout& L, const UnitDesc& ud, char* base, int T_old, int n,
                                                  int n_rot, const uint16_t* kin, const uint16_t* vin,
                                                  int64_t in_stride, const float* Rs, float* xs, uint16_t* rot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T_new = T_old + n;
  const int S = L.S, W = L.W;
  uint16_t* win_k = reinterpret_cast<uint16_t*>(base + L.off_win_k);
  uint16_t* win_v = reinterpret_cast<uint16_t*>(base + L.off_win_v);

  // Phase A: window tokens that leave the window, in position order.
  const int e_lo = max(S, T_old - W), e_hi = min(T_old, T_new - W);
  if (warp < 2) {
    for (int e = e_lo; e < e_hi; ++e) {
      const int slot = (e - S) % W;
      const uint16_t* row = (warp == 0 ? win_k : win_v) + (int64_t)slot * D;
      compress_vec(L, ud, base, e, row, warp, lane, warp == 0);
    }
  }
  __syncthreads();

  // Phase B: rotate the new tokens (k' = k R_k^T, v' = v R_v^T).
  for (int i = tid; i < n_rot * 2 * D; i += blockDim.x) {
    const int t = i / (2 * D), w = (i / D) & 1, c = i % D;
    const uint16_t* src = (w == 0 ? kin : vin) + (int64_t)t * in_stride;
    xs[(t * 2 + w) * D + c] = bf2f(src[c]);
  }
  cp_async_wait_all();
  __syncthreads();
  {
    // thread (w, ch): channel ch of the rotated key (w = 0) or value (w = 1)
    const int w = tid >> 7, ch = tid & 127;
    const float* RT = Rs + w * D * D;
    for (int i = 0; i < n_rot; ++i) {
      float acc = 0.0f;
#pragma unroll 8
      for (int j = 0; j < D; ++j) acc = fmaf(xs[(i * 2 + w) * D + j], RT[j * D + ch], acc);
      rot[(i * 2 + w) * D + ch] = f2bf(acc);
    }
  }
  __syncthreads();

  // Route: sinks and window dense, the rest compressed in position order.
  uint16_t* sink_k = reinterpret_cast<uint16_t*>(base + L.off_sink_k);
  uint16_t* sink_v = reinterpret_cast<uint16_t*>(base + L.off_sink_v);
  for (int i = 0; i < n_rot; ++i) {
    const int p = T_old + i;
    if (p < S || p >= T_new - W) {
      uint16_t* dk = p < S ? sink_k + (int64_t)p * D : win_k + (int64_t)((p - S) % W) * D;
      uint16_t* dv = p < S ? sink_v + (int64_t)p * D : win_v + (int64_t)((p - S) % W) * D;
      if (tid < D) dk[tid] = rot[(i * 2) * D + tid];
      else dv[tid - D] = rot[(i * 2 + 1) * D + tid - D];
    } else if (warp < 2) {
      compress_vec(L, ud, base, p, rot + (i * 2 + warp) * D, warp, lane, warp == 0);
    }
  }
  __syncthreads();
}

// The decode step's append of one token to a unit whose window is full
// (T_old >= S + W, W > 0), for the fused append + selection: the token at
// T_old - W leaves the window into the middle and the new token takes its
// window slot.  Warps 0 and 1 compress the leaving key (with the block
// min/max) and value while warps 2-5 rotate the new token; only the window
// write waits for both.  Same arithmetic as append_small_body with n = 1.
// Called by all 256 threads; Rs = [R_k^T | R_v^T] in shared memory,
// xs: 2*128 floats of shared scratch.  Shared memory is not touched after
// the one barrier inside, so the caller may reuse it at once.  Optional:
// warp 6 waits on `lbar` (a copy the caller started) before that barrier,
// and warp 0 returns its lane's part of the block's new min/max rows in
// meta_out[0..1].
__device__ __forceinline__ void append_one_body(const Layout& L, const UnitDesc& ud, char* base, int T_old,
                                                const uint16_t* kin, const uint16_t* vin, const float* Rs,
                                                float* xs, uint64_t* lbar = nullptr, uint2* meta_out = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = T_old - L.W;
  const int slot = (e - L.S) % L.W;
  uint16_t* win_k = reinterpret_cast<uint16_t*>(base + L.off_win_k) + (int64_t)slot * D;
  uint16_t* win_v = reinterpret_cast<uint16_t*>(base + L.off_win_v) + (int64_t)slot * D;
  const int ch = tid - 64;  // warps 2-5: channel of k' and v'
  float ak = 0.0f, av = 0.0f;
  if (warp < 2) {
    compress_vec(L, ud, base, e, warp == 0 ? win_k : win_v, warp, lane, warp == 0, warp == 0 ? meta_out : nullptr);
  } else if (warp == 6 && lbar) {
    if (!mbar_wait(lbar, 0)) {
      if (lane == 0) set_error(L, ERR_COPY_WAIT, -1, -6, (int32_t)MK_ETIMEOUT);
      (void)mbar_wait(lbar, 0);
    }
  } else if (warp >= 2 && warp < 6) {
    xs[ch] = bf2f(kin[ch]);
    xs[D + ch] = bf2f(vin[ch]);
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
#pragma unroll 8
    for (int j = 0; j < D; ++j) {
      ak = fmaf(xs[j], Rs[j * D + ch], ak);
      av = fmaf(xs[D + j], Rs[D * D + j * D + ch], av);
    }
  }
  __syncthreads();  // the leaving rows were read, and shared memory is free
  if (warp >= 2 && warp < 6) {
    win_k[ch] = f2bf(ak);
    win_v[ch] = f2bf(av);
  }
}

}  // namespace mk
