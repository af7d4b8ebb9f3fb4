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

// Grouped top-r for the bitmap format ([S] sec. 5.1: one bit per group of g
// adjacent channels), g = 2, 4 or 8, on a vector held 4 bf16 channels per lane
// (4*lane .. 4*lane+3).  Keeps the r/g groups with the largest energy, the
// fp32 sum of the group's squares in channel order (each product and sum
// rounded: a bf16 square is exact), ties to the lower group.  Groups from
// keep/g on count 0; with r <= keep the ties at 0 go to lower groups, so they
// are never taken.  The energies are non-negative floats, ordered as their
// bit patterns, so the (r/g)-th largest is found by a 31-bit search from the
// top.  Returns this lane's channel keep bits.
__device__ __forceinline__ unsigned warp_top_groups(const uint16_t v[4], int g, int r, int keep, int lane) {
  float sq[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x = bf2f(v[i]);
    sq[i] = __fmul_rn(x, x);
  }
  uint32_t key[2] = {0u, 0u};
  unsigned valid = 0u;  // bit s: key[s] is a group of this lane
  if (g == 2) {         // groups 2 lane, 2 lane + 1
    key[0] = 4 * lane < keep ? __float_as_uint(__fadd_rn(sq[0], sq[1])) : 0u;
    key[1] = 4 * lane + 2 < keep ? __float_as_uint(__fadd_rn(sq[2], sq[3])) : 0u;
    valid = 3u;
  } else {
    float e = __fadd_rn(__fadd_rn(__fadd_rn(sq[0], sq[1]), sq[2]), sq[3]);
    if (g == 4) {       // group lane
      key[0] = 4 * lane < keep ? __float_as_uint(e) : 0u;
      valid = 1u;
    } else {            // group lane / 2: the odd lane continues the even lane's sum
      const float lo = __shfl_xor_sync(FULL, e, 1);
      e = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(lo, sq[0]), sq[1]), sq[2]), sq[3]);
      key[0] = 4 * (lane - 1) < keep ? __float_as_uint(e) : 0u;
      valid = lane & 1;
    }
  }
  const int k = r / g;
  uint32_t t = 0u;
#pragma unroll 1
  for (int bit = 30; bit >= 0; --bit) {
    const uint32_t cand = t | (1u << bit);
    const unsigned c = (unsigned)((valid & 1u) && key[0] >= cand) + (unsigned)((valid & 2u) && key[1] >= cand);
    if ((int)__reduce_add_sync(FULL, c) >= k) t = cand;
  }
  const unsigned gt = (unsigned)((valid & 1u) && key[0] > t) + (unsigned)((valid & 2u) && key[1] > t);
  const unsigned eq = (unsigned)((valid & 1u) && key[0] == t) + (unsigned)((valid & 2u) && key[1] == t);
  const int need = k - (int)__reduce_add_sync(FULL, gt);
  int run = warp_excl_scan((int)eq, lane);
  unsigned kg = 0u;  // kept groups of this lane (bit s: key[s])
#pragma unroll
  for (int s2 = 0; s2 < 2; ++s2) {
    if (!(valid >> s2 & 1u)) continue;
    if (key[s2] > t) {
      kg |= 1u << s2;
    } else if (key[s2] == t) {
      if (run < need) kg |= 1u << s2;
      ++run;
    }
  }
  if (g == 2) return (kg & 1u ? 3u : 0u) | (kg & 2u ? 12u : 0u);
  if (g == 8) kg = __shfl_sync(FULL, kg, lane | 1);
  return kg ? 0xfu : 0u;
}

// Stores the position bitmap of one vector ([S] sec. 5.1): 128/g bits, bit j
// (byte j/8, bit j%8) set when group j is kept.  kbits: this lane's channel
// keep bits (channels 4*lane .. 4*lane+3, whole groups).  Called by one full
// warp; dst is aligned to the bitmap's size.
__device__ __forceinline__ void store_bitmap(uint8_t* dst, unsigned kbits, int g, int lane) {
  uint32_t w;
  int lpw;  // lanes whose group bits share one 32-bit word
  if (g == 1) {
    w = kbits << (4 * (lane & 7));
    lpw = 8;
  } else if (g == 2) {
    w = ((kbits & 1u) | ((kbits >> 1) & 2u)) << (2 * (lane & 15));
    lpw = 16;
  } else if (g == 4) {
    w = (kbits & 1u) << lane;
    lpw = 32;
  } else {
    w = (kbits & 1u) << (lane >> 1);
    lpw = 32;
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_xor_sync(FULL, w, off);
    if (off < lpw) w |= o;
  }
  if ((lane & (lpw - 1)) == 0) {
    if (g == 8)
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w;
    else
      reinterpret_cast<uint32_t*>(dst)[lane / lpw] = w;
  }
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
  if (!in_bounds(L, m >= 0 && b < L.nblk_cap, SITE_DECODE_PAGE, pos)) return 0u;  // (warp-uniform)
  const int sg = seg_of_block(ud, b);
  const int r = ud.r[sg], keep = seg_keep(ud, sg);
  char* page = base + L.off_pages + (int64_t)b * L.page_stride;
  const int gg = L.bm_g ? seg_group(ud, sg) : 0;  // bitmap pages: the segment's element-group size
  uint16_t* val = reinterpret_cast<uint16_t*>(page + (is_v ? page_vval(L, r, gg) : 0));
  uint8_t* idx = reinterpret_cast<uint8_t*>(page + (is_v ? page_vpos(L, r, gg) : page_kpos(L, r)));
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
    if (gg > 1) {
      kbits = warp_top_groups(v, gg, r, keep, lane);
      rank = warp_excl_scan(__popc(kbits), lane);
    } else {
      kbits = warp_topr(mag, r, lane, rank);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (kbits >> i & 1u) {
        val[t * r + rank] = v[i];
        if (!gg) idx[t * r + rank] = (uint8_t)(4 * lane + i);
        ++rank;
      }
    }
    if (gg) store_bitmap(idx + t * pos_bytes(L, r, gg), kbits, gg, lane);
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
  if (!in_bounds(L, e >= L.S, SITE_WINDOW, e)) return;  // (block-uniform: the caller's full window)
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
