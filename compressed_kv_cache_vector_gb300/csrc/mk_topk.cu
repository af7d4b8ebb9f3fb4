// Top-k block selection over the block-score keys of each (sequence, kv
// head): the k largest scores, ties to the lower block id, ids ascending.
//
// Method: "MosaicKV：...阅读笔记" (zhongzhuzhou.org), Eq. (12) (the k blocks
// with the largest bound are attended); "MosaicKV: Serving Long-Context LLM
// with Dynamic Two-D KV Cache Compression" (paperlayer.ai), sec. 4.2 stage 2
// (top-k token blocks before each decode attention layer).
//
// GB300 structure: C CTAs of 1024 threads per (sequence, kv head) (one per
// 4096 blocks of the context, up to 8), launched right behind the scoring
// kernel (programmatic dependent launch).  The
// scoring kernel leaves, per unit, an order-preserving 32-bit key per block
// (0 = not a candidate) and a 4096-bin histogram of the keys' top 12 bits.
//  * One bulk copy each stages the histogram and the keys; thread t takes
//    the 16-byte chunks j * 1024 + t (round j), so every read of a round is
//    conflict free and the block's key order is (j, t).
//  * Threshold: the histogram's coarse bin holds the k-th key.  Two passes
//    over the keys of that bin histogram their next 10 bits and then their
//    last 10 bits (1024 bins each, atomics aggregated per warp over equal
//    bins), and a block scan of each picks the bin that holds the k-th key:
//    the threshold key and the number of its ties to take come out exact.
//  * Output: every CTA of the unit finds the same threshold and writes the
//    ids of its share of the blocks.  A key above the threshold goes to
//    position (keys above it before it) + min(ties before it, need); a tie is
//    taken while fewer than `need` ties precede it.  The counts before a key
//    come from a counting pass over the blocks below the share, per-round
//    per-warp totals (one block scan) and warp scans.
// This code runs once per launch on its SM, so the passes are short loops
// (instructions not yet in the instruction cache cost a fetch each).
#include <algorithm>

#include "mk_internal.cuh"

namespace mk {

namespace {
constexpr int kTkThreads = 1024, kTkWarps = kTkThreads / 32;
constexpr int kTkRoundsMax = 32;                              // nch <= 32768: nblk <= 131072
constexpr int kTkSmemMax = 200 * 1024;                        // keys staged when they fit

// Exclusive prefix sums of two per-thread counts over the 1024 threads.
__device__ __forceinline__ int2 block_excl_scan2_1024(int a, int b, int2* wsum) {
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
  if (warp == 0) {
    const int2 w = wsum[lane];
    int sa = w.x, sb = w.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(FULL, sa, o), yb = __shfl_up_sync(FULL, sb, o);
      if (lane >= o) {
        sa += ya;
        sb += yb;
      }
    }
    wsum[lane] = make_int2(sa - w.x, sb - w.y);
  }
  __syncthreads();
  const int2 base = wsum[warp];
  __syncthreads();  // wsum may be reused right after
  return make_int2(base.x + xa - a, base.y + xb - b);
}
}  // namespace

// grid: C CTAs per (sequence, kv head) of the call; 1024 threads.  Each
// finds the threshold by itself and writes the ids of its share of the
// blocks.  With APPEND the scoring kernel appended cs.n_new[ci] tokens first:
// the length it read is advanced here, after every scoring CTA has read it.
// PERSEG: per-segment sequence retention, each scored segment selected on
// its own (its own k over its own blocks); else one top-k over all of them.
template <bool APPEND, bool PERSEG>
__global__ void __launch_bounds__(kTkThreads, 1) k_topk(Layout L, int layer, CallSeqs cs, int32_t* __restrict__ ids,
                                                        int32_t* __restrict__ n_sel, int dyn_bytes, int C) {
  extern __shared__ __align__(16) unsigned char smem[];   // staged keys
  __shared__ __align__(16) uint32_t hc[kKeyBins];
  __shared__ __align__(16) uint32_t fh[2][1024];           // fine histograms
  __shared__ __align__(16) int2 wtab[kTkThreads];          // per (round, warp): totals, then their bases
  __shared__ int2 wsum[kTkWarps];
  __shared__ __align__(16) UnitDesc ud;
  __shared__ int s_abort, s_bin, s_rem, s_last;
  __shared__ __align__(8) uint64_t bar;

  const int unit = blockIdx.x / C, part = blockIdx.x - unit * C;
  const int ci = unit / L.n_kv, kvh = unit - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = unit_index(L, layer, seq, kvh);
  const int64_t slot = (int64_t)seq * L.n_kv + kvh;
  // The unit's descriptor was last written two or more launches back (by
  // the append or by this kernel in an earlier call), never by the scoring
  // kernel this launch waits on, so it is read before the wait point.
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
    uint4 dd[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) dd[i] = __ldcg(reinterpret_cast<const uint4*>(L.desc + u) + i);
#pragma unroll
    for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(&ud)[i] = dd[i];
  }
  __syncthreads();
  const int T_cur = ud.T + (APPEND ? cs.n_new[ci] : 0);
  const int nblk = n_mid_blocks(L, T_cur);
  const int n_cand = n_scored_blocks(ud, nblk);
  const int k = n_select(L, n_cand);
  const bool all = k >= n_cand;  // every candidate is taken
  const int nch = (nblk + 3) >> 2;
  const int rounds = (nch + kTkThreads - 1) / kTkThreads;
  uint32_t* kw = L.keys + slot * L.keys_stride;
  uint32_t* gh = L.khist + slot * kKeyBins;
  int32_t* out = ids + ((int64_t)ci * L.n_kv + kvh) * L.k_max;
  const bool staged = (int64_t)nch * 16 <= (int64_t)dyn_bytes;
  const uint4* ks = reinterpret_cast<const uint4*>(smem);
  pdl_wait();
  pdl_trigger();

  // The histogram and the keys, one bulk copy each, in flight while the
  // error word is read.
  if (tid == 0) {
    fence_proxy_async_all();
    const unsigned kb = staged ? (unsigned)nch * 16u : 0u;
    mbar_expect_tx(&bar, kKeyBins * 4u + kb);
    bulk_g2s(hc, gh, kKeyBins * 4, &bar);
    if (kb) bulk_g2s(smem, kw, kb, &bar);
    s_abort = __ldcg(L.err);
  }
  fh[0][tid] = 0u;
  fh[1][tid] = 0u;
  const bool landed = mbar_wait(&bar, 0);
  if (!landed) {
    if (tid == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, -2, (int32_t)MK_ETIMEOUT);
    (void)mbar_wait(&bar, 0);
    return;
  }
  __syncthreads();
  if (s_abort) return;
  // The last of the unit's CTAs to have staged the histogram clears it for
  // the next call (no CTA waits); part 0 advances the length after the
  // fused append.
  int32_t* arrived = L.counters + (int64_t)L.max_seqs * L.n_kv + slot;
  if (tid == 0) s_last = atomicAdd(arrived, 1) == C - 1;
  __syncthreads();
  if (s_last) {
    reinterpret_cast<uint4*>(gh)[tid] = make_uint4(0, 0, 0, 0);
    if (tid == 0) *arrived = 0;
  }
  if (APPEND && part == 0 && tid == 0) L.desc[u].T = T_cur;

  // Chunk c (keys 4c .. 4c+3), keys past nblk zero; with PERSEG, keys
  // outside the blocks [r_lo, r_hi) of the segment being selected zero too.
  int r_lo = 0, r_hi = nblk;
  auto chunk_at = [&](int c) -> uint4 {
    if (c >= nch) return make_uint4(0, 0, 0, 0);
    uint4 v = staged ? ks[c] : __ldcg(reinterpret_cast<const uint4*>(kw) + c);
    if constexpr (PERSEG) {
      const int b0 = 4 * c;
      if (b0 < r_lo || b0 >= r_hi) v.x = 0u;
      if (b0 + 1 < r_lo || b0 + 1 >= r_hi) v.y = 0u;
      if (b0 + 2 < r_lo || b0 + 2 >= r_hi) v.z = 0u;
      if (b0 + 3 < r_lo || b0 + 3 >= r_hi) v.w = 0u;
    } else {
      if (4 * c + 1 >= nblk) v.y = 0u;
      if (4 * c + 2 >= nblk) v.z = 0u;
      if (4 * c + 3 >= nblk) v.w = 0u;
    }
    return v;
  };
  // Histogram into h, by bits [shift, shift + 10), of the keys whose bits
  // from shift + 10 up equal pre (0 is never a candidate).  When all of a
  // warp's keys in range share one bin they add once, so runs of equal keys
  // do not serialise on one address.
  auto fine_pass = [&](uint32_t* h, uint32_t pre, int shift) {
#pragma unroll 1
    for (int j = 0; j < rounds; ++j) {
      const uint4 v = chunk_at(j * kTkThreads + tid);
      const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool in = e[q] != 0u && (e[q] >> (shift + 10)) == pre;
        const unsigned act = __ballot_sync(FULL, in);
        if (act) {
          const uint32_t bin = (e[q] >> shift) & 1023u;
          const uint32_t bmin = __reduce_min_sync(FULL, in ? bin : 1023u);
          const uint32_t bmax = __reduce_max_sync(FULL, in ? bin : 0u);
          if (bmin == bmax) {
            if (lane == __ffs(act) - 1) atomicAdd(&h[bin], (uint32_t)__popc(act));
          } else if (in) {
            atomicAdd(&h[bin], 1u);
          }
        }
      }
    }
    __syncthreads();
  };
  // The bin of h (descending) that holds the rem-th largest of its keys:
  // s_bin, and s_rem = its rank inside that bin.
  auto fine_find = [&](const uint32_t* h, int rem) {
    const int c = (int)h[1023 - tid];
    const int ex = block_excl_scan2_1024(c, 0, wsum).x;  // keys in higher bins
    if (ex < rem && ex + c >= rem) {
      s_bin = 1023 - tid;
      s_rem = rem - ex;
    }
    __syncthreads();
  };

  // The selection of k_r keys of the current range (all of them when
  // all_r), its ids written from out[out_off] on: thr, the threshold key;
  // need, the ties at thr it takes.
  uint32_t thr = 1u;  // every candidate (key >= 1) when all are taken
  int need = 0;       // keys equal to thr to take
  bool all_r = all;
  // Keys above thr (all candidates when every one is taken) and ties of one
  // chunk, as 4-bit masks.
  auto masks = [&](int c, uint32_t& gm, uint32_t& em) {
    const uint4 v = chunk_at(c);
    const uint32_t e[4] = {v.x, v.y, v.z, v.w};
    gm = 0u;
    em = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      gm |= (all_r ? e[q] != 0u : e[q] > thr) ? 1u << q : 0u;
      em |= (!all_r && e[q] == thr) ? 1u << q : 0u;
    }
  };
  auto run_range = [&](int k_r, int out_off) {
    thr = 1u;
    need = 0;
    if (!all_r) {
      // Coarse bin of the k-th largest key: thread t holds bins 4095 - 4t - 3 .. 4095 - 4t.
      {
        const uint4 h4 = reinterpret_cast<const uint4*>(hc)[kKeyBins / 4 - 1 - tid];
        const int c = (int)(h4.x + h4.y + h4.z + h4.w);
        const int ex = block_excl_scan2_1024(c, 0, wsum).x;  // keys in higher bins
        if (ex < k_r && ex + c >= k_r) {
          const uint32_t hv[4] = {h4.w, h4.z, h4.y, h4.x};  // descending bin order
          int acc = ex;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (acc < k_r && acc + (int)hv[i] >= k_r) {
              s_bin = kKeyBins - 1 - 4 * tid - i;
              s_rem = k_r - acc;
            }
            acc += (int)hv[i];
          }
        }
        __syncthreads();
      }
      const uint32_t b = (uint32_t)s_bin;
      const int rem0 = s_rem;
      fine_pass(fh[0], b, 10);
      fine_find(fh[0], rem0);
      const uint32_t ba = (uint32_t)s_bin;
      const int rem1 = s_rem;
      fine_pass(fh[1], (b << 10) | ba, 0);
      fine_find(fh[1], rem1);
      thr = (b << 20) | (ba << 10) | (uint32_t)s_bin;
      need = s_rem;
    }



    // This CTA's share of the chunks, and the keys taken before it.
    const int per = (nch + C - 1) / C;
    const int c_lo = min(nch, part * per), c_hi = min(nch, c_lo + per);
    const int own_rounds = (c_hi - c_lo + kTkThreads - 1) / kTkThreads;
    int2 before;
    {
      int g0 = 0, e0 = 0;
      for (int c = tid; c < c_lo; c += kTkThreads) {
        uint32_t gm, em;
        masks(c, gm, em);
        g0 += __popc(gm);
        e0 += __popc(em);
      }
      const int2 ex = block_excl_scan2_1024(g0, e0, wsum);
      if (tid == kTkThreads - 1) wsum[0] = make_int2(ex.x + g0, ex.y + e0);
      __syncthreads();
      before = wsum[0];
      __syncthreads();
    }
    // Per (round, warp) of the share: totals of (above, ties); then their
    // exclusive scan in (round, warp) order, one entry per thread.
#pragma unroll 1
    for (int j = 0; j < own_rounds; ++j) {
      uint32_t gm = 0u, em = 0u;
      const int c = c_lo + j * kTkThreads + tid;
      if (c < c_hi) masks(c, gm, em);
      const int tg = (int)__reduce_add_sync(FULL, (unsigned)__popc(gm));
      const int te = (int)__reduce_add_sync(FULL, (unsigned)__popc(em));
      if (lane == 0) wtab[j * kTkWarps + warp] = make_int2(tg, te);
    }
    __syncthreads();
    {
      const int2 v = tid < own_rounds * kTkWarps ? wtab[tid] : make_int2(0, 0);
      const int2 ex = block_excl_scan2_1024(v.x, v.y, wsum);
      wtab[tid] = make_int2(ex.x + before.x, ex.y + before.y);
    }
    __syncthreads();
#pragma unroll 1
    for (int j = 0; j < own_rounds; ++j) {
      uint32_t gm = 0u, em = 0u;
      const int c = c_lo + j * kTkThreads + tid;
      if (c < c_hi) masks(c, gm, em);
      const int og = __popc(gm), oe = __popc(em);
      int ig = og, ie = oe;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yg = __shfl_up_sync(FULL, ig, o), ye = __shfl_up_sync(FULL, ie, o);
        if (lane >= o) {
          ig += yg;
          ie += ye;
        }
      }
      const int2 base = wtab[j * kTkWarps + warp];
      const int g_before = base.x + ig - og, e_before = base.y + ie - oe;
      const int take_eq = max(0, min(oe, need - e_before));  // ties still below `need`
      uint32_t tm = em;
      while (__popc(tm) > take_eq) tm &= ~(1u << (31 - __clz(tm)));  // keep the lowest ids
      const uint32_t take = gm | tm;
      const int p0 = g_before + min(e_before, need);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int p = p0 + __popc(take & ((1u << q) - 1u));
        if (((take >> q) & 1u) && out_off + p < L.k_max) out[out_off + p] = 4 * c + q;
      }
    }
  };
  if constexpr (!PERSEG) {
    run_range(k, 0);
  } else {
    // Each scored segment on its own: its keys' coarse histogram (the
    // scoring kernel's covers all segments), then its selection, its ids
    // after those of the segments before it.
    int32_t* ssel = L.seg_sel + (((int64_t)layer * L.max_seqs + seq) * L.n_kv + kvh) * MK_MAX_SEGMENTS;
    int off = 0;
    for (int sgi = 0; sgi < ud.n_seg; ++sgi) {
      if (part == 0 && tid == 0 && any_own(ud)) ssel[sgi] = off;  // ids below the segment's first block
      if (seg_always(ud, sgi)) continue;
      const int lo = min(ud.first_block[sgi], nblk);
      const int hi = sgi + 1 < ud.n_seg ? min(ud.first_block[sgi + 1], nblk) : nblk;
      if (hi <= lo) continue;
      const int k_s = n_select_segment(L, sgi, hi - lo);
      r_lo = lo;
      r_hi = hi;
      all_r = k_s >= hi - lo;
      fh[0][tid] = 0u;
      fh[1][tid] = 0u;
      if (!all_r) {
        for (int i = tid; i < kKeyBins; i += kTkThreads) hc[i] = 0u;
        __syncthreads();
#pragma unroll 1
        for (int j = 0; j < rounds; ++j) {
          const uint4 v = chunk_at(j * kTkThreads + tid);
          const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            // lanes with equal bins add once (runs of equal keys, e.g. ties)
            const bool in = e[q] != 0u;
            const unsigned act = __ballot_sync(FULL, in);
            if (in) {
              const unsigned peers = __match_any_sync(act, e[q] >> 20);
              if (lane == __ffs(peers) - 1) atomicAdd(&hc[e[q] >> 20], (uint32_t)__popc(peers));
            }
          }
        }
      }
      __syncthreads();
      run_range(k_s, off);
      off += k_s;
    }
    if (part == 0 && tid == 0) {
      n_sel[(int64_t)ci * L.n_kv + kvh] = off;
      if (any_own(ud))
        for (int sgi = ud.n_seg; sgi < MK_MAX_SEGMENTS; ++sgi) ssel[sgi] = off;
    }
    return;
  }
  if (part == 0 && tid == 0) n_sel[(int64_t)ci * L.n_kv + kvh] = k;
  // With segments stored under their own rotation, part 0 also records where
  // each segment's ids start in the ids row (the ids taken below its first
  // block): the attention gives each rotation its own CTAs.
  if (part == 0 && any_own(ud)) {
    int32_t* dst = L.seg_sel + (((int64_t)layer * L.max_seqs + seq) * L.n_kv + kvh) * MK_MAX_SEGMENTS;
    for (int sgi = 0; sgi < MK_MAX_SEGMENTS; ++sgi) {
      const int bnd = sgi < ud.n_seg ? min(ud.first_block[sgi], nblk) : nblk;
      int g0 = 0, e0 = 0;
      for (int c = tid; 4 * c < bnd; c += kTkThreads) {
        uint32_t gm, em;
        masks(c, gm, em);
        const uint32_t below = 4 * c + 4 <= bnd ? 0xfu : (1u << (bnd - 4 * c)) - 1u;
        g0 += __popc(gm & below);
        e0 += __popc(em & below);
      }
      const int2 ex = block_excl_scan2_1024(g0, e0, wsum);
      if (tid == kTkThreads - 1) dst[sgi] = ex.x + g0 + min(ex.y + e0, need);
      __syncthreads();
    }
  }
}

bool topk_plan_ok(const Layout& L) { return (L.nblk_cap + 3) / 4 <= kTkThreads * kTkRoundsMax; }

cudaError_t launch_topk(const Layout& L, int layer, const CallSeqs& cs, int32_t* ids, int32_t* n_sel, bool append,
                        cudaStream_t s) {
  const int dyn = (int)std::min<int64_t>(kTkSmemMax, (int64_t)16 * ((L.nblk_cap + 3) / 4));
  auto kern = append ? (L.per_seg_k ? k_topk<true, true> : k_topk<true, false>)
                     : (L.per_seg_k ? k_topk<false, true> : k_topk<false, false>);
  cudaError_t e = kernel_smem_attr((const void*)kern, dyn, kTkThreads, nullptr, nullptr);
  if (e != cudaSuccess) return e;
  // CTAs per unit: one per round of 4096 keys (the output pass is then one
  // round each), as many as the SMs allow.
  const int units = cs.n * L.n_kv;
  const int rounds = ((L.nblk_cap + 3) / 4 + kTkThreads - 1) / kTkThreads;
  const int C = std::max(1, std::min(rounds, std::min(8, 152 / std::max(1, units))));
  return launch_pdl(kern, dim3(units * C), dim3(kTkThreads), dyn, s, 0, L, layer, cs, ids, n_sel, dyn, C);
}

}  // namespace mk
