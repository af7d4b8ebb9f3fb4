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
// GB300 structure: P CTAs per (sequence, kv head).
//  * Each CTA stages R_k^T by one bulk copy and forms q' for the group's
//    heads before the wait point (this prologue runs between the previous
//    layer's attention and the scoring: the two kernels' CTAs do not fit on
//    one SM together).
//  * Scoring is a dense contraction: for block b and head h,
//      sum_j max(q'_hj mn_bj, q'_hj mx_bj) = [mn_b | mx_b] . [min(q'_h,0) | max(q'_h,0)]
//    over K = 256.  Meta tiles of 16 blocks are staged by bulk copies (one
//    per block row, double-buffered per warp) and multiplied on the tensor
//    cores (mma.sync m16n8k16).  With channel-compressed keys the staged rows
//    are rebuilt into the same dense tile, dropped channels zero.  The fp32 operand is
//    split exactly into three bf16 parts (24 = 3 x 8 significant bits) and the
//    meta values are bf16, so every product is exact and the accumulation is
//    fp32: the scores keep fp32 accuracy.
//  * Each score is written as an order-preserving 32-bit key (0 for blocks of
//    always-attended segments, which are not candidates) and counted in a
//    4096-bin histogram of the keys' top 12 bits, kept in shared memory and
//    added to the unit's histogram in global memory when the CTA is done.
//  * The top k of each (sequence, kv head) follow in a second kernel
//    (mk_topk.cu) launched right behind this one.
//  * With APPEND, CTA 0 of each unit first appends the step's new token (see
//    k_select) and scores the unit's last tile.
#include <algorithm>

#include "mk_append_body.cuh"

namespace mk {

namespace {
constexpr int kSelWarps = 8;
constexpr int kMT = 16;                       // blocks per MMA tile
constexpr int kMetaRow = 2 * D + 8;           // padded bf16 row (528 bytes): ldmatrix conflict-free
constexpr int kMetaTile = kMT * kMetaRow * 2; // bytes per staged tile
constexpr int kSelSmem = kSelWarps * 2 * kMetaTile;  // double-buffered tiles (also holds R_k^T)
static_assert(kSelSmem >= 2 * D * D * 4 + 2 * D * 4 + 2 * D * 2, "R_k^T, R_v^T and the append scratch fit in the tile area");

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
// for normal x: each part takes the next 8 significant bits).  A part is the
// remainder truncated to its upper 16 bits (bf16 rounded toward zero), and
// the subtraction that leaves the next remainder is exact.
__device__ __forceinline__ void split3(float x, uint16_t (&p)[3]) {
  float r = x;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const uint32_t b = __float_as_uint(r) & 0xffff0000u;
    p[i] = (uint16_t)(b >> 16);
    r -= __uint_as_float(b);
  }
}

}  // namespace

// grid: P CTAs per (sequence, kv head) of the call; 256 threads.
// With APPEND, the kernel first appends one new token per sequence (the
// decode step's append, fused): CTA 0 of each unit evicts the window token
// that leaves the window, rotates and stores the new one, and scores the
// unit's last tiles afterwards (the evicted token lands in the last block);
// the top-k kernel advances the device length.  kin/vin: [n_seqs][n_kv][128]
// bf16.
template <int G, bool APPEND, bool OWN>
__global__ void __launch_bounds__(256, 1) k_select(Layout L, int layer, CallSeqs cs, int P,
                                                   const uint16_t* __restrict__ q, int32_t* __restrict__ ids,
                                                   int32_t* __restrict__ n_sel, float* __restrict__ scores_out,
                                                   int dyn_bytes, const uint16_t* __restrict__ kin,
                                                   const uint16_t* __restrict__ vin) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ __align__(16) float qs[D][G];  // q, channel-major: one vector load per channel
  __shared__ float qr[2][G][D];
  __shared__ UnitDesc ud;
  __shared__ __align__(16) uint32_t hc[kKeyBins];   // coarse key histogram
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_rbar;
  __shared__ __align__(8) uint64_t s_tbar[kSelWarps][2];  // each warp's two meta-tile stages
  __shared__ __align__(16) uint32_t bqs[3][16][2][32];  // B fragments, staged once (then: the early last tile)
  __shared__ __align__(8) uint64_t s_lbar;            // the early last tile's copy
  // OWN (some segment stored under its own rotation): q, and q' in each such segment's basis.
  __shared__ float qraw[OWN ? G : 1][OWN ? D : 1];
  __shared__ float qrc[OWN ? MK_MAX_SEGMENTS - 1 : 1][OWN ? G : 1][OWN ? D : 1];

  const int unit_call = blockIdx.x / P, part = blockIdx.x - unit_call * P;
  const int ci = unit_call / L.n_kv, kvh = unit_call - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t u = unit_index(L, layer, seq, kvh);
  const int64_t slot = (int64_t)seq * L.n_kv + kvh;
  const char* base = unit_base(L, u);
  // R_k^T (and, for the appending CTA, R_v^T right after it in the unit) by
  // one bulk copy, in flight while q is converted and the histogram cleared.
  const unsigned r_bytes = (unsigned)((APPEND && part == 0) ? 2 : 1) * D * D * 4;
  if (tid == 0) {
    mbar_init(&s_rbar, 1);
    mbar_init(&s_lbar, 1);
    for (int w = 0; w < kSelWarps; ++w) {
      mbar_init(&s_tbar[w][0], 1);
      mbar_init(&s_tbar[w][1], 1);
    }
    mbar_init_fence();
    mbar_expect_tx(&s_rbar, r_bytes);
    bulk_g2s(smem, base + L.off_rkt, r_bytes, &s_rbar);
  }
  for (int i = tid; i < G * D; i += blockDim.x) {
    const float x = bf2f(q[((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D + i]);
    qs[i % D][i / D] = x;
    if constexpr (OWN) qraw[i / D][i % D] = x;
  }
  for (int i = tid; i < kKeyBins / 4; i += blockDim.x) reinterpret_cast<uint4*>(hc)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();  // the barrier's initialisation is visible before anyone waits on it
  if (!mbar_wait(&s_rbar, 0)) {
    if (tid == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, -4, (int32_t)MK_ETIMEOUT);
    (void)mbar_wait(&s_rbar, 0);
    return;
  }

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
      for (int h = 0; h < G; ++h) acc[h] = fmaf(qs[j][h], rr, acc[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) qr[half][h][c] = acc[h];
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    const float v = qr[0][h][c] + qr[1][h][c];
    qr[0][h][c] = v;
    qs[c][h] = v;  // q' channel-major too, for the direct scoring of compressed block keys
  }
  __syncthreads();

  // B fragments of [min(q',0) | max(q',0)] (k = 0..255, n = head), 3 exact
  // parts: built once per (chunk, half, lane) by a short loop into shared
  // memory, then loaded into the registers of every warp.
  for (int i = tid; i < 16 * 2 * 32; i += blockDim.x) {
    const int ln = i & 31, hf2 = (i >> 5) & 1, kc = i >> 6;
    const int n = ln >> 2, k = kc * 16 + hf2 * 8 + 2 * (ln & 3);
    uint16_t e0[3] = {0, 0, 0}, e1[3] = {0, 0, 0};
    if (n < G) {
      const float x0 = k < D ? fminf(qr[0][n][k], 0.0f) : fmaxf(qr[0][n][k - D], 0.0f);
      const float x1 = (k + 1) < D ? fminf(qr[0][n][k + 1], 0.0f) : fmaxf(qr[0][n][k + 1 - D], 0.0f);
      split3(x0, e0);
      split3(x1, e1);
    }
#pragma unroll
    for (int s = 0; s < 3; ++s) bqs[s][kc][hf2][ln] = (uint32_t)e0[s] | ((uint32_t)e1[s] << 16);
  }
  __syncthreads();
  uint32_t bq[3][16][2];
#pragma unroll
  for (int s = 0; s < 3; ++s)
#pragma unroll
    for (int kc = 0; kc < 16; ++kc)
#pragma unroll
      for (int hf2 = 0; hf2 < 2; ++hf2) bq[s][kc][hf2] = bqs[s][kc][hf2][lane];
  // Everything above used only q and R_k.  From here on the kernel reads
  // what the append kernel wrote (lengths, block keys).
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    s_abort = has_error(L);
    ud = L.desc[u];
  }
  if (part == 0)
    for (int i = tid; i < G * D; i += blockDim.x) qrot_of(L, layer, slot)[i] = qr[0][i / D][i % D];
  __syncthreads();  // also: the R_k^T area becomes the tile stages
  if (s_abort) return;

  int T_cur = ud.T;
  // The appending CTA's last tile, staged early (see below): its index, rows,
  // and warp 0's part of the leaving token's new min/max row.
  bool early = false;
  int tl = 0;
  uint2 mrow[2] = {make_uint2(0, 0), make_uint2(0, 0)};
  uint16_t* lt = reinterpret_cast<uint16_t*>(&bqs[0][0][0][0]);
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
      const bool one = n == 1 && L.W > 0 && T_cur >= L.S + L.W;
      // With full keys and other CTAs to share the rest, warp 6 stages the
      // unit's last tile (which holds the leaving token's block) while the
      // append runs; warp 0 then patches that block's row with the new
      // min/max it computed, instead of reading back what it wrote.
      early = one && P > 1 && L.meta_c == 0 && !(OWN && any_own(ud));
      if (early) {
        const int nb_new = n_mid_blocks(L, T_cur + 1);
        tl = (nb_new - 1) / kMT;
        const int nrow = nb_new - tl * kMT;
        if (warp == 6) {
          if (lane == 0) {
            fence_proxy_async();  // the area was last read as the B fragments
            mbar_expect_tx(&s_lbar, (unsigned)nrow * 2u * D * 2u);
          }
          __syncwarp();
          const uint16_t* meta0 = reinterpret_cast<const uint16_t*>(base + L.off_meta);
          if (lane < nrow)
            bulk_g2s(lt + lane * kMetaRow, meta0 + (int64_t)(tl * kMT + lane) * 2 * D, 2 * D * 2, &s_lbar);
        }
      }
      if (one)
        append_one_body(L, ud, const_cast<char*>(base), T_cur, kin + row0, vin + row0,
                        reinterpret_cast<const float*>(smem), xs, early ? &s_lbar : nullptr, mrow);
      else
        append_small_body(L, ud, const_cast<char*>(base), T_cur, n, n, kin + row0, vin + row0, in_stride,
                          reinterpret_cast<const float*>(smem), xs, rot);
      if (early) {
        if (warp == 0) {  // the copy landed before the append's barrier
          const int be = (T_cur - L.W - L.S) / L.B;
          uint16_t* rowp = lt + (be - tl * kMT) * kMetaRow;
          *reinterpret_cast<uint2*>(rowp + 4 * lane) = mrow[0];
          *reinterpret_cast<uint2*>(rowp + D + 4 * lane) = mrow[1];
          __syncwarp();
        }
      } else {
        __threadfence();          // the updated block min/max before this CTA's own tiles are read,
        fence_proxy_async_all();  // which the bulk copies (async proxy) do
      }
    }
    T_cur += n;
  }
  // Segments stored under their own rotation (re-compressed closed
  // segments): q'_c = q R_c^T for each, R_c^T staged by one bulk copy over
  // the (now free) first 64 KB of the tile area; part 0 keeps q'_c in the
  // workspace for the attention.
  const bool own = OWN && any_own(ud);
  unsigned r_phase = 1u;
  if (own) {
    __syncthreads();  // the append (part 0) is done with the staged rotations
    for (int sg = 0; sg + 1 < ud.n_seg; ++sg) {
      if (!seg_own(ud, sg)) continue;
      if (tid == 0) {
        fence_proxy_async();
        mbar_expect_tx(&s_rbar, (unsigned)(D * D * 4));
        bulk_g2s(smem, base + segrot_off(L, sg), (unsigned)(D * D * 4), &s_rbar);
      }
      if (!__syncthreads_and(mbar_wait(&s_rbar, r_phase & 1u) ? 1 : 0)) {
        if (tid == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, -6, (int32_t)MK_ETIMEOUT);
        (void)mbar_wait(&s_rbar, r_phase & 1u);
        return;  // no CTA of this kernel waits on another
      }
      ++r_phase;
      const float* Rs = reinterpret_cast<const float*>(smem);
      {
        const int c = tid & (D - 1), half = tid >> 7;
        float acc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = 0.0f;
        for (int j = half * 64; j < half * 64 + 64; ++j) {
          const float rr = Rs[j * D + c];
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h] = fmaf(qraw[OWN ? h : 0][OWN ? j : 0], rr, acc[h]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) qr[half][h][c] = acc[h];
      }
      __syncthreads();
      for (int i = tid; i < G * D; i += blockDim.x) {
        const int h = i / D, c = i % D;
        const float v = qr[0][h][c] + qr[1][h][c];
        if constexpr (OWN) qrc[sg][h][c] = v;
        if (part == 0) qrot_of(L, layer, slot, sg + 1)[i] = v;
      }
      __syncthreads();  // the staging area is read; qr is free again
    }
  }
  const int nblk = n_mid_blocks(L, T_cur);
  const int ntiles = (nblk + kMT - 1) / kMT;
  // With APPEND, CTA 0 scores only the last tile (after its own append: the
  // evicted token lands in the last block) and the other CTAs share the rest.
  int t0, t1;
  if (APPEND && P > 1) {
    const int tp = (ntiles - 1 + P - 2) / (P - 1);
    t0 = part == 0 ? max(0, ntiles - 1) : min(ntiles - 1, (part - 1) * tp);
    t1 = part == 0 ? ntiles : min(ntiles - 1, part * tp);
  } else {
    const int tper = (ntiles + P - 1) / P;
    t0 = min(ntiles, part * tper);
    t1 = min(ntiles, t0 + tper);
  }
  if (early) t1 = t0;  // the last tile is already staged (scored below by warp 0)
  const uint16_t* meta = reinterpret_cast<const uint16_t*>(base + L.off_meta);
  uint32_t* kw = L.keys + slot * L.keys_stride;
  float* so = scores_out ? scores_out + ((int64_t)ci * L.n_kv + kvh) * L.nblk_cap : nullptr;
  unsigned char* stg = smem + (size_t)warp * 2 * kMetaTile;
  // Tile t (16 blocks) into stage sidx: one 512-byte bulk copy per block row
  // (rows padded to kMetaRow for conflict-free ldmatrix), on the stage's
  // barrier; rows past the last block are not loaded (and not scored).
  uint32_t tph = 0, tpend = 0;  // per stage: phase parity, copy in flight
  // With channel-compressed keys (L.meta_c > 0) a stage holds the tile's
  // compressed rows (one bulk copy), rebuilt into one dense tile after it.
  const bool cmp = L.meta_c > 0;
  const int mc = L.meta_c;
  const char* cmeta = base + L.off_cmeta;
  auto cstage = [&](int sidx) { return stg + kMetaTile + (size_t)sidx * kMT * L.cmeta_row; };
  auto issue = [&](int t, int sidx) {
    if (t >= t1) return;
    const int nrow = min(kMT, nblk - t * kMT);
    if (cmp) {
      if (lane == 0) {
        fence_proxy_async();  // the stage was last read by the rebuild
        mbar_expect_tx(&s_tbar[warp][sidx], (unsigned)(nrow * L.cmeta_row));
        bulk_g2s(cstage(sidx), cmeta + (int64_t)t * kMT * L.cmeta_row, (unsigned)(nrow * L.cmeta_row),
                 &s_tbar[warp][sidx]);
      }
      __syncwarp();
    } else {
      unsigned char* dst = stg + (size_t)sidx * kMetaTile;
      if (lane == 0) {
        fence_proxy_async();  // the stage was last read by ldmatrix
        mbar_expect_tx(&s_tbar[warp][sidx], (unsigned)nrow * 2u * D * 2u);
      }
      __syncwarp();
      if (lane < nrow)
        bulk_g2s(dst + lane * kMetaRow * 2, meta + (int64_t)(t * kMT + lane) * 2 * D, 2 * D * 2, &s_tbar[warp][sidx]);
    }
    tpend |= 1u << sidx;
  };
  // Write block b's score: the user's fp32 copy, the key, the histogram count.
  auto emit = [&](int b, float sc) {
    if (!in_bounds(L, b >= 0 && b < L.nblk_cap, SITE_SELECT_KEY, b)) return;
    if (so) so[b] = sc;
    const uint32_t key = seg_always(ud, seg_of_block(ud, b)) ? 0u : ordered_key(sc);
    kw[b] = key;
    if (key) atomicAdd(&hc[key >> 20], 1u);
  };
  const float inv_sqrt_d = 0.08838834764831845f;
  // Scores of tile t (16 dense [min | max] rows) into keys, histogram, scores.
  // Scores of tile t; with cf >= 0 only the rows whose blocks belong to
  // rotation class cf are written.
  auto score_tile = [&](const uint16_t* tile, int t, int cf = -1) {
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
      if (b0 < nblk && (cf < 0 || seg_class(ud, seg_of_block(ud, b0)) == cf)) emit(b0, b_lo * inv_sqrt_d);
      if (b1 < nblk && (cf < 0 || seg_class(ud, seg_of_block(ud, b1)) == cf)) emit(b1, b_hi * inv_sqrt_d);
    }
  };
  // With segments under their own rotation, a tile is scored once per
  // rotation class among its blocks; the B fragments are rebuilt (from the
  // class's q') when the class changes.
  int cur_cls = 0;
  auto build_bq = [&](int c) {
    const int n = lane >> 2;
#pragma unroll
    for (int kc = 0; kc < 16; ++kc)
#pragma unroll
      for (int hf2 = 0; hf2 < 2; ++hf2) {
        const int k = kc * 16 + hf2 * 8 + 2 * (lane & 3);
        uint16_t e0[3] = {0, 0, 0}, e1[3] = {0, 0, 0};
        if (n < G) {
          const float a0 = (!OWN || c == 0) ? qs[k % D][n] : qrc[OWN ? c - 1 : 0][OWN ? n : 0][OWN ? k % D : 0];
          const float a1 = (!OWN || c == 0) ? qs[(k + 1) % D][n]
                                            : qrc[OWN ? c - 1 : 0][OWN ? n : 0][OWN ? (k + 1) % D : 0];
          split3(k < D ? fminf(a0, 0.0f) : fmaxf(a0, 0.0f), e0);
          split3((k + 1) < D ? fminf(a1, 0.0f) : fmaxf(a1, 0.0f), e1);
        }
#pragma unroll
        for (int p3 = 0; p3 < 3; ++p3) bq[p3][kc][hf2] = (uint32_t)e0[p3] | ((uint32_t)e1[p3] << 16);
      }
  };
  auto score_tile_own = [&](const uint16_t* tile, int t) {
    const int b0 = t * kMT + g, b1 = b0 + 8;
    const int c0 = b0 < nblk ? seg_class(ud, seg_of_block(ud, b0)) : -1;
    const int c1 = b1 < nblk ? seg_class(ud, seg_of_block(ud, b1)) : -1;
    for (int c = 0; c < ud.n_seg; ++c) {
      if (!__any_sync(FULL, c0 == c || c1 == c)) continue;
      if (c != cur_cls) {
        build_bq(c);
        cur_cls = c;
      }
      score_tile(tile, t, c);
    }
  };
  if (early && warp == 0) score_tile(lt, tl);
  int st = 0;
  int t = t0 + warp;
  issue(t, 0);
  for (; t < t1; t += kSelWarps) {
    issue(t + kSelWarps, st ^ 1);
    if (!mbar_wait_warp(&s_tbar[warp][st], (tph >> st) & 1u)) {
      if (lane == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, -5, (int32_t)MK_ETIMEOUT);
      break;
    }
    tph ^= 1u << st;
    tpend &= ~(1u << st);
    const uint16_t* tile = reinterpret_cast<const uint16_t*>(stg + (size_t)st * kMetaTile);
    if (cmp) {
      // Compressed rows, scored directly: lane (row, half) sums over half of
      // the row's kept channels, q' gathered by channel from shared memory
      // (the dropped channels contribute zero), and the halves add by one
      // shuffle.
      const int nrow = min(kMT, nblk - t * kMT);
      const unsigned char* cst = cstage(st);
      const int row = lane & 15, hf = lane >> 4;
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.0f;
      if (row < nrow) {
        const unsigned char* crow = cst + row * L.cmeta_row;
        const uint16_t* cv = reinterpret_cast<const uint16_t*>(crow);
        const int j0 = hf ? (mc + 1) / 2 : 0, j1 = hf ? mc : (mc + 1) / 2;
        const int rc = own ? seg_class(ud, seg_of_block(ud, t * kMT + row)) : 0;
        for (int j = j0; j < j1; ++j) {
          const float mn = bf2f(cv[j]), mx = bf2f(cv[mc + j]);
          const int ch = crow[4 * mc + j];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float qv = (!OWN || rc == 0) ? qs[ch][h] : qrc[OWN ? rc - 1 : 0][OWN ? h : 0][OWN ? ch : 0];
            acc[h] += fmaxf(qv * mn, qv * mx);
          }
        }
      }
      float sc = -INFINITY;
#pragma unroll
      for (int h = 0; h < G; ++h) sc = fmaxf(sc, acc[h] + __shfl_xor_sync(FULL, acc[h], 16));
      if (hf == 0 && row < nrow) emit(t * kMT + row, sc * inv_sqrt_d);
    } else if (own) {
      score_tile_own(tile, t);
    } else {
      score_tile(tile, t);
    }
    __syncwarp();
    st ^= 1;
  }
  // Only after a timed-out wait can copies still be landing: let them.
  for (int i = 0; i < 2; ++i)
    if ((tpend >> i) & 1u) (void)mbar_wait(&s_tbar[warp][i], (tph >> i) & 1u);
  __syncthreads();
  // Add this CTA's histogram to the unit's (the top-k kernel reads it).
  uint32_t* gh = L.khist + slot * kKeyBins;
  for (int i = tid; i < kKeyBins / 4; i += blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(hc)[i];
    if (v.x) atomicAdd(gh + 4 * i, v.x);
    if (v.y) atomicAdd(gh + 4 * i + 1, v.y);
    if (v.z) atomicAdd(gh + 4 * i + 2, v.z);
    if (v.w) atomicAdd(gh + 4 * i + 3, v.w);
  }
}

bool select_plan_ok(const Layout& L) { return topk_plan_ok(L); }

cudaError_t launch_block_select(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* q,
                                int32_t* ids, int32_t* n_sel, float* scores_out, int max_nblk,
                                cudaStream_t s, const uint16_t* kin, const uint16_t* vin, bool own) {
  const int units = cs.n * L.n_kv;
  const int tiles = (max_nblk + kMT - 1) / kMT;
  int P = std::max(1, 152 / units);
  P = std::min(P, std::max(1, (tiles + kSelWarps - 1) / kSelWarps));
  const dim3 grid(units * P);
  // Dynamic shared memory: the meta tile stages (they also hold R_k^T and
  // R_v^T plus the append scratch before the scoring).
  const int dyn = kSelSmem;
  const bool append = kin != nullptr;
#define MK_SEL_CASE(GG)                                                                                       \
  case GG: {                                                                                                  \
    auto kern = append ? (own ? k_select<GG, true, true> : k_select<GG, true, false>)                       \
                       : (own ? k_select<GG, false, true> : k_select<GG, false, false>);                                             \
    cudaError_t e = kernel_smem_attr((const void*)kern, dyn, 256, nullptr, nullptr);                           \
    if (e != cudaSuccess) return e;                                                                            \
    e = launch_pdl(kern, grid, dim3(256), dyn, s, 0, L, layer, cs, P, q, ids, n_sel, scores_out,   \
                               dyn, kin, vin);                                                                 \
    if (e != cudaSuccess) return e;                                                                            \
    return launch_topk(L, layer, cs, ids, n_sel, append, s);                                                   \
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
