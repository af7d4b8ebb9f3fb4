// PackedAttention: decode attention straight from the packed pages, with
// dense sink and window tokens, online softmax, the rotated values
// accumulated by their channel indices, and the un-rotation by R_v.  The same
// kernel with dense items only and no rotation is the uncompressed reference.
//
// Method: "MosaicKV：...阅读笔记" (zhongzhuzhou.org), Eq. (1) (dense
// attention), Eq. (13) (attention on the kept tokens' compressed vectors),
// Eq. (14) (output = o R_v); "MosaicKV: Serving Long-Context LLM with Dynamic
// Two-D KV Cache Compression" (paperlayer.ai), sec. 5.3 (PackedAttention:
// attention on packed vectors with positions rebuilt on the fly, inverse
// rotation merged into the query).
//
// GB300 structure.
//  * Work items of one (sequence, kv head): dense chunks of 16 tokens (sinks,
//    window), then 16-token groups of the selected / always-attended pages.
//    They are split over Q clusters of C CTAs (8 warps each); every warp
//    double-buffers its items into shared memory with cp.async.
//  * Per group the warp rebuilds the positions: it zero-fills a 16 x 128 bf16
//    K tile and V tile and scatters the kept values by their channel indices
//    (lanes 0-15 keys, lanes 16-31 values).  Logits S^T[16 tok x 8 heads] and
//    the value sum O'^T[128 x 8 heads] then run on the tensor cores
//    (mma.sync m16n8k16, bf16 in, fp32 accumulate).  The fp32 operands q' and
//    p are split into bf16 hi + lo parts (two MMAs), so the products keep
//    ~16 significant bits: the rounding stays far below the 5e-3 tolerance.
//  * The split-T log-sum-exp merge: warps -> CTA in shared memory, CTAs ->
//    cluster through distributed shared memory (CTA `rank` owns output
//    channels [rank*128/C, (rank+1)*128/C)), clusters -> unit through the
//    workspace when Q > 1: the last cluster to arrive (atomic counter, no
//    waiting) merges and un-rotates.
#include <algorithm>
#include <cstdio>
#include <cstdlib>

#include <cooperative_groups.h>

#include "mk_internal.cuh"

namespace cg = cooperative_groups;

namespace mk {

namespace {
constexpr int kWarps = 8;
constexpr int kTG = 16;                      // tokens per group (one MMA tile)
constexpr int kRow = D + 8;                  // padded bf16 row: 272 bytes, ldmatrix conflict-free
constexpr int kTile = kTG * kRow;            // one 16-row tile (bf16 elements)
constexpr int kDenseStage = 2 * kTile * 2;   // staged dense chunk: K tile + V tile (bytes)
constexpr float kScaleLog2 = 0.08838834764831845f * 1.4426950408889634f;  // log2(e)/sqrt(128)

__device__ __forceinline__ int always_block(const UnitDesc& ud, int nblk, int i) {
  for (int s = 0; s < ud.n_seg; ++s) {
    if (!ud.always[s]) continue;
    const int lo = min(ud.first_block[s], nblk);
    const int hi = (s + 1 < ud.n_seg) ? min(ud.first_block[s + 1], nblk) : nblk;
    if (i < hi - lo) return lo + i;
    i -= max(0, hi - lo);
  }
  return -1;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// fp32 -> (hi, lo) bf16 pair with hi + lo ~ x to ~16 bits.
__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
}
__device__ __forceinline__ uint32_t pack2(uint16_t lo16, uint16_t hi16) {
  return (uint32_t)lo16 | ((uint32_t)hi16 << 16);
}

struct Task {
  int kind;      // 0 none, 1 dense chunk, 2 packed group, 3 skipped (bad block id)
  int item;
  int j0, nd;    // dense: first dense token and count
  int b, r, tg, n_live;
};

size_t smem_for(const Layout& L, int nst) {
  const size_t sb = (size_t)((std::max(6 * kTG * L.r_max, kDenseStage) + 15) / 16 * 16);
  const size_t per_warp = nst * sb + (size_t)kDenseStage + 2 * 8 * kTG * 2;  // stages, K/V tiles, P hi/lo
  return (size_t)kWarps * per_warp
         + (size_t)L.G * D * 4          // q' (fp32) for building the B fragments
         + (size_t)kWarps * 8 * 2 * 4   // per-warp (m, l) for 8 head slots
         + 8 * 2 * 4                    // CTA (m, l)
         + (size_t)2 * L.G * D * 4      // CTA acc, merged o'
         + 16;                          // flags
}
}  // namespace

// Shared-memory plan; fills attn_nst / attn_sb and returns the dynamic shared
// memory size (0 if nothing fits).
size_t attn_plan(Layout& L, int /*r_min*/) {
  for (int nst = 2; nst >= 1; --nst) {
    const size_t s = smem_for(L, nst);
    if (s <= 227 * 1024) {
      L.attn_tg = kTG;
      L.attn_nst = nst;
      L.attn_nc = 1;
      L.attn_sb = (int)((std::max(6 * kTG * L.r_max, kDenseStage) + 15) / 16 * 16);
      return s;
    }
  }
  return 0;
}

size_t attn_smem_bytes(const Layout& L, int) { return smem_for(L, L.attn_nst); }

template <int G, bool DENSE>
__global__ void __launch_bounds__(256, 1) k_attn(Layout L, int layer, CallSeqs cs, int Q,
                                                 const int32_t* __restrict__ ids,
                                                 const int32_t* __restrict__ n_sel_in,
                                                 const uint16_t* __restrict__ q_in, const uint16_t* __restrict__ Kd,
                                                 const uint16_t* __restrict__ Vd, int64_t t_stride,
                                                 uint16_t* __restrict__ out) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int NST = L.attn_nst, SB = L.attn_sb;

  extern __shared__ __align__(16) unsigned char smem[];
  const size_t per_warp = (size_t)NST * SB + kDenseStage + 2 * 8 * kTG * 2;
  unsigned char* warp_area = smem;                                             // [kWarps][per_warp]
  float* qs = reinterpret_cast<float*>(smem + kWarps * per_warp);              // [G][D]
  float* mlw = qs + G * D;                                                     // [kWarps][8][2]
  float* cl_ml = mlw + kWarps * 16;                                            // [8][2]
  float* cl_acc = cl_ml + 16;                                                  // [G][D]
  float* ofull = cl_acc + G * D;                                               // [G][D]
  int* flag = reinterpret_cast<int*>(ofull + G * D);
  __shared__ UnitDesc ud;
  __shared__ int s_abort, s_ns;

  const int per_unit = Q * C;
  const int unit_call = blockIdx.x / per_unit;
  const int kq = blockIdx.x - unit_call * per_unit;   // CTA index within the unit: q*C + rank
  const int qi = kq / C;
  const int ci = unit_call / L.n_kv, kvh = unit_call - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t u = DENSE ? 0 : unit_index(L, layer, seq, kvh);
  const int64_t slot = (int64_t)seq * L.n_kv + kvh;

  if (!DENSE && rank == 0 && qi == 0) {   // R_v is static: warm L2 before the wait
    const char* rv = unit_base(L, u) + L.off_rv;
    for (int i = tid; i < D * D * 4 / 128; i += blockDim.x) prefetch_l2(rv + (size_t)i * 128);
  }
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    s_abort = has_error(L);
    if (!DENSE) ud = L.desc[u];
    s_ns = DENSE ? 0 : n_sel_in[(int64_t)ci * L.n_kv + kvh];
  }
  __syncthreads();
  // Every CTA must reach the cluster barriers below: an abort only empties the work.
  bool skip = s_abort != 0;

  const int S = L.S, W = L.W, B = L.B;
  int n_sink = 0, win_lo = 0, n_dense, nblk = 0, n_mid = 0, ns = s_ns, n_always = 0;
  if (DENSE) {
    n_dense = cs.T_old[ci];
  } else {
    const int T = ud.T;
    n_sink = min(S, T);
    n_mid = n_mid_tokens(L, T);
    win_lo = S + n_mid;
    n_dense = n_sink + max(0, T - win_lo);
    nblk = n_mid_blocks(L, T);
    n_always = nblk - n_scored_blocks(ud, nblk);
    if (ns < 0 || ns > L.k_max) {
      if (tid == 0) set_error(L, ERR_BAD_NSEL, (int32_t)u, ns);
      skip = true;
      ns = 0;
    }
  }
  const int n_dch = (n_dense + kTG - 1) / kTG;
  const int n_items = skip ? 0 : n_dch + ns + n_always;
  const int per = (n_items + per_unit - 1) / per_unit;
  const int i0 = kq * per, i1 = min(n_items, i0 + per);

  for (int i = tid; i < G * D; i += blockDim.x) {
    float v = 0.0f;
    if (!skip) {
      if (DENSE) v = bf2f(q_in[((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D + i]);
      else v = L.qrot[slot * G * D + i];
    }
    qs[i] = v;
  }
  __syncthreads();

  // q'^T B fragments (k = channel, n = head), hi and lo parts: 8 k-chunks.
  uint32_t bqh[8][2], bql[8][2];
#pragma unroll
  for (int kc = 0; kc < 8; ++kc)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint16_t h0 = 0, l0 = 0, h1 = 0, l1 = 0;
      if (g < G) {
        const int c = kc * 16 + half * 8 + 2 * tig;
        split_bf16(qs[g * D + c], h0, l0);
        split_bf16(qs[g * D + c + 1], h1, l1);
      }
      bqh[kc][half] = pack2(h0, h1);
      bql[kc][half] = pack2(l0, l1);
    }

  const char* base = DENSE ? nullptr : unit_base(L, u);
  const int32_t* my_ids = DENSE ? nullptr : ids + ((int64_t)ci * L.n_kv + kvh) * L.k_max;
  unsigned char* my_area = warp_area + (size_t)warp * per_warp;
  uint16_t* tiles = reinterpret_cast<uint16_t*>(my_area + (size_t)NST * SB);           // K tile, V tile
  uint16_t* ps = reinterpret_cast<uint16_t*>(my_area + (size_t)NST * SB + kDenseStage);  // [2][8][16]

  float o[8][4];  // O'^T fragments: m-tile mt, rows = channels, cols = heads
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[mt][k] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;  // heads 2*tig, 2*tig+1

  auto make_task = [&](int it, int tg) -> Task {
    Task t{};
    if (it >= i1) return t;
    t.item = it;
    if (it < n_dch) {
      t.kind = 1;
      t.j0 = it * kTG;
      t.nd = min(kTG, n_dense - t.j0);
      return t;
    }
    const int pi = it - n_dch;
    const int b = pi < ns ? __ldg(my_ids + pi) : always_block(ud, nblk, pi - ns);
    if (b < 0 || b >= nblk) {
      if (lane == 0) set_error(L, ERR_BAD_BLOCK, (int32_t)u, b);
      t.kind = 3;
      return t;
    }
    t.kind = 2;
    t.b = b;
    t.r = ud.r[seg_of_block(ud, b)];
    t.tg = tg;
    t.n_live = min(B, n_mid - b * B);
    return t;
  };
  auto advance = [&](const Task& t) -> Task {
    if (t.kind == 2 && t.tg + kTG < t.n_live) return make_task(t.item, t.tg + kTG);
    return make_task(t.item + kWarps, 0);
  };
  auto dense_rows = [&](int j, const uint16_t*& kr, const uint16_t*& vr) {
    if (DENSE) {
      const int64_t off = (((int64_t)ci * L.n_kv + kvh) * t_stride + j) * D;
      kr = Kd + off;
      vr = Vd + off;
    } else if (j < n_sink) {
      kr = reinterpret_cast<const uint16_t*>(base + L.off_sink_k) + (int64_t)j * D;
      vr = reinterpret_cast<const uint16_t*>(base + L.off_sink_v) + (int64_t)j * D;
    } else {
      const int p = win_lo + (j - n_sink);
      const int64_t sl = (int64_t)((p - S) % W) * D;
      kr = reinterpret_cast<const uint16_t*>(base + L.off_win_k) + sl;
      vr = reinterpret_cast<const uint16_t*>(base + L.off_win_v) + sl;
    }
  };
  auto issue = [&](const Task& t, unsigned char* dst) {
    if (t.kind == 1) {
      // K tile then V tile, rows padded to 272 bytes.
      for (int i = lane; i < t.nd * 16; i += 32) {
        const int row = i >> 4, part = i & 15;
        const uint16_t *kr, *vr;
        dense_rows(t.j0 + row, kr, vr);
        cp_async16(dst + row * kRow * 2 + part * 16, kr + part * 8);
        cp_async16(dst + kTile * 2 + row * kRow * 2 + part * 16, vr + part * 8);
      }
    } else if (t.kind == 2) {
      // This group's rows of the page's four sub-arrays (B is a multiple of
      // 16, so a whole group stays inside the page; sizes and offsets are
      // multiples of 16 bytes).
      const int Br = B * t.r, gr = kTG * t.r;
      const char* page = base + L.off_pages + (int64_t)t.b * L.page_stride;
      const char* src[4] = {page + 2 * t.tg * t.r, page + 2 * Br + t.tg * t.r, page + 3 * Br + 2 * t.tg * t.r,
                            page + 5 * Br + t.tg * t.r};
      const int len[4] = {2 * gr, gr, 2 * gr, gr};
      int off = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        for (int i = lane * 16; i < len[q]; i += 32 * 16) cp_async16(dst + off + i, src[q] + i);
        off += len[q];
      }
    }
  };

  Task cur = make_task(i0 + warp, 0);
  int st = 0;
  issue(cur, my_area);
  cp_async_commit();
  while (cur.kind != 0) {
    const Task nxt = advance(cur);
    if (NST == 2) {
      issue(nxt, my_area + (size_t)(st ^ 1) * SB);
      cp_async_commit();
      asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    } else {
      cp_async_wait_all();
    }
    __syncwarp();
    const unsigned char* buf = my_area + (size_t)st * SB;
    if (cur.kind == 1 || cur.kind == 2) {
      const uint16_t* Kt;
      const uint16_t* Vt;
      int ntok;
      if (cur.kind == 1) {
        Kt = reinterpret_cast<const uint16_t*>(buf);
        Vt = Kt + kTile;
        ntok = cur.nd;
        if (ntok < kTG) {
          // rows past the chunk hold stale bytes: zero them (0 * NaN would poison P.V)
          uint16_t* kb = const_cast<uint16_t*>(Kt);
          for (int i = lane; i < (kTG - ntok) * 16; i += 32) {
            const int row = ntok + (i >> 4), part = i & 15;
            *reinterpret_cast<uint4*>(kb + row * kRow + part * 8) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(kb + kTile + row * kRow + part * 8) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
      } else {
        // Rebuild positions: zero both tiles, scatter kept values by index.
        uint4* z = reinterpret_cast<uint4*>(tiles);
#pragma unroll
        for (int i = lane; i < kDenseStage / 16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
        __syncwarp();
        const int r = cur.r, gr = kTG * r;
        ntok = min(kTG, cur.n_live - cur.tg);
        const int t = lane & 15;
        const bool is_v = lane >= 16;
        if (t < ntok) {
          const uint16_t* val = reinterpret_cast<const uint16_t*>(buf + (is_v ? 3 * gr : 0)) + t * r;
          const uint8_t* idx = buf + (is_v ? 5 * gr : 2 * gr) + t * r;
          uint16_t* row = tiles + (is_v ? kTile : 0) + t * kRow;
          if ((r & 1) == 0) {
            const uint16_t* i2 = reinterpret_cast<const uint16_t*>(idx);
            const uint32_t* v2 = reinterpret_cast<const uint32_t*>(val);
#pragma unroll 4
            for (int jj = 0; jj < (r >> 1); ++jj) {
              const uint32_t ip = i2[jj], vp = v2[jj];
              row[ip & 0xff] = (uint16_t)(vp & 0xffff);
              row[ip >> 8] = (uint16_t)(vp >> 16);
            }
          } else {
            for (int jj = 0; jj < r; ++jj) row[idx[jj]] = val[jj];
          }
        }
        __syncwarp();
        Kt = tiles;
        Vt = tiles + kTile;
      }

      // Logits S^T[token][head] = sum_c K[token][c] q'[head][c] (hi + lo parts).
      float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      {
        const int mi = lane >> 3, ri = lane & 7;
        const uint16_t* arow = Kt + (ri + (mi & 1) * 8) * kRow + (mi >> 1) * 8;
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {
          uint32_t a[4];
          ldsm_x4(a, arow + kc * 16);
          mma_bf16(s, a, bqh[kc][0], bqh[kc][1]);
          mma_bf16(s, a, bql[kc][0], bql[kc][1]);
        }
      }
      // Online softmax over this group's tokens (g, g+8) for heads 2tig, 2tig+1.
      const bool v_lo = g < ntok, v_hi = g + 8 < ntok;
      const float s00 = v_lo ? s[0] * kScaleLog2 : -INFINITY, s01 = v_lo ? s[1] * kScaleLog2 : -INFINITY;
      const float s10 = v_hi ? s[2] * kScaleLog2 : -INFINITY, s11 = v_hi ? s[3] * kScaleLog2 : -INFINITY;
      float x0 = fmaxf(s00, s10), x1 = fmaxf(s01, s11);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(FULL, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(FULL, x1, off));
      }
      const float mn0 = fmaxf(m0, x0), mn1 = fmaxf(m1, x1);
      const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
      const float p00 = exp2f(s00 - mn0), p01 = exp2f(s01 - mn1);
      const float p10 = exp2f(s10 - mn0), p11 = exp2f(s11 - mn1);
      float y0 = p00 + p10, y1 = p01 + p11;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        y0 += __shfl_xor_sync(FULL, y0, off);
        y1 += __shfl_xor_sync(FULL, y1, off);
      }
      l0 = l0 * a0 + y0;
      l1 = l1 * a1 + y1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
      // P (hi, lo) to shared memory as [head][token], read back as B fragments.
      {
        uint16_t h, lw;
        const int h0 = 2 * tig, h1 = 2 * tig + 1;
        split_bf16(p00, h, lw); ps[h0 * kTG + g] = h; ps[128 + h0 * kTG + g] = lw;
        split_bf16(p01, h, lw); ps[h1 * kTG + g] = h; ps[128 + h1 * kTG + g] = lw;
        split_bf16(p10, h, lw); ps[h0 * kTG + g + 8] = h; ps[128 + h0 * kTG + g + 8] = lw;
        split_bf16(p11, h, lw); ps[h1 * kTG + g + 8] = h; ps[128 + h1 * kTG + g + 8] = lw;
      }
      __syncwarp();
      const uint32_t* ps32 = reinterpret_cast<const uint32_t*>(ps);
      const uint32_t pbh0 = ps32[(g * kTG + 2 * tig) >> 1], pbh1 = ps32[(g * kTG + 2 * tig + 8) >> 1];
      const uint32_t pbl0 = ps32[(128 + g * kTG + 2 * tig) >> 1], pbl1 = ps32[(128 + g * kTG + 2 * tig + 8) >> 1];
      // O'^T[channel][head] += sum_token V[token][channel] P[token][head].
      {
        const int mi = lane >> 3, ri = lane & 7;
        const uint16_t* vrow = Vt + (ri + (mi >> 1) * 8) * kRow + (mi & 1) * 8;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t a[4];
          ldsm_x4_t(a, vrow + mt * 16);
          mma_bf16(o[mt], a, pbh0, pbh1);
          mma_bf16(o[mt], a, pbl0, pbl1);
        }
      }
    }
    __syncwarp();
    if (NST == 1) {
      issue(nxt, my_area);
      cp_async_commit();
    }
    cur = nxt;
    st ^= (NST - 1);
  }
  cp_async_wait_all();
  __syncwarp();

  // ---- merge: warps -> CTA ------------------------------------------------
  if (g == 0) {
    mlw[(warp * 8 + 2 * tig) * 2] = m0;
    mlw[(warp * 8 + 2 * tig) * 2 + 1] = l0;
    mlw[(warp * 8 + 2 * tig + 1) * 2] = m1;
    mlw[(warp * 8 + 2 * tig + 1) * 2 + 1] = l1;
  }
  __syncthreads();
  float* dump = reinterpret_cast<float*>(warp_area);  // [kWarps][G][D], main loop is over
  {
    float e0 = 0.0f, e1 = 0.0f;
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    float M0 = -INFINITY, M1 = -INFINITY;
    for (int w = 0; w < kWarps; ++w) {
      M0 = fmaxf(M0, mlw[(w * 8 + h0) * 2]);
      M1 = fmaxf(M1, mlw[(w * 8 + h1) * 2]);
    }
    if (m0 != -INFINITY) e0 = exp2f(m0 - M0);
    if (m1 != -INFINITY) e1 = exp2f(m1 - M1);
    float* dw = dump + (size_t)warp * G * D;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int c = mt * 16 + g;
      if (h0 < G) {
        dw[h0 * D + c] = o[mt][0] * e0;
        dw[h0 * D + c + 8] = o[mt][2] * e0;
      }
      if (h1 < G) {
        dw[h1 * D + c] = o[mt][1] * e1;
        dw[h1 * D + c + 8] = o[mt][3] * e1;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += blockDim.x) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) a += dump[(size_t)w * G * D + i];
    cl_acc[i] = a;
  }
  if (tid < G) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mlw[(w * 8 + tid) * 2]);
    float ls = 0.0f;
    if (M != -INFINITY)
      for (int w = 0; w < kWarps; ++w) {
        const float mw = mlw[(w * 8 + tid) * 2];
        if (mw != -INFINITY) ls += mlw[(w * 8 + tid) * 2 + 1] * exp2f(mw - M);
      }
    cl_ml[tid * 2] = M;
    cl_ml[tid * 2 + 1] = ls;
  }
  cluster.sync();

  // ---- merge: CTAs -> cluster, for this CTA's channel slice ---------------
  const int w = D / C, c_lo = rank * w;
  float* part_acc = L.part_acc + slot * MK_MAX_SPLITS * G * D;
  float* part_ml = L.part_ml + slot * MK_MAX_SPLITS * G * 2;
  for (int i = tid; i < G * w; i += blockDim.x) {
    const int h = i / w, c = c_lo + (i - h * w);
    float M = -INFINITY;
    for (int r2 = 0; r2 < C; ++r2) M = fmaxf(M, cluster.map_shared_rank(cl_ml, r2)[h * 2]);
    float a = 0.0f, ls = 0.0f;
    if (M != -INFINITY)
      for (int r2 = 0; r2 < C; ++r2) {
        const float* ml = cluster.map_shared_rank(cl_ml, r2);
        const float mr = ml[h * 2];
        if (mr == -INFINITY) continue;
        const float e = exp2f(mr - M);
        a = fmaf(cluster.map_shared_rank(cl_acc, r2)[h * D + c], e, a);
        ls = fmaf(ml[h * 2 + 1], e, ls);
      }
    if (Q == 1) {
      const float v = ls > 0.0f ? a / ls : 0.0f;
      for (int r2 = 0; r2 < C; ++r2) cluster.map_shared_rank(ofull, r2)[h * D + c] = v;
    } else {
      part_acc[((size_t)qi * G + h) * D + c] = a;
      if (i - h * w == 0 && rank == 0) {
        part_ml[((size_t)qi * G + h) * 2] = M;
        part_ml[((size_t)qi * G + h) * 2 + 1] = ls;
      }
    }
  }
  if (Q > 1) {
    // ---- merge: clusters -> unit (last cluster to arrive) -----------------
    __threadfence();
    cluster.sync();
    if (rank == 0 && tid == 0) {
      const int prev = atomicAdd(&L.counters[slot], 1);
      *flag = (prev == Q - 1);
      if (prev == Q - 1) L.counters[slot] = 0;
    }
    cluster.sync();
    const int last = *cluster.map_shared_rank(flag, 0);
    if (!last) {
      cluster.sync();  // same barrier count in every CTA of the cluster
      return;
    }
    __threadfence();
    for (int i = tid; i < G * w; i += blockDim.x) {
      const int h = i / w, c = c_lo + (i - h * w);
      float M = -INFINITY;
      for (int q2 = 0; q2 < Q; ++q2) M = fmaxf(M, __ldcg(part_ml + ((size_t)q2 * G + h) * 2));
      float a = 0.0f, ls = 0.0f;
      if (M != -INFINITY)
        for (int q2 = 0; q2 < Q; ++q2) {
          const float mq = __ldcg(part_ml + ((size_t)q2 * G + h) * 2);
          if (mq == -INFINITY) continue;
          const float e = exp2f(mq - M);
          a = fmaf(__ldcg(part_acc + ((size_t)q2 * G + h) * D + c), e, a);
          ls = fmaf(__ldcg(part_ml + ((size_t)q2 * G + h) * 2 + 1), e, ls);
        }
      const float v = ls > 0.0f ? a / ls : 0.0f;
      for (int r2 = 0; r2 < C; ++r2) cluster.map_shared_rank(ofull, r2)[h * D + c] = v;
    }
  }
  cluster.sync();
  if (s_abort) return;

  // ---- output channels [c_lo, c_lo + w): out_j = sum_c o'_c R_v[c][j] ------
  uint16_t* orow = out + ((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D;
  if (DENSE) {
    for (int i = tid; i < G * w; i += blockDim.x) {
      const int h = i / w, j = c_lo + (i - h * w);
      orow[h * D + j] = f2bf(ofull[h * D + j]);
    }
    return;
  }
  float* rvs = reinterpret_cast<float*>(warp_area);   // [128][w] staged R_v columns
  float* red = rvs + D * w;                           // [parts][G*w]
  const float* Rv = reinterpret_cast<const float*>(base + L.off_rv);
  const int w4 = w / 4;
  for (int i = tid; i < D * w4; i += blockDim.x) {
    const int c = i / w4, q4 = i - c * w4;
    cp_async16(rvs + c * w + 4 * q4, Rv + (size_t)c * D + c_lo + 4 * q4);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  const int outs = G * w;
  const int parts = max(1, (int)blockDim.x / outs);
  const int cper = D / parts;
  for (int i = tid; i < outs * parts; i += blockDim.x) {
    const int oo = i % outs, pidx = i / outs;
    const int h = oo / w, jl = oo - h * w;
    float a = 0.0f;
    for (int c = pidx * cper; c < (pidx + 1) * cper; ++c) a = fmaf(ofull[h * D + c], rvs[c * w + jl], a);
    red[pidx * outs + oo] = a;
  }
  __syncthreads();
  for (int oo = tid; oo < outs; oo += blockDim.x) {
    float a = 0.0f;
    for (int pidx = 0; pidx < parts; ++pidx) a += red[pidx * outs + oo];
    const int h = oo / w, jl = oo - h * w;
    orow[h * D + c_lo + jl] = f2bf(a);
  }
}

namespace {
// Cluster size C and clusters per unit Q: every cluster resident at once
// (checked against cudaOccupancyMaxActiveClusters), as many CTAs as the SMs
// allow, preferring larger clusters when the CTA count is within 90%.
template <int G, bool DENSE>
void choose_grid(int units, int max_items, size_t smem, int& C, int& Q) {
  static int max_active[17];
  static size_t for_smem = 0;
  if (for_smem != smem) {
    for (int c = 1; c <= 16; c *= 2) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c, 1, 1);
      cfg.blockDim = dim3(256, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = c;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k_attn<G, DENSE>, &cfg);
      if (e != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      max_active[c] = n;
      if (std::getenv("MK_LOG"))
        std::fprintf(stderr, "[mosaickv] attention G=%d dense=%d smem=%zu: cluster %d -> %d resident\n", G,
                     (int)DENSE, smem, c, n);
    }
    for_smem = smem;
  }
  int best = 0;
  for (int c = 1; c <= 16; c *= 2) {
    if (max_active[c] < units) continue;
    int q = std::min(MK_MAX_SPLITS, max_active[c] / units);
    q = std::min(q, std::max(1, max_items / (2 * c)));
    best = std::max(best, units * q * c);
  }
  C = 1;
  Q = 1;
  for (int c = 16; c >= 1; c /= 2) {
    if (max_active[c] < units) continue;
    int q = std::min(MK_MAX_SPLITS, max_active[c] / units);
    q = std::min(q, std::max(1, max_items / (2 * c)));
    if ((int64_t)units * q * c * 10 >= (int64_t)best * 9) {
      C = c;
      Q = q;
      break;
    }
  }
}

template <int G, bool DENSE>
cudaError_t launch_one(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids, const int32_t* n_sel,
                       const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t t_stride, uint16_t* out,
                       int max_items, size_t smem, cudaStream_t s) {
  static size_t set_bytes = 0;
  if (smem > set_bytes) {
    cudaError_t e = cudaFuncSetAttribute(k_attn<G, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_attn<G, DENSE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    set_bytes = smem;
  }
  const int units = cs.n * L.n_kv;
  int C = 1, Q = 1;
  choose_grid<G, DENSE>(units, max_items, smem, C, Q);
  if (std::getenv("MK_LOG"))
    std::fprintf(stderr, "[mosaickv] attention launch: %d units x Q=%d clusters x C=%d CTAs\n", units, Q, C);
  return launch_pdl(k_attn<G, DENSE>, dim3(units * Q * C), dim3(256), smem, s, C, L, layer, cs, Q, ids, n_sel, q,
                    K, V, t_stride, out);
}

template <bool DENSE>
cudaError_t launch_attn_g(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids, const int32_t* n_sel,
                          const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t t_stride, uint16_t* out,
                          int max_items, cudaStream_t s) {
  const size_t smem = attn_smem_bytes(L, 0);
  if (smem == 0 || smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  switch (L.G) {
    case 1: return launch_one<1, DENSE>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, max_items, smem, s);
    case 2: return launch_one<2, DENSE>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, max_items, smem, s);
    case 4: return launch_one<4, DENSE>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, max_items, smem, s);
    case 8: return launch_one<8, DENSE>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, max_items, smem, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_decode_attn(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids,
                               const int32_t* n_sel, uint16_t* out, int max_items, cudaStream_t s) {
  return launch_attn_g<false>(L, layer, cs, ids, n_sel, nullptr, nullptr, nullptr, 0, out, max_items, s);
}

cudaError_t launch_dense_attn(const Layout& L, const CallSeqs& cs, const uint16_t* q, const uint16_t* K,
                              const uint16_t* V, int64_t t_stride, uint16_t* out, int max_items, cudaStream_t s) {
  return launch_attn_g<true>(L, 0, cs, nullptr, nullptr, q, K, V, t_stride, out, max_items, s);
}

}  // namespace mk
