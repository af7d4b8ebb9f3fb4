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
//  * Work items of one (sequence, kv head): dense chunks of 8 tokens (sinks,
//    window), then 16-token groups of the selected / always-attended pages.
//    P CTAs (8 warps, two CTAs per SM) share them; each warp double-buffers
//    its items into shared memory with cp.async.
//  * Per group the warp rebuilds positions in one 16 x 128 bf16 tile: it
//    zero-fills it and scatters the kept key values by their channel indices
//    (two lanes per token), computes the logits S^T[16 tok x 8 heads] on the
//    tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate), then does the
//    same for the values and accumulates O'^T[128 x 8 heads].  The fp32
//    operands q' and p are split into bf16 hi + lo parts (two MMAs), keeping
//    ~16 significant bits, far below the 5e-3 tolerance.
//  * Split-T merge: warps -> CTA in shared memory, CTA partials (m, l, acc)
//    -> workspace; the last CTA of the unit to arrive (atomic counter, no
//    waiting) stages all partials with one cp.async burst, merges them
//    (log-sum-exp), un-rotates (out = o' R_v) and stores bf16.
#include <algorithm>
#include <cstdio>
#include <cstdlib>

#include "mk_internal.cuh"

namespace mk {

namespace {
constexpr int kWarps = 8;
constexpr int kTG = 16;                      // tokens per packed group (one MMA tile)
constexpr int kDC = 8;                       // tokens per dense chunk
constexpr int kRow = D + 8;                  // padded bf16 row: 272 bytes, ldmatrix conflict-free
constexpr int kTileBytes = kTG * kRow * 2;   // 16-row tile
constexpr int kDenseStage = 2 * kDC * kRow * 2;  // staged dense chunk: 8 K rows + 8 V rows
constexpr int kPsBytes = 2 * 8 * kTG * 2;    // P hi/lo as [8 heads][16 tokens]
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

// Rebuild one token's dense row from its packed (values, indices): the row is
// zero already.  Lanes t and t + 16 share token t and split its elements.
__device__ __forceinline__ void scatter_row(uint16_t* row, const uint16_t* val, const uint8_t* idx, int r,
                                            int lane) {
  const int h2 = (r >> 1) & ~1;
  const int j0 = lane < 16 ? 0 : h2, j1 = lane < 16 ? h2 : r;
  if ((r & 1) == 0) {
    for (int jj = j0; jj < j1; jj += 2) {
      const uint32_t ip = *reinterpret_cast<const uint16_t*>(idx + jj);
      const uint32_t vp = *reinterpret_cast<const uint32_t*>(val + jj);
      row[ip & 0xff] = (uint16_t)(vp & 0xffff);
      row[ip >> 8] = (uint16_t)(vp >> 16);
    }
  } else {
    for (int jj = j0; jj < j1; ++jj) row[idx[jj]] = val[jj];
  }
}

struct Task {
  int kind;      // 0 none, 1 dense chunk, 2 packed group, 3 skipped (bad block id)
  int item;
  int j0, nd;    // dense: first dense token and count
  int b, r, tg, n_live;
};

int stage_bytes(const Layout& L) { return (std::max(6 * kTG * L.r_max, kDenseStage) + 15) / 16 * 16; }
size_t per_warp_bytes(const Layout& L, int nst) { return (size_t)nst * stage_bytes(L) + kTileBytes + kPsBytes; }
size_t smem_for(const Layout& L, int nst) {
  return (size_t)kWarps * per_warp_bytes(L, nst) + (size_t)kWarps * 8 * 2 * 4 + kRow * 2 + 64;
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
      L.attn_sb = stage_bytes(L);
      return s;
    }
  }
  return 0;
}

size_t attn_smem_bytes(const Layout& L, int) { return smem_for(L, L.attn_nst); }

// Largest number of CTAs per unit whose partials the merging CTA can stage
// (next to the merged o' and the un-rotation halves).
int attn_max_parts(const Layout& L) {
  const int64_t avail = (int64_t)kWarps * per_warp_bytes(L, L.attn_nst) - (int64_t)3 * L.G * D * 4 - 64;  // o', halves
  return (int)std::max<int64_t>(1, std::min<int64_t>(MK_MAX_SPLITS, avail / ((int64_t)L.G * (D + 2) * 4)));
}

template <int G, bool DENSE>
__global__ void __launch_bounds__(256, 2) k_attn(Layout L, int layer, CallSeqs cs, int P,
                                                 const int32_t* __restrict__ ids,
                                                 const int32_t* __restrict__ n_sel_in,
                                                 const uint16_t* __restrict__ q_in, const uint16_t* __restrict__ Kd,
                                                 const uint16_t* __restrict__ Vd, int64_t t_stride,
                                                 uint16_t* __restrict__ out) {
  const int NST = L.attn_nst, SB = L.attn_sb;
  extern __shared__ __align__(16) unsigned char smem[];
  const size_t pwb = (size_t)NST * SB + kTileBytes + kPsBytes;
  unsigned char* warp_area = smem;                                       // [kWarps][pwb]
  float* mlw = reinterpret_cast<float*>(smem + kWarps * pwb);            // [kWarps][8][2]
  uint16_t* zrow = reinterpret_cast<uint16_t*>(mlw + kWarps * 16);      // one zero row (272 B)
  __shared__ UnitDesc ud;
  __shared__ int s_abort, s_ns, s_last;
  __shared__ float s_m[8], s_l[8];

  const int unit_call = blockIdx.x / P;
  const int part = blockIdx.x - unit_call * P;
  const int ci = unit_call / L.n_kv, kvh = unit_call - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t u = DENSE ? 0 : unit_index(L, layer, seq, kvh);
  const int64_t slot = (int64_t)seq * L.n_kv + kvh;

  if (!DENSE && part == 0) {  // R_v is static: warm L2 for the final un-rotation
    const char* rv = unit_base(L, u) + L.off_rv;
    for (int i = tid; i < D * D * 4 / 128; i += blockDim.x) prefetch_l2(rv + (size_t)i * 128);
  }
  for (int i = tid; i < kRow / 8; i += blockDim.x) reinterpret_cast<uint4*>(zrow)[i] = make_uint4(0, 0, 0, 0);
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    s_abort = has_error(L);
    if (!DENSE) ud = L.desc[u];
    s_ns = DENSE ? 0 : n_sel_in[(int64_t)ci * L.n_kv + kvh];
  }
  __syncthreads();
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
  const int n_dch = (n_dense + kDC - 1) / kDC;
  const int n_items = skip ? 0 : n_dch + ns + n_always;
  const int per = (n_items + P - 1) / P;
  const int i0 = part * per, i1 = min(n_items, i0 + per);

  const char* base = DENSE ? nullptr : unit_base(L, u);
  const int32_t* my_ids = DENSE ? nullptr : ids + ((int64_t)ci * L.n_kv + kvh) * L.k_max;
  unsigned char* my_area = warp_area + (size_t)warp * pwb;
  uint16_t* tile = reinterpret_cast<uint16_t*>(my_area + (size_t)NST * SB);
  uint16_t* ps = reinterpret_cast<uint16_t*>(my_area + (size_t)NST * SB + kTileBytes);

  auto make_task = [&](int it, int tg) -> Task {
    Task t{};
    if (it >= i1) return t;
    t.item = it;
    if (it < n_dch) {
      t.kind = 1;
      t.j0 = it * kDC;
      t.nd = min(kDC, n_dense - t.j0);
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
      // 8 K rows then 8 V rows, padded to 272 bytes.
      for (int i = lane; i < t.nd * 16; i += 32) {
        const int row = i >> 4, prt = i & 15;
        const uint16_t *kr, *vr;
        dense_rows(t.j0 + row, kr, vr);
        cp_async16(dst + row * kRow * 2 + prt * 16, kr + prt * 8);
        cp_async16(dst + (kDC + row) * kRow * 2 + prt * 16, vr + prt * 8);
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

  // Start the first item's copies before reading q'.
  Task cur = make_task(i0 + warp, 0);
  int st = 0;
  issue(cur, my_area);
  cp_async_commit();

  // q'^T B fragments (k = channel, n = head), hi and lo parts: 8 k-chunks.
  uint32_t bqh[8][2], bql[8][2];
  {
    const float* qrot = L.qrot + slot * G * D;
    const uint16_t* qin = DENSE ? q_in + ((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D : nullptr;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint16_t h0 = 0, l0 = 0, h1 = 0, l1 = 0;
        if (g < G && !skip) {
          const int c = kc * 16 + hf * 8 + 2 * tig;
          float x0, x1;
          if (DENSE) {
            x0 = bf2f(qin[g * D + c]);
            x1 = bf2f(qin[g * D + c + 1]);
          } else {
            const float2 v = *reinterpret_cast<const float2*>(qrot + g * D + c);
            x0 = v.x;
            x1 = v.y;
          }
          split_bf16(x0, h0, l0);
          split_bf16(x1, h1, l1);
        }
        bqh[kc][hf] = pack2(h0, h1);
        bql[kc][hf] = pack2(l0, l1);
      }
  }

  float o[8][4];  // O'^T fragments: m-tile mt, rows = channels, cols = heads
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[mt][k] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;  // heads 2*tig, 2*tig+1

  const int mi = lane >> 3, ri = lane & 7;
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
      int ntok;
      const uint16_t* arow_k;   // this lane's ldmatrix row address for the key tile
      if (cur.kind == 1) {
        ntok = cur.nd;
        const int row = ri + (mi & 1) * 8;
        const uint16_t* kb = reinterpret_cast<const uint16_t*>(buf);
        arow_k = (row < ntok ? kb + row * kRow : zrow) + (mi >> 1) * 8;
      } else {
        ntok = min(kTG, cur.n_live - cur.tg);
        // Rebuild key positions: zero the tile, scatter by channel index.
        uint4* z = reinterpret_cast<uint4*>(tile);
        for (int i = lane; i < kTileBytes / 16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
        __syncwarp();
        const int r = cur.r, t = lane & 15;
        if (t < ntok)
          scatter_row(tile + t * kRow, reinterpret_cast<const uint16_t*>(buf) + t * r, buf + 2 * kTG * r + t * r, r,
                      lane);
        __syncwarp();
        arow_k = tile + (ri + (mi & 1) * 8) * kRow + (mi >> 1) * 8;
      }

      // Logits S^T[token][head] = sum_c K[token][c] q'[head][c] (hi + lo parts).
      float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        uint32_t a[4];
        ldsm_x4(a, arow_k + kc * 16);
        mma_bf16(s, a, bqh[kc][0], bqh[kc][1]);
        mma_bf16(s, a, bql[kc][0], bql[kc][1]);
      }
      // Online softmax over this item's tokens (g, g+8) for heads 2tig, 2tig+1.
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
      // Value tile: dense rows in the stage, or rebuilt in the (now free) tile.
      const int vrow = ri + (mi >> 1) * 8;  // ldmatrix.trans rows are tokens
      const uint16_t* vrow_base;
      if (cur.kind == 1) {
        const uint16_t* vb = reinterpret_cast<const uint16_t*>(buf) + kDC * kRow;
        vrow_base = (vrow < ntok ? vb + vrow * kRow : zrow) + (mi & 1) * 8;
        __syncwarp();
      } else {
        __syncwarp();  // the key tile's ldmatrix reads are done
        uint4* z = reinterpret_cast<uint4*>(tile);
        for (int i = lane; i < kTileBytes / 16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
        __syncwarp();
        const int r = cur.r, t = lane & 15, gr = kTG * r;
        if (t < ntok)
          scatter_row(tile + t * kRow, reinterpret_cast<const uint16_t*>(buf + 3 * gr) + t * r, buf + 5 * gr + t * r,
                      r, lane);
        __syncwarp();
        vrow_base = tile + vrow * kRow + (mi & 1) * 8;
      }
      const uint32_t* ps32 = reinterpret_cast<const uint32_t*>(ps);
      const uint32_t pbh0 = ps32[(g * kTG + 2 * tig) >> 1], pbh1 = ps32[(g * kTG + 2 * tig + 8) >> 1];
      const uint32_t pbl0 = ps32[(128 + g * kTG + 2 * tig) >> 1], pbl1 = ps32[(128 + g * kTG + 2 * tig + 8) >> 1];
      // O'^T[channel][head] += sum_token V[token][channel] P[token][head].
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4];
        ldsm_x4_t(a, vrow_base + mt * 16);
        mma_bf16(o[mt], a, pbh0, pbh1);
        mma_bf16(o[mt], a, pbl0, pbl1);
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

  // ---- warps -> CTA partial ------------------------------------------------
  if (g == 0) {
    mlw[(warp * 8 + 2 * tig) * 2] = m0;
    mlw[(warp * 8 + 2 * tig) * 2 + 1] = l0;
    mlw[(warp * 8 + 2 * tig + 1) * 2] = m1;
    mlw[(warp * 8 + 2 * tig + 1) * 2 + 1] = l1;
  }
  __syncthreads();
  float* dump = reinterpret_cast<float*>(warp_area);  // [kWarps][G][D] (main loop is over)
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
  if (tid < G) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mlw[(w * 8 + tid) * 2]);
    float ls = 0.0f;
    if (M != -INFINITY)
      for (int w = 0; w < kWarps; ++w) {
        const float mw = mlw[(w * 8 + tid) * 2];
        if (mw != -INFINITY) ls += mlw[(w * 8 + tid) * 2 + 1] * exp2f(mw - M);
      }
    s_m[tid] = M;
    s_l[tid] = ls;
  }
  __syncthreads();
  float* pacc = L.part_acc + slot * MK_MAX_SPLITS * G * D;   // [part][G][D]
  float* pml = L.part_ml + slot * MK_MAX_SPLITS * G * 2;     // [part][G][2]
  for (int i = tid; i < G * D; i += blockDim.x) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) a += dump[(size_t)w * G * D + i];
    pacc[(size_t)part * G * D + i] = a;
  }
  if (tid < G) {
    pml[(part * G + tid) * 2] = s_m[tid];
    pml[(part * G + tid) * 2 + 1] = s_l[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&L.counters[slot], 1);
    s_last = (prev == P - 1);
    if (prev == P - 1) L.counters[slot] = 0;
  }
  __syncthreads();
  if (!s_last || s_abort) return;
  __threadfence();

  // ---- the last CTA: merge the P partials, un-rotate, store ----------------
  float* ofull = reinterpret_cast<float*>(warp_area);       // [G][D]
  float* red = ofull + G * D;                                // [2][G][D]
  float* sacc = red + 2 * G * D;                             // [P][G][D]
  float* sml = sacc + (size_t)P * G * D;                     // [P][G][2]
  for (int i = tid; i < P * G * D / 4; i += blockDim.x) cp_async16(sacc + 4 * i, pacc + 4 * i);
  for (int i = tid; i < (P * G * 2 + 3) / 4; i += blockDim.x) cp_async16(sml + 4 * i, pml + 4 * i);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int p = 0; p < P; ++p) M = fmaxf(M, sml[(p * G + tid) * 2]);
    float ls = 0.0f;
    if (M != -INFINITY)
      for (int p = 0; p < P; ++p) {
        const float mp = sml[(p * G + tid) * 2];
        if (mp != -INFINITY) ls += sml[(p * G + tid) * 2 + 1] * exp2f(mp - M);
      }
    s_m[tid] = M;
    s_l[tid] = ls;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int h = i / D;
    const float M = s_m[h], ls = s_l[h];
    float a = 0.0f;
    if (M != -INFINITY && ls > 0.0f) {
      for (int p = 0; p < P; ++p) {
        const float mp = sml[(p * G + h) * 2];
        if (mp != -INFINITY) a = fmaf(sacc[(size_t)p * G * D + i], exp2f(mp - M), a);
      }
      a /= ls;
    }
    ofull[i] = a;
  }
  __syncthreads();
  uint16_t* orow = out + ((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D;
  if (DENSE) {
    for (int i = tid; i < G * D; i += blockDim.x) orow[i] = f2bf(ofull[i]);
    return;
  }
  // out[h][j] = sum_c o'[h][c] R_v[c][j]: R_v staged over the partials (one
  // cp.async burst) when it fits, then thread (j, half of c), halves summed.
  const float* Rv = reinterpret_cast<const float*>(base + L.off_rv);
  const bool rv_smem = (size_t)(3 * G * D) * 4 + (size_t)D * D * 4 <= (size_t)kWarps * pwb;
  if (rv_smem) {
    for (int i = tid; i < D * D / 4; i += blockDim.x) cp_async16(sacc + 4 * i, Rv + 4 * i);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
  }
  const float* Rsrc = rv_smem ? sacc : Rv;
  {
    const int j = tid & (D - 1), half = tid >> 7;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.0f;
    const float* Rc = Rsrc + (size_t)half * 64 * D + j;
#pragma unroll 16
    for (int c = 0; c < 64; ++c) {
      const float rr = Rc[(size_t)c * D];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = fmaf(ofull[h * D + half * 64 + c], rr, acc[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) red[(half * G + h) * D + j] = acc[h];
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += blockDim.x) orow[i] = f2bf(red[i] + red[G * D + i]);
}

namespace {
template <int G, bool DENSE>
cudaError_t launch_one(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids, const int32_t* n_sel,
                       const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t t_stride, uint16_t* out,
                       int max_items, size_t smem, cudaStream_t s) {
  static size_t set_bytes = 0;
  static int occ = 1, sms = 0;
  if (smem > set_bytes) {
    cudaError_t e = cudaFuncSetAttribute(k_attn<G, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    set_bytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_attn<G, DENSE>, 256, smem) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 1;
    }
    occ = std::max(1, n);
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) ==
                                                  cudaSuccess)
      sms = v;
  }
  const int units = cs.n * L.n_kv;
  int P = std::max(1, (std::max(sms, 1) * occ) / units);
  P = std::min(P, std::max(1, max_items / 2));
  P = std::min(P, attn_max_parts(L));
  if (std::getenv("MK_LOG"))
    std::fprintf(stderr, "[mosaickv] attention: %d units x %d CTAs (%d per SM), %zu B smem\n", units, P, occ, smem);
  return launch_pdl(k_attn<G, DENSE>, dim3(units * P), dim3(256), smem, s, 0, L, layer, cs, P, ids, n_sel, q, K, V,
                    t_stride, out);
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
