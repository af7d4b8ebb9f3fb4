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
//  * Work items of one (sequence, kv head): the selected and always-attended
//    pages (16-token groups), then dense chunks of 8 tokens (sinks, window).
//    P CTAs (one per SM) share them.  Short selections use 12 warps, each
//    double-buffering its items into shared memory by bulk copies; long ones
//    16 warps with one stage each, the next copy issued as soon as the stage
//    is consumed.
//  * Per group the warp rebuilds positions in a 16 x 128 bf16 key tile and a
//    value tile: it zero-fills them and scatters the kept values by their
//    channel indices, lanes taking consecutive packed elements (coalesced
//    loads, few bank conflicts).  Kept channels are stored ascending, so a
//    token's last index is its highest channel; only the 16-channel chunks up
//    to the group's highest one are zeroed, loaded and multiplied (in the
//    rotated basis the kept channels gather in the leading ones).
//  * The logits are computed as S[head][token] = q' K^T on the tensor cores
//    (mma.sync m16n8k16, bf16 in, fp32 accumulate; q' is the A operand, the
//    key tile the B operand), which leaves each lane holding the softmax
//    weights of one head for four tokens in exactly the B-operand layout of
//    the value product: P never leaves the registers.  Then
//    O'^T[128 x 8] += V^T P accumulates on the tensor cores.  The fp32
//    operands q' and p are split into bf16 hi + lo parts (~16 significant
//    bits, far below the 5e-3 tolerance): q' hi in A rows 0-7 and lo in rows
//    8-15, so one MMA per 16 channels yields both partial logits; with G <= 4
//    heads, P hi fills B columns 0-3 and P lo columns 4-7, so one MMA per 16
//    channels accumulates both (the columns are added once at the end).
//  * Online softmax with a lazily raised running max: the accumulators are
//    rescaled only when a group's max exceeds the running one by more than
//    2^8 (weights stay <= 2^8, exact in the hi + lo split), so most groups
//    skip the rescale.
//  * Split-T merge: warps -> CTA in shared memory; each CTA un-rotates its
//    partial (o'_p R_v, with R_v staged by a bulk copy) and writes (m, l,
//    acc) to the workspace; the last CTA of the unit to arrive (atomic
//    counter, no waiting) stages all partials with one bulk copy, merges
//    them (log-sum-exp weights) and stores bf16.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>

#include "mk_internal.cuh"

namespace mk {

namespace {
// Kernel variants of the packed path: uint8 indices, every segment in the
// head's rotation; uint8 indices with rotation classes (segments under their
// own rotation); bitmap pages (rotation classes checked at run time).
constexpr int kModePlain = 0, kModeOwn = 1, kModeBitmap = 2;
constexpr int kMaxWarps = 16;                // one CTA per SM, 4 to 16 warps (shared memory decides)
constexpr int kTG = 16;                      // tokens per packed group (one MMA tile)
constexpr int kDC = 8;                       // tokens per dense chunk
constexpr int kRow = D + 8;                  // padded bf16 row: 272 bytes, ldmatrix conflict-free
constexpr int kTileBytes = kTG * kRow * 2;   // 16-row tile
constexpr int kDenseStage = 2 * kDC * kRow * 2;  // staged dense chunk: 8 K rows + 8 V rows
constexpr int kIdsCap = 256;                 // block ids a CTA caches in shared memory
constexpr int kLongSelTokens = 32768;        // selected tokens per unit from which 16 warps pay off
constexpr float kLazy = 8.0f;                // log2 headroom before the running max is raised
constexpr float kScaleLog2 = 0.08838834764831845f * 1.4426950408889634f;  // log2(e)/sqrt(128)

__device__ __forceinline__ int always_block(const UnitDesc& ud, int nblk, int i) {
  for (int s = 0; s < ud.n_seg; ++s) {
    if (!seg_always(ud, s)) continue;
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
// (x0, x1) -> packed bf16x2 hi parts and lo parts (x ~ hi + lo to ~16 bits).
__device__ __forceinline__ void split2_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  unsigned short v;
  asm("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_u16(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;\n" ::"r"(a), "h"((unsigned short)v) : "memory");
}
// Rebuild a group's dense key and value rows from their packed (values,
// indices): the rows are zero already.  Element e = t * r + j (token t, rank
// j) is the e-th entry of the packed arrays; lane l takes the pairs (e, e + 1)
// with e = 2 l + 64 i, so each load of the warp reads one contiguous 128-byte
// (values) or 64-byte (indices) run.  t = floor(e / r) = umulhi(2e, rm) with
// rm = ceil(2^31 / r) (exact for e < 2^20).  Keys and values share e, so their
// loads and stores interleave.
// Addresses are shared-window bytes: tk, tv (tiles), kv/ki/vv/vi (packed
// values and indices); two pairs per lane per step, loads first.
__device__ __forceinline__ void scatter_kv(const Layout& L, uint32_t tk, uint32_t tv, uint32_t kv, uint32_t ki,
                                           uint32_t vv, uint32_t vi, int n_el, uint32_t rm, int lane) {
  for (int e = 2 * lane; e < n_el; e += 128) {
    const int e2 = e + 64;
    const bool has2 = e2 < n_el;
    const uint32_t kp = lds_u32(kv + 2 * e), vp = lds_u32(vv + 2 * e);
    uint32_t kx = lds_u16(ki + e), vx = lds_u16(vi + e);
    uint32_t kp2 = 0, vp2 = 0, kx2 = 0, vx2 = 0;
    if (has2) {
      kp2 = lds_u32(kv + 2 * e2);
      vp2 = lds_u32(vv + 2 * e2);
      kx2 = lds_u16(ki + e2);
      vx2 = lds_u16(vi + e2);
    }
#if MK_CHECKS
    // channels from the pages' index bytes stay inside the row (else the
    // element goes to channel 0 and the error word records it)
    if (!in_bounds(L, ((kx | vx | kx2 | vx2) & 0x8080u) == 0u, SITE_ATTN_TILE, (int64_t)(kx | vx << 16))) {
      kx &= 0x7f7fu;
      vx &= 0x7f7fu;
      kx2 &= 0x7f7fu;
      vx2 &= 0x7f7fu;
    }
#else
    (void)L;
#endif
    const uint32_t r0 = __umulhi(2u * (uint32_t)e, rm) * (kRow * 2), r1 = __umulhi(2u * (uint32_t)e + 2u, rm) * (kRow * 2);
    sts_u16(tk + r0 + 2 * (kx & 0xff), kp);
    sts_u16(tv + r0 + 2 * (vx & 0xff), vp);
    if (e + 1 < n_el) {
      sts_u16(tk + r1 + 2 * (kx >> 8), kp >> 16);
      sts_u16(tv + r1 + 2 * (vx >> 8), vp >> 16);
    }
    if (has2) {
      const uint32_t q0 = __umulhi(2u * (uint32_t)e2, rm) * (kRow * 2), q1 = __umulhi(2u * (uint32_t)e2 + 2u, rm) * (kRow * 2);
      sts_u16(tk + q0 + 2 * (kx2 & 0xff), kp2);
      sts_u16(tv + q0 + 2 * (vx2 & 0xff), vp2);
      if (e2 + 1 < n_el) {
        sts_u16(tk + q1 + 2 * (kx2 >> 8), kp2 >> 16);
        sts_u16(tv + q1 + 2 * (vx2 >> 8), vp2 >> 16);
      }
    }
  }
}

// Rebuild one token's dense row from its position bitmap ([S] sec. 5.1; the
// row is zero already).  Bit j of the bitmap (group j, channels GG j ..
// GG j + GG - 1) takes the next GG packed values, so the lane walks its set
// bits from the lowest and copies GG values per bit: n = r / GG iterations
// for every live token.  vals, bm, row: shared-window byte addresses of the
// token's packed values, its bitmap and its dense row.
template <int GG>
__device__ __forceinline__ void unpack_bitmap_row(uint32_t vals, uint32_t bm, uint32_t row, int r) {
  uint64_t cur, nxt = 0ull;
  if (GG == 1) {
    uint32_t w0, w1, w2, w3;
    asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3) : "r"(bm));
    cur = (uint64_t)w0 | ((uint64_t)w1 << 32);
    nxt = (uint64_t)w2 | ((uint64_t)w3 << 32);
  } else if (GG == 2) {
    uint32_t w0, w1;
    asm("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(w0), "=r"(w1) : "r"(bm));
    cur = (uint64_t)w0 | ((uint64_t)w1 << 32);
  } else if (GG == 4) {
    cur = lds_u32(bm);
  } else {
    cur = lds_u16(bm);
  }
  int cb = 0;
  for (int k = 0; k < r; k += GG) {
    if (GG == 1 && cur == 0ull) {
      cur = nxt;
      cb = 64;
    }
    // (the mask keeps a malformed bitmap with too few bits inside the row)
    const int c = ((cb + __ffsll((long long)cur) - 1) & (128 / GG - 1)) * GG;
    cur &= cur - 1ull;
    const uint32_t src = vals + 2 * k, dst = row + 2 * c;
    if (GG == 1) {
      sts_u16(dst, lds_u16(src));
    } else if (GG == 2) {
      asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(dst), "r"(lds_u32(src)) : "memory");
    } else if (GG == 4) {
      uint32_t a, b;
      asm("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(a), "=r"(b) : "r"(src));
      asm volatile("st.shared.v2.u32 [%0], {%1, %2};\n" ::"r"(dst), "r"(a), "r"(b) : "memory");
    } else {
      uint32_t a, b, c2, d;
      asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(a), "=r"(b), "=r"(c2), "=r"(d) : "r"(src));
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(a), "r"(b), "r"(c2), "r"(d)
                   : "memory");
    }
  }
}
// Highest channel a token's bitmap keeps (0 for an empty bitmap).
__device__ __forceinline__ int bitmap_top_channel(uint32_t bm, int gg) {
  const int nw = gg == 1 ? 4 : gg == 2 ? 2 : 1;
  int top = -1;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i < nw) {
      const uint32_t w = gg == 8 ? lds_u16(bm) : lds_u32(bm + 4 * i);
      if (w) top = 32 * i + 31 - __clz(w);
    }
  }
  return top < 0 ? 0 : top * gg + gg - 1;
}

struct Task {
  int kind;      // 0 none, 1 dense chunk, 2 packed group, 3 skipped (bad block id)
                 // (kind 1 with b >= 0: rows j0.. of an uncompressed page, the Quest comparator)
  int item;
  int j0, nd;    // dense: first dense token and count
  int b, r, tg, n_live;
  int g;         // bitmap pages: the block's element-group size
};

int stage_bytes(const Layout& L) {
  return (std::max(L.dense_pages ? 0 : kTG * (4 * L.r_max + 2 * pos_bytes(L, L.r_max, L.bm_g)), kDenseStage) + 15) / 16 *
         16;
}
// Per warp: the stages, then the key tile and the value tile.
size_t per_warp_bytes(const Layout& L, int nst) {
  return (size_t)nst * stage_bytes(L) + 2 * kTileBytes + ((size_t)nst * 8 + 15) / 16 * 16;  // + stage barriers
}
size_t smem_for(const Layout& L, int nst, int nw) {
  return (size_t)nw * per_warp_bytes(L, nst) + (size_t)nw * 8 * 2 * 4 + kRow * 2 + 64;
}
}  // namespace

// Shared-memory plan; fills attn_nst / attn_sb and returns the dynamic shared
// memory size (0 if nothing fits).
size_t attn_plan(Layout& L, int64_t attend_max) {
  // Double-buffered stages first (they hide the copy latency), then as many
  // warps as fit.
  // Warps per CTA are a multiple of 4, an equal share for each of the SM's
  // four sub-partitions.
  // Long selections (many 16-token groups per warp; attend_max: the page
  // tokens a unit may attend, selected and always-attended) are bound by the
  // main loop's densify work: more warps with one stage each (the next copy
  // goes out as soon as a stage is consumed) beat fewer with two.  Short ones
  // are bound by each warp's latency chain: two stages, 12 warps (which also
  // get more registers).
  const bool long_sel = std::max<int64_t>((int64_t)L.k_max * L.B, attend_max) >= kLongSelTokens;
  int plans[8][2] = {{2, 12}, {2, 8}, {2, 4}, {0, 0}, {0, 0}, {0, 0}, {0, 0}, {0, 0}};
  if (long_sel) {
    const int lp[5][2] = {{1, 16}, {1, 12}, {2, 8}, {2, 4}, {1, 4}};
    for (int i = 0; i < 5; ++i) {
      plans[i][0] = lp[i][0];
      plans[i][1] = lp[i][1];
    }
  }
  if (const char* e = std::getenv("MK_ATTN_PLAN")) {  // tuning override: "stages,warps"
    int a = 0, b = 0;
    // one stage (the one-stage kernel, up to 16 warps) or two or more with at most 12 warps
    if (std::sscanf(e, "%d,%d", &a, &b) == 2 && b >= 4 && b <= kMaxWarps && b % 4 == 0 &&
        (a == 1 || (b <= 12 && a >= 2))) {
      plans[0][0] = a;
      plans[0][1] = b;
    }
  }
  for (const auto& pl : plans) {
    if (pl[0] == 0) break;
    const size_t s = smem_for(L, pl[0], pl[1]);
    if (s <= 225 * 1024) {  // leaves room for the static shared memory
      L.attn_tg = kTG;
      L.attn_nst = pl[0];
      L.attn_nc = pl[1];  // warps per CTA
      L.attn_sb = stage_bytes(L);
      return s;
    }
  }
  return 0;
}

size_t attn_smem_bytes(const Layout& L, int) { return smem_for(L, L.attn_nst, L.attn_nc); }

// Largest number of CTAs per unit whose partials the merging CTA can stage
// (next to the warps' dump, R_v and the CTA's o').
int attn_max_parts(const Layout& L) {
  const int64_t dump = ((int64_t)L.attn_nc * L.G * D * 4 + 15) / 16 * 16;
  const int64_t avail = (int64_t)L.attn_nc * per_warp_bytes(L, L.attn_nst) - dump - (int64_t)D * D * 4 -
                        (int64_t)L.G * D * 4 - 64;  // dump, R_v, o'
  return (int)std::max<int64_t>(1, std::min<int64_t>(MK_MAX_SPLITS, avail / ((int64_t)L.G * (D + 2) * 4)));
}

template <int G, bool DENSE, int MAXW, int MODE>
__global__ void __launch_bounds__(MAXW * 32, 1) k_attn(Layout L, int layer, CallSeqs cs, AttnSplit split,
                                                 const int32_t* __restrict__ ids,
                                                 const int32_t* __restrict__ n_sel_in,
                                                 const uint16_t* __restrict__ q_in, const uint16_t* __restrict__ Kd,
                                                 const uint16_t* __restrict__ Vd, int64_t t_stride,
                                                 uint16_t* __restrict__ out) {
  const int NST = L.attn_nst, SB = L.attn_sb;
  const int kWarps = blockDim.x >> 5;
  extern __shared__ __align__(16) unsigned char smem[];
  const size_t pwb = (size_t)NST * SB + 2 * kTileBytes + ((size_t)NST * 8 + 15) / 16 * 16;
  unsigned char* warp_area = smem;                                       // [kWarps][pwb]
  float* mlw = reinterpret_cast<float*>(smem + kWarps * pwb);            // [kWarps][8][2]
  uint16_t* zrow = reinterpret_cast<uint16_t*>(mlw + kWarps * 16);      // one zero row (272 B)
  __shared__ __align__(16) UnitDesc ud;
  __shared__ int s_abort, s_ns, s_last;
  __shared__ int s_segsel[MK_MAX_SEGMENTS + 1];  // first position of each segment's ids (own-rotation segments)
  __shared__ float s_m[8], s_l[8];
  __shared__ int32_t s_ids[kIdsCap];
  __shared__ uint64_t s_bar, s_bar2;  // R_v staging (every CTA), partials staging (the merging CTA)  // this CTA's selected block ids (its j-th item: ids[part + j P])

  // This CTA's sequence (the last with off <= blockIdx.x), kv head and part.
  int ci = 0;
  {
    int hi = cs.n - 1;
    const int bid = (int)blockIdx.x;
    while (ci < hi) {
      const int mid = (ci + hi + 1) >> 1;
      if (split.off[mid] <= bid) ci = mid; else hi = mid - 1;
    }
  }
  const int P = (split.off[ci + 1] - split.off[ci]) / L.n_kv;
  const int local = (int)blockIdx.x - split.off[ci];
  const int kvh = local / P, part = local - kvh * P;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t u = DENSE ? 0 : unit_index(L, layer, seq, kvh);
  const int64_t slot = (int64_t)seq * L.n_kv + kvh;
  const int32_t* my_ids = DENSE ? nullptr : ids + ((int64_t)ci * L.n_kv + kvh) * L.k_max;

  if (!DENSE && part == 0) {  // R_v is static: warm L2 for the partials' un-rotation
    const char* rv = unit_base(L, u) + L.off_rv;
    for (int i = tid; i < D * D * 4 / 128; i += blockDim.x) prefetch_l2(rv + (size_t)i * 128);
  }
  for (int i = tid; i < kRow / 8; i += blockDim.x) reinterpret_cast<uint4*>(zrow)[i] = make_uint4(0, 0, 0, 0);
  // Barriers before the wait point (their init fence stays off the critical path).
  unsigned char* const my_area0 = warp_area + (size_t)warp * pwb;
  uint64_t* const bars0 = reinterpret_cast<uint64_t*>(my_area0 + (size_t)NST * SB + 2 * kTileBytes);
  if (lane == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(&bars0[i], 1);
    if (tid == 0) {
      mbar_init(&s_bar, 1);
      mbar_init(&s_bar2, 1);
    }
    mbar_init_fence();
  }
  // q' as the A operand of the logits (k = channel): row g holds the bf16 hi
  // part and row g + 8 the lo part of head hq = g % G (rows repeat when
  // G < 8), so one MMA gives both partial sums in the same lane.  The
  // selection kernel wrote q' two launches back (the top-k kernel runs in
  // between and leaves it alone), so it is read before the wait point; the
  // caller's q of the dense reference is read after it.
  const int hq = g % G;
  uint32_t aq[8][4];
  auto load_q = [&](int cls_q) {
    const float* qrot = qrot_of(L, layer, slot, cls_q);
    const uint16_t* qin = DENSE ? q_in + ((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D : nullptr;
    float2 qx[8][2];
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int c = kc * 16 + hf * 8 + 2 * tig;
        if (DENSE) {
          qx[kc][hf] = make_float2(bf2f(qin[hq * D + c]), bf2f(qin[hq * D + c + 1]));
        } else {
          qx[kc][hf] = __ldcg(reinterpret_cast<const float2*>(qrot + hq * D + c));
        }
      }
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) split2_bf16(qx[kc][hf].x, qx[kc][hf].y, aq[kc][2 * hf], aq[kc][2 * hf + 1]);
  };
  if (!DENSE) load_q(0);
  pdl_wait();
  pdl_trigger();
  // One round of independent loads (L2 path: the previous kernel wrote them):
  // state, selection count, this CTA's block ids.
  if (tid == 0) {
    // all three loads in flight before the first use
    const int32_t err = __ldcg(L.err);
    uint4 dd[4] = {};
    if (!DENSE)
#pragma unroll
      for (int i = 0; i < 4; ++i) dd[i] = __ldcg(reinterpret_cast<const uint4*>(L.desc + u) + i);
    const int32_t ns0 = DENSE ? 0 : __ldcg(n_sel_in + (int64_t)ci * L.n_kv + kvh);
    s_abort = err;
    if (!DENSE)
#pragma unroll
      for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(&ud)[i] = dd[i];
    s_ns = ns0;
  }
  if (!DENSE)
    for (int j = tid; j < kIdsCap && part + j * P < L.k_max; j += blockDim.x) s_ids[j] = __ldcg(my_ids + part + j * P);
  if (DENSE) load_q(0);
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
  // Items of the unit: the selected pages, the always-attended pages, then
  // the dense chunks.  CTA `part` takes items part, part + P, ...; its warps
  // take its j-th items round robin (j = warp, warp + kWarps, ...).
  const int n_dch = (n_dense + kDC - 1) / kDC;
  // Rotation classes.  With segments stored under their own rotation
  // (re-compressed closed segments), every rotation gets its own CTAs of the
  // unit: a CTA takes the items of one class only, rotates the query into
  // that class's basis and un-rotates its partial by the class's R_v, so
  // the merge stays a weighted sum.  Class 0 is the head's rotation (with the
  // sinks and the window); class s + 1 is segment s's own.  Each class holds
  // at least one CTA (the host gives such units enough), the rest go by the
  // classes' work.  Without such segments: one class, the unit's P CTAs.
  int cls = 0, pc = part, Pc = P;
  int ns_c = ns, nalw_c = n_always, ndch_c = n_dch;
  const bool own_mode = MODE != kModePlain && !DENSE && !skip && any_own(ud);
  if (own_mode) {
    if (tid == 0)
      for (int i = 0; i < MK_MAX_SEGMENTS; ++i)
        s_segsel[i] = __ldcg(L.seg_sel + (((int64_t)layer * L.max_seqs + seq) * L.n_kv + kvh) * MK_MAX_SEGMENTS + i);
    __syncthreads();
    const int nseg = ud.n_seg;
    int ss[MK_MAX_SEGMENTS + 1];
#pragma unroll
    for (int i = 0; i <= MK_MAX_SEGMENTS; ++i) ss[i] = i < nseg ? min(max(s_segsel[i], 0), ns) : ns;
    const int mine = tid <= MK_MAX_SEGMENTS ? (tid < nseg ? min(max(s_segsel[tid], 0), ns) : ns) : 0;
    __syncthreads();
    if (tid <= MK_MAX_SEGMENTS) s_segsel[tid] = mine;  // clamped, kept for the item mapping below
    int csel[MK_MAX_SEGMENTS], calw[MK_MAX_SEGMENTS], wcls[MK_MAX_SEGMENTS];
#pragma unroll
    for (int c = 0; c < MK_MAX_SEGMENTS; ++c) csel[c] = calw[c] = 0;
#pragma unroll
    for (int sg = 0; sg < MK_MAX_SEGMENTS; ++sg) {
      if (sg >= nseg) continue;
      const int lo = min(ud.first_block[sg], nblk), hi = sg + 1 < nseg ? min(ud.first_block[sg + 1], nblk) : nblk;
      const int c = seg_class(ud, sg);
#pragma unroll
      for (int k = 0; k < MK_MAX_SEGMENTS; ++k)
        if (k == c) {
          if (seg_always(ud, sg)) calw[k] += max(0, hi - lo);
          else csel[k] += ss[sg + 1] - ss[sg];
        }
    }
    int nact = 0, wsum_c = 0;
#pragma unroll
    for (int c = 0; c < MK_MAX_SEGMENTS; ++c) {
      const bool act = c < nseg && (c == 0 || seg_own(ud, c - 1));
      wcls[c] = act ? (csel[c] + calw[c]) * ((B + kDC - 1) / kDC) + (c == 0 ? n_dch : 0) : -1;
      nact += act ? 1 : 0;
      wsum_c += act ? wcls[c] : 0;
    }
    const int extra = max(0, P - nact);
    int start = 0, used = 0;
    int pcs[MK_MAX_SEGMENTS];
#pragma unroll
    for (int c = 0; c < MK_MAX_SEGMENTS; ++c) {
      pcs[c] = wcls[c] < 0 ? 0 : 1 + (wsum_c > 0 ? (int)(((int64_t)extra * wcls[c]) / wsum_c) : 0);
      used += pcs[c];
    }
    pcs[0] += max(0, P - used);  // what the rounding left
#pragma unroll
    for (int c = 0; c < MK_MAX_SEGMENTS; ++c) {
      if (pcs[c] > 0 && part >= start && part < start + pcs[c]) {
        cls = c;
        pc = part - start;
        Pc = pcs[c];
        ns_c = csel[c];
        nalw_c = calw[c];
        ndch_c = c == 0 ? n_dch : 0;
      }
      start += pcs[c];
    }
    if (part >= start) {  // more CTAs than classes can use (cannot happen with P >= the class count): idle
      ns_c = nalw_c = ndch_c = 0;
    }
  }
  // The i-th selected id of this CTA's class: its position in the ids row.
  auto sel_pos = [&](int i) -> int {
    if (!own_mode) return i;
    int pos = -1;
#pragma unroll
    for (int sg = 0; sg < MK_MAX_SEGMENTS; ++sg) {
      if (sg < ud.n_seg && seg_class(ud, sg) == cls && !seg_always(ud, sg) && pos < 0) {
        const int n = s_segsel[sg + 1] - s_segsel[sg];
        if (i < n) pos = s_segsel[sg] + i;
        else i -= n;
      }
    }
    return pos;
  };
  // The i-th always-attended block of this CTA's class.
  auto alw_block = [&](int i) -> int {
    if (!own_mode) return always_block(ud, nblk, i);
    int b = -1;
#pragma unroll
    for (int sg = 0; sg < MK_MAX_SEGMENTS; ++sg) {
      if (sg < ud.n_seg && seg_class(ud, sg) == cls && seg_always(ud, sg) && b < 0) {
        const int lo = min(ud.first_block[sg], nblk), hi = sg + 1 < ud.n_seg ? min(ud.first_block[sg + 1], nblk) : nblk;
        const int n = max(0, hi - lo);
        if (i < n) b = lo + i;
        else i -= n;
      }
    }
    return b;
  };
  if (own_mode) {
    // This CTA's block ids and query, for its class.
    __syncthreads();
    for (int j = tid; j < kIdsCap && pc + j * Pc < ns_c; j += blockDim.x) s_ids[j] = __ldcg(my_ids + sel_pos(pc + j * Pc));
    if (cls != 0) load_q(cls);
    __syncthreads();
  }
  const int n_items = skip ? 0 : ns_c + nalw_c + ndch_c;
  const int n_mine = n_items > pc ? (n_items - pc + Pc - 1) / Pc : 0;

  const char* base = DENSE ? nullptr : unit_base(L, u);
  unsigned char* my_area = warp_area + (size_t)warp * pwb;
  uint16_t* tk = reinterpret_cast<uint16_t*>(my_area + (size_t)NST * SB);  // dense key tile
  uint16_t* tv = tk + kTG * kRow;                                           // dense value tile

  auto make_task = [&](int j, int tg) -> Task {
    Task t{};
    if (j >= n_mine) return t;
    t.item = j;
    const int it = pc + j * Pc;
    if (it >= ns_c + nalw_c) {
      t.kind = 1;
      t.b = -1;
      t.j0 = (it - ns_c - nalw_c) * kDC;
      t.nd = min(kDC, n_dense - t.j0);
      return t;
    }
    const int b = it < ns_c ? (j < kIdsCap ? s_ids[j] : __ldcg(my_ids + sel_pos(it))) : alw_block(it - ns_c);
    if (b < 0 || b >= nblk) {
      if (lane == 0) set_error(L, ERR_BAD_BLOCK, (int32_t)u, b);
      t.kind = 3;
      return t;
    }
    t.b = b;
    t.n_live = min(B, n_mid - b * B);
    if (!DENSE && L.dense_pages) {  // whole rows: staged like the dense chunks
      t.kind = 1;
      t.j0 = tg;
      t.nd = min(kDC, t.n_live - tg);
      return t;
    }
    t.kind = 2;
    const int sgb = seg_of_block(ud, b);
    t.r = ud.r[sgb];
    t.g = MODE == kModeBitmap ? seg_group(ud, sgb) : 0;
    t.tg = tg;
    return t;
  };
  auto advance = [&](const Task& t) -> Task {
    if (t.kind == 0) return t;
    if (t.kind == 2 && t.tg + kTG < t.n_live) {
      Task n = t;
      n.tg += kTG;
      return n;
    }
    if (t.kind == 1 && t.b >= 0 && t.j0 + kDC < t.n_live) {
      Task n = t;
      n.j0 += kDC;
      n.nd = min(kDC, t.n_live - n.j0);
      return n;
    }
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
  // Bulk copies of a task into stage sidx; its barrier expects the bytes.
  uint64_t* bars = reinterpret_cast<uint64_t*>(my_area + (size_t)NST * SB + 2 * kTileBytes);
  auto issue = [&](const Task& t, int sidx) {
    unsigned char* dst = my_area + (size_t)sidx * SB;
    if (t.kind == 1) {
      // nd K rows then nd V rows, 256 bytes each, into rows padded to 272 bytes.
      if (lane == 0) {
        fence_proxy_async();
        mbar_expect_tx(&bars[sidx], 2u * (unsigned)t.nd * D * 2);
      }
      __syncwarp();
      if (lane < 2 * t.nd) {
        const int row = lane >> 1, isv = lane & 1;
        const uint16_t *kr, *vr;
        if (t.b >= 0) {
          kr = reinterpret_cast<const uint16_t*>(base + L.off_pages + (int64_t)t.b * L.page_stride) +
               (int64_t)(t.j0 + row) * D;
          vr = kr + (int64_t)B * D;
        } else {
          dense_rows(t.j0 + row, kr, vr);
        }
        bulk_g2s(dst + (isv * kDC + row) * kRow * 2, isv ? vr : kr, D * 2, &bars[sidx]);
      }
    } else if (t.kind == 2) {
      // This group's rows of the page's four sub-arrays (B is a multiple of
      // 16, so a whole group stays inside the page; sizes and offsets are
      // multiples of 16 bytes), back to back in the stage:
      // [K val 2gr][K pos gp][V val 2gr][V pos gp] bytes (gp = 16 position
      // rows: gr uint8 indices or 16 bitmaps); lane q copies run q.
      const int gr = kTG * t.r, pb = MODE == kModeBitmap ? 16 / t.g : t.r, gp = kTG * pb;
      if (lane == 0) {
        fence_proxy_async();
        mbar_expect_tx(&bars[sidx], (unsigned)(4 * gr + 2 * gp));
      }
      __syncwarp();
      if (lane < 4) {
        const int tr = t.tg * t.r, tp = t.tg * pb, Br = B * t.r, Bp = B * pb;  // page: [2Br][Bp][2Br][Bp]
        const char* page = base + L.off_pages + (int64_t)t.b * L.page_stride;
        const int soff = lane == 0 ? 2 * tr : lane == 1 ? 2 * Br + tp : lane == 2 ? 2 * Br + Bp + 2 * tr
                                                                                    : 4 * Br + Bp + tp;
        const int doff = lane == 0 ? 0 : lane == 1 ? 2 * gr : lane == 2 ? 2 * gr + gp : 4 * gr + gp;
        bulk_g2s(dst + doff, page + soff, (lane & 1) ? gp : 2 * gr, &bars[sidx]);
      }
    }
  };
  auto has_copy = [](const Task& t) { return t.kind == 1 || t.kind == 2; };

  // Ring of NST stages: the task being consumed sits in stage st, the next
  // NST - 1 tasks are in flight.  With one stage, the next task's copy goes
  // out as soon as the current one's stage is consumed (after the scatter of
  // a packed group, after the value product of a dense chunk).  ph: parity of
  // each stage's next phase; pend: stages with copies in flight.
  Task cur = make_task(warp, 0), ahead = cur;
  int st = 0;
  uint32_t ph = 0, pend = 0;
  bool broken = false;
  issue(cur, 0);
  if (has_copy(cur)) pend |= 1u;
  for (int i = 1; i < NST - 1; ++i) {
    ahead = advance(ahead);
    issue(ahead, i);
    if (has_copy(ahead)) pend |= 1u << i;
  }

  // O'^T fragments, m-tile mt: rows = channels mt*16 + g (+8), columns 2tig,
  // 2tig+1.  With G <= 4, column n holds the hi part (n < 4) or the lo part
  // (n >= 4) of head n % G; with G = 8, column n is head n.
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[mt][k] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;  // head hq: running max (log2 units) and sum

  const int mi = lane >> 3, ri = lane & 7;
  const int ktok = ri + (mi >> 1) * 8, kch = (mi & 1) * 8;  // ldmatrix rows for the key B fragments
  const int vtok = ri + (mi >> 1) * 8, vch = (mi & 1) * 8;  // ldmatrix.trans rows for the value A fragments
  // The 16-warp plan has one stage (kOneStage); the 12-warp plans two or more.
  constexpr bool kOneStage = MAXW > 12;
  while (cur.kind != 0) {
    bool next_out = !kOneStage;
    auto issue_next = [&]() {  // one stage: the next task into the consumed stage
      if (!kOneStage || next_out) return;
      __syncwarp();
      ahead = advance(cur);
      issue(ahead, st);
      if (has_copy(ahead)) pend |= 1u << st;
      next_out = true;
    };
    if (!kOneStage) {
      const int sn = st + NST - 1 < NST ? st + NST - 1 : st - 1;  // (st + NST - 1) mod NST
      ahead = advance(ahead);
      issue(ahead, sn);
      if (has_copy(ahead)) pend |= 1u << sn;
    }
    if (has_copy(cur)) {
      if (!mbar_wait_warp(&bars[st], (ph >> st) & 1u)) {
        if (lane == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, st, (int32_t)MK_ETIMEOUT);
        broken = true;
        break;
      }
      ph ^= 1u << st;
      pend &= ~(1u << st);
    }
    const unsigned char* buf = my_area + (size_t)st * SB;
    if (cur.kind == 1 || cur.kind == 2) {
      int ntok, nck_k = 8, nck_v = 8;  // 16-channel chunks that can hold a nonzero
      const uint16_t *krow, *vrow;      // this lane's ldmatrix rows
      if (cur.kind == 1) {
        ntok = cur.nd;
        const uint16_t* kb = reinterpret_cast<const uint16_t*>(buf);
        const uint16_t* vb = kb + kDC * kRow;
        krow = (ktok < ntok ? kb + ktok * kRow : zrow) + kch;
        vrow = (vtok < ntok ? vb + vtok * kRow : zrow) + vch;
      } else {
        ntok = min(kTG, cur.n_live - cur.tg);
        const int r = cur.r, gr = kTG * r, pb = MODE == kModeBitmap ? 16 / cur.g : r, gp = kTG * pb;
        const uint16_t* kval = reinterpret_cast<const uint16_t*>(buf);
        const uint8_t* kidx = buf + 2 * gr;
        const uint16_t* vval = reinterpret_cast<const uint16_t*>(buf + 2 * gr + gp);
        const uint8_t* vidx = buf + 4 * gr + gp;
        // Kept channels are stored in ascending order, so a token's last
        // index (its bitmap's top bit) is its highest channel: the group's
        // rows are zero from the chunk after the largest one on.
        const int tt = lane & 15, gg = MODE == kModeBitmap ? cur.g : 0;
        uint32_t hk = 0, hv = 0;
        if (tt < ntok) {
          if (gg) {
            const uint32_t hc = (uint32_t)bitmap_top_channel(smem_u32((lane >> 4) ? vidx : kidx) + tt * pb, gg);
            (lane >> 4 ? hv : hk) = hc;
          } else {
            hk = kidx[tt * r + r - 1];
            hv = vidx[tt * r + r - 1];
          }
        }
        nck_k = (int)(__reduce_max_sync(FULL, hk) >> 4) + 1;
        nck_v = (int)(__reduce_max_sync(FULL, hv) >> 4) + 1;
        // Zero those chunks of all 16 rows (lane: row tt, 16-byte half lane >> 4).
        uint4* zk = reinterpret_cast<uint4*>(tk + tt * kRow) + (lane >> 4);
        uint4* zv = reinterpret_cast<uint4*>(tv + tt * kRow) + (lane >> 4);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (c < nck_k) zk[2 * c] = make_uint4(0, 0, 0, 0);
          if (c < nck_v) zv[2 * c] = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        if (gg) {
          // Lane (token tt, tensor lane / 16) rebuilds that row.
          if (tt < ntok) {
            const bool isv = lane >> 4;
            const uint32_t vals = smem_u32(isv ? vval : kval) + 2 * tt * r;
            const uint32_t bm = smem_u32(isv ? vidx : kidx) + tt * pb;
            const uint32_t row = smem_u32(isv ? tv : tk) + tt * kRow * 2;
            if (gg == 1) unpack_bitmap_row<1>(vals, bm, row, r);
            else if (gg == 2) unpack_bitmap_row<2>(vals, bm, row, r);
            else if (gg == 4) unpack_bitmap_row<4>(vals, bm, row, r);
            else unpack_bitmap_row<8>(vals, bm, row, r);
          }
        } else {
          const int n_el = ntok * r;
          const uint32_t rm = (0x80000000u + (uint32_t)r - 1u) / (uint32_t)r;
          scatter_kv(L, smem_u32(tk), smem_u32(tv), smem_u32(kval), smem_u32(kidx), smem_u32(vval),
                     smem_u32(vidx), n_el, rm, lane);
        }
        __syncwarp();
        issue_next();  // the packed group now lives in the tiles
        krow = tk + ktok * kRow + kch;
        vrow = tv + vtok * kRow + vch;
      }

      // S[head][token] = sum_c q'[head][c] K[token][c] over the nonzero
      // chunks: tokens 0-7 (s0), 8-15 (s1); c0/c1 hi part, c2/c3 lo part.
      float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        if (kc < nck_k) {
          uint32_t b[4];
          ldsm_x4(b, krow + kc * 16);
          mma_bf16(s0, aq[kc], b[0], b[1]);
          mma_bf16(s1, aq[kc], b[2], b[3]);
        }
      }
      // Online softmax for head hq over tokens 2tig, 2tig+1, 8+2tig, 9+2tig
      // (the four lanes of a quad hold the group's 16 tokens).
      const int t0 = 2 * tig;
      const float v0 = t0 < ntok ? (s0[0] + s0[2]) * kScaleLog2 : -INFINITY;
      const float v1 = t0 + 1 < ntok ? (s0[1] + s0[3]) * kScaleLog2 : -INFINITY;
      const float v2 = t0 + 8 < ntok ? (s1[0] + s1[2]) * kScaleLog2 : -INFINITY;
      const float v3 = t0 + 9 < ntok ? (s1[1] + s1[3]) * kScaleLog2 : -INFINITY;
      float x = fmaxf(fmaxf(v0, v1), fmaxf(v2, v3));
      x = fmaxf(x, __shfl_xor_sync(FULL, x, 1));
      x = fmaxf(x, __shfl_xor_sync(FULL, x, 2));
      const bool raise = x > m_run + kLazy;  // false for an all-masked group (x = -inf)
      const float m_new = raise ? x : m_run;
      const float a = raise ? exp2f(m_run - m_new) : 1.0f;
      const float p0 = exp2f(v0 - m_new), p1 = exp2f(v1 - m_new);
      const float p2 = exp2f(v2 - m_new), p3 = exp2f(v3 - m_new);
      float y = (p0 + p1) + (p2 + p3);
      y += __shfl_xor_sync(FULL, y, 1);
      y += __shfl_xor_sync(FULL, y, 2);
      l_run = l_run * a + y;
      m_run = m_new;
      if (__any_sync(FULL, raise)) {
        // Column n's head is n % G, whose factor quad n (g = n) holds.
        const float a0 = __shfl_sync(FULL, a, (2 * tig) << 2), a1 = __shfl_sync(FULL, a, (2 * tig + 1) << 2);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][0] *= a0;
          o[mt][1] *= a1;
          o[mt][2] *= a0;
          o[mt][3] *= a1;
        }
      }
      // P as the B operand of the value product: k = token, n = column g.
      uint32_t ph0, pl0, ph1, pl1;
      split2_bf16(p0, p1, ph0, pl0);
      split2_bf16(p2, p3, ph1, pl1);
      // O'^T[channel][column] += sum_token V[token][channel] P[token][column].
      if (G <= 4) {
        const bool lo = g >= 4;
        const uint32_t pb0 = lo ? pl0 : ph0, pb1 = lo ? pl1 : ph1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          if (mt < nck_v) {
            uint32_t av[4];
            ldsm_x4_t(av, vrow + mt * 16);
            mma_bf16(o[mt], av, pb0, pb1);
          }
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          if (mt < nck_v) {
            uint32_t av[4];
            ldsm_x4_t(av, vrow + mt * 16);
            mma_bf16(o[mt], av, ph0, ph1);
            mma_bf16(o[mt], av, pl0, pl1);
          }
        }
      }
    }
    issue_next();  // dense chunk, skipped item: after every use of the stage
    __syncwarp();
    cur = advance(cur);
    st = st + 1 < NST ? st + 1 : 0;
  }
  if (broken) {
    // Let the copies still in flight land before the stages are reused.
    for (int i = 0; i < NST; ++i)
      if ((pend >> i) & 1u) (void)mbar_wait(&bars[i], (ph >> i) & 1u);
  }
  __syncwarp();
  if (G <= 4) {
    // Fold the lo columns (lanes tig + 2) into the hi ones.
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[mt][k] += __shfl_xor_sync(FULL, o[mt][k], 2);
  }
  // This lane's columns now hold heads 2tig, 2tig+1 (valid below G, and for
  // G <= 4 only in lanes tig < 2).
  const bool col_ok0 = 2 * tig < G && (G == 8 || tig < 2), col_ok1 = 2 * tig + 1 < G && (G == 8 || tig < 2);

  // ---- warps -> CTA partial ------------------------------------------------
  if (tig == 0) {
    mlw[(warp * 8 + g) * 2] = m_run;
    mlw[(warp * 8 + g) * 2 + 1] = l_run;
  }
  __syncthreads();
  // Every CTA stages R_v above the dump area now, for the un-rotation of its
  // partial after the cross-warp sums.
  const size_t dump_bytes = ((size_t)kWarps * G * D * 4 + 15) / 16 * 16;
  float* rvs = reinterpret_cast<float*>(warp_area + dump_bytes);
  if (!DENSE && tid == 0) {
    fence_proxy_async();  // the stages and tiles were written by the main loop
    mbar_expect_tx(&s_bar, (unsigned)(D * D * 4));
    bulk_g2s(rvs, base + (cls == 0 ? L.off_rv : segrot_off(L, cls - 1) + (int64_t)D * D * 4), (unsigned)(D * D * 4),
             &s_bar);
  }
  float* dump = reinterpret_cast<float*>(warp_area);  // [kWarps][G][D] (main loop is over)
  {
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMaxWarps; ++w)
      if (w < kWarps) {
        M0 = fmaxf(M0, mlw[(w * 8 + h0) * 2]);
        M1 = fmaxf(M1, mlw[(w * 8 + h1) * 2]);
      }
    const float mw0 = mlw[(warp * 8 + h0) * 2], mw1 = mlw[(warp * 8 + h1) * 2];
    const float e0 = mw0 != -INFINITY ? exp2f(mw0 - M0) : 0.0f;
    const float e1 = mw1 != -INFINITY ? exp2f(mw1 - M1) : 0.0f;
    float* dw = dump + (size_t)warp * G * D;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int c = mt * 16 + g;
      if (col_ok0) {
        dw[h0 * D + c] = o[mt][0] * e0;
        dw[h0 * D + c + 8] = o[mt][2] * e0;
      }
      if (col_ok1) {
        dw[h1 * D + c] = o[mt][1] * e1;
        dw[h1 * D + c + 8] = o[mt][3] * e1;
      }
    }
  }
  for (int h = warp; h < G; h += kWarps) {
    // warp h: head h's (m, l) over the CTA's warps, lanes = warps
    const float mw = lane < kWarps ? mlw[(lane * 8 + h) * 2] : -INFINITY;
    const float lw = lane < kWarps ? mlw[(lane * 8 + h) * 2 + 1] : 0.0f;
    const float M = warp_max(mw);
    const float ls = warp_sum(mw != -INFINITY ? lw * exp2f(mw - M) : 0.0f);
    if (lane == 0) {
      s_m[h] = M;
      s_l[h] = ls;
    }
  }
  __syncthreads();
  // The CTA's partial: o' summed over its warps, then (MosaicKV) un-rotated
  // here, out_p = o'_p R_v, so that the merge is a weighted sum of rows that
  // are already in the output basis (the un-rotation is linear).
  // Shared memory above the dump: R_v [D][D] | o' [D][G] | partials
  // [P][G][D] | (m, l) [P][G][2] (merging CTA).
  float* pacc = L.part_acc + slot * MK_MAX_SPLITS * G * D;   // [part][G][D]
  float* pml = L.part_ml + slot * MK_MAX_SPLITS * G * 2;     // [part][G][2]
  float* ofull = rvs + (DENSE ? 0 : D * D);
  float* sacc = ofull + G * D;
  float* sml = sacc + (size_t)P * G * D;
  for (int i = tid; i < G * D; i += blockDim.x) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < kMaxWarps; ++w)
      if (w < kWarps) a += dump[(size_t)w * G * D + i];
    if (DENSE)
      pacc[(size_t)part * G * D + i] = a;
    else
      ofull[(i % D) * G + i / D] = a;  // [channel][head]: one vector load per channel below
  }
  if (!DENSE) {
    if (!mbar_wait(&s_bar, 0)) {
      if (tid == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, -3, (int32_t)MK_ETIMEOUT);
      (void)mbar_wait(&s_bar, 0);
    }
    __syncthreads();
    // out_p[h][j] = sum_c o'_p[h][c] R_v[c][j]: lane = four columns j, warp =
    // slice of c; the slice sums go over the dump area (read above) and are
    // added in slice order.
    {
      float* slc = dump;  // [kWarps][G][D]
      const int kC = (D + kWarps - 1) / kWarps;
      const int c0 = warp * kC, c1 = min(D, c0 + kC);
      float acc[G][4];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.0f;
#pragma unroll 4
      for (int c = c0; c < c1; ++c) {
        const float4 rr = *reinterpret_cast<const float4*>(rvs + c * D + 4 * lane);
        float oc[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int h = 0; h < G; h += 4) {
            const float4 t = *reinterpret_cast<const float4*>(ofull + c * G + h);
            oc[h] = t.x;
            oc[h + 1] = t.y;
            oc[h + 2] = t.z;
            oc[h + 3] = t.w;
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h) oc[h] = ofull[c * G + h];
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          acc[h][0] = fmaf(oc[h], rr.x, acc[h][0]);
          acc[h][1] = fmaf(oc[h], rr.y, acc[h][1]);
          acc[h][2] = fmaf(oc[h], rr.z, acc[h][2]);
          acc[h][3] = fmaf(oc[h], rr.w, acc[h][3]);
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h)
        *reinterpret_cast<float4*>(slc + ((size_t)warp * G + h) * D + 4 * lane) =
            make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      __syncthreads();
      for (int i = tid; i < G * D; i += blockDim.x) {
        float a = 0.0f;
#pragma unroll
        for (int w = 0; w < kMaxWarps; ++w)
          if (w < kWarps) a += slc[(size_t)w * G * D + i];
        pacc[(size_t)part * G * D + i] = a;
      }
    }
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

  // ---- the last CTA: merge the P partials and store -------------------------
  {
    const unsigned b_acc = (unsigned)(P * G * D * 4), b_ml = ((unsigned)(P * G * 2 * 4) + 15u) & ~15u;
    if (tid == 0) {
      fence_proxy_async_all();  // partials written through the generic proxy
      mbar_expect_tx(&s_bar2, b_acc + b_ml);
      bulk_g2s(sacc, pacc, b_acc, &s_bar2);
      bulk_g2s(sml, pml, b_ml, &s_bar2);
    }
    if (!mbar_wait(&s_bar2, 0)) {
      if (tid == 0) set_error(L, ERR_COPY_WAIT, (int32_t)u, -1, (int32_t)MK_ETIMEOUT);
      (void)mbar_wait(&s_bar2, 0);
      return;
    }
  }
  // Per (partial, head) weight exp2(m_p - M) / l, computed once; written over
  // the m entries.
  for (int h = warp; h < G; h += kWarps) {
    // warp h: head h over the partials, lanes p, p + 32 (P <= 64)
    float mp[2], lp[2];
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int p = lane + 32 * k2;
      mp[k2] = p < P ? sml[(p * G + h) * 2] : -INFINITY;
      lp[k2] = p < P ? sml[(p * G + h) * 2 + 1] : 0.0f;
    }
    const float M = warp_max(fmaxf(mp[0], mp[1]));
    float part_l = 0.0f;
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2)
      if (mp[k2] != -INFINITY) part_l += lp[k2] * exp2f(mp[k2] - M);
    const float ls = warp_sum(part_l);
    const float inv = (M != -INFINITY && ls > 0.0f) ? 1.0f / ls : 0.0f;
    __syncwarp();
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int p = lane + 32 * k2;
      if (p < P) sml[(p * G + h) * 2] = (mp[k2] != -INFINITY && inv != 0.0f) ? exp2f(mp[k2] - M) * inv : 0.0f;
    }
  }
  __syncthreads();
  uint16_t* orow = out + ((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D;
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int h = i / D;
    float a = 0.0f;
#pragma unroll 8
    for (int p = 0; p < P; ++p) a = fmaf(sacc[(size_t)p * G * D + i], sml[(p * G + h) * 2], a);
    orow[i] = f2bf(a);
  }
}

namespace {
template <int G, bool DENSE, int MAXW, int MODE>
cudaError_t launch_one(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids, const int32_t* n_sel,
                       const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t t_stride, uint16_t* out,
                       const int32_t* items, const int32_t* min_parts, size_t smem, cudaStream_t s) {
  int occ = 1, sms = 0;
  cudaError_t e = kernel_smem_attr((const void*)k_attn<G, DENSE, MAXW, MODE>, (int)smem, L.attn_nc * 32, &occ, &sms);
  if (e != cudaSuccess) return e;
  // CTAs per (sequence, kv head) in proportion to its items: one wave of
  // CTAs when the units fit on the SMs; with more units than CTA slots (many
  // sequences), about four CTAs' worth of work per slot, so long sequences
  // split and the SMs finish together.
  const int slots = std::max(1, std::max(sms, 1) * occ);
  const int units = cs.n * L.n_kv;
  int64_t work = 0;
  for (int i = 0; i < cs.n; ++i) work += (int64_t)std::max(1, items[i]) * L.n_kv;
  const double per_cta = (double)work / ((double)slots * (units > slots ? 4 : 1));
  const int cap = attn_max_parts(L);
  AttnSplit split;
  split.off[0] = 0;
  int p_min = 1 << 30, p_max = 0;
  for (int i = 0; i < cs.n; ++i) {
    const int it = std::max(1, items[i]);
    int P = (int)std::floor((double)it / per_cta);
    P = std::max(1, std::min(P, std::min(cap, std::max(1, it / 2))));
    if (min_parts) P = std::max(P, std::min(cap, min_parts[i]));
    p_min = std::min(p_min, P);
    p_max = std::max(p_max, P);
    split.off[i + 1] = split.off[i] + P * L.n_kv;
  }
  if (std::getenv("MK_LOG"))
    std::fprintf(stderr, "[mosaickv] attention: %d units, %d to %d CTAs each, %d CTAs (%d per SM), %zu B smem\n",
                 units, p_min, p_max, split.off[cs.n], occ, smem);
  return launch_pdl(k_attn<G, DENSE, MAXW, MODE>, dim3(split.off[cs.n]), dim3(L.attn_nc * 32), smem, s, 0, L, layer, cs,
                    split, ids, n_sel, q, K, V, t_stride, out);
}

template <bool DENSE>
cudaError_t launch_attn_g(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids, const int32_t* n_sel,
                          const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t t_stride, uint16_t* out,
                          const int32_t* items, const int32_t* min_parts, cudaStream_t s) {
  const size_t smem = attn_smem_bytes(L, 0);
  if (smem == 0 || smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  // One stage per warp: the one-stage kernel (launch bounds of 16 warps, at
  // most 128 registers), launched with the plan's 12 or 16 warps.
  const bool wide = L.attn_nst == 1;
  // The variant with rotation classes only where some unit of the call has a
  // segment under its own rotation (its CTAs need one per class).
  bool own = false;
  if (!DENSE && min_parts)
    for (int i = 0; i < cs.n; ++i) own = own || min_parts[i] > 1;
  const int mode = DENSE ? kModePlain : L.bm_g ? kModeBitmap : own ? kModeOwn : kModePlain;
#define MK_ATTN_ONE(GG, MM)                                                                                      \
  return wide ? launch_one<GG, DENSE, 16, MM>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, items, min_parts, \
                                              smem, s)                                                           \
              : launch_one<GG, DENSE, 12, MM>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, items, min_parts, \
                                              smem, s);
#define MK_ATTN_CASE(GG)                                                                                         \
  case GG:                                                                                                       \
    if constexpr (!DENSE) {                                                                                      \
      if (mode == kModeBitmap) MK_ATTN_ONE(GG, kModeBitmap)                                                      \
      if (mode == kModeOwn) MK_ATTN_ONE(GG, kModeOwn)                                                            \
    }                                                                                                            \
    MK_ATTN_ONE(GG, kModePlain)
  switch (L.G) {
    MK_ATTN_CASE(1)
    MK_ATTN_CASE(2)
    MK_ATTN_CASE(4)
    MK_ATTN_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef MK_ATTN_CASE
#undef MK_ATTN_ONE
}
}  // namespace

cudaError_t launch_decode_attn(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids,
                               const int32_t* n_sel, uint16_t* out, const int32_t* items, cudaStream_t s,
                               const int32_t* min_parts) {
  return launch_attn_g<false>(L, layer, cs, ids, n_sel, nullptr, nullptr, nullptr, 0, out, items, min_parts, s);
}

cudaError_t launch_dense_attn(const Layout& L, const CallSeqs& cs, const uint16_t* q, const uint16_t* K,
                              const uint16_t* V, int64_t t_stride, uint16_t* out, const int32_t* items, cudaStream_t s) {
  return launch_attn_g<true>(L, 0, cs, nullptr, nullptr, q, K, V, t_stride, out, items, nullptr, s);
}

}  // namespace mk
