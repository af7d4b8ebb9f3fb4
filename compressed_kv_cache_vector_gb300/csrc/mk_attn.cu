// PackedAttention: decode attention straight from the packed pages, with
// dense sink and window tokens, online softmax, scatter accumulation of the
// rotated values by their channel indices, and the un-rotation by R_v.  The
// same kernel with dense items only and no rotation is the uncompressed
// reference.
//
// Method: "MosaicKV：...阅读笔记" (zhongzhuzhou.org), Eq. (1) (dense
// attention), Eq. (13) (attention on the kept tokens' compressed vectors),
// Eq. (14) (output = o R_v); "MosaicKV: Serving Long-Context LLM with Dynamic
// Two-D KV Cache Compression" (paperlayer.ai), sec. 5.3 (PackedAttention:
// attention on packed vectors with positions rebuilt on the fly, inverse
// rotation merged into the query).
//
// GB300 structure: one thread-block cluster of C <= 16 CTAs per (sequence,
// kv head).  Each CTA takes a contiguous share of the work items (dense
// chunks of 16 tokens, then packed page groups of TG tokens); each warp
// double-buffers its items into shared memory with cp.async.  The split-T
// log-sum-exp merge and the un-rotation go through distributed shared
// memory: CTA `rank` merges and un-rotates output channels
// [rank*128/C, (rank+1)*128/C).  No global partials, no counters, no waits
// other than cluster barriers.
#include <algorithm>
#include <cstdio>
#include <cstdlib>

#include <cooperative_groups.h>

#include "mk_internal.cuh"

namespace cg = cooperative_groups;

namespace mk {

namespace {
constexpr int kWarps = 8;
constexpr int kDC = 16;                     // dense chunk (tokens)
constexpr int kKRow = D + 8;                // padded K row (bf16) in a staged dense chunk: 272 bytes
constexpr int kDenseStage = kDC * (kKRow + D) * 2;
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

template <int G>
__device__ __forceinline__ void load_q(const float* qs, int c, float (&qv)[G]) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int h = 0; h < G; h += 4) {
      const float4 t = *reinterpret_cast<const float4*>(qs + c * G + h);
      qv[h] = t.x; qv[h + 1] = t.y; qv[h + 2] = t.z; qv[h + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) qv[h] = qs[c * G + h];
  }
}

template <int G>
__device__ __forceinline__ void fma_vec(float* a, const float (&p)[G], float v) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int h = 0; h < G; h += 4) {
      float4 t = *reinterpret_cast<float4*>(a + h);
      t.x = fmaf(p[h], v, t.x); t.y = fmaf(p[h + 1], v, t.y);
      t.z = fmaf(p[h + 2], v, t.z); t.w = fmaf(p[h + 3], v, t.w);
      *reinterpret_cast<float4*>(a + h) = t;
    }
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) a[h] = fmaf(p[h], v, a[h]);
  }
}

// One work item of a warp: a dense chunk or one TG-token group of a page.
struct Task {
  int kind;      // 0 none, 1 dense, 2 sparse group, 3 skipped (bad block id)
  int item;      // item index in this unit's list
  int j0, nd;    // dense: first dense token and count
  int b, r, tg, n_live;
};

struct UnitInfo {
  int n_sink, win_lo, n_dense, n_dch, nblk, n_mid, ns, n_items;
};

size_t smem_for(const Layout& L, int tg, int nst, int nc) {
  const int G = L.G;
  const size_t sb = (size_t)((std::max(6 * tg * L.r_max, kDenseStage) + 15) / 16 * 16);
  return (size_t)D * G * 4                         // q'
         + (size_t)kWarps * nc * D * G * 4         // per-warp accumulators
         + (size_t)kWarps * 32 * G * 4             // per-token softmax weights
         + (size_t)kWarps * nst * sb               // stages
         + (size_t)kWarps * G * 2 * 4              // per-warp (m, l)
         + 16 * ((G * 2 * 4 + 15) / 16)            // CTA (m, l)
         + (size_t)2 * G * D * 4;                  // CTA acc, merged o'
}
}  // namespace

// Shared-memory plan of the attention kernel; fills the attn_* fields of the
// layout and returns the dynamic shared memory size (0 if nothing fits).
size_t attn_plan(Layout& L, int r_min) {
  const int nc = r_min >= 32 ? 2 : (r_min >= 16 ? 3 : 1);
  const int tgs[2] = {32, 16};
  for (int nst = 2; nst >= 1; --nst)
    for (int ti = 0; ti < 2; ++ti) {
      const int tg = tgs[ti];
      if (tg > L.B) continue;
      const size_t s = smem_for(L, tg, nst, nc);
      if (s <= 227 * 1024) {
        L.attn_tg = tg;
        L.attn_nst = nst;
        L.attn_nc = nc;
        L.attn_sb = (int)((std::max(6 * tg * L.r_max, kDenseStage) + 15) / 16 * 16);
        return s;
      }
    }
  return 0;
}

size_t attn_smem_bytes(const Layout& L, int) { return smem_for(L, L.attn_tg, L.attn_nst, L.attn_nc); }

template <int G, bool DENSE>
__global__ void __launch_bounds__(256, 1) k_attn(Layout L, int layer, CallSeqs cs, const int32_t* __restrict__ ids,
                                                 const int32_t* __restrict__ n_sel_in,
                                                 const uint16_t* __restrict__ q_in, const uint16_t* __restrict__ Kd,
                                                 const uint16_t* __restrict__ Vd, int64_t t_stride,
                                                 uint16_t* __restrict__ out) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int NC = L.attn_nc, NST = L.attn_nst, TG = L.attn_tg, SB = L.attn_sb;

  extern __shared__ __align__(16) unsigned char smem[];
  float* qs = reinterpret_cast<float*>(smem);                       // [D][G]
  float* accw = qs + D * G;                                         // [kWarps][NC][D][G]
  float* ptok = accw + kWarps * NC * D * G;                         // [kWarps][32][G]
  unsigned char* stages = reinterpret_cast<unsigned char*>(ptok + kWarps * 32 * G);  // [kWarps][NST][SB]
  float* mlw = reinterpret_cast<float*>(stages + (size_t)kWarps * NST * SB);         // [kWarps][G][2]
  float* cl_ml = mlw + kWarps * G * 2;                              // [G][2] (padded to 16 B)
  float* cl_acc = cl_ml + 4 * ((G * 2 + 3) / 4);                    // [G][D]
  float* ofull = cl_acc + G * D;                                    // [G][D]
  __shared__ UnitDesc ud;
  __shared__ int s_abort, s_ns;

  const int unit_call = blockIdx.x / C;
  const int ci = unit_call / L.n_kv, kvh = unit_call - ci * L.n_kv;
  const int seq = cs.seq[ci];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = DENSE ? 0 : unit_index(L, layer, seq, kvh);
  const int64_t slot = (int64_t)seq * L.n_kv + kvh;

  if (tid == 0) {
    s_abort = has_error(L);
    if (!DENSE) {
      ud = L.desc[u];
      s_ns = n_sel_in[(int64_t)ci * L.n_kv + kvh];
    } else {
      s_ns = 0;
    }
  }
  __syncthreads();
  // Every CTA of the cluster must reach the cluster barriers below, so an
  // abort only skips the work, never the barriers.
  bool skip = s_abort != 0;

  const int S = L.S, W = L.W, B = L.B;
  UnitInfo ui{};
  if (DENSE) {
    ui.n_dense = cs.T_old[ci];
  } else {
    const int T = ud.T;
    ui.n_sink = min(S, T);
    ui.n_mid = n_mid_tokens(L, T);
    ui.win_lo = S + ui.n_mid;
    ui.n_dense = ui.n_sink + max(0, T - ui.win_lo);
    ui.nblk = n_mid_blocks(L, T);
    ui.ns = s_ns;
    if (ui.ns < 0 || ui.ns > L.k_max) {
      if (tid == 0) set_error(L, ERR_BAD_NSEL, (int32_t)u, ui.ns);
      skip = true;
      ui.ns = 0;
    }
  }
  ui.n_dch = (ui.n_dense + kDC - 1) / kDC;
  const int n_always = DENSE ? 0 : ui.nblk - n_scored_blocks(ud, ui.nblk);
  ui.n_items = skip ? 0 : ui.n_dch + ui.ns + n_always;
  const int per = (ui.n_items + C - 1) / C;
  const int i0 = rank * per, i1 = min(ui.n_items, i0 + per);

  for (int i = tid; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    float v = 0.0f;
    if (!skip) {
      if (DENSE) v = bf2f(q_in[((int64_t)ci * L.n_kv * G + (int64_t)kvh * G + h) * D + c]);
      else v = L.qrot[(slot * G + h) * D + c];
    }
    qs[c * G + h] = v;
  }
  for (int i = tid; i < kWarps * NC * D * G; i += blockDim.x) accw[i] = 0.0f;
  __syncthreads();

  const char* base = DENSE ? nullptr : unit_base(L, u);
  const int32_t* my_ids = DENSE ? nullptr : ids + ((int64_t)ci * L.n_kv + kvh) * L.k_max;
  float* acc = accw + warp * NC * D * G;
  float* pt = ptok + warp * 32 * G;
  unsigned char* stg = stages + (size_t)warp * NST * SB;
  float m[G], l[G], racc[4][G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) racc[i][h] = 0.0f;
  }

  auto make_task = [&](int it, int tg) -> Task {
    Task t{};
    if (it >= i1) return t;
    t.item = it;
    if (it < ui.n_dch) {
      t.kind = 1;
      t.j0 = it * kDC;
      t.nd = min(kDC, ui.n_dense - t.j0);
      return t;
    }
    const int pi = it - ui.n_dch;
    const int b = pi < ui.ns ? __ldg(my_ids + pi) : always_block(ud, ui.nblk, pi - ui.ns);
    if (b < 0 || b >= ui.nblk) {
      if (lane == 0) set_error(L, ERR_BAD_BLOCK, (int32_t)u, b);
      t.kind = 3;
      return t;
    }
    t.kind = 2;
    t.b = b;
    t.r = ud.r[seg_of_block(ud, b)];
    t.tg = tg;
    t.n_live = min(B, ui.n_mid - b * B);
    return t;
  };
  auto advance = [&](const Task& t) -> Task {
    if (t.kind == 2 && t.tg + TG < t.n_live) return make_task(t.item, t.tg + TG);
    return make_task(t.item + kWarps, 0);
  };
  // Dense rows of token j of this unit (sinks, then the window ring).
  auto dense_rows = [&](int j, const uint16_t*& kr, const uint16_t*& vr) {
    if (DENSE) {
      const int64_t off = (((int64_t)ci * L.n_kv + kvh) * t_stride + j) * D;
      kr = Kd + off;
      vr = Vd + off;
    } else if (j < ui.n_sink) {
      kr = reinterpret_cast<const uint16_t*>(base + L.off_sink_k) + (int64_t)j * D;
      vr = reinterpret_cast<const uint16_t*>(base + L.off_sink_v) + (int64_t)j * D;
    } else {
      const int p = ui.win_lo + (j - ui.n_sink);
      const int64_t sl = (int64_t)((p - S) % W) * D;
      kr = reinterpret_cast<const uint16_t*>(base + L.off_win_k) + sl;
      vr = reinterpret_cast<const uint16_t*>(base + L.off_win_v) + sl;
    }
  };
  auto issue = [&](const Task& t, unsigned char* dst) {
    if (t.kind == 1) {
      // K rows padded to 272 bytes, then V rows of 256 bytes.
      for (int i = lane; i < t.nd * 16; i += 32) {
        const int row = i >> 4, part = i & 15;
        const uint16_t *kr, *vr;
        dense_rows(t.j0 + row, kr, vr);
        cp_async16(dst + row * kKRow * 2 + part * 16, kr + part * 8);
        cp_async16(dst + kDC * kKRow * 2 + row * D * 2 + part * 16, vr + part * 8);
      }
    } else if (t.kind == 2) {
      // This group's rows of the page's four sub-arrays.  B is a multiple of
      // TG, so whole groups stay inside the page; sizes and offsets are
      // multiples of 16 bytes.
      const int Br = B * t.r, gr = TG * t.r;
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
  // Online-softmax update of this warp's state (log2 domain).
  auto softmax_update = [&](const float (&s)[G], bool valid, float (&p)[G], float (&alpha)[G]) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float sh = valid ? s[h] : -INFINITY;
      const float mn = fmaxf(m[h], warp_max(sh));
      alpha[h] = exp2f(m[h] - mn);
      p[h] = valid ? exp2f(sh - mn) : 0.0f;
      l[h] = l[h] * alpha[h] + warp_sum(p[h]);
      m[h] = mn;
    }
  };
  auto rescale = [&](const float (&alpha)[G]) {
    for (int k = 0; k < NC; ++k)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int h = 0; h < G; ++h) acc[(k * D + 4 * lane + i) * G + h] *= alpha[h];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < G; ++h) racc[i][h] *= alpha[h];
  };

  Task cur = make_task(i0 + warp, 0);
  int st = 0;
  issue(cur, stg);
  cp_async_commit();
  while (cur.kind != 0) {
    const Task nxt = advance(cur);
    if (NST == 2) {
      issue(nxt, stg + (size_t)(st ^ 1) * SB);
      cp_async_commit();
      asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    } else {
      cp_async_wait_all();
    }
    __syncwarp();
    const unsigned char* buf = stg + (size_t)st * SB;
    if (cur.kind == 1) {
      // Dense chunk.  K: lane = token, 8 channels per 16-byte load (rows
      // padded so the 8 lanes of a phase hit distinct banks).  V: lanes own
      // channels 4*lane .. 4*lane+3 and accumulate in registers.
      const uint16_t* Ks = reinterpret_cast<const uint16_t*>(buf);
      const uint16_t* Vs = reinterpret_cast<const uint16_t*>(buf + kDC * kKRow * 2);
      const bool valid = lane < cur.nd;
      float s[G];
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = 0.0f;
      if (valid) {
#pragma unroll 2
        for (int c8 = 0; c8 < D; c8 += 8) {
          const uint4 kk = *reinterpret_cast<const uint4*>(Ks + lane * kKRow + c8);
          const float kf[8] = {bf2f(kk.x & 0xffff), bf2f(kk.x >> 16), bf2f(kk.y & 0xffff), bf2f(kk.y >> 16),
                               bf2f(kk.z & 0xffff), bf2f(kk.z >> 16), bf2f(kk.w & 0xffff), bf2f(kk.w >> 16)};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float qv[G];
            load_q<G>(qs, c8 + i, qv);
#pragma unroll
            for (int h = 0; h < G; ++h) s[h] = fmaf(qv[h], kf[i], s[h]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] *= kScaleLog2;
      float p[G], alpha[G];
      softmax_update(s, valid, p, alpha);
      rescale(alpha);
#pragma unroll
      for (int h = 0; h < G; ++h) pt[lane * G + h] = p[h];
      __syncwarp();
      for (int t = 0; t < cur.nd; ++t) {
        float pp[G];
        load_q<G>(pt, t, pp);
        const uint2 v4 = *reinterpret_cast<const uint2*>(Vs + t * D + 4 * lane);
        const float vf[4] = {bf2f(v4.x & 0xffff), bf2f(v4.x >> 16), bf2f(v4.y & 0xffff), bf2f(v4.y >> 16)};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int h = 0; h < G; ++h) racc[i][h] = fmaf(pp[h], vf[i], racc[i][h]);
      }
    } else if (cur.kind == 2) {
      const int r = cur.r, gr = TG * r;
      const uint16_t* Kv = reinterpret_cast<const uint16_t*>(buf);
      const uint8_t* Ki = buf + 2 * gr;
      const uint16_t* Vv = reinterpret_cast<const uint16_t*>(buf + 3 * gr);
      const uint8_t* Vi = buf + 5 * gr;
      const int ntok = min(TG, cur.n_live - cur.tg);
      const bool valid = lane < ntok;
      float s[G];
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = 0.0f;
      if (valid) {
        const int row = lane * r;
        if ((r & 1) == 0) {
          const uint16_t* ki2 = reinterpret_cast<const uint16_t*>(Ki + row);
          const uint32_t* kv2 = reinterpret_cast<const uint32_t*>(Kv + row);
#pragma unroll 2
          for (int jj = 0; jj < (r >> 1); ++jj) {
            const uint32_t ip = ki2[jj], vp = kv2[jj];
            float q0[G], q1[G];
            load_q<G>(qs, ip & 0xff, q0);
            load_q<G>(qs, ip >> 8, q1);
            const float v0 = bf2f(vp & 0xffff), v1 = bf2f(vp >> 16);
#pragma unroll
            for (int h = 0; h < G; ++h) s[h] = fmaf(q1[h], v1, fmaf(q0[h], v0, s[h]));
          }
        } else {
          for (int jj = 0; jj < r; ++jj) {
            float qv[G];
            load_q<G>(qs, Ki[row + jj], qv);
            const float kv = bf2f(Kv[row + jj]);
#pragma unroll
            for (int h = 0; h < G; ++h) s[h] = fmaf(qv[h], kv, s[h]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] *= kScaleLog2;
      float p[G], alpha[G];
      softmax_update(s, valid, p, alpha);
      rescale(alpha);
#pragma unroll
      for (int h = 0; h < G; ++h) pt[lane * G + h] = p[h];
      __syncwarp();
      if (NC > 1) {
        // Flattened element stream: element e = t*r + j of this group.  The
        // 32 elements of one instruction span at most NC consecutive tokens,
        // each writing its own accumulator copy (t mod NC), so no two lanes
        // of an instruction touch the same address.
        const int total = ntok * r;
        int t = lane / r, j = lane - t * r, k = t % NC;
        for (int e = lane; e < total; e += 32) {
          float pp[G];
          load_q<G>(pt, t, pp);
          fma_vec<G>(acc + (k * D + Vi[e]) * G, pp, bf2f(Vv[e]));
          j += 32;
          while (j >= r) {
            j -= r;
            ++t;
            if (++k == NC) k = 0;
          }
        }
      } else {
        for (int t = 0; t < ntok; ++t) {
          float pp[G];
          load_q<G>(pt, t, pp);
          for (int jj = lane; jj < r; jj += 32) fma_vec<G>(acc + Vi[t * r + jj] * G, pp, bf2f(Vv[t * r + jj]));
          __syncwarp();
        }
      }
    }
    __syncwarp();
    if (NST == 1) {
      // single stage: fetch the next item only once this one is consumed
      issue(nxt, stg);
      cp_async_commit();
    }
    cur = nxt;
    st ^= (NST - 1);
  }
  cp_async_wait_all();
  __syncwarp();

  // Fold the accumulator copies and the register (dense) accumulators into copy 0.
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int c = 4 * lane + i;
      float a = acc[c * G + h] + racc[i][h];
      for (int k = 1; k < NC; ++k) a += acc[(k * D + c) * G + h];
      acc[c * G + h] = a;
    }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      mlw[(warp * G + h) * 2] = m[h];
      mlw[(warp * G + h) * 2 + 1] = l[h];
    }
  }
  __syncthreads();
  // CTA partial: (m, l, acc) merged over the warps.
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mlw[(w * G + h) * 2]);
    float a = 0.0f, ls = 0.0f;
    if (M != -INFINITY) {
      for (int w = 0; w < kWarps; ++w) {
        const float mw = mlw[(w * G + h) * 2];
        if (mw == -INFINITY) continue;
        const float e = exp2f(mw - M);
        a = fmaf(accw[(w * NC * D + c) * G + h], e, a);
        ls = fmaf(mlw[(w * G + h) * 2 + 1], e, ls);
      }
    }
    cl_acc[h * D + c] = a;
    if (c == 0) {
      cl_ml[h * 2] = M;
      cl_ml[h * 2 + 1] = ls;
    }
  }
  cluster.sync();

  // Merge the cluster's partials for this CTA's channel slice and broadcast
  // the normalised o' slice to every CTA of the cluster.
  const int w = D / C;
  const int c_lo = rank * w;
  for (int i = tid; i < G * w; i += blockDim.x) {
    const int h = i / w, c = c_lo + (i - h * w);
    float M = -INFINITY;
    for (int r2 = 0; r2 < C; ++r2) M = fmaxf(M, cluster.map_shared_rank(cl_ml, r2)[h * 2]);
    float o = 0.0f, ls = 0.0f;
    if (M != -INFINITY) {
      for (int r2 = 0; r2 < C; ++r2) {
        const float* ml = cluster.map_shared_rank(cl_ml, r2);
        const float mr = ml[h * 2];
        if (mr == -INFINITY) continue;
        const float e = exp2f(mr - M);
        o = fmaf(cluster.map_shared_rank(cl_acc, r2)[h * D + c], e, o);
        ls = fmaf(ml[h * 2 + 1], e, ls);
      }
    }
    const float v = ls > 0.0f ? o / ls : 0.0f;
    for (int r2 = 0; r2 < C; ++r2) cluster.map_shared_rank(ofull, r2)[h * D + c] = v;
  }
  cluster.sync();
  if (s_abort) return;

  // Output channels [c_lo, c_lo + w): out_j = sum_c o'_c R_v[c][j].
  uint16_t* orow = out + ((int64_t)ci * L.n_kv * G + (int64_t)kvh * G) * D;
  if (DENSE) {
    for (int i = tid; i < G * w; i += blockDim.x) {
      const int h = i / w, j = c_lo + (i - h * w);
      orow[h * D + j] = f2bf(ofull[h * D + j]);
    }
    return;
  }
  float* rvs = reinterpret_cast<float*>(stages);  // [128][w]: staged R_v columns
  const float* Rv = reinterpret_cast<const float*>(base + L.off_rv);
  const int w4 = w / 4;
  for (int i = tid; i < D * w4; i += blockDim.x) {
    const int c = i / w4, q4 = i - c * w4;
    cp_async16(rvs + c * w + 4 * q4, Rv + (size_t)c * D + c_lo + 4 * q4);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  // Each output (h, j) is split over `parts` threads, combined through smem.
  const int outs = G * w;
  const int parts = max(1, (int)blockDim.x / outs);
  const int cper = D / parts;
  float* red = accw;  // free now: [parts][outs]
  for (int i = tid; i < outs * parts; i += blockDim.x) {
    const int o = i % outs, pidx = i / outs;
    const int h = o / w, jl = o - h * w;
    float a = 0.0f;
    for (int c = pidx * cper; c < (pidx + 1) * cper; ++c) a = fmaf(ofull[h * D + c], rvs[c * w + jl], a);
    red[pidx * outs + o] = a;
  }
  __syncthreads();
  for (int o = tid; o < outs; o += blockDim.x) {
    float a = 0.0f;
    for (int pidx = 0; pidx < parts; ++pidx) a += red[pidx * outs + o];
    const int h = o / w, jl = o - h * w;
    orow[h * D + c_lo + jl] = f2bf(a);
  }
}

namespace {
template <int G, bool DENSE>
cudaError_t launch_one(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids, const int32_t* n_sel,
                       const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t t_stride, uint16_t* out,
                       int cluster, size_t smem, cudaStream_t s) {
  static size_t set_bytes = 0;
  if (smem > set_bytes) {
    cudaError_t e = cudaFuncSetAttribute(k_attn<G, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_attn<G, DENSE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    set_bytes = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Halve the cluster until one cluster of it can be resident (checked once
  // per cluster size and shared-memory size).
  static int verified[17] = {0};
  static size_t verified_smem = 0;
  if (verified_smem != smem) {
    for (int i = 0; i < 17; ++i) verified[i] = 0;
    verified_smem = smem;
  }
  while (cluster > 1) {
    if (verified[cluster] == 0) {
      cfg.gridDim = dim3(cluster, 1, 1);
      attr[0].val.clusterDim.x = cluster;
      int n = 0;
      const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k_attn<G, DENSE>, &cfg);
      if (e != cudaSuccess) (void)cudaGetLastError();
      verified[cluster] = (e == cudaSuccess && n > 0) ? 1 : -1;
      if (std::getenv("MK_LOG"))
        std::fprintf(stderr, "[mosaickv] attention G=%d dense=%d smem=%zu cluster=%d: max active clusters %d (%s)\n",
                     G, (int)DENSE, smem, cluster, n, cudaGetErrorString(e));
    }
    if (verified[cluster] == 1) break;
    cluster /= 2;
  }
  cfg.gridDim = dim3(cluster * cs.n * L.n_kv, 1, 1);
  attr[0].val.clusterDim.x = cluster;
  return cudaLaunchKernelEx(&cfg, k_attn<G, DENSE>, L, layer, cs, ids, n_sel, q, K, V, t_stride, out);
}

template <bool DENSE>
cudaError_t launch_attn_g(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids, const int32_t* n_sel,
                          const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t t_stride, uint16_t* out,
                          int cluster, cudaStream_t s) {
  const size_t smem = attn_smem_bytes(L, 0);
  if (smem == 0 || smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  switch (L.G) {
    case 1: return launch_one<1, DENSE>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, cluster, smem, s);
    case 2: return launch_one<2, DENSE>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, cluster, smem, s);
    case 4: return launch_one<4, DENSE>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, cluster, smem, s);
    case 8: return launch_one<8, DENSE>(L, layer, cs, ids, n_sel, q, K, V, t_stride, out, cluster, smem, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

// Cluster size per (sequence, kv head): a power of two <= 16 (so that 128
// output channels split evenly) giving at most about one CTA per SM.
int attn_cluster_size(int n_units) {
  int c = 1;
  while (c < 16 && (int64_t)n_units * c * 2 <= 152) c *= 2;
  return c;
}

cudaError_t launch_decode_attn(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids,
                               const int32_t* n_sel, uint16_t* out, int cluster, cudaStream_t s) {
  return launch_attn_g<false>(L, layer, cs, ids, n_sel, nullptr, nullptr, nullptr, 0, out, cluster, s);
}

cudaError_t launch_dense_attn(const Layout& L, const CallSeqs& cs, const uint16_t* q, const uint16_t* K,
                              const uint16_t* V, int64_t t_stride, uint16_t* out, int cluster, cudaStream_t s) {
  return launch_attn_g<true>(L, 0, cs, nullptr, nullptr, q, K, V, t_stride, out, cluster, s);
}

}  // namespace mk
