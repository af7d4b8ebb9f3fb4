// Host side of the C ABI (include/mosaickv.h): configuration checks, arena
// and workspace layout, per-call validation, the host view of sequence
// lengths and strategy segments, and kernel launches.  No device memory is
// allocated here: the caller owns the arena and the workspace.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "mk_internal.cuh"

using mk::CallSeqs;
using mk::Layout;
using mk::UnitDesc;

struct mk_ctx {
  mk_config cfg;
  Layout L;
  size_t arena_bytes = 0, ws_bytes = 0;
  int64_t n_units = 0;
  std::vector<int32_t> T;            // [layers][max_seqs]
  std::vector<int32_t> T0;           // prefill length, 0 = not started
  std::vector<int32_t> firsts;       // [layers][max_seqs][MK_MAX_SEGMENTS]
  std::vector<uint8_t> rot_set;      // [layers][max_seqs][n_kv]
  std::vector<std::vector<int32_t>> sel_seqs;  // per layer: sequence list of its last selection
  std::vector<uint8_t> own_rot;      // [units][MK_MAX_SEGMENTS]: segment stored under its own rotation
};

namespace {

constexpr int64_t kAlign = 256;
inline int64_t align_up(int64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Plan {
  Layout L;
  int64_t n_units, units_off, arena_bytes, ws_bytes;
};

// Element-group size of segment i of a bitmap-page configuration: its own,
// else the configuration's, else 1.
int seg_group_of(const mk_config* c, int i) {
  return c->seg[i].elem_group ? c->seg[i].elem_group : (c->elem_group ? c->elem_group : 1);
}
int log2_group(int g) { return g >= 8 ? 3 : g >= 4 ? 2 : g >= 2 ? 1 : 0; }

mk_status check_config(const mk_config* c) {
  if (!c) return MK_EINVAL;
  if (c->head_dim != MK_HEAD_DIM) return MK_EINVAL;
  if (c->n_kv_heads < 1 || c->n_q_heads < 1 || c->n_q_heads % c->n_kv_heads) return MK_EINVAL;
  const int G = c->n_q_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return MK_EINVAL;
  if (c->n_layers < 1 || c->max_seqs < 1 || c->max_seqs > MK_MAX_CALL_SEQS) return MK_EINVAL;
  if (c->max_tokens < 1 || c->n_sink < 0 || c->window < 1) return MK_EINVAL;
  if (c->block != 16 && c->block != 32 && c->block != 64) return MK_EINVAL;
  if (c->topk_fixed < 0 || c->retain_permille < 0 || c->retain_permille > 1000) return MK_EINVAL;
  if (c->topk_fixed == 0 && c->retain_permille == 0) return MK_EINVAL;
  if (c->n_segments < 1 || c->n_segments > MK_MAX_SEGMENTS) return MK_EINVAL;
  if (c->meta_channels < 0 || c->meta_channels > MK_MAX_META_CHANNELS) return MK_EINVAL;
  int prev = 0;
  for (int i = 0; i < c->n_segments; ++i) {
    const mk_segment& s = c->seg[i];
    if (s.r < 1 || s.r > MK_HEAD_DIM || (s.always != 0 && s.always != 1)) return MK_EINVAL;
    if (s.keep_channels != 0 && (s.keep_channels < s.r || s.keep_channels > MK_HEAD_DIM)) return MK_EINVAL;
    if (s.begin_permille < 0 || s.begin_permille > 1000) return MK_EINVAL;
    // Per-segment retention: a scored segment's own rate, not with a fixed k.
    if (s.retain_permille < 0 || s.retain_permille > 1000 || (s.always && s.retain_permille)) return MK_EINVAL;
    if (s.retain_permille && c->topk_fixed > 0) return MK_EINVAL;
    if (i == 0 && s.begin_permille != 0) return MK_EINVAL;
    if (s.begin_permille < prev) return MK_EINVAL;
    prev = s.begin_permille;
    if (c->page_format == MK_PAGES_DENSE && (s.r != MK_HEAD_DIM || s.keep_channels != 0)) return MK_EINVAL;
    if (c->page_format == MK_PAGES_BITMAP) {
      const int g = seg_group_of(c, i);
      if (g != 1 && g != 2 && g != 4 && g != 8) return MK_EINVAL;
      if (s.r % g || s.keep_channels % g) return MK_EINVAL;
    } else if (s.elem_group != 0) {
      return MK_EINVAL;
    }
  }
  if (c->page_format != MK_PAGES_PACKED && c->page_format != MK_PAGES_DENSE && c->page_format != MK_PAGES_BITMAP)
    return MK_EINVAL;
  if (c->page_format == MK_PAGES_DENSE && c->meta_channels != 0) return MK_EINVAL;
  if (c->page_format == MK_PAGES_BITMAP) {
    const int g = c->elem_group;
    if (g != 0 && g != 1 && g != 2 && g != 4 && g != 8) return MK_EINVAL;
  } else if (c->elem_group != 0) {
    return MK_EINVAL;
  }
  return MK_OK;
}

Plan make_plan(const mk_config* c) {
  Plan p{};
  Layout& L = p.L;
  L.S = c->n_sink;
  L.W = c->window;
  L.B = c->block;
  L.n_kv = c->n_kv_heads;
  L.G = c->n_q_heads / c->n_kv_heads;
  L.max_seqs = c->max_seqs;
  L.cap_tokens = c->max_tokens;
  L.n_layers = c->n_layers;
  L.topk_fixed = c->topk_fixed;
  L.retain_permille = c->retain_permille;
  int r_max = 0;
  for (int i = 0; i < c->n_segments; ++i) r_max = std::max(r_max, (int)c->seg[i].r);
  L.r_max = r_max;
  L.nblk_cap = mk::n_mid_blocks(L, c->max_tokens);
  L.per_seg_k = 0;
  for (int i = 0; i < c->n_segments; ++i) {
    L.seg_retain[i] = c->seg[i].retain_permille;
    if (c->seg[i].retain_permille && !c->seg[i].always) L.per_seg_k = 1;
  }
  for (int i = c->n_segments; i < MK_MAX_SEGMENTS; ++i) L.seg_retain[i] = 0;
  if (!L.per_seg_k) {
    L.k_max = std::max(1, mk::n_select(L, L.nblk_cap));
  } else {  // each scored segment's k is at most its rate of the capacity; all of them at most the blocks
    int64_t km = 0;
    for (int i = 0; i < c->n_segments; ++i)
      if (!c->seg[i].always) km += mk::n_select_segment(L, i, L.nblk_cap);
    L.k_max = (int)std::max<int64_t>(1, std::min<int64_t>(km, L.nblk_cap));
  }
  L.keys_stride = (std::max(1, L.nblk_cap) + 3) & ~3;
  L.dense_pages = c->page_format == MK_PAGES_DENSE ? 1 : 0;
  L.bm_g = 0;
  if (c->page_format == MK_PAGES_BITMAP) {  // the smallest group size: the largest bitmap
    L.bm_g = 8;
    for (int i = 0; i < c->n_segments; ++i) L.bm_g = std::min(L.bm_g, seg_group_of(c, i));
  }
  // packed: K and V values (2 r bytes each) and positions, sized for the
  // largest r and the largest positions; dense: 2 x 256 bytes per token
  L.page_stride = L.dense_pages ? (int64_t)4 * L.B * MK_HEAD_DIM
                                : page_vpos(L, r_max, L.bm_g) + (int64_t)L.B * pos_bytes(L, r_max, L.bm_g);
  const int64_t D = MK_HEAD_DIM;
  int64_t off = 0;
  L.off_rkt = off; off += D * D * 4;
  L.off_rvt = off; off += D * D * 4;
  L.off_rv = off; off += D * D * 4;
  L.off_rkp = off; off += 3 * D * D * 2;
  L.off_rvp = off; off += 3 * D * D * 2;
  L.off_sink_k = off; off = align_up(off + std::max<int64_t>(1, L.S) * D * 2);
  L.off_sink_v = off; off = align_up(off + std::max<int64_t>(1, L.S) * D * 2);
  L.off_win_k = off; off = align_up(off + (int64_t)L.W * D * 2);
  L.off_win_v = off; off = align_up(off + (int64_t)L.W * D * 2);
  L.off_meta = off; off = align_up(off + (int64_t)std::max(1, L.nblk_cap) * 2 * D * 2);
  L.off_pages = off; off = align_up(off + (int64_t)std::max(1, L.nblk_cap) * L.page_stride);
  L.meta_c = c->meta_channels;
  L.cmeta_row = L.meta_c > 0 ? (5 * L.meta_c + 15) / 16 * 16 : 0;
  L.off_cmeta = off; off = align_up(off + (int64_t)std::max(1, L.nblk_cap) * L.cmeta_row);
  // Own rotations of the closed segments (re-compression under a segment's own rotation).
  L.n_cls = c->n_segments > 1 ? c->n_segments : 1;
  L.off_segrot = off; off = align_up(off + (int64_t)(L.n_cls - 1) * 2 * D * D * 4);
  L.unit_stride = off;
  p.n_units = (int64_t)c->n_layers * c->max_seqs * c->n_kv_heads;
  p.units_off = align_up(kAlign + p.n_units * (int64_t)sizeof(UnitDesc));
  p.arena_bytes = p.units_off + p.n_units * L.unit_stride;
  const int64_t slots = (int64_t)c->max_seqs * c->n_kv_heads;
  int64_t w = 0;
  w = align_up(w + (int64_t)L.n_cls * c->n_layers * slots * L.G * D * 4);  // qrot, per class and layer
  w = align_up(w + (int64_t)c->n_layers * slots * MK_MAX_SEGMENTS * 4);     // seg_sel
  w = align_up(w + slots * (int64_t)L.keys_stride * 4);        // block keys
  w = align_up(w + slots * (int64_t)mk::kKeyBins * 4);         // coarse key histograms
  w = align_up(w + slots * MK_MAX_SPLITS * L.G * D * 4);       // part_acc
  w = align_up(w + slots * MK_MAX_SPLITS * L.G * 2 * 4);       // part_ml
  w = align_up(w + slots * 4 * 2);                             // counters: attention, selection
  p.ws_bytes = w;
  return p;
}

void bind_pointers(Plan& p, void* arena, void* ws) {
  Layout& L = p.L;
  char* a = static_cast<char*>(arena);
  L.arena = a;
  L.err = reinterpret_cast<int32_t*>(a);
  L.desc = reinterpret_cast<UnitDesc*>(a + kAlign);
  L.units = a + p.units_off;
  const int64_t D = MK_HEAD_DIM;
  const int64_t slots = (int64_t)L.max_seqs * L.n_kv;
  char* w = static_cast<char*>(ws);
  int64_t o = 0;
  L.qrot = reinterpret_cast<float*>(w + o); o = align_up(o + (int64_t)L.n_cls * L.n_layers * slots * L.G * D * 4);
  L.seg_sel = reinterpret_cast<int32_t*>(w + o); o = align_up(o + (int64_t)L.n_layers * slots * MK_MAX_SEGMENTS * 4);
  L.keys = reinterpret_cast<uint32_t*>(w + o); o = align_up(o + slots * (int64_t)L.keys_stride * 4);
  L.khist = reinterpret_cast<uint32_t*>(w + o); o = align_up(o + slots * (int64_t)mk::kKeyBins * 4);
  L.part_acc = reinterpret_cast<float*>(w + o); o = align_up(o + slots * MK_MAX_SPLITS * L.G * D * 4);
  L.part_ml = reinterpret_cast<float*>(w + o); o = align_up(o + slots * MK_MAX_SPLITS * L.G * 2 * 4);
  L.counters = reinterpret_cast<int32_t*>(w + o);
}

// Segment rule: segment i >= 1 starts at the first block boundary at or after
// begin_permille/1000 of the prefill length T0, clamped to [previous start,
// number of middle blocks at T0]; segment 0 starts at block 0.
void segment_firsts(const mk_config& c, const Layout& L, int T0, int32_t* out) {
  const int nb0 = mk::n_mid_blocks(L, T0);
  int prev = 0;
  for (int i = 0; i < MK_MAX_SEGMENTS; ++i) {
    int b = 0;
    if (i > 0 && i < c.n_segments) {
      const int64_t pos = (int64_t)c.seg[i].begin_permille * T0 / 1000;
      const int64_t rel = std::max<int64_t>(0, pos - L.S);
      b = (int)((rel + L.B - 1) / L.B);
      b = std::min(std::max(b, prev), nb0);
    } else if (i >= c.n_segments) {
      b = prev;
    }
    out[i] = b;
    prev = b;
  }
}

UnitDesc host_desc(const mk_ctx* ctx, int layer, int seq) {
  UnitDesc d{};
  const size_t i = (size_t)layer * ctx->cfg.max_seqs + seq;
  d.T = ctx->T[i];
  d.T0 = ctx->T0[i];
  d.n_seg = ctx->cfg.n_segments;
  for (int s = 0; s < MK_MAX_SEGMENTS; ++s) {
    d.first_block[s] = ctx->firsts[i * MK_MAX_SEGMENTS + s];
    d.r[s] = s < ctx->cfg.n_segments ? ctx->cfg.seg[s].r : 0;
    if (s < ctx->cfg.n_segments) {
      const mk_segment& g = ctx->cfg.seg[s];
      d.sflags[s] = mk::seg_flags(g.always != 0, g.keep_channels ? g.keep_channels : MK_HEAD_DIM,
                                  ctx->cfg.page_format == MK_PAGES_BITMAP ? log2_group(seg_group_of(&ctx->cfg, s))
                                                                          : 0);
    } else {
      d.sflags[s] = mk::seg_flags(false, MK_HEAD_DIM);
    }
  }
  return d;
}

mk_status check_seqs(const mk_ctx* ctx, int32_t layer, int32_t n_seqs, const int32_t* seq_ids) {
  if (!ctx || !seq_ids) return MK_EINVAL;
  if (layer < 0 || layer >= ctx->cfg.n_layers) return MK_EINVAL;
  if (n_seqs < 1 || n_seqs > MK_MAX_CALL_SEQS || n_seqs > ctx->cfg.max_seqs) return MK_EINVAL;
  std::vector<uint8_t> seen(ctx->cfg.max_seqs, 0);
  for (int i = 0; i < n_seqs; ++i) {
    const int s = seq_ids[i];
    if (s < 0 || s >= ctx->cfg.max_seqs || seen[s]) return MK_EINVAL;
    seen[s] = 1;
  }
  return MK_OK;
}

inline mk_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MK_OK : MK_ECUDA; }

// Whether some unit of the call has a segment stored under its own rotation.
bool call_has_own(const mk_ctx* ctx, int layer, int n_seqs, const int32_t* seq_ids) {
  for (int i = 0; i < n_seqs; ++i)
    for (int h = 0; h < ctx->cfg.n_kv_heads; ++h) {
      const int64_t u = mk::unit_index(ctx->L, layer, seq_ids[i], h);
      for (int sg = 0; sg < MK_MAX_SEGMENTS; ++sg)
        if (ctx->own_rot[(size_t)u * MK_MAX_SEGMENTS + sg]) return true;
    }
  return false;
}

}  // namespace

namespace mk {

cudaError_t kernel_smem_attr(const void* fn, int bytes, int threads, int* occ, int* sms) {
  struct Entry {
    int attr_bytes = -1;             // limit set on this device
    int occ_bytes = -1, occ_threads = 0, occ = 1, sms = 0;
  };
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, Entry> seen;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  Entry& en = seen[{fn, dev}];
  if (en.attr_bytes < bytes) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    en.attr_bytes = bytes;
  }
  if ((occ || sms) && (en.occ_bytes != bytes || en.occ_threads != threads)) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, (size_t)bytes) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 1;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      v = 0;
    }
    en.occ = n > 0 ? n : 1;
    en.sms = v;
    en.occ_bytes = bytes;
    en.occ_threads = threads;
  }
  if (occ) *occ = en.occ;
  if (sms) *sms = en.sms;
  return cudaSuccess;
}

}  // namespace mk

extern "C" {

const char* mk_status_str(mk_status s) {
  switch (s) {
    case MK_OK: return "ok";
    case MK_EINVAL: return "invalid argument";
    case MK_ENOMEM: return "buffer too small or capacity exceeded";
    case MK_ESTATE: return "call out of order";
    case MK_ECUDA: return "CUDA runtime error";
    case MK_EDEVICE: return "device error word set";
    case MK_ETIMEOUT: return "device wait timed out";
    case MK_ENOTSUP: return "not supported";
  }
  return "unknown status";
}

mk_status mk_arena_bytes(const mk_config* cfg, size_t* bytes) {
  mk_status st = check_config(cfg);
  if (st != MK_OK || !bytes) return st != MK_OK ? st : MK_EINVAL;
  *bytes = (size_t)make_plan(cfg).arena_bytes;
  return MK_OK;
}

mk_status mk_workspace_bytes(const mk_config* cfg, size_t* bytes) {
  mk_status st = check_config(cfg);
  if (st != MK_OK || !bytes) return st != MK_OK ? st : MK_EINVAL;
  *bytes = (size_t)make_plan(cfg).ws_bytes;
  return MK_OK;
}

mk_status mk_max_select(const mk_config* cfg, int32_t* k_max) {
  mk_status st = check_config(cfg);
  if (st != MK_OK || !k_max) return st != MK_OK ? st : MK_EINVAL;
  *k_max = make_plan(cfg).L.k_max;
  return MK_OK;
}

mk_status mk_create(const mk_config* cfg, void* arena, size_t arena_bytes, void* workspace,
                    size_t workspace_bytes, mk_ctx** out) {
  mk_status st = check_config(cfg);
  if (st != MK_OK) return st;
  if (!arena || !workspace || !out) return MK_EINVAL;
  if (((uintptr_t)arena % kAlign) || ((uintptr_t)workspace % kAlign)) return MK_EINVAL;
  Plan p = make_plan(cfg);
  if ((int64_t)arena_bytes < p.arena_bytes || (int64_t)workspace_bytes < p.ws_bytes) return MK_ENOMEM;
  // Page tokens a unit may attend: its selection plus the always-attended
  // segments (a fraction of the prefill, at most of the capacity).
  int64_t attend_max = (int64_t)p.L.k_max * cfg->block;
  for (int i = 0; i < cfg->n_segments; ++i)
    if (cfg->seg[i].always) {
      const int end = i + 1 < cfg->n_segments ? cfg->seg[i + 1].begin_permille : 1000;
      attend_max += (int64_t)(end - cfg->seg[i].begin_permille) * cfg->max_tokens / 1000 + 2 * cfg->block;
    }
  if (mk::attn_plan(p.L, attend_max) == 0) return MK_ENOTSUP;
  if (!mk::select_plan_ok(p.L)) return MK_ENOTSUP;
  bind_pointers(p, arena, workspace);
  mk_ctx* ctx = new (std::nothrow) mk_ctx();
  if (!ctx) return MK_ENOMEM;
  ctx->cfg = *cfg;
  ctx->L = p.L;
  ctx->arena_bytes = arena_bytes;
  ctx->ws_bytes = workspace_bytes;
  ctx->n_units = p.n_units;
  const size_t ls = (size_t)cfg->n_layers * cfg->max_seqs;
  ctx->T.assign(ls, 0);
  ctx->T0.assign(ls, 0);
  ctx->firsts.assign(ls * MK_MAX_SEGMENTS, 0);
  ctx->rot_set.assign(ls * cfg->n_kv_heads, 0);
  ctx->sel_seqs.assign(cfg->n_layers, std::vector<int32_t>());
  ctx->own_rot.assign((size_t)p.n_units * MK_MAX_SEGMENTS, 0);
  cudaError_t e = cudaMemset(arena, 0, (size_t)p.units_off);
  if (e == cudaSuccess) e = cudaMemset(ctx->L.counters, 0, sizeof(int32_t) * 2 * cfg->max_seqs * cfg->n_kv_heads);
  if (e == cudaSuccess)
    e = cudaMemset(ctx->L.khist, 0, sizeof(uint32_t) * mk::kKeyBins * cfg->max_seqs * cfg->n_kv_heads);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    delete ctx;
    return MK_ECUDA;
  }
  *out = ctx;
  return MK_OK;
}

mk_status mk_destroy(mk_ctx* ctx) {
  delete ctx;
  return MK_OK;
}

mk_status mk_set_rotation(mk_ctx* ctx, int32_t layer, int32_t seq, int32_t kv_head, const float* Rk,
                          const float* Rv, mk_stream stream) {
  if (!ctx || !Rk || !Rv) return MK_EINVAL;
  if (layer < 0 || layer >= ctx->cfg.n_layers || seq < 0 || seq >= ctx->cfg.max_seqs || kv_head < 0 ||
      kv_head >= ctx->cfg.n_kv_heads)
    return MK_EINVAL;
  const size_t ls = (size_t)layer * ctx->cfg.max_seqs + seq;
  if (ctx->T[ls] != 0) return MK_ESTATE;
  const int D = MK_HEAD_DIM;
  // R_k^T, R_v^T, R_v (fp32), then R_k and R_v each split exactly into three
  // bf16 parts (x = p0 + p1 + p2: 8 significant bits each, truncated) in the
  // tensor cores' K-major operand layout (B operand of k' = k R^T: row = output
  // channel, K = input channel), contiguous after them in the unit.
  std::vector<float> buf((size_t)3 * D * D + (size_t)3 * D * D);  // 3 fp32 matrices + 6 bf16 parts
  uint16_t* parts = reinterpret_cast<uint16_t*>(buf.data() + (size_t)3 * D * D);
  auto split3 = [](float x, uint16_t p[3]) {
    float r = x;
    for (int i = 0; i < 3; ++i) {
      uint32_t b;
      std::memcpy(&b, &r, 4);
      p[i] = (uint16_t)(b >> 16);
      const uint32_t hb = b & 0xffff0000u;
      float h;
      std::memcpy(&h, &hb, 4);
      r -= h;
    }
  };
  for (int i = 0; i < D; ++i)
    for (int j = 0; j < D; ++j) {
      buf[(size_t)j * D + i] = Rk[(size_t)i * D + j];                 // R_k^T
      buf[(size_t)D * D + (size_t)j * D + i] = Rv[(size_t)i * D + j];  // R_v^T
      buf[(size_t)2 * D * D + (size_t)i * D + j] = Rv[(size_t)i * D + j];
      const int off = mk::umma_kmajor_offset(i, j) / 2;  // element (row i, k j), in bf16 units
      uint16_t pk[3], pv[3];
      split3(Rk[(size_t)i * D + j], pk);
      split3(Rv[(size_t)i * D + j], pv);
      for (int q = 0; q < 3; ++q) {
        parts[(size_t)q * D * D + off] = pk[q];
        parts[(size_t)(3 + q) * D * D + off] = pv[q];
      }
    }
  const int64_t u = mk::unit_index(ctx->L, layer, seq, kv_head);
  char* dst = ctx->L.units + u * ctx->L.unit_stride + ctx->L.off_rkt;
  cudaError_t e = cudaMemcpyAsync(dst, buf.data(), buf.size() * sizeof(float), cudaMemcpyHostToDevice,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return MK_ECUDA;
  ctx->rot_set[ls * ctx->cfg.n_kv_heads + kv_head] = 1;
  return MK_OK;
}

mk_status mk_append_compress(mk_ctx* ctx, int32_t layer, int32_t n_seqs, const int32_t* seq_ids,
                             const int32_t* n_new, const void* k, const void* v, mk_stream stream) {
  mk_status st = check_seqs(ctx, layer, n_seqs, seq_ids);
  if (st != MK_OK) return st;
  if (!n_new) return MK_EINVAL;
  int64_t total = 0;
  int max_new = 0;
  for (int i = 0; i < n_seqs; ++i) {
    if (n_new[i] < 0) return MK_EINVAL;
    total += n_new[i];
    max_new = std::max(max_new, (int)n_new[i]);
    const size_t ls = (size_t)layer * ctx->cfg.max_seqs + seq_ids[i];
    if ((int64_t)ctx->T[ls] + n_new[i] > ctx->cfg.max_tokens) return MK_ENOMEM;
    for (int h = 0; h < ctx->cfg.n_kv_heads; ++h)
      if (!ctx->rot_set[ls * ctx->cfg.n_kv_heads + h]) return MK_ESTATE;
  }
  if (total == 0) return MK_OK;
  if (!k || !v || total > INT32_MAX) return MK_EINVAL;
  // The bulk path reads 16-byte vectors of k and v.
  if (max_new > mk::kSmallAppend && (((uintptr_t)k | (uintptr_t)v) & 15u) != 0) return MK_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  CallSeqs* cs = new (std::nothrow) CallSeqs();
  if (!cs) return MK_ENOMEM;
  cs->n = n_seqs;
  int row = 0, tiles = 0;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < n_seqs; ++i) {
    const size_t ls = (size_t)layer * ctx->cfg.max_seqs + seq_ids[i];
    cs->seq[i] = seq_ids[i];
    cs->n_new[i] = n_new[i];
    cs->row_off[i] = row;
    cs->T_old[i] = ctx->T[ls];
    cs->tile_off[i] = tiles;
    row += n_new[i];
    tiles += mk::n_tiles(ctx->T[ls], ctx->T[ls] + n_new[i], ctx->L.S);
    if (ctx->T0[ls] == 0 && n_new[i] > 0) {
      ctx->T0[ls] = n_new[i];
      segment_firsts(ctx->cfg, ctx->L, n_new[i], &ctx->firsts[ls * MK_MAX_SEGMENTS]);
      if (e == cudaSuccess) e = mk::launch_init_desc(ctx->L, layer, seq_ids[i], host_desc(ctx, layer, seq_ids[i]), s);
    }
  }
  cs->tile_off[n_seqs] = tiles;
  const uint16_t* kk = static_cast<const uint16_t*>(k);
  const uint16_t* vv = static_cast<const uint16_t*>(v);
  if (e == cudaSuccess) {
    if (max_new <= mk::kSmallAppend) {
      e = mk::launch_append_small(ctx->L, layer, *cs, kk, vv, 0, s);
    } else {
      e = mk::launch_append_small(ctx->L, layer, *cs, kk, vv, 1, s);
      if (e == cudaSuccess && tiles > 0) e = mk::launch_append_bulk(ctx->L, layer, *cs, kk, vv, tiles, s);
    }
  }
  delete cs;
  if (e != cudaSuccess) return MK_ECUDA;
  for (int i = 0; i < n_seqs; ++i) ctx->T[(size_t)layer * ctx->cfg.max_seqs + seq_ids[i]] += n_new[i];
  return MK_OK;
}

mk_status mk_block_select(mk_ctx* ctx, int32_t layer, int32_t n_seqs, const int32_t* seq_ids, const void* q,
                          int32_t* ids, int32_t* n_sel, float* scores, mk_stream stream) {
  mk_status st = check_seqs(ctx, layer, n_seqs, seq_ids);
  if (st != MK_OK) return st;
  if (!q || !ids || !n_sel) return MK_EINVAL;
  CallSeqs* cs = new (std::nothrow) CallSeqs();
  if (!cs) return MK_ENOMEM;
  cs->n = n_seqs;
  int max_nblk = 0;
  for (int i = 0; i < n_seqs; ++i) {
    const size_t ls = (size_t)layer * ctx->cfg.max_seqs + seq_ids[i];
    if (ctx->T[ls] == 0) {
      delete cs;
      return MK_ESTATE;
    }
    cs->seq[i] = seq_ids[i];
    cs->T_old[i] = ctx->T[ls];
    max_nblk = std::max(max_nblk, mk::n_mid_blocks(ctx->L, ctx->T[ls]));
  }
  cudaError_t e = mk::launch_block_select(ctx->L, layer, *cs, static_cast<const uint16_t*>(q), ids, n_sel, scores,
                                          std::max(1, max_nblk), (cudaStream_t)stream, nullptr, nullptr,
                                          call_has_own(ctx, layer, n_seqs, seq_ids));
  delete cs;
  if (e != cudaSuccess) return MK_ECUDA;
  ctx->sel_seqs[layer].assign(seq_ids, seq_ids + n_seqs);
  return MK_OK;
}

mk_status mk_append_select(mk_ctx* ctx, int32_t layer, int32_t n_seqs, const int32_t* seq_ids, const void* k,
                           const void* v, const void* q, int32_t* ids, int32_t* n_sel, float* scores,
                           mk_stream stream) {
  mk_status st = check_seqs(ctx, layer, n_seqs, seq_ids);
  if (st != MK_OK) return st;
  if (!k || !v || !q || !ids || !n_sel) return MK_EINVAL;
  int max_nblk = 0;
  for (int i = 0; i < n_seqs; ++i) {
    const size_t ls = (size_t)layer * ctx->cfg.max_seqs + seq_ids[i];
    if (ctx->T[ls] == 0) return MK_ESTATE;  // the prefill comes first
    if ((int64_t)ctx->T[ls] + 1 > ctx->cfg.max_tokens) return MK_ENOMEM;
    for (int h = 0; h < ctx->cfg.n_kv_heads; ++h)
      if (!ctx->rot_set[ls * ctx->cfg.n_kv_heads + h]) return MK_ESTATE;
    max_nblk = std::max(max_nblk, mk::n_mid_blocks(ctx->L, ctx->T[ls] + 1));
  }
  CallSeqs* cs = new (std::nothrow) CallSeqs();
  if (!cs) return MK_ENOMEM;
  cs->n = n_seqs;
  for (int i = 0; i < n_seqs; ++i) {
    const size_t ls = (size_t)layer * ctx->cfg.max_seqs + seq_ids[i];
    cs->seq[i] = seq_ids[i];
    cs->n_new[i] = 1;
    cs->row_off[i] = i;
    cs->T_old[i] = ctx->T[ls];
  }
  cudaError_t e = mk::launch_block_select(ctx->L, layer, *cs, static_cast<const uint16_t*>(q), ids, n_sel, scores,
                                          std::max(1, max_nblk), (cudaStream_t)stream,
                                          static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v),
                                          call_has_own(ctx, layer, n_seqs, seq_ids));
  delete cs;
  if (e != cudaSuccess) return MK_ECUDA;
  for (int i = 0; i < n_seqs; ++i) ctx->T[(size_t)layer * ctx->cfg.max_seqs + seq_ids[i]] += 1;
  ctx->sel_seqs[layer].assign(seq_ids, seq_ids + n_seqs);
  return MK_OK;
}

mk_status mk_decode_attn(mk_ctx* ctx, int32_t layer, int32_t n_seqs, const int32_t* seq_ids, const int32_t* ids,
                         const int32_t* n_sel, void* out, mk_stream stream) {
  mk_status st = check_seqs(ctx, layer, n_seqs, seq_ids);
  if (st != MK_OK) return st;
  if (!ids || !n_sel || !out) return MK_EINVAL;
  const std::vector<int32_t>& last = ctx->sel_seqs[layer];
  if ((int)last.size() != n_seqs || !std::equal(last.begin(), last.end(), seq_ids)) return MK_ESTATE;
  CallSeqs* cs = new (std::nothrow) CallSeqs();
  if (!cs) return MK_ENOMEM;
  cs->n = n_seqs;
  int32_t items[MK_MAX_CALL_SEQS], min_parts[MK_MAX_CALL_SEQS];
  for (int i = 0; i < n_seqs; ++i) {
    cs->seq[i] = seq_ids[i];
    const size_t ls = (size_t)layer * ctx->cfg.max_seqs + seq_ids[i];
    // one CTA per rotation class of the unit with the most own-rotation segments
    min_parts[i] = 1;
    for (int h = 0; h < ctx->cfg.n_kv_heads; ++h) {
      const int64_t u = mk::unit_index(ctx->L, layer, seq_ids[i], h);
      int n_own = 0;
      for (int sg = 0; sg < MK_MAX_SEGMENTS; ++sg) n_own += ctx->own_rot[(size_t)u * MK_MAX_SEGMENTS + sg];
      min_parts[i] = std::max(min_parts[i], 1 + n_own);
    }
    const int T = ctx->T[ls];
    const int nblk = mk::n_mid_blocks(ctx->L, T);
    const UnitDesc d = host_desc(ctx, layer, seq_ids[i]);
    const int scored = mk::n_scored_blocks(d, nblk);
    const int dense = std::min(ctx->L.S, T) + std::max(0, T - (ctx->L.S + mk::n_mid_tokens(ctx->L, T)));
    const int groups = (ctx->L.B + mk::kDenseChunk - 1) / mk::kDenseChunk;
    items[i] = (dense + mk::kDenseChunk - 1) / mk::kDenseChunk +
               (mk::n_select_unit(ctx->L, d, nblk) + (nblk - scored)) * groups;
  }
  cudaError_t e = mk::launch_decode_attn(ctx->L, layer, *cs, ids, n_sel, static_cast<uint16_t*>(out), items,
                                         (cudaStream_t)stream, min_parts);
  delete cs;
  return cuda_status(e);
}

mk_status mk_dense_decode_attn(mk_ctx* ctx, int32_t n_seqs, const int32_t* T, const void* q, const void* K,
                               const void* V, int64_t t_stride, void* out, mk_stream stream) {
  if (!ctx || !T || !q || !K || !V || !out) return MK_EINVAL;
  if (((uintptr_t)q | (uintptr_t)K | (uintptr_t)V | (uintptr_t)out) & 15) return MK_EINVAL;  // bulk-copied rows
  if (n_seqs < 1 || n_seqs > ctx->cfg.max_seqs || t_stride < 1) return MK_EINVAL;
  CallSeqs* cs = new (std::nothrow) CallSeqs();
  if (!cs) return MK_ENOMEM;
  cs->n = n_seqs;
  int32_t items[MK_MAX_CALL_SEQS];
  for (int i = 0; i < n_seqs; ++i) {
    if (T[i] < 1 || T[i] > t_stride) {
      delete cs;
      return MK_EINVAL;
    }
    cs->seq[i] = i;
    cs->T_old[i] = T[i];
    items[i] = (T[i] + mk::kDenseChunk - 1) / mk::kDenseChunk;
  }
  cudaError_t e = mk::launch_dense_attn(ctx->L, *cs, static_cast<const uint16_t*>(q),
                                        static_cast<const uint16_t*>(K), static_cast<const uint16_t*>(V), t_stride,
                                        static_cast<uint16_t*>(out), items, (cudaStream_t)stream);
  delete cs;
  return cuda_status(e);
}

mk_status mk_gram(const void* x, int64_t n_rows, int64_t row_stride, float* gram, mk_stream stream) {
  if (!x || !gram || n_rows < 1 || row_stride < MK_HEAD_DIM || row_stride % 8 || ((uintptr_t)x & 15))
    return MK_EINVAL;
  return cuda_status(mk::launch_gram(static_cast<const uint16_t*>(x), n_rows, row_stride, gram,
                                     (cudaStream_t)stream));
}

mk_status mk_poll_error(mk_ctx* ctx, int32_t* detail) {
  if (!ctx) return MK_EINVAL;
  int32_t w[4] = {0, 0, 0, 0};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(w, ctx->L.err, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return MK_ECUDA;
  if (detail) *detail = w[1];
  return w[0] == 0 ? MK_OK : (mk_status)w[0];
}

mk_status mk_clear_error(mk_ctx* ctx) {
  if (!ctx) return MK_EINVAL;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemset(ctx->L.err, 0, 4 * sizeof(int32_t));
  // Kernels that gave up may have left arrival counters and key histograms
  // part-way: back to zero.
  const size_t slots = (size_t)ctx->cfg.max_seqs * ctx->cfg.n_kv_heads;
  if (e == cudaSuccess) e = cudaMemset(ctx->L.counters, 0, sizeof(int32_t) * 2 * slots);
  if (e == cudaSuccess) e = cudaMemset(ctx->L.khist, 0, sizeof(uint32_t) * mk::kKeyBins * slots);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return cuda_status(e);
}

mk_status mk_sync_state(mk_ctx* ctx) {
  if (!ctx) return MK_EINVAL;
  std::vector<UnitDesc> d((size_t)ctx->n_units);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(d.data(), ctx->L.desc, d.size() * sizeof(UnitDesc), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return MK_ECUDA;
  for (int l = 0; l < ctx->cfg.n_layers; ++l)
    for (int s = 0; s < ctx->cfg.max_seqs; ++s) {
      const size_t ls = (size_t)l * ctx->cfg.max_seqs + s;
      if (ctx->T0[ls] > 0) ctx->T[ls] = d[(size_t)mk::unit_index(ctx->L, l, s, 0)].T;
    }
  return MK_OK;
}

mk_status mk_seq_length(mk_ctx* ctx, int32_t layer, int32_t seq, int32_t* T) {
  if (!ctx || !T || layer < 0 || layer >= ctx->cfg.n_layers || seq < 0 || seq >= ctx->cfg.max_seqs)
    return MK_EINVAL;
  *T = ctx->T[(size_t)layer * ctx->cfg.max_seqs + seq];
  return MK_OK;
}

mk_status mk_layout(mk_ctx* ctx, int32_t layer, int32_t seq, int32_t kv_head, mk_layout_info* out) {
  if (!ctx || !out || layer < 0 || layer >= ctx->cfg.n_layers || seq < 0 || seq >= ctx->cfg.max_seqs ||
      kv_head < 0 || kv_head >= ctx->cfg.n_kv_heads)
    return MK_EINVAL;
  const Layout& L = ctx->L;
  const int64_t base = (L.units - L.arena) + mk::unit_index(L, layer, seq, kv_head) * L.unit_stride;
  std::memset(out, 0, sizeof(*out));
  out->rkt = base + L.off_rkt;
  out->rvt = base + L.off_rvt;
  out->rv = base + L.off_rv;
  out->sink_k = base + L.off_sink_k;
  out->sink_v = base + L.off_sink_v;
  out->win_k = base + L.off_win_k;
  out->win_v = base + L.off_win_v;
  out->meta = base + L.off_meta;
  out->pages = base + L.off_pages;
  out->page_stride = L.page_stride;
  out->nblk_cap = L.nblk_cap;
  const size_t ls = (size_t)layer * ctx->cfg.max_seqs + seq;
  out->T = ctx->T[ls];
  for (int s = 0; s < MK_MAX_SEGMENTS; ++s) out->seg_first_block[s] = ctx->firsts[ls * MK_MAX_SEGMENTS + s];
  out->n_segments = ctx->cfg.n_segments;
  out->cmeta = base + L.off_cmeta;
  out->cmeta_row = L.cmeta_row;
  out->meta_channels = L.meta_c;
  return MK_OK;
}

mk_status mk_record_event(void* event, mk_stream stream) {
  if (!event) return MK_EINVAL;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing((cudaStream_t)stream, &cap);
  if (e != cudaSuccess) return MK_ECUDA;
  const unsigned flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  return cuda_status(cudaEventRecordWithFlags((cudaEvent_t)event, (cudaStream_t)stream, flags));
}

}  // extern "C"

mk_status mk_swap_segment(mk_ctx* ctx, int32_t layer, int32_t seq, int32_t kv_head, int32_t segment, int32_t r,
                          int32_t keep_channels, const float* R_k, const float* R_v, const void* pages,
                          const void* meta, const void* cmeta, mk_stream stream) {
  if (!ctx || !pages || !meta) return MK_EINVAL;
  const mk_config& c = ctx->cfg;
  const Layout& L = ctx->L;
  if (L.dense_pages) return MK_ENOTSUP;  // uncompressed pages have nothing to re-compress
  if (layer < 0 || layer >= c.n_layers || seq < 0 || seq >= c.max_seqs || kv_head < 0 || kv_head >= c.n_kv_heads)
    return MK_EINVAL;
  if (segment < 0 || segment >= c.n_segments) return MK_EINVAL;
  if (r < 1 || r > L.r_max) return MK_EINVAL;  // the pages hold at most r_max entries per token
  if (keep_channels != 0 && (keep_channels < r || keep_channels > MK_HEAD_DIM)) return MK_EINVAL;
  if (L.bm_g) {  // the segment keeps its element-group size: whole groups only
    const int g = seg_group_of(&c, segment);
    if (r % g || keep_channels % g) return MK_EINVAL;
  }
  if (L.meta_c > 0 && !cmeta) return MK_EINVAL;
  if ((R_k == nullptr) != (R_v == nullptr)) return MK_EINVAL;
  const size_t ls = (size_t)layer * c.max_seqs + seq;
  if (ctx->T0[ls] == 0 || segment == c.n_segments - 1) return MK_ESTATE;
  const int fb = ctx->firsts[ls * MK_MAX_SEGMENTS + segment], lb = ctx->firsts[ls * MK_MAX_SEGMENTS + segment + 1];
  const int n = lb - fb;
  if (n <= 0) return MK_ESTATE;
  // The attention trusts the positions it reads from the pages: check them
  // here, before any copy (a closed segment's blocks are complete).  uint8
  // indices must name channels below 128; a bitmap row must hold exactly
  // r / g groups.
  {
    const int g = L.bm_g ? seg_group_of(&c, segment) : 0;
    const int pb = g ? MK_HEAD_DIM / g / 8 : r;
    const int64_t Br = (int64_t)L.B * r, Bp = (int64_t)L.B * pb;
    const unsigned char* pg = static_cast<const unsigned char*>(pages);
    for (int b = 0; b < n; ++b) {
      const unsigned char* page = pg + (int64_t)b * L.page_stride;
      for (int w = 0; w < 2; ++w) {
        const unsigned char* pos = page + (w == 0 ? 2 * Br : 4 * Br + Bp);
        for (int t = 0; t < L.B; ++t) {
          const unsigned char* row = pos + (int64_t)t * pb;
          if (g) {
            int bits = 0;
            for (int i = 0; i < pb; ++i) bits += __builtin_popcount(row[i]);
            if (bits != r / g) return MK_EINVAL;
          } else {
            for (int i = 0; i < r; ++i)
              if (row[i] >= MK_HEAD_DIM) return MK_EINVAL;
          }
        }
      }
    }
  }
  const int64_t u = mk::unit_index(L, layer, seq, kv_head);
  char* base = L.units + u * L.unit_stride;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(base + L.off_pages + (int64_t)fb * L.page_stride, pages,
                                  (size_t)n * (size_t)L.page_stride, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + L.off_meta + (int64_t)fb * 2 * MK_HEAD_DIM * 2, meta,
                        (size_t)n * 2 * MK_HEAD_DIM * 2, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && L.meta_c > 0)
    e = cudaMemcpyAsync(base + L.off_cmeta + (int64_t)fb * L.cmeta_row, cmeta, (size_t)n * (size_t)L.cmeta_row,
                        cudaMemcpyHostToDevice, s);
  const bool own = R_k != nullptr;
  if (own && e == cudaSuccess) {
    // The segment's rotation in the layouts the kernels read: R_k^T for the
    // selection's query rotation, R_v for the attention's un-rotation.  The
    // copy is from pageable memory, so the data has been taken when it
    // returns (it waits for the stream's earlier work, as a rotation change
    // should).
    std::vector<float> rt((size_t)2 * MK_HEAD_DIM * MK_HEAD_DIM);
    for (int i = 0; i < MK_HEAD_DIM; ++i)
      for (int j = 0; j < MK_HEAD_DIM; ++j) {
        rt[(size_t)j * MK_HEAD_DIM + i] = R_k[(size_t)i * MK_HEAD_DIM + j];
        rt[(size_t)MK_HEAD_DIM * MK_HEAD_DIM + (size_t)i * MK_HEAD_DIM + j] = R_v[(size_t)i * MK_HEAD_DIM + j];
      }
    e = cudaMemcpyAsync(base + mk::segrot_off(L, segment), rt.data(), rt.size() * sizeof(float),
                        cudaMemcpyHostToDevice, s);
  }
  if (e == cudaSuccess)
    e = mk::launch_set_segment(L, u, segment, r, keep_channels ? keep_channels : MK_HEAD_DIM, own ? 1 : 0, s);
  if (e == cudaSuccess) ctx->own_rot[(size_t)u * MK_MAX_SEGMENTS + segment] = own ? 1 : 0;
  return cuda_status(e);
}
