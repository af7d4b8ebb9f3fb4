// Internal declarations shared by the kernels and the host layer of
// libmosaickv.so.  Not part of the public ABI (include/mosaickv.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/mosaickv.h"

namespace mk {

constexpr int D = MK_HEAD_DIM;
constexpr int kDenseChunk = 16;        // tokens per dense work item in attention
constexpr int kTileTokens = 128;       // tokens per bulk-append tile (one 128-row tensor-core tile)
constexpr int kSmallAppend = 16;       // largest per-sequence append handled by the decode kernel
constexpr int kKeyBins = 4096;         // coarse key histogram of the block selection (top 12 key bits)
constexpr uint32_t FULL = 0xffffffffu;

// Device error codes (detail word); the status word holds MK_EDEVICE.
enum DevErr : int32_t {
  ERR_NONE = 0,
  ERR_CAPACITY = 1,    // append past max_tokens
  ERR_BAD_BLOCK = 2,   // selected block id out of range
  ERR_BAD_NSEL = 3,    // n_sel larger than the ids row
  ERR_NO_ROTATION = 4,
  ERR_COPY_WAIT = 5,   // a bulk copy did not complete within the wait bound (status MK_ETIMEOUT)
  ERR_BOUNDS = 6,      // checked build: an index failed its bounds check (unit = site, aux = index)
};

// Sites of the checked build's bounds checks (reported in the error word).
enum CheckSite : int32_t {
  SITE_DECODE_PAGE = 1,   // a decode-path packed row (page slot, rank)
  SITE_DECODE_META = 2,   // a decode-path block min/max row
  SITE_WINDOW = 3,        // a window ring or sink row
  SITE_PREFILL_PAGE = 4,  // a prefill packed row (page, or its staging run)
  SITE_PREFILL_OUT = 5,   // a prefill bulk store of a block's run
  SITE_PREFILL_META = 6,  // a prefill block min/max row
  SITE_ATTN_TILE = 7,     // an attention dense-tile element (token row, channel)
  SITE_ATTN_PART = 8,     // an attention split-T partial or output row
  SITE_SELECT_KEY = 9,    // a block-selection key or score
};

// Per (layer, seq, kv head) state kept on the device (64 bytes).
struct UnitDesc {
  int32_t T;                        // tokens held
  int32_t T0;                       // prefill length (fixes the segments)
  int32_t n_seg;
  int32_t rot_set;
  int32_t first_block[MK_MAX_SEGMENTS];
  int32_t r[MK_MAX_SEGMENTS];
  int32_t sflags[MK_MAX_SEGMENTS];  // per segment: bit 0 always attended; bit 1 stored under its own rotation
                                    // (a re-compressed closed segment); bits 4-5 log2 of the element-group size
                                    // (bitmap pages); bits 8-15 channels eligible for the top-r
};
static_assert(sizeof(UnitDesc) == 64, "UnitDesc is 64 bytes");

__host__ __device__ inline int32_t seg_flags(bool always, int keep, int g_log2 = 0) {
  return (always ? 1 : 0) | (g_log2 << 4) | (keep << 8);
}
// Element-group size of segment s (bitmap pages: 1, 2, 4 or 8).
__host__ __device__ inline int seg_group(const UnitDesc& u, int s) { return 1 << ((u.sflags[s] >> 4) & 3); }
__host__ __device__ inline bool seg_always(const UnitDesc& u, int s) { return (u.sflags[s] & 1) != 0; }
__host__ __device__ inline int seg_keep(const UnitDesc& u, int s) { return (u.sflags[s] >> 8) & 0xff; }
__host__ __device__ inline bool seg_own(const UnitDesc& u, int s) { return (u.sflags[s] & 2) != 0; }
// Rotation class of segment s: 0 for the head's rotation, s + 1 for a
// segment stored under its own.
__host__ __device__ inline int seg_class(const UnitDesc& u, int s) { return seg_own(u, s) ? s + 1 : 0; }
__host__ __device__ inline bool any_own(const UnitDesc& u) {
  bool a = false;
  for (int s = 0; s < u.n_seg; ++s) a = a || seg_own(u, s);
  return a;
}

// Everything a kernel needs to find data in the arena and workspace.
struct Layout {
  char* arena;
  int32_t* err;                 // [0] status, [1] detail, [2] unit, [3] aux
  UnitDesc* desc;               // [n_layers][max_seqs][n_kv]
  char* units;                  // first unit region
  int64_t unit_stride;
  int64_t off_rkt, off_rvt, off_rv, off_sink_k, off_sink_v, off_win_k, off_win_v;
  int64_t off_rkp, off_rvp;     // R_k, R_v as three bf16 parts each, tensor-core operand layout
  int64_t off_meta, off_pages;
  int64_t off_cmeta;            // compressed per-block keys (meta_c > 0): [nblk_cap][cmeta_row] bytes
  int64_t off_segrot;           // own rotations of closed segments s < n_seg - 1: [s] x {R_k^T, R_v} fp32 [128][128]
  int32_t n_cls;                // rotation classes: 1 + closed segments (1 with a single segment)
  int32_t meta_c, cmeta_row;    // channels a compressed key keeps (0 = none), bytes per row
  int64_t page_stride;
  int32_t S, W, B, n_kv, G, max_seqs, nblk_cap, cap_tokens, n_layers, k_max;
  int32_t topk_fixed, retain_permille, r_max;
  int32_t per_seg_k;                         // 1: each scored segment keeps its own k (per-segment retention)
  int32_t seg_retain[MK_MAX_SEGMENTS];       // per-segment retention (0: the cache's retain_permille)
  int32_t dense_pages;          // 1: uncompressed middle pages [K B x 128][V B x 128] (Quest comparator)
  int32_t bm_g;                 // 0: uint8 channel indices; else bitmap pages (128/g bits per vector, g per
                                // segment), and this is the smallest g (the largest bitmap, for sizes)
  int32_t attn_tg;              // attention: tokens per staged page group (32 or 16)
  int32_t attn_nst, attn_nc, attn_sb;  // attention: stages per warp, warps per CTA, stage bytes
  // workspace
  float* qrot;                  // [n_cls][n_layers][max_seqs][n_kv][G][128]: q' of each layer's last selection,
                                // per rotation class
  int32_t* seg_sel;             // [n_layers][max_seqs][n_kv][MK_MAX_SEGMENTS]: selected ids below each segment's
                                // first block (written by the top-k when a segment has its own rotation)
  uint32_t* keys;               // [max_seqs][n_kv][keys_stride]: ordered block-score keys, 0 = not a candidate
  int32_t keys_stride;          // nblk_cap rounded up to a multiple of 4
  uint32_t* khist;              // [max_seqs][n_kv][kKeyBins]: key counts by top 12 bits (zero between calls)
  float* part_acc;              // [max_seqs][n_kv][MK_MAX_SPLITS][G][128]
  float* part_ml;               // [max_seqs][n_kv][MK_MAX_SPLITS][G][2]
  int32_t* counters;            // [2][max_seqs][n_kv]: attention merge, selection top-k
};

// Per-call sequence list, passed by value.
struct CallSeqs {
  int32_t n;
  int32_t seq[MK_MAX_CALL_SEQS];
  int32_t n_new[MK_MAX_CALL_SEQS];
  int32_t row_off[MK_MAX_CALL_SEQS];   // first input row of the sequence
  int32_t T_old[MK_MAX_CALL_SEQS];     // host view, used by the bulk path only
  int32_t tile_off[MK_MAX_CALL_SEQS + 1];
};

__host__ __device__ inline int64_t unit_index(const Layout& L, int layer, int seq, int kvh) {
  return ((int64_t)layer * L.max_seqs + seq) * L.n_kv + kvh;
}
// q' of (layer, sequence slot), written by the selection, read by attention.
__host__ __device__ inline float* qrot_of(const Layout& L, int layer, int64_t slot, int cls = 0) {
  return L.qrot + (((int64_t)cls * L.n_layers + layer) * L.max_seqs * L.n_kv + slot) * L.G * 128;
}
// Packed page of a block with r kept channels: [K val B r bf16][K pos B pb]
// [V val B r bf16][V pos B pb], pb = pos_bytes (r uint8 indices, or a bitmap
// of 16/g bytes, g the block's element-group size).
__host__ __device__ inline int pos_bytes(const Layout& L, int r, int g) { return L.bm_g ? 16 / g : r; }
__host__ __device__ inline int64_t page_kpos(const Layout& L, int r) { return (int64_t)2 * L.B * r; }
__host__ __device__ inline int64_t page_vval(const Layout& L, int r, int g) {
  return (int64_t)2 * L.B * r + (int64_t)L.B * pos_bytes(L, r, g);
}
__host__ __device__ inline int64_t page_vpos(const Layout& L, int r, int g) {
  return (int64_t)4 * L.B * r + (int64_t)L.B * pos_bytes(L, r, g);
}
// Own rotation of closed segment s: R_k^T then R_v, fp32 [128][128] each.
__host__ __device__ inline int64_t segrot_off(const Layout& L, int s) {
  return L.off_segrot + (int64_t)s * 2 * 128 * 128 * 4;
}
__host__ __device__ inline int n_mid_tokens(const Layout& L, int T) {
  int m = T - L.W - L.S;
  return m > 0 ? m : 0;
}
__host__ __device__ inline int n_mid_blocks(const Layout& L, int T) {
  return (n_mid_tokens(L, T) + L.B - 1) / L.B;
}
__host__ __device__ inline int seg_of_block(const UnitDesc& u, int b) {
  int s = 0;
  for (int i = 1; i < u.n_seg; ++i)
    if (b >= u.first_block[i]) s = i;
  return s;
}
// Number of top-k candidates (blocks of scored segments) among the first nblk blocks.
__host__ __device__ inline int n_scored_blocks(const UnitDesc& u, int nblk) {
  int n = 0;
  for (int i = 0; i < u.n_seg; ++i) {
    int lo = u.first_block[i];
    int hi = (i + 1 < u.n_seg) ? u.first_block[i + 1] : nblk;
    if (hi > nblk) hi = nblk;
    if (lo > nblk) lo = nblk;
    if (!seg_always(u, i) && hi > lo) n += hi - lo;
  }
  return n;
}
// k of scored segment s with n of its blocks present (per-segment retention).
__host__ __device__ inline int n_select_segment(const Layout& L, int s, int n) {
  if (n <= 0) return 0;
  const int ret = L.seg_retain[s] ? L.seg_retain[s] : L.retain_permille;
  long long k = ((long long)ret * n + 999) / 1000;
  if (k < 1) k = 1;
  if (k > n) k = n;
  return (int)k;
}
__host__ __device__ inline int n_select(const Layout& L, int n_scored) {
  if (n_scored <= 0) return 0;
  if (L.topk_fixed > 0) return L.topk_fixed < n_scored ? L.topk_fixed : n_scored;
  long long k = ((long long)L.retain_permille * n_scored + 999) / 1000;
  if (k < 1) k = 1;
  if (k > n_scored) k = n_scored;
  return (int)k;
}
// Blocks a unit's selection keeps among its first nblk blocks: one top-k
// over every scored block, or (per-segment retention) each scored segment's
// own k.
__host__ __device__ inline int n_select_unit(const Layout& L, const UnitDesc& u, int nblk) {
  if (!L.per_seg_k) return n_select(L, n_scored_blocks(u, nblk));
  int k = 0;
  for (int i = 0; i < u.n_seg; ++i) {
    if (seg_always(u, i)) continue;
    int lo = u.first_block[i];
    int hi = (i + 1 < u.n_seg) ? u.first_block[i + 1] : nblk;
    if (hi > nblk) hi = nblk;
    if (lo > nblk) lo = nblk;
    if (hi > lo) k += n_select_segment(L, i, hi - lo);
  }
  return k;
}
// Bulk-append tiles: [T_old, f), [f, f+128), ... with f the first position
// S + 128j (or S) past T_old, so that every middle block sits in one tile.
__host__ __device__ inline int tile_first_boundary(int T_old, int S) {
  if (T_old < S) return S;
  return S + ((T_old - S) / kTileTokens + 1) * kTileTokens;
}
__host__ __device__ inline int n_tiles(int T_old, int T_new, int S) {
  if (T_new <= T_old) return 0;
  int f = tile_first_boundary(T_old, S);
  if (T_new <= f) return 1;
  return 1 + (T_new - f + kTileTokens - 1) / kTileTokens;
}

#ifdef __CUDACC__
__device__ __forceinline__ float bf2f(uint32_t b16) { return __uint_as_float(b16 << 16); }
// Round to nearest even; a zero result is stored as +0.
__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  uint16_t b = __bfloat16_as_ushort(h);
  return b == 0x8000 ? (uint16_t)0 : b;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ int warp_excl_scan(int v, int lane) {
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(FULL, x, o);
    if (lane >= o) x += y;
  }
  return x - v;
}
__device__ __forceinline__ void set_error(const Layout& L, int32_t detail, int32_t unit, int32_t aux,
                                          int32_t status = (int32_t)MK_EDEVICE) {
  if (atomicCAS(&L.err[0], 0, status) == 0) {
    L.err[1] = detail;
    L.err[2] = unit;
    L.err[3] = aux;
  }
}
// The checked build (compiled with MK_CHECKS=1 into a separate library for
// the tests) tests an index before its access: a failed check records the
// site and the index in the error word and the caller skips the access.  The
// default build compiles every check to true.
#ifndef MK_CHECKS
#define MK_CHECKS 0
#endif
__device__ __forceinline__ bool in_bounds(const Layout& L, bool ok, int32_t site, int64_t index) {
#if MK_CHECKS
  if (!ok) set_error(L, ERR_BOUNDS, site, (int32_t)index);
  return ok;
#else
  (void)L;
  (void)site;
  (void)index;
  return true;
#endif
}
__device__ __forceinline__ bool has_error(const Layout& L) {
  return *(volatile int32_t*)L.err != 0;
}
// 16-byte asynchronous global -> shared copies (cp.async, L2-only caching).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}
// Bulk (TMA) global -> shared copies completing on an mbarrier.  One request
// moves a whole contiguous run (16-byte aligned addresses, size a multiple of
// 16), so a single SM keeps far more bytes in flight than with 16-byte
// cp.async requests.
__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Makes initialised barriers visible to the asynchronous (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// Orders this thread's earlier shared-memory accesses before later bulk
// copies into the same bytes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
// Same for every state space: global data this CTA (or, through an acquired
// counter, another CTA) wrote becomes visible to later bulk copies.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;\n" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// Bulk shared -> global copy (16-byte aligned addresses, size a multiple of
// 16), tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Waits until this thread's bulk copies have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// Waits until this thread's bulk copies are complete (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// ---- 5th-generation tensor cores (tcgen05), single CTA --------------------
// Shared-memory matrix descriptor, K-major operand without swizzle: 8-row x
// 16-byte core matrices stored contiguously (128 bytes each); lbo = bytes
// between core matrices adjacent along K, sbo = bytes between 8-row groups.
__device__ __forceinline__ uint64_t umma_desc(const void* p, unsigned lbo, unsigned sbo) {
  uint64_t d = (uint64_t)((smem_u32(p) >> 4) & 0x3fffu);
  d |= (uint64_t)((lbo >> 4) & 0x3fffu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3fffu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of tcgen05; base offset 0, no swizzle
  return d;
}
// Instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier when every MMA issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// Whole warp: allocate ncols (power of two >= 32) TMEM columns, address to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, unsigned ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, unsigned ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
// Whole warp: 32 consecutive fp32 columns of this warp's 32 TMEM lanes
// (lane quarter = warp % 4), one lane per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
// Byte offset of element (row, k) of a 128-column bf16 matrix in the K-major
// core-matrix layout above (lbo = 128, sbo = 2048).
__host__ __device__ constexpr int umma_kmajor_offset(int row, int k) {
  return ((row >> 3) * 16 + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

// Bounded wait for the phase with the given parity to complete: false once
// 20 ms have passed (far above any real copy time).
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > 20000000ull) return false;
  return true;
}
// The same for a full warp whose lanes then branch together on the result:
// if any lane gave up, all report failure (a lane that saw the phase
// complete finds it complete again in the caller's drain).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, unsigned parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity)) != 0;
}
// Programmatic dependent launch: a kernel launched with the
// programmatic-serialization attribute may start while the previous kernel
// in the stream finishes.  It must call pdl_wait() before touching anything
// the previous kernel writes; it calls pdl_trigger() right after its own wait,
// so that whatever a kernel reads before its wait was complete two launches
// earlier.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ char* unit_base(const Layout& L, int64_t u) {
  return L.units + u * L.unit_stride;
}
#endif

#ifdef __CUDACC__
// Launch with programmatic stream serialization (and an optional cluster size).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
#endif

// Raises a kernel's dynamic shared memory limit to `bytes` on the current
// device (cudaFuncSetAttribute acts on one device only), once per (kernel,
// device) and size, under a lock, and reports the kernel's resident blocks per
// SM at that size with `threads` threads (occ) and the device's SM count (sms).
// Defined in mk_api.cu.
cudaError_t kernel_smem_attr(const void* fn, int bytes, int threads, int* occ, int* sms);

// Kernel launchers (defined in the .cu files); they return cudaGetLastError().
cudaError_t launch_init_desc(const Layout& L, int layer, int seq, const UnitDesc& d, cudaStream_t s);
cudaError_t launch_set_segment(const Layout& L, int64_t u, int seg, int r, int keep, int own, cudaStream_t s);
cudaError_t launch_append_small(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* k,
                                const uint16_t* v, int evict_only, cudaStream_t s);
cudaError_t launch_append_bulk(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* k,
                               const uint16_t* v, int total_tiles, cudaStream_t s);
// Whether the block selection can handle the context's largest block count.
bool select_plan_ok(const Layout& L);
bool topk_plan_ok(const Layout& L);
// The top-k kernel behind the scoring kernel (append: the scoring kernel
// appended cs.n_new tokens; the top-k kernel then advances the lengths).
cudaError_t launch_topk(const Layout& L, int layer, const CallSeqs& cs, int32_t* ids, int32_t* n_sel, bool append,
                        cudaStream_t s);
// kin/vin non-null: append one new token per sequence first (fused decode
// append, see k_select).  own: some unit of the call has a segment stored
// under its own rotation (the variant that scores by rotation class).
cudaError_t launch_block_select(const Layout& L, int layer, const CallSeqs& cs, const uint16_t* q,
                                int32_t* ids, int32_t* n_sel, float* scores_out, int max_nblk,
                                cudaStream_t s, const uint16_t* kin = nullptr, const uint16_t* vin = nullptr,
                                bool own = false);
// items[i]: the attention work of each (sequence i, kv head) of the call, in
// items of up to kDenseChunk tokens (dense chunks, page groups), host array.
// A sequence gets CTAs per kv head in proportion to its items.
// min_parts[i] (optional): the fewest CTAs per kv head sequence i needs (one
// per rotation class when some segment is stored under its own rotation).
cudaError_t launch_decode_attn(const Layout& L, int layer, const CallSeqs& cs, const int32_t* ids,
                               const int32_t* n_sel, uint16_t* out, const int32_t* items, cudaStream_t s,
                               const int32_t* min_parts = nullptr);
cudaError_t launch_dense_attn(const Layout& L, const CallSeqs& cs, const uint16_t* q,
                              const uint16_t* K, const uint16_t* V, int64_t t_stride,
                              uint16_t* out, const int32_t* items, cudaStream_t s);

// Attention CTAs of a call: sequence i (call order) owns CTAs off[i] ..
// off[i + 1] - 1, n_kv x P_i of them (kv head major, then part).
struct AttnSplit {
  int32_t off[MK_MAX_CALL_SEQS + 1];
};
size_t attn_plan(Layout& L, int64_t attend_max);
cudaError_t launch_gram(const uint16_t* x, int64_t n_rows, int64_t row_stride, float* gram,
                        cudaStream_t s);
size_t attn_smem_bytes(const Layout& L, int r_max);

}  // namespace mk
