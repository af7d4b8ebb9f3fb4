// Uncompressed decode attention for callers that cannot allocate device
// memory.  Same kernel and same results as mk_dense_decode_attn, but the
// scratch it needs (split-T partials, arrival counters, the error word) lives
// in one static device array of this library instead of a context's
// workspace, and no context is needed.
//
// Who needs it: code that runs where device allocation is not allowed or not
// possible - inside a host framework's plugin whose enqueue step forbids
// allocation, in a runtime with a fixed memory plan decided before serving
// starts, or in a process whose allocator belongs to someone else - and that
// only has its inputs and outputs at hand.
#include <algorithm>
#include <mutex>

#include "mk_internal.cuh"

namespace {

// The scratch: held by every GPU that loads this library, until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).  In host code the array's name is
// only a host-side stand-in, never a device address.
mk_status scratch_for_current_device(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MK_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MK_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  return MK_OK;
}

inline int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" mk_status mk_dense_decode_attn_noalloc(int32_t n_q_heads, int32_t n_kv_heads, int32_t n_seqs,
                                                  const int32_t* T, const void* q, const void* K, const void* V,
                                                  int64_t t_stride, void* out, mk_stream stream) {
  if (!T || !q || !K || !V || !out) return MK_EINVAL;
  // K and V rows arrive by bulk copies, which need 16-byte aligned sources.
  if (((uintptr_t)q | (uintptr_t)K | (uintptr_t)V | (uintptr_t)out) & 15) return MK_EINVAL;
  if (n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads) return MK_EINVAL;
  const int G = n_q_heads / n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return MK_EINVAL;
  if (n_seqs < 1 || n_seqs > MK_MAX_CALL_SEQS || t_stride < 1) return MK_EINVAL;
  int32_t items[MK_MAX_CALL_SEQS];
  for (int i = 0; i < n_seqs; ++i) {
    if (T[i] < 1 || T[i] > t_stride) return MK_EINVAL;
    items[i] = (T[i] + mk::kDenseChunk - 1) / mk::kDenseChunk;
  }
  // Size limit: n_seqs * n_q_heads <= MK_NOALLOC_MAX_QUERY_HEADS.
  if ((int64_t)n_seqs * n_q_heads > MK_NOALLOC_MAX_QUERY_HEADS) return MK_ENOMEM;
  // Scratch plan: error word, two counter banks, split-T partials.
  const int64_t slots = (int64_t)n_seqs * n_kv_heads;
  const int64_t off_cnt = 256;
  const int64_t off_acc = align256(off_cnt + slots * 2 * 4);
  const int64_t off_ml = align256(off_acc + slots * MK_MAX_SPLITS * G * mk::D * 4);
  const int64_t need = align256(off_ml + slots * MK_MAX_SPLITS * G * 2 * 4);
  if (need > (int64_t)MK_NOALLOC_SCRATCH_BYTES) return MK_ENOMEM;

  unsigned char* scratch = nullptr;
  mk_status st = scratch_for_current_device(&scratch);
  if (st != MK_OK) return st;

  mk::Layout L{};
  L.n_kv = n_kv_heads;
  L.G = G;
  L.max_seqs = n_seqs;
  L.S = 0;
  L.W = 1;
  L.B = 16;
  L.r_max = 1;
  L.err = reinterpret_cast<int32_t*>(scratch);
  L.counters = reinterpret_cast<int32_t*>(scratch + off_cnt);
  L.part_acc = reinterpret_cast<float*>(scratch + off_acc);
  L.part_ml = reinterpret_cast<float*>(scratch + off_ml);
  if (mk::attn_plan(L, 0) == 0) return MK_ENOTSUP;

  mk::CallSeqs cs{};  // on the stack: nothing is allocated, host or device
  cs.n = n_seqs;
  for (int i = 0; i < n_seqs; ++i) {
    cs.seq[i] = i;
    cs.T_old[i] = T[i];
  }
  // What must start at zero: the arrival counters (a previous call that
  // failed part-way may have left them set).  The error word before them is
  // kept: a device-side failure stays recorded until mk_noalloc_poll_error
  // reads and clears it, and meanwhile every call leaves its output alone.
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch + off_cnt, 0, (size_t)(off_acc - off_cnt), s);
  if (e == cudaSuccess)
    e = mk::launch_dense_attn(L, cs, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(K),
                              static_cast<const uint16_t*>(V), t_stride, static_cast<uint16_t*>(out), items, s);
  return e == cudaSuccess ? MK_OK : MK_ECUDA;
}

extern "C" mk_status mk_noalloc_poll_error(int32_t* detail) {
  unsigned char* scratch = nullptr;
  mk_status st = scratch_for_current_device(&scratch);
  if (st != MK_OK) return st;
  int32_t w[4] = {0, 0, 0, 0};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(w, scratch, sizeof(w), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && w[0] != 0) e = cudaMemset(scratch, 0, sizeof(w));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return MK_ECUDA;
  if (detail) *detail = w[1];
  return w[0] == 0 ? MK_OK : (mk_status)w[0];
}
