// ll_attend_chunk_noalloc: the chunk attention of ll_attend_chunk for callers
// that may not allocate device memory.
//
// Who they are: a host program whose memory manager owns the GPU's whole
// budget (a serving runtime that reserves nearly all of HBM in its own pool
// at start-up and hands out slices), a plugin interface that gives a kernel
// library a stream and buffers but forbids it to allocate, or a real-time
// loop whose per-frame deadline cannot absorb cudaMalloc / cudaFree (they can
// block the host and synchronise the device).  Such a caller cannot create an
// ll_cache either, since that allocates the cache: it keeps the K/V rows in
// memory it owns, in the head-major layout of the cache, and places frames
// with the host helpers ll_frame_slot / ll_resident_frames.
//
// The tensor-core attention splits the work items left over after its whole
// rounds across SMs and merges their partial results (combine pass).  Those
// partial results need scratch memory; ll_attend_chunk takes it from the
// cache, this entry point from the file-scope array below, which every GPU
// that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "ll.h"
#include "ll_internal.h"

namespace {

// 256-byte header (the fallback device error word), then the partial results.
constexpr size_t kHeaderBytes = 256;
constexpr size_t kPartialBytes = (size_t)LL_NOALLOC_PARTIAL_SLOTS * 256 * (128 + 2) * sizeof(float);
static_assert(LL_NOALLOC_SCRATCH_BYTES == kHeaderBytes + kPartialBytes, "scratch size in ll.h");

static __device__ __align__(256) unsigned char g_noalloc_scratch[LL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr long long kTimeoutNs = 2000000000LL;  // same bound as the cache path's waits

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {nullptr};  // device address of the array, per device

// Device address of the array on the current device (looked up once per device).
ll_status scratch_address(int dev, unsigned char** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_dev[dev]);
  return LL_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// true when the byte ranges [a, a + na) and [b, b + nb) share a byte
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" ll_status ll_attend_chunk_noalloc(const void* q, const void* k_cached, const void* v_cached,
                                             int cached_tokens, int64_t cached_head_stride, const void* k,
                                             const void* v, int chunk_tokens, void* out, int heads,
                                             int head_dim, unsigned* err_word, void* stream) {
  if (!q || !k || !v || !out) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LL_ERR_INVALID_ARG;
  if (heads < 1 || chunk_tokens < 1 || cached_tokens < 0) return LL_ERR_INVALID_ARG;
  // out shares no byte with any input (bf16 rows of heads * head_dim elements)
  if (head_dim > 0) {
    const size_t chunk_bytes = (size_t)chunk_tokens * heads * head_dim * 2;
    if (overlap(out, chunk_bytes, q, chunk_bytes) || overlap(out, chunk_bytes, k, chunk_bytes) ||
        overlap(out, chunk_bytes, v, chunk_bytes))
      return LL_ERR_INVALID_ARG;
    if (cached_tokens > 0 && cached_head_stride > 0) {
      const size_t cached_bytes = ((size_t)(heads - 1) * cached_head_stride + (size_t)cached_tokens * head_dim) * 2;
      if ((k_cached && overlap(out, chunk_bytes, k_cached, cached_bytes)) ||
          (v_cached && overlap(out, chunk_bytes, v_cached, cached_bytes)))
        return LL_ERR_INVALID_ARG;
    }
  }
  if (head_dim != 64 && head_dim != 128) return LL_ERR_UNSUPPORTED;
  if ((int64_t)cached_tokens + chunk_tokens > (1LL << 30)) return LL_ERR_UNSUPPORTED;
  if (cached_tokens > 0) {
    if (!k_cached || !v_cached || !aligned16(k_cached) || !aligned16(v_cached)) return LL_ERR_INVALID_ARG;
    // rows of one head are contiguous; head starts are 16-byte aligned (tensor-map strides)
    if (cached_head_stride < (int64_t)cached_tokens * head_dim || (cached_head_stride * 2) % 16 != 0)
      return LL_ERR_INVALID_ARG;
  }
  if (err_word && (reinterpret_cast<uintptr_t>(err_word) & 3u)) return LL_ERR_INVALID_ARG;

  // The launch uses two partial-result slots per CTA and as many CTAs as
  // ll_attend_chunk would (one per SM, at most one per work item).  Reject the
  // request if the array cannot hold them at this head_dim.
  const int64_t items = (int64_t)((chunk_tokens + 255) / 256) * heads;
  int64_t need = ll::attend_scratch_slots_wanted();
  if (2 * items < need) need = 2 * items;
  const int64_t have = (int64_t)(kPartialBytes / ll::attend_scratch_bytes(head_dim, 1));
  if (need > have) return LL_ERR_UNSUPPORTED;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LL_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LL_ERR_UNSUPPORTED;
  unsigned char* base = nullptr;
  if (ll_status s = scratch_address(dev, &base)) return s;

  ll::AttendArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.out = out;
  if (cached_tokens > 0) {
    a.kc = k_cached;
    a.vc = v_cached;
    a.cache_head_elems = cached_head_stride;
  } else {
    // no cached rows: the cache tensor map still needs a valid base; it is never read
    a.kc = k;
    a.vc = v;
    a.cache_head_elems = head_dim;
  }
  a.La = cached_tokens;
  a.kn = k;
  a.vn = v;
  a.Lb = chunk_tokens;
  a.Lq = chunk_tokens;
  a.heads = heads;
  a.head_dim = head_dim;
  a.mode = 0;
  a.block_tokens = chunk_tokens;
  a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)head_dim));
  a.out_f32 = 0;
  a.err = err_word ? err_word : reinterpret_cast<unsigned*>(base);
  a.stall_inject = 0;
  a.timeout_ns = kTimeoutNs;
  a.scratch = reinterpret_cast<float*>(base + kHeaderBytes);
  a.scratch_slots = (int)have;
  return ll::launch_attend_bf16_tc(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}
