// Host side of libll: the cache object, argument and state checks, the
// frame-to-slot bookkeeping, and the C ABI declared in include/ll.h.
//
// Cache rule ("LongLive: Real-time Interactive Long Video Generation", §3.3
// Efficient Long Inference, "Frame sink" and "Short window attention"): the
// first S frames of a layer are a sink that is never evicted; the next frames
// roll through a window of W slots, frame f >= S living in slot
// S + ((f - S) mod W).  After n commits the resident frames are
// 0..min(S,n)-1 and max(S, n-W)..n-1, and their slots always form the prefix
// [0, R) of the slot range, so the attention kernels read the resident keys as
// one contiguous run of R*T rows per head.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "ll.h"
#include "ll_internal.h"

namespace ll {

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace ll

struct ll_cache {
  int L, H, D, T, S, W, C;
  ll_dtype dtype;
  int eb;                 // element bytes of the token tensors
  int keb;                // element bytes of the K cache (1: e4m3 keys, LL_BF16_K8 and LL_FP8)
  int veb;                // element bytes of the V cache (1: e4m3 values, LL_FP8)
  int device;
  size_t layer_elems;     // elements of one layer's K (= V)
  void* k = nullptr;      // [L][H][S+W][T][D]
  void* v = nullptr;
  uint8_t* q8 = nullptr;  // e4m3 caches: q and the chunk's (or recache window's) keys rounded to e4m3
  uint8_t* k8 = nullptr;
  uint8_t* v8 = nullptr;  // LL_FP8: the values rounded to e4m3
  std::vector<int64_t> n;               // frames committed per layer
  std::vector<int64_t> fos;             // frame_of_slot, L x (S+W)
  unsigned* err_host = nullptr;         // mapped host word written by kernels
  unsigned* err_dev = nullptr;
  float* scratch = nullptr;             // partial results of split attention work items
  int scratch_slots = 0;
  int stall_inject = 0;
  int stall_timeout_us = 0;
  int use_simt = 0;
  int pair = 0;           // head_dim 128 on the CTA-pair tensor-core kernel (test hook)
  int out_f32 = 0;        // outputs in fp32 on a bf16 cache
  int chunk_mask = LL_MASK_CHUNK;
  int recache_scope = LL_RECACHE_RESIDENT;
  bool poison = false;    // empty slots hold all-ones bytes (NaN in every dtype): a stray read shows
  // per-kernel timing (ll_profile_enable / ll_profile_read)
  struct Mark {
    int kind;
    cudaEvent_t start, stop;
  };
  bool profiling = false;
  int profile_every = 1;                    // bracket one launch in every `profile_every` of a kind
  uint64_t profile_seen[LL_KERNEL_KINDS] = {0, 0, 0};
  std::vector<Mark> marks;
  std::vector<cudaEvent_t> event_pool;
};

namespace {

constexpr long long kDefaultTimeoutNs = 2000000000LL;  // 2 s: no legal wait comes near it

// An NVTX range around each entry point that works with the device (a no-op unless a
// profiler or another NVTX tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

// ---------------------------------------------------------------------------
// Fault injection on the host (ll_debug_inject_fault, or LL_FAULT=alloc:N,launch:N in
// the environment when the library loads): the N-th next device allocation, or kernel
// launch step, of the library reports failure as if the CUDA call had failed.  No
// device fault is involved: the failing call is never made.
// ---------------------------------------------------------------------------
std::atomic<long long> g_fault_alloc{0}, g_fault_launch{0};  // countdown; 0 = off

bool fault_hit(std::atomic<long long>& c) {
  long long v = c.load();
  while (v > 0) {
    if (c.compare_exchange_weak(v, v - 1)) return v == 1;
  }
  return false;
}

struct FaultFromEnv {
  FaultFromEnv() {
    const char* e = std::getenv("LL_FAULT");
    if (!e) return;
    // comma-separated "alloc:N" / "launch:N"
    for (const char* p = e; *p;) {
      long long n = 0;
      if (std::strncmp(p, "alloc:", 6) == 0 && (n = std::atoll(p + 6)) > 0) g_fault_alloc = n;
      if (std::strncmp(p, "launch:", 7) == 0 && (n = std::atoll(p + 7)) > 0) g_fault_launch = n;
      const char* q = std::strchr(p, ',');
      if (!q) break;
      p = q + 1;
    }
  }
} g_fault_from_env;

cudaError_t dev_alloc(void** p, size_t n) {
  if (fault_hit(g_fault_alloc)) return cudaErrorMemoryAllocation;
  return cudaMalloc(p, n);
}
cudaError_t host_alloc_mapped(void** p, size_t n) {
  if (fault_hit(g_fault_alloc)) return cudaErrorMemoryAllocation;
  return cudaHostAlloc(p, n, cudaHostAllocMapped);
}
bool launch_fault() { return fault_hit(g_fault_launch); }

bool env_poison() {
  const char* e = std::getenv("LL_POISON");
  return e && *e && std::strcmp(e, "0") != 0;
}

int64_t resident_count(int S, int W, int64_t n) {
  const int64_t sink = n < S ? n : S;
  int64_t win = n - S;
  if (win < 0) win = 0;
  if (win > W) win = W;
  return sink + win;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// true when the byte ranges [a, a + na) and [b, b + nb) share a byte
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// An output of `rows` token rows may share no byte with the inputs of `rows` rows
// (an input pointer may be NULL).
bool output_overlaps_inputs(const ll_cache* c, int64_t rows, const void* out, const void* a, const void* b,
                            const void* d) {
  const size_t row_elems = (size_t)c->H * c->D;
  const size_t in_bytes = (size_t)rows * row_elems * c->eb;
  const size_t out_bytes = (size_t)rows * row_elems * ((c->dtype == LL_FP32 || c->out_f32) ? 4 : c->eb);
  for (const void* p : {a, b, d})
    if (p && overlap(out, out_bytes, p, in_bytes)) return true;
  return false;
}

ll_status take_device_error(ll_cache* c) {
  volatile unsigned* e = c->err_host;
  const unsigned v = *e;
  if (v != 0) {
    *e = 0;
    return LL_ERR_DEVICE_TIMEOUT;
  }
  return LL_OK;
}

ll_status set_device(const ll_cache* c) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return LL_ERR_CUDA;
  if (cur != c->device && cudaSetDevice(c->device) != cudaSuccess) return LL_ERR_CUDA;
  return LL_OK;
}

ll::AttendArgs base_args(ll_cache* c, int layer) {
  ll::AttendArgs a;
  std::memset(&a, 0, sizeof(a));
  const size_t off = c->layer_elems * (size_t)layer;
  a.kc = static_cast<const char*>(c->k) + off * c->keb;
  a.vc = static_cast<const char*>(c->v) + off * c->veb;
  a.cache_head_elems = (int64_t)(c->S + c->W) * c->T * c->D;
  a.qk_fp8 = (c->dtype == LL_BF16_K8 || c->dtype == LL_FP8) ? 1 : 0;
  a.v_fp8 = c->dtype == LL_FP8 ? 1 : 0;
  a.heads = c->H;
  a.head_dim = c->D;
  a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)c->D));
  a.err = c->err_dev;
  a.out_f32 = (c->dtype == LL_FP32 || c->out_f32) ? 1 : 0;
  a.scratch = c->scratch;
  a.scratch_slots = c->scratch_slots;
  a.pair = c->pair;
  a.stall_inject = c->stall_inject;
  a.timeout_ns = c->stall_inject ? (long long)c->stall_timeout_us * 1000LL : kDefaultTimeoutNs;
  c->stall_inject = 0;  // one launch only
  return a;
}

cudaEvent_t pooled_event(ll_cache* c) {
  if (!c->event_pool.empty()) {
    cudaEvent_t e = c->event_pool.back();
    c->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one launch with events when profiling is on.
struct ProfileScope {
  ll_cache* c;
  cudaStream_t st;
  int kind;
  cudaEvent_t start = nullptr;
  ProfileScope(ll_cache* c_, cudaStream_t st_, int kind_) : c(c_), st(st_), kind(kind_) {
    if (!c->profiling) return;
    if (c->profile_seen[kind]++ % (uint64_t)c->profile_every != 0) return;  // not sampled
    if ((start = pooled_event(c)) != nullptr) cudaEventRecord(start, st);
  }
  void done() {
    if (!start) return;
    cudaEvent_t stop = pooled_event(c);
    if (!stop) return;
    cudaEventRecord(stop, st);
    c->marks.push_back({kind, start, stop});
  }
};

// kind: LL_KERNEL_ATTEND (chunk attention) or LL_KERNEL_PREFILL (recache prefill)
ll_status launch_attend(ll_cache* c, const ll::AttendArgs& a, cudaStream_t st, int kind) {
  if (launch_fault()) return LL_ERR_CUDA;
  ProfileScope prof(c, st, kind);
  cudaError_t e;
  if (c->dtype == LL_BF16_K8 || c->dtype == LL_FP8) {
    // keys (and with LL_FP8 values) in e4m3: the attention reads q and its fresh
    // keys (and values) rounded the same way, from the cache's staging buffers
    // (which a commit copy then reads); every caller here has as many fresh keys
    // as queries
    ll::AttendArgs a8 = a;
    const bool v8 = c->dtype == LL_FP8;
    const void* src[3] = {a.q, a.kn, v8 ? a.vn : nullptr};
    void* const dst[3] = {c->q8, c->k8, v8 ? c->v8 : nullptr};
    e = ll::launch_quantize_e4m3(src, dst, (int64_t)a.Lq * c->H * c->D, st);
    a8.q = c->q8;
    a8.kn = c->k8;
    if (v8) a8.vn = c->v8;
    if (e == cudaSuccess) e = ll::launch_attend_bf16_tc(a8, st);
  } else if (c->use_simt || (c->dtype == LL_FP32 && c->D != 64)) {
    // the CUDA-core kernel: fp32 at head_dim 128 (two fp32 query tiles and a K/V
    // ring do not fit one CTA's shared memory), or on request (tests)
    e = ll::launch_attend_simt(a, c->eb, st);
  } else if (c->dtype == LL_FP32) {
    e = ll::launch_attend_tf32_tc(a, st);
  } else {
    e = ll::launch_attend_bf16_tc(a, st);
  }
  prof.done();
  return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

ll_status launch_copy(ll_cache* c, int layer, const void* k, const void* v, const std::vector<int>& slot_of,
                      cudaStream_t st) {
  ll::CopyFramesArgs a;
  std::memset(&a, 0, sizeof(a));
  const size_t off = c->layer_elems * (size_t)layer;
  a.src_k = k;
  a.src_v = v;
  a.dst_k = static_cast<char*>(c->k) + off * c->keb;
  a.dst_v = static_cast<char*>(c->v) + off * c->veb;
  a.k_elem_bytes = c->keb;
  a.frames = (int)slot_of.size();
  a.tokens_per_frame = c->T;
  a.heads = c->H;
  a.head_dim = c->D;
  a.slots = c->S + c->W;
  a.elem_bytes = c->veb;
  for (size_t i = 0; i < slot_of.size(); ++i) a.slot_of[i] = slot_of[i];
  if (launch_fault()) return LL_ERR_CUDA;
  ProfileScope prof(c, st, LL_KERNEL_COPY);
  const cudaError_t e = ll::launch_copy_frames(a, st);
  prof.done();
  return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

ll_status check_layer(const ll_cache* c, int layer) {
  if (!c) return LL_ERR_INVALID_ARG;
  if (layer < 0 || layer >= c->L) return LL_ERR_INVALID_ARG;
  return LL_OK;
}

// All slots of every layer back to all-ones bytes (NaN in bf16, fp32 and e4m3), after
// the device has finished with them.
ll_status poison_slots(ll_cache* c) {
  if (ll_status s = set_device(c)) return s;
  const size_t kbytes = c->layer_elems * c->L * c->keb, vbytes = c->layer_elems * c->L * c->veb;
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemset(c->k, 0xFF, kbytes) != cudaSuccess ||
      cudaMemset(c->v, 0xFF, vbytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return LL_ERR_CUDA;
  return LL_OK;
}

// Poison every slot (of every layer and head) that holds no resident frame.
ll_status poison_resident_gaps(ll_cache* c) {
  if (ll_status s = set_device(c)) return s;
  if (cudaDeviceSynchronize() != cudaSuccess) return LL_ERR_CUDA;
  const int slots = c->S + c->W;
  const size_t rows = (size_t)c->T * c->D;  // elements of one (head, slot)
  for (int layer = 0; layer < c->L; ++layer)
    for (int slot = 0; slot < slots; ++slot) {
      if (c->fos[(size_t)layer * slots + slot] >= 0) continue;
      for (int h = 0; h < c->H; ++h) {
        const size_t e = c->layer_elems * layer + ((size_t)h * slots + slot) * rows;
        if (cudaMemset(static_cast<char*>(c->k) + e * c->keb, 0xFF, rows * c->keb) != cudaSuccess ||
            cudaMemset(static_cast<char*>(c->v) + e * c->veb, 0xFF, rows * c->veb) != cudaSuccess)
          return LL_ERR_CUDA;
      }
    }
  return cudaDeviceSynchronize() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* ll_status_str(ll_status s) {
  switch (s) {
    case LL_OK: return "LL_OK";
    case LL_ERR_INVALID_ARG: return "LL_ERR_INVALID_ARG";
    case LL_ERR_UNSUPPORTED: return "LL_ERR_UNSUPPORTED";
    case LL_ERR_OOM: return "LL_ERR_OOM";
    case LL_ERR_STATE: return "LL_ERR_STATE";
    case LL_ERR_CUDA: return "LL_ERR_CUDA";
    case LL_ERR_DEVICE_TIMEOUT: return "LL_ERR_DEVICE_TIMEOUT";
  }
  return "LL_ERR_UNKNOWN";
}

int ll_frame_slot(int S, int W, int64_t f) {
  if (f < 0) return -1;
  if (f < S) return (int)f;
  if (W <= 0) return -1;
  return S + (int)((f - S) % W);
}

int ll_resident_frames(int S, int W, int64_t n, int64_t* frames) {
  int cnt = 0;
  const int64_t sink = n < S ? n : S;
  for (int64_t f = 0; f < sink; ++f) frames[cnt++] = f;
  int64_t lo = n - W;
  if (lo < S) lo = S;
  for (int64_t f = lo; f < n; ++f) frames[cnt++] = f;
  return cnt;
}

uint64_t ll_launch_count(void) { return ll::g_launches.load(std::memory_order_relaxed); }

ll_status ll_cache_create(ll_cache** out, int layers, int heads, int head_dim, int tokens_per_frame,
                          int sink_frames, int window_frames, int chunk_frames, ll_dtype dtype) {
  NvtxRange range("ll_cache_create");
  if (!out) return LL_ERR_INVALID_ARG;
  *out = nullptr;
  if (layers < 1 || heads < 1 || tokens_per_frame < 1 || chunk_frames < 1 || sink_frames < 0 ||
      window_frames < 0)
    return LL_ERR_INVALID_ARG;
  if (dtype != LL_BF16 && dtype != LL_FP32 && dtype != LL_BF16_K8 && dtype != LL_FP8) return LL_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return LL_ERR_UNSUPPORTED;
  if ((dtype == LL_BF16_K8 || dtype == LL_FP8) && head_dim != 128) return LL_ERR_UNSUPPORTED;
  const int slots = sink_frames + window_frames;
  if (slots > ll::kMaxFrameTable || chunk_frames > ll::kMaxFrameTable) return LL_ERR_UNSUPPORTED;
  // kernel grids: (frames x heads) copy blocks; 32-bit token counts per call
  if ((int64_t)ll::kMaxFrameTable * heads > 65535) return LL_ERR_UNSUPPORTED;
  if ((int64_t)(slots + chunk_frames) * tokens_per_frame > (1LL << 30)) return LL_ERR_UNSUPPORTED;

  ll_cache* c = new ll_cache();
  c->L = layers;
  c->H = heads;
  c->D = head_dim;
  c->T = tokens_per_frame;
  c->S = sink_frames;
  c->W = window_frames;
  c->C = chunk_frames;
  c->dtype = dtype;
  c->eb = dtype == LL_FP32 ? 4 : 2;
  c->keb = (dtype == LL_BF16_K8 || dtype == LL_FP8) ? 1 : c->eb;
  c->veb = dtype == LL_FP8 ? 1 : c->eb;
  c->layer_elems = (size_t)heads * slots * tokens_per_frame * head_dim;
  c->n.assign(layers, 0);
  c->fos.assign((size_t)layers * slots, -1);
  if (cudaGetDevice(&c->device) != cudaSuccess) {
    delete c;
    return LL_ERR_CUDA;
  }
  // at least one 256-byte block, so a cache without slots (S = W = 0) still
  // hands the kernels a valid base address
  size_t kbytes = c->layer_elems * layers * c->keb, vbytes = c->layer_elems * layers * c->veb;
  if (kbytes < 256) kbytes = 256;
  if (vbytes < 256) vbytes = 256;
  auto fail = [&](ll_status st) {
    cudaGetLastError();
    cudaFree(c->k);
    cudaFree(c->v);
    cudaFree(c->scratch);
    cudaFree(c->q8);
    delete c;
    return st;
  };
  if (dev_alloc(&c->k, kbytes) != cudaSuccess || dev_alloc(&c->v, vbytes) != cudaSuccess) return fail(LL_ERR_OOM);
  c->poison = env_poison();
  const int fill = c->poison ? 0xFF : 0;
  if (cudaMemset(c->k, fill, kbytes) != cudaSuccess || cudaMemset(c->v, fill, vbytes) != cudaSuccess)
    return fail(LL_ERR_CUDA);
  if (dtype != LL_FP32 || head_dim == 64) {
    // the tensor-core kernel splits left-over work items across SMs and merges
    // their partial results: two slots per SM
    c->scratch_slots = ll::attend_scratch_slots_wanted();
    if (dev_alloc(reinterpret_cast<void**>(&c->scratch), ll::attend_scratch_bytes(head_dim, c->scratch_slots)) !=
        cudaSuccess)
      return fail(LL_ERR_OOM);
  }
  if (dtype == LL_BF16_K8 || dtype == LL_FP8) {
    // staging for q and the fresh keys (and values) rounded to e4m3: a chunk, or a
    // recache window
    const int frames = chunk_frames > slots ? chunk_frames : slots;
    const size_t n = (size_t)frames * tokens_per_frame * heads * head_dim;
    if (dev_alloc(reinterpret_cast<void**>(&c->q8), (dtype == LL_FP8 ? 3 : 2) * n) != cudaSuccess)
      return fail(LL_ERR_OOM);
    c->k8 = c->q8 + n;
    if (dtype == LL_FP8) c->v8 = c->q8 + 2 * n;
  }
  if (host_alloc_mapped(reinterpret_cast<void**>(&c->err_host), 256) != cudaSuccess ||
      cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->err_dev), c->err_host, 0) != cudaSuccess) {
    if (c->err_host) cudaFreeHost(c->err_host);
    return fail(LL_ERR_CUDA);
  }
  *c->err_host = 0;
  *out = c;
  return LL_OK;
}

void ll_cache_destroy(ll_cache* c) {
  NvtxRange range("ll_cache_destroy");
  if (!c) return;
  set_device(c);
  cudaDeviceSynchronize();
  for (auto& m : c->marks) {
    cudaEventDestroy(m.start);
    cudaEventDestroy(m.stop);
  }
  for (auto e : c->event_pool) cudaEventDestroy(e);
  cudaFree(c->k);
  cudaFree(c->v);
  cudaFree(c->scratch);
  cudaFree(c->q8);
  cudaFreeHost(c->err_host);
  delete c;
}

ll_status ll_attend_chunk(ll_cache* c, int layer, const void* q, const void* k, const void* v, void* out,
                          int commit, void* stream) {
  NvtxRange range("ll_attend_chunk");
  if (ll_status s = check_layer(c, layer)) return s;
  if (!q || !k || !v || !out) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LL_ERR_INVALID_ARG;
  if (output_overlaps_inputs(c, (int64_t)c->C * c->T, out, q, k, v)) return LL_ERR_INVALID_ARG;
  if (ll_status s = take_device_error(c)) return s;
  if (ll_status s = set_device(c)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t t0 = c->n[layer];
  const int64_t R = resident_count(c->S, c->W, t0);
  ll::AttendArgs a = base_args(c, layer);
  a.q = q;
  a.out = out;
  a.La = (int)(R * c->T);
  a.kn = k;
  a.vn = v;
  a.Lb = c->C * c->T;
  a.Lq = c->C * c->T;
  a.mode = 0;
  a.block_tokens = c->C * c->T;
  if (c->chunk_mask == LL_MASK_FRAME && c->C > 1) {
    // frame-causal chunk: cached keys all visible, the chunk's own keys up to the query's frame
    a.mode = 2;
    a.block_tokens = c->T;
  }
  if (ll_status s = launch_attend(c, a, st, LL_KERNEL_ATTEND)) return s;
  if (!commit) return LL_OK;

  // Commit: frames t0 .. t0+C-1.  A frame that the same commit would already
  // evict (W < C) is not written, so the copy has no write-write conflicts.
  const int64_t n1 = t0 + c->C;
  int64_t win_lo = n1 - c->W;
  if (win_lo < c->S) win_lo = c->S;
  std::vector<int> slot_of(c->C, -1);
  for (int i = 0; i < c->C; ++i) {
    const int64_t f = t0 + i;
    if (f < c->S || f >= win_lo) slot_of[i] = ll_frame_slot(c->S, c->W, f);
  }
  // an e4m3 cache takes the keys (and values) the attention just rounded
  const bool k8 = c->dtype == LL_BF16_K8 || c->dtype == LL_FP8;
  if (ll_status s = launch_copy(c, layer, k8 ? c->k8 : k, c->dtype == LL_FP8 ? c->v8 : v, slot_of, st)) return s;
  int64_t* fos = &c->fos[(size_t)layer * (c->S + c->W)];
  for (int i = 0; i < c->C; ++i)
    if (slot_of[i] >= 0) fos[slot_of[i]] = t0 + i;
  c->n[layer] = n1;
  return LL_OK;
}

static ll_status recache_common(ll_cache* c, int layer, const void* q_win, const void* k_win,
                                const void* v_win, void* out_win, void* stream) {
  if (ll_status s = check_layer(c, layer)) return s;
  if (!k_win || !v_win) return LL_ERR_INVALID_ARG;
  if (!aligned16(k_win) || !aligned16(v_win)) return LL_ERR_INVALID_ARG;
  if (q_win && (!out_win || !aligned16(q_win) || !aligned16(out_win))) return LL_ERR_INVALID_ARG;
  const int64_t n = c->n[layer];
  std::vector<int64_t> frames(c->S + c->W + 1);
  int R = ll_resident_frames(c->S, c->W, n, frames.data());
  const int sink = (int)(n < c->S ? n : c->S);  // resident sink frames: the first `sink` of the list
  if (c->recache_scope == LL_RECACHE_WINDOW) {
    // keep-sink scope: only the window frames are rewritten
    frames.erase(frames.begin(), frames.begin() + sink);
    R -= sink;
  }
  if (R == 0) return LL_ERR_STATE;
  if (q_win && output_overlaps_inputs(c, (int64_t)R * c->T, out_win, q_win, k_win, v_win)) return LL_ERR_INVALID_ARG;
  if (ll_status s = take_device_error(c)) return s;
  if (ll_status s = set_device(c)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q_win) {
    ll::AttendArgs a = base_args(c, layer);
    a.q = q_win;
    a.out = out_win;
    a.kn = k_win;
    a.vn = v_win;
    a.Lb = R * c->T;
    a.Lq = R * c->T;
    a.block_tokens = (c->chunk_mask == LL_MASK_FRAME ? 1 : c->C) * c->T;
    // keep-sink scope: the window queries also see the cached sink rows (slots [0, sink))
    a.La = c->recache_scope == LL_RECACHE_WINDOW ? sink * c->T : 0;
    a.mode = 1;
    if (ll_status s = launch_attend(c, a, st, LL_KERNEL_PREFILL)) return s;
  }
  std::vector<int> slot_of(R);
  for (int i = 0; i < R; ++i) slot_of[i] = ll_frame_slot(c->S, c->W, frames[i]);
  if (c->dtype == LL_BF16_K8 || c->dtype == LL_FP8) {
    // the keys (and with LL_FP8 the values) go in rounded to e4m3 (the prefill
    // above already rounded them)
    const bool v8 = c->dtype == LL_FP8;
    const void* src[3] = {nullptr, k_win, v8 ? v_win : nullptr};
    void* const dst[3] = {nullptr, c->k8, v8 ? c->v8 : nullptr};
    if (!q_win && ll::launch_quantize_e4m3(src, dst, (int64_t)R * c->T * c->H * c->D, st) != cudaSuccess)
      return LL_ERR_CUDA;
    return launch_copy(c, layer, c->k8, v8 ? c->v8 : v_win, slot_of, st);
  }
  return launch_copy(c, layer, k_win, v_win, slot_of, st);
}

ll_status ll_recache_tokens(const ll_cache* c, int layer, int64_t* tokens) {
  if (ll_status s = check_layer(c, layer)) return s;
  if (!tokens) return LL_ERR_INVALID_ARG;
  const int64_t n = c->n[layer];
  int64_t R = resident_count(c->S, c->W, n);
  if (c->recache_scope == LL_RECACHE_WINDOW) R -= n < c->S ? n : c->S;  // the sink keeps its K/V
  *tokens = R * c->T;
  return LL_OK;
}

ll_status ll_recache(ll_cache* c, int layer, const void* k_win, const void* v_win, void* stream) {
  NvtxRange range("ll_recache");
  return recache_common(c, layer, nullptr, k_win, v_win, nullptr, stream);
}

ll_status ll_recache_attend(ll_cache* c, int layer, const void* q_win, const void* k_win, const void* v_win,
                            void* out_win, void* stream) {
  NvtxRange range("ll_recache_attend");
  if (!q_win || !out_win) return LL_ERR_INVALID_ARG;
  return recache_common(c, layer, q_win, k_win, v_win, out_win, stream);
}

ll_status ll_set_output_dtype(ll_cache* c, ll_dtype dtype) {
  if (!c) return LL_ERR_INVALID_ARG;
  if (dtype == LL_FP32) {
    c->out_f32 = 1;
  } else if (dtype == LL_BF16 && (c->dtype == LL_BF16 || c->dtype == LL_BF16_K8 || c->dtype == LL_FP8)) {
    c->out_f32 = 0;
  } else {
    return LL_ERR_INVALID_ARG;
  }
  return LL_OK;
}

ll_status ll_set_chunk_mask(ll_cache* c, int mode) {
  if (!c || (mode != LL_MASK_CHUNK && mode != LL_MASK_FRAME)) return LL_ERR_INVALID_ARG;
  c->chunk_mask = mode;
  return LL_OK;
}

ll_status ll_set_recache_scope(ll_cache* c, int scope) {
  if (!c || (scope != LL_RECACHE_RESIDENT && scope != LL_RECACHE_WINDOW)) return LL_ERR_INVALID_ARG;
  c->recache_scope = scope;
  return LL_OK;
}

ll_status ll_reset(ll_cache* c) {
  if (!c) return LL_ERR_INVALID_ARG;
  std::fill(c->n.begin(), c->n.end(), 0);
  std::fill(c->fos.begin(), c->fos.end(), -1);
  if (c->poison) return poison_slots(c);
  return LL_OK;
}

ll_status ll_sync(ll_cache* c) {
  NvtxRange range("ll_sync");
  if (!c) return LL_ERR_INVALID_ARG;
  if (ll_status s = set_device(c)) return s;
  if (cudaDeviceSynchronize() != cudaSuccess) return LL_ERR_CUDA;
  return take_device_error(c);
}

ll_status ll_cache_state(ll_cache* c, int layer, int64_t* frames_committed, int64_t* frame_of_slot) {
  if (ll_status s = check_layer(c, layer)) return s;
  if (ll_status s = ll_sync(c)) return s;
  if (frames_committed) *frames_committed = c->n[layer];
  if (frame_of_slot) {
    const int slots = c->S + c->W;
    for (int i = 0; i < slots; ++i) frame_of_slot[i] = c->fos[(size_t)layer * slots + i];
  }
  return LL_OK;
}

ll_status ll_cache_read(ll_cache* c, int layer, void* host_k, void* host_v) {
  NvtxRange range("ll_cache_read");
  if (ll_status s = check_layer(c, layer)) return s;
  const size_t kbytes = c->layer_elems * c->keb, vbytes = c->layer_elems * c->veb;
  if (kbytes == 0) return ll_sync(c);  // no slots (S = W = 0): nothing to copy
  if (!host_k || !host_v) return LL_ERR_INVALID_ARG;
  if (ll_status s = ll_sync(c)) return s;
  if (cudaMemcpy(host_k, static_cast<char*>(c->k) + kbytes * (size_t)layer, kbytes, cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemcpy(host_v, static_cast<char*>(c->v) + vbytes * (size_t)layer, vbytes, cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return LL_ERR_CUDA;
  return LL_OK;
}

ll_status ll_cache_info(const ll_cache* c, int* slots, size_t* layer_bytes, int* elem_bytes) {
  if (!c) return LL_ERR_INVALID_ARG;
  if (slots) *slots = c->S + c->W;
  if (layer_bytes) *layer_bytes = c->layer_elems * c->keb;
  if (elem_bytes) *elem_bytes = c->keb;
  return LL_OK;
}

ll_status ll_debug_inject_stall(ll_cache* c, int enable, int timeout_us) {
  if (!c || timeout_us < 0) return LL_ERR_INVALID_ARG;
  c->stall_inject = enable ? 1 : 0;
  c->stall_timeout_us = timeout_us;
  return LL_OK;
}

ll_status ll_profile_enable(ll_cache* c, int enable) {
  if (!c) return LL_ERR_INVALID_ARG;
  c->profiling = enable > 0;
  if (enable > 0) {
    c->profile_every = enable;
    for (auto& n : c->profile_seen) n = 0;
  }
  return LL_OK;
}

ll_status ll_profile_read(ll_cache* c, int kind, int64_t* launches, double* total_ms) {
  if (!c || kind < 0 || kind >= LL_KERNEL_KINDS) return LL_ERR_INVALID_ARG;
  if (ll_status s = ll_sync(c)) return s;
  int64_t n = 0;
  double ms = 0.0;
  std::vector<ll_cache::Mark> keep;
  for (auto& m : c->marks) {
    if (m.kind != kind) {
      keep.push_back(m);
      continue;
    }
    float t = 0.f;
    if (cudaEventElapsedTime(&t, m.start, m.stop) == cudaSuccess) {
      ms += t;
      ++n;
    }
    c->event_pool.push_back(m.start);
    c->event_pool.push_back(m.stop);
  }
  c->marks.swap(keep);
  if (launches) *launches = n;
  if (total_ms) *total_ms = ms;
  return LL_OK;
}

int ll_debug_attend_schedule(int Lq, int La, int Lb, int heads, int max_ctas, int mode, int block_tokens,
                             int* grid, int* pieces, int cap, int* splits, int split_cap, int* split_ints) {
  if (Lq < 1 || La < 0 || Lb < 1 || heads < 1 || max_ctas < 1 || !grid || !split_ints) return -1;
  if (mode < 0 || mode > 2) return -1;
  if (mode != 0 && block_tokens < 1) return -1;
  return ll::attend_schedule_dump(Lq, La, Lb, heads, max_ctas, mode, block_tokens, grid, pieces, cap, splits,
                                  split_cap, split_ints);
}

ll_status ll_debug_use_simt(ll_cache* c, int enable) {
  if (!c) return LL_ERR_INVALID_ARG;
  c->use_simt = enable ? 1 : 0;
  return LL_OK;
}

ll_status ll_debug_poison(ll_cache* c, int enable) {
  if (!c) return LL_ERR_INVALID_ARG;
  c->poison = enable != 0;
  if (!c->poison) return LL_OK;
  // every slot not holding a resident frame gets the poison now
  if (ll_status s = poison_resident_gaps(c)) return s;
  return LL_OK;
}

ll_status ll_debug_inject_fault(int kind, int n) {
  if (n < 0) return LL_ERR_INVALID_ARG;
  if (kind == LL_FAULT_ALLOC) {
    g_fault_alloc = n;
  } else if (kind == LL_FAULT_LAUNCH) {
    g_fault_launch = n;
  } else {
    return LL_ERR_INVALID_ARG;
  }
  return LL_OK;
}

ll_status ll_debug_pair_kernel(ll_cache* c, int enable) {
  if (!c) return LL_ERR_INVALID_ARG;
  c->pair = enable ? 1 : 0;
  return LL_OK;
}

}  // extern "C"
