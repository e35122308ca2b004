// Commit / recache write: move whole frames of K and V from the caller's
// token-major tensors into their cache slots.
//
// "LongLive", §3.3 "Frame sink": the sink frames stay in the cache for good and
// the other frames roll through a short window with FIFO eviction; §3.1 "KV
// recache" rewrites the resident frames in place.  Both reduce to the same
// HBM-bound copy with a per-frame destination slot chosen on the host.
//
// Layout: source [frames*T][H][d]; destination [H][slots*T][d].  Each thread
// moves 16-byte vectors; consecutive threads walk the d-vectors of one row and
// then consecutive tokens of one head, so each warp writes 512 contiguous bytes
// of the cache and reads two whole 256-byte rows of the source (bf16, d = 128).
// A block's slab is one (frame, head) pair: a frame's T tokens of one head are
// contiguous in the cache.
//
// The copy is launched as a programmatic dependent of the kernel before it on the
// stream (the attention launch of the same call, for a commit): its blocks may be
// scheduled while that kernel drains, and each one waits (griddepcontrol.wait)
// until the predecessor has completed and its memory is visible before it reads
// or writes anything, so the launch latency is hidden and the order is kept.
#include "ll_internal.h"

namespace ll {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte vectors per thread per tensor

// grid.y = source frame * heads + head; grid.x covers that (frame, head) slab of
// T rows x vpr vectors.  All index math stays in 32 bits within one slab.  When K
// and V have the same element size one block moves both tensors' vectors; with an
// e4m3 key cache (K one byte per element, V two) grid.z = 2 and each block moves
// one tensor's slab (z = 0: K, z = 1: V).
__global__ void __launch_bounds__(kThreads) copy_frames_kernel(const __grid_constant__ CopyFramesArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int f = blockIdx.y / a.heads;
  const int h = blockIdx.y - f * a.heads;
  const int slot = a.slot_of[f];
  if (slot < 0) return;
  const int i0 = blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
  if (a.k_elem_bytes != 0 && a.k_elem_bytes != a.elem_bytes) {
    const bool is_v = blockIdx.z != 0;
    const int vpr = a.head_dim * (is_v ? a.elem_bytes : a.k_elem_bytes) / 16;
    const int slab = a.tokens_per_frame * vpr;
    if (i0 >= slab) return;
    const uint4* src = static_cast<const uint4*>(is_v ? a.src_v : a.src_k);
    uint4* dst = static_cast<uint4*>(is_v ? a.dst_v : a.dst_k);
    const int64_t src_base = ((int64_t)f * a.tokens_per_frame * a.heads + h) * vpr;
    const int64_t src_tok = (int64_t)a.heads * vpr;
    const int64_t dst_base = ((int64_t)h * a.slots + slot) * a.tokens_per_frame * vpr;
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kThreads;
      if (i < slab) {
        const int t = i / vpr;
        x[u] = __ldcs(src + src_base + t * src_tok + (i - t * vpr));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kThreads;
      if (i < slab) __stcg(dst + dst_base + i, x[u]);
    }
    return;
  }
  const int vpr = a.head_dim * a.elem_bytes / 16;  // 16-byte vectors per (token, head) row
  const int slab = a.tokens_per_frame * vpr;
  const uint4* sk = static_cast<const uint4*>(a.src_k);
  const uint4* sv = static_cast<const uint4*>(a.src_v);
  uint4* dk = static_cast<uint4*>(a.dst_k);
  uint4* dv = static_cast<uint4*>(a.dst_v);
  const int64_t src_base = ((int64_t)f * a.tokens_per_frame * a.heads + h) * vpr;
  const int64_t src_tok = (int64_t)a.heads * vpr;
  const int64_t dst_base = ((int64_t)h * a.slots + slot) * a.tokens_per_frame * vpr;
  uint4 kx[kUnroll], vx[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int i = i0 + u * kThreads;
    if (i < slab) {
      const int t = i / vpr;
      const int c = i - t * vpr;
      const int64_t s = src_base + t * src_tok + c;
      kx[u] = __ldcs(sk + s);
      vx[u] = __ldcs(sv + s);
    }
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int i = i0 + u * kThreads;
    if (i < slab) {
      __stcg(dk + dst_base + i, kx[u]);
      __stcg(dv + dst_base + i, vx[u]);
    }
  }
}

// Rounds bf16 values to e4m3 (cvt.rn.satfinite: nearest, ties to even, beyond
// +-448 clamped to +-448).  blockIdx.y picks the tensor; each thread converts 16
// consecutive values (two 16-byte loads, one 16-byte store).  Launched as a
// programmatic dependent: it waits for the kernel before it on the stream.
struct QuantArgs {
  const uint4* src[3];
  uint4* dst[3];
  int64_t groups;  // 16-value groups per tensor
};

__device__ __forceinline__ uint32_t e4m3x4(uint32_t bf_lo, uint32_t bf_hi) {
  // four bf16 (two words) -> four e4m3 bytes, lowest element in the lowest byte
  const float a0 = __uint_as_float(bf_lo << 16), a1 = __uint_as_float(bf_lo & 0xFFFF0000u);
  const float a2 = __uint_as_float(bf_hi << 16), a3 = __uint_as_float(bf_hi & 0xFFFF0000u);
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a1), "f"(a0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a3), "f"(a2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__global__ void __launch_bounds__(kThreads) quantize_e4m3_kernel(const __grid_constant__ QuantArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (i >= a.groups || !a.src[t]) return;
  const uint4 x = a.src[t][2 * i], y = a.src[t][2 * i + 1];
  uint4 o;
  o.x = e4m3x4(x.x, x.y);
  o.y = e4m3x4(x.z, x.w);
  o.z = e4m3x4(y.x, y.y);
  o.w = e4m3x4(y.z, y.w);
  a.dst[t][i] = o;
}

}  // namespace

cudaError_t launch_copy_frames(const CopyFramesArgs& a, cudaStream_t stream) {
  if (a.frames <= 0) return cudaSuccess;
  const bool split = a.k_elem_bytes != 0 && a.k_elem_bytes != a.elem_bytes;
  const int vpr = a.head_dim * a.elem_bytes / 16;  // V's (the larger) vectors per row when split
  const int slab = a.tokens_per_frame * vpr;
  const dim3 grid((unsigned)((slab + kThreads * kUnroll - 1) / (kThreads * kUnroll)),
                  (unsigned)(a.frames * a.heads), split ? 2u : 1u);
  const cudaError_t e = launch_dependent(copy_frames_kernel, grid, dim3(kThreads), 0, stream, a);
  count_launch();
  return e;
}

cudaError_t launch_quantize_e4m3(const void* const src[3], void* const dst[3], int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (n % 16 != 0) return cudaErrorInvalidValue;
  QuantArgs q;
  unsigned tensors = 0;
  for (int t = 0; t < 3; ++t) {
    q.src[t] = static_cast<const uint4*>(src[t]);
    q.dst[t] = static_cast<uint4*>(dst[t]);
    if (src[t]) tensors = (unsigned)t + 1;
  }
  if (tensors == 0) return cudaSuccess;
  q.groups = n / 16;
  const dim3 grid((unsigned)((q.groups + kThreads - 1) / kThreads), tensors);
  const cudaError_t e = launch_dependent(quantize_e4m3_kernel, grid, dim3(kThreads), 0, stream, q);
  count_launch();
  return e;
}

}  // namespace ll
