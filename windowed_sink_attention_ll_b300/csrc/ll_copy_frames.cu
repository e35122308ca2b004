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
// T rows x vpr vectors.  All index math stays in 32 bits within one slab.
__global__ void __launch_bounds__(kThreads) copy_frames_kernel(const __grid_constant__ CopyFramesArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int f = blockIdx.y / a.heads;
  const int h = blockIdx.y - f * a.heads;
  const int slot = a.slot_of[f];
  if (slot < 0) return;
  const int vpr = a.head_dim * a.elem_bytes / 16;  // 16-byte vectors per (token, head) row
  const int slab = a.tokens_per_frame * vpr;
  const uint4* sk = static_cast<const uint4*>(a.src_k);
  const uint4* sv = static_cast<const uint4*>(a.src_v);
  uint4* dk = static_cast<uint4*>(a.dst_k);
  uint4* dv = static_cast<uint4*>(a.dst_v);
  const int64_t src_base = ((int64_t)f * a.tokens_per_frame * a.heads + h) * vpr;
  const int64_t src_tok = (int64_t)a.heads * vpr;
  const int64_t dst_base = ((int64_t)h * a.slots + slot) * a.tokens_per_frame * vpr;
  const int i0 = blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
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

}  // namespace

cudaError_t launch_copy_frames(const CopyFramesArgs& a, cudaStream_t stream) {
  if (a.frames <= 0) return cudaSuccess;
  const int vpr = a.head_dim * a.elem_bytes / 16;
  const int slab = a.tokens_per_frame * vpr;
  const dim3 grid((unsigned)((slab + kThreads * kUnroll - 1) / (kThreads * kUnroll)),
                  (unsigned)(a.frames * a.heads));
  const cudaError_t e = launch_dependent(copy_frames_kernel, grid, dim3(kThreads), 0, stream, a);
  count_launch();
  return e;
}

}  // namespace ll
