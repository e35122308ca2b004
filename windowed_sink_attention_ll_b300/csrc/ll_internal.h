// Internal declarations shared by the host layer and the kernels of libll.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ll {

// Largest number of frames one copy launch may place (C for a commit, S + W for a recache).
constexpr int kMaxFrameTable = 512;

// Device error word codes (OR-ed together by kernels, read and cleared by the host).
constexpr unsigned kErrTimeout = 1u;

// ---------------------------------------------------------------------------
// Frame copy: chunk/recache K,V [frames*T][H][d] (token-major) -> cache slots
// [H][slots*T][d] (head-major).  slot_of[i] is the destination slot of source
// frame i, or -1 to skip it.
// ---------------------------------------------------------------------------
struct CopyFramesArgs {
  const void* src_k;
  const void* src_v;
  void* dst_k;  // this layer's K cache: head 0, slot 0
  void* dst_v;
  int frames;
  int tokens_per_frame;
  int heads;
  int head_dim;
  int slots;         // S + W
  int elem_bytes;    // of V (and of K unless k_elem_bytes says otherwise): 2 or 4
  int k_elem_bytes;  // of K: 0 = elem_bytes; 1 = e4m3 keys
  int slot_of[kMaxFrameTable];
};

cudaError_t launch_copy_frames(const CopyFramesArgs& a, cudaStream_t stream);

// Round `n` bf16 values of each of up to three tensors to e4m3 (round to nearest
// even, saturating at +-448), as the FP8 caches store keys (and values) and the
// kind::f8f6f4 Q K^T product reads q and the chunk's keys.  Null entries of src
// are skipped.
cudaError_t launch_quantize_e4m3(const void* const src[3], void* const dst[3], int64_t n, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Attention over two key/value sources:
//   source A: rows [0, La) of this layer's head-major cache (the resident slots,
//             which always form a prefix of the slots);
//   source B: rows [0, Lb) of a caller tensor [Lb][H][d] (the chunk's own K/V,
//             or the recache window in prefill mode).
// mode 0 (attend): every query sees all La + Lb keys.
// mode 1 (prefill): every key of source A (La = 0 except in the keep-sink
//             prefill) and keys j of source B with j / block_tokens <=
//             i / block_tokens (prefill schedule: unequal items, none split).
// mode 2 (masked attend): the same mask with the attend schedule.
// ---------------------------------------------------------------------------
struct AttendArgs {
  const void* q;      // [Lq][H][d]
  void* out;          // [Lq][H][d]
  const void* kc;     // cache K of this layer (head 0, slot 0)
  const void* vc;
  int64_t cache_head_elems;  // elements between consecutive heads in the cache
  int La;
  const void* kn;     // [Lb][H][d]
  const void* vn;
  int Lb;
  int Lq;
  int heads;
  int head_dim;
  int mode;
  int block_tokens;
  float scale_log2;   // log2(e) / sqrt(d)
  int out_f32;        // out is fp32 (else the cache dtype)
  unsigned* err;      // device-visible error word
  int stall_inject;   // test hook: skip one barrier arrival
  long long timeout_ns;
  float* scratch;     // partial results of split work items (tensor-core kernel)
  int scratch_slots;  // partial-result slots the scratch holds
  int pair;           // head_dim 128: the CTA-pair tensor-core kernel instead of the one-CTA kernel
  int qk_fp8;         // q, kn and the cache K hold e4m3 bytes (Q K^T on kind::f8f6f4); head_dim 128
  int v_fp8;          // with qk_fp8: vn and the cache V hold e4m3 bytes too (P V on fp16 operands)
};

// bf16 attention on the tensor cores: the one-CTA kernel, or for head_dim 128 with
// a.pair the CTA-pair kernel.
cudaError_t launch_attend_bf16_tc(const AttendArgs& a, cudaStream_t stream);
cudaError_t launch_attend_bf16_pair(const AttendArgs& a, cudaStream_t stream);
// fp32 attention on the tensor cores (tf32 operands), head_dim 64.
cudaError_t launch_attend_tf32_tc(const AttendArgs& a, cudaStream_t stream);
// Scratch of the tensor-core kernel: bytes for `slots` partial results, and the
// slot count it uses on the current device (two per SM).
size_t attend_scratch_bytes(int head_dim, int slots);
int attend_scratch_slots_wanted();
// Host replay of the schedule of an attend (mode 0) or prefill (mode 1) launch
// (tests): pieces as (cta, item, j0, j1, partial, slot) sextuples, split items
// as (item, parts, slots...).
int attend_schedule_dump(int Lq, int La, int Lb, int heads, int max_ctas, int mode, int block_tokens, int* grid,
                         int* out, int cap, int* splits, int split_cap, int* split_ints);
cudaError_t launch_attend_simt(const AttendArgs& a, int elem_bytes, cudaStream_t stream);

void count_launch();

// Launch `kernel` as a programmatic dependent of the kernel before it on `stream`
// (programmatic stream serialization): its blocks may be scheduled while that
// kernel drains.  The kernel must execute griddepcontrol.wait before its first
// access to memory that earlier work on the stream writes or reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace ll
