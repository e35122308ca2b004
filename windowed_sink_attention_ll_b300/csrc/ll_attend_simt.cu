// Attention for the fp32 cache dtype (and a bf16 instantiation used only to
// cross-check the tensor-core kernel): one warp per (query row, head), fp32
// online softmax, dot products reduced with warp shuffles.
//
// "LongLive", §3.3 "Frame sink" / "Short window attention": each query of the
// chunk attends to [resident sink + window frames of the cache || the chunk's
// own K/V]; in prefill mode (§3.1 "KV recache") it attends block-causally over
// the recache window, and in mode 2 it sees every cached key and the chunk's
// own keys block-causally.  The key/value list is read from the two sources that
// AttendArgs describes; the order of keys does not change the softmax.
#include <cuda_bf16.h>

#include "ll_internal.h"

namespace ll {

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

constexpr int kWarps = 8;

// Each lane owns D/32 consecutive elements of the query row and of the output.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) attend_simt_kernel(const __grid_constant__ AttendArgs a) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t task = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (task >= (int64_t)a.Lq * a.heads) return;
  const int row = (int)(task / a.heads);
  const int h = (int)(task - (int64_t)row * a.heads);
  const T* q = static_cast<const T*>(a.q) + ((int64_t)row * a.heads + h) * D + lane * E;
  float qv[E], o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qv[e] = to_f(q[e]);
    o[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const float sl2 = a.scale_log2;

  auto visit = [&](const T* krow, const T* vrow) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) s = fmaf(qv[e], to_f(krow[e]), s);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const float x = s * sl2;
    const float mn = fmaxf(m, x);
    const float alpha = exp2f(m - mn);  // 0 on the first key (m = -inf)
    const float p = exp2f(x - mn);
    l = l * alpha + p;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = fmaf(o[e], alpha, p * to_f(vrow[e]));
    m = mn;
  };

  // source A: the cache's resident rows of head h
  const T* kc = static_cast<const T*>(a.kc) + (int64_t)h * a.cache_head_elems + lane * E;
  const T* vc = static_cast<const T*>(a.vc) + (int64_t)h * a.cache_head_elems + lane * E;
  for (int j = 0; j < a.La; ++j) visit(kc + (int64_t)j * D, vc + (int64_t)j * D);
  // source B: caller tensor rows, all of them (attend) or a block-causal prefix (prefill)
  int end = a.Lb;
  if (a.mode != 0) {
    const int64_t e = ((int64_t)row / a.block_tokens + 1) * a.block_tokens;
    end = e < a.Lb ? (int)e : a.Lb;
  }
  const T* kn = static_cast<const T*>(a.kn) + (int64_t)h * D + lane * E;
  const T* vn = static_cast<const T*>(a.vn) + (int64_t)h * D + lane * E;
  const int64_t stride = (int64_t)a.heads * D;
  for (int j = 0; j < end; ++j) visit(kn + j * stride, vn + j * stride);

  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int64_t ob = ((int64_t)row * a.heads + h) * D + lane * E;
  if (a.out_f32) {
    float* out = static_cast<float*>(a.out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = o[e] * inv;
  } else {
    T* out = static_cast<T*>(a.out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = from_f<T>(o[e] * inv);
  }
}

template <typename T, int D>
cudaError_t launch(const AttendArgs& a, cudaStream_t stream) {
  const int64_t tasks = (int64_t)a.Lq * a.heads;
  const int64_t blocks = (tasks + kWarps - 1) / kWarps;
  attend_simt_kernel<T, D><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend_simt(const AttendArgs& a, int elem_bytes, cudaStream_t stream) {
  if (elem_bytes == 4) {
    return a.head_dim == 64 ? launch<float, 64>(a, stream) : launch<float, 128>(a, stream);
  }
  return a.head_dim == 64 ? launch<__nv_bfloat16, 64>(a, stream) : launch<__nv_bfloat16, 128>(a, stream);
}

}  // namespace ll
