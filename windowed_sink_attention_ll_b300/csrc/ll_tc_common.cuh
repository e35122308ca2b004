// Pieces shared by the two tensor-core attention kernels (ll_attend_tc.cu: one CTA
// per work item; ll_attend_pair.cu: a CTA pair per work item): inline-PTX
// wrappers for mbarriers, TMA, tcgen05 and tensor memory, the matrix and
// instruction descriptors, the persistent work schedule, the merge of split
// work items, and the tensor-map encoder.
//
// Work item = one head x 256 query rows ("LongLive", §3.3: every query of the
// chunk attends to the same key list, so items differ only in their rows).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstring>

#include "ll_internal.h"

namespace ll {
namespace tc {

constexpr int kItemRows = 256;  // query rows per work item
constexpr int kKeyTile = 128;   // keys per K/V tile
constexpr int kAtom = 16384;    // one 128-row x 128-byte swizzled TMA box
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kDrainNs = 200000000LL;  // 0.2 s for copies/MMAs already in flight
constexpr int kMaxSplit = 256;               // most workers of a persistent attend launch
constexpr int kMinTailTiles = 16;            // shortest run of key tiles a tail worker takes

// ----------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct Ctl {
  volatile int* abort;
  unsigned* err;
  long long timeout_ns;
};

template <bool kCluster>
__device__ __forceinline__ bool mbar_try_t(uint32_t bar, uint32_t parity);
template <>
__device__ __forceinline__ bool mbar_try_t<false>(uint32_t bar, uint32_t parity) {
  return mbar_try(bar, parity);
}
// acquire at cluster scope: the phase may have been completed by arrivals from the peer CTA
template <>
__device__ __forceinline__ bool mbar_try_t<true>(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

template <bool kCluster>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Ctl& c) {
  const uint64_t t0 = now_ns();
  while (true) {
    if (mbar_try_t<kCluster>(bar, parity)) return true;
    if (*c.abort) return false;
    if ((long long)(now_ns() - t0) > c.timeout_ns) {
      *c.abort = 1;
      *reinterpret_cast<volatile unsigned*>(c.err) = kErrTimeout;
      __threadfence_system();
      return false;
    }
  }
}
// Bounded wait for the phase of `bar` with the given parity; false = abort.
template <bool kCluster = false>
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (mbar_try_t<kCluster>(bar, parity)) return true;
  return wait_slow<kCluster>(bar, parity, c);
}
// Bounded wait that ignores the abort flag (teardown of work in flight).
static __device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = now_ns();
  while (!mbar_try(bar, parity)) {
    if ((long long)(now_ns() - t0) > kDrainNs) return;
  }
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define LL_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define LL_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                 "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : LL_R8(0), LL_R8(8), LL_R8(16), LL_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : LL_R8(0), LL_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      LL_W8(0), LL_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Orders later uses of loaded registers after tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence(uint32_t* r, int n) {
#pragma unroll
  for (int i = 0; i < n; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max of three floats in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
// (d0, d1) = (a0, a1) * b + c, two lanes per instruction
__device__ __forceinline__ void fma_f32x2(float& d0, float& d1, float a0, float a1, uint64_t b, uint64_t c) {
  asm("{\n\t.reg .b64 a, d;\n\tmov.b64 a, {%2, %3};\n\tfma.rn.f32x2 d, a, %4, %5;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "l"(b), "l"(c));
}
// s0 += low bf16 of pk, s1 += high bf16 of pk (widened exactly, fp32 adds)
__device__ __forceinline__ void add_bf16x2(float& s0, float& s1, uint32_t pk) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.bf16 %0, lo, %0;\n\t"
      "add.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "r"(pk));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// s0 += low f16 of pk, s1 += high f16 of pk (widened exactly, fp32 adds)
__device__ __forceinline__ void add_f16x2(float& s0, float& s1, uint32_t pk) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.f16 %0, lo, %0;\n\t"
      "add.rn.f32.f16 %1, hi, %1;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "r"(pk));
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start
// address, leading and stride byte offsets in 16-byte units, version 1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ uint64_t make_desc(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
// Instruction descriptor, kind::f8f6f4: e4m3 A and B (format code 0), fp32 D, M x N,
// both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor, kind::tf32: tf32 A and B (format code 2), fp32 D, M x N,
// both operands K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor, kind::f16: f16 A and B (format code 0), fp32 D, M x N, A/B major-ness.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M x N, A/B major-ness.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ----------------------------------------------------------------------------
// Work schedule (both kernels; a "worker" is a CTA of the one-CTA kernel or a
// CTA pair of the pair kernel)
// ----------------------------------------------------------------------------
// Attend mode: an item is (head, 256-row query block); every item has the same
// nkv key tiles.  The grid is persistent (at most one worker per SM or SM pair).
// Whole rounds of items come first -- worker c takes item r*grid + c in round
// r, so the workers sweep the K/V tiles of a few heads in step and each tile is
// fetched from HBM about once -- and the items left over (fewer than the grid)
// are cut into equal runs of key tiles across `tail_ctas` workers.  A run that
// covers only part of an item leaves a partial result (unnormalised O,
// reference max m and sum l per row) in scratch slot 2*c + (0: first run of
// worker c, 1: its last run); combine_kernel merges the parts of each split
// item.  Mode 2 (masked attend) uses the same schedule.
// Prefill mode (mode 1): items are numbered from the last query block to the
// first, i.e. longest first (block g of a block-causal prefill sees g + 1
// blocks of keys); round r gives worker c item r*grid + c (r even) or
// r*grid + grid - 1 - c (r odd), which keeps every worker's total within one
// item of the mean without splitting any item.
struct Sched {
  int nqb;               // query blocks of 256 rows per head
  int nkv;               // attend: key tiles per item
  int grid;              // workers launched
  int rounds;            // attend: whole-item rounds
  int tail_ctas;         // attend: workers sharing the left-over items
  long long tail_iters;  // attend: key tiles of the left-over items
};

struct Piece {
  int item;
  int j0, j1;   // key tiles [j0, j1) of the item
  int partial;  // 1: write a partial result to scratch slot `slot`
  int slot;
};

struct Walker {
  int r;
  long long it, end, begin;
  int prefill;
};

__host__ __device__ __forceinline__ void walker_init(Walker& w, const AttendArgs& a, const Sched& s, int cta) {
  w.r = 0;
  w.prefill = a.mode == 1;
  w.begin = w.end = 0;
  if (!w.prefill && cta < s.tail_ctas) {
    w.begin = (s.tail_iters * cta) / s.tail_ctas;
    w.end = (s.tail_iters * (cta + 1)) / s.tail_ctas;
  }
  w.it = w.begin;
}

// Key tiles a prefill item of query block qb needs: every cached tile (source A,
// fully visible) and the fresh tiles up to the end of the block of its last row.
__host__ __device__ __forceinline__ int prefill_nkv(const AttendArgs& a, int qb) {
  const int qend = (qb + 1) * kItemRows;
  const int qlast = (qend < a.Lq ? qend : a.Lq) - 1;
  const long long e = ((long long)qlast / a.block_tokens + 1) * a.block_tokens;
  const int kv_end = (int)(e < a.Lb ? e : a.Lb);
  return (a.La + kKeyTile - 1) / kKeyTile + (kv_end + kKeyTile - 1) / kKeyTile;
}

__host__ __device__ __forceinline__ bool walker_next(Walker& w, const AttendArgs& a, const Sched& s, Piece& pc,
                                                     int cta) {
  if (w.prefill) {
    // items come longest first; round r hands them out left to right (even r) or
    // right to left (odd r), so each worker's total stays close to the mean
    const int items = s.nqb * a.heads;
    while (w.r * s.grid < items) {
      const int r = w.r++;
      const int item = r * s.grid + ((r & 1) ? s.grid - 1 - cta : cta);
      if (item >= items) continue;
      pc.item = item;
      pc.j0 = 0;
      pc.j1 = prefill_nkv(a, s.nqb - 1 - item / a.heads);
      pc.partial = 0;
      pc.slot = 0;
      return true;
    }
    return false;
  }
  if (w.r < s.rounds) {
    pc.item = w.r * s.grid + cta;
    pc.j0 = 0;
    pc.j1 = s.nkv;
    pc.partial = 0;
    pc.slot = 0;
    ++w.r;
    return true;
  }
  if (w.it >= w.end) return false;
  const long long ti = w.it / s.nkv;
  const int j0 = (int)(w.it - ti * s.nkv);
  const long long stop = w.end - ti * s.nkv;
  const int j1 = (int)(stop < s.nkv ? stop : s.nkv);
  pc.item = s.rounds * s.grid + (int)ti;
  pc.j0 = j0;
  pc.j1 = j1;
  pc.partial = !(j0 == 0 && j1 == s.nkv);
  pc.slot = 2 * cta + (w.it == w.begin ? 0 : 1);
  w.it = ti * s.nkv + j1;
  return true;
}

// head, first query row and cache-tile count of an item
__device__ __forceinline__ void item_geom(const AttendArgs& a, const Sched& s, int item, int& head, int& q0,
                                          int& nA) {
  if (a.mode != 1) {
    head = item / s.nqb;
    q0 = (item - head * s.nqb) * kItemRows;
  } else {
    const int qb = s.nqb - 1 - item / a.heads;
    head = item - (item / a.heads) * a.heads;
    q0 = qb * kItemRows;
  }
  nA = (a.La + kKeyTile - 1) / kKeyTile;
}

struct CombineParams {
  void* out;
  const float* part;
  int grid;  // the attend launch's workers; scratch slots = 2 * grid
  int nqb;
  int Lq;
  int heads;
  int out_f32;
  int nsplit;
  int item[kMaxSplit];
  int first[kMaxSplit + 1];  // parts of split k: slot[first[k] .. first[k+1])
  int slot[2 * kMaxSplit];
};

// Schedule of an attend launch with at most max_workers workers (see "Work
// schedule"); fills s and the split list.
inline void plan_attend(const AttendArgs& a, Sched& s, CombineParams& cp, int max_workers) {
  const int items = s.nqb * a.heads;
  s.nkv = (a.La + kKeyTile - 1) / kKeyTile + (a.Lb + kKeyTile - 1) / kKeyTile;
  int g = max_workers < kMaxSplit ? max_workers : kMaxSplit;
  if (g > items) g = items;
  if (g < 1) g = 1;
  s.grid = g;
  s.rounds = items / g;
  const int rem = items - s.rounds * g;
  s.tail_iters = (long long)rem * s.nkv;
  long long tc = s.tail_iters / kMinTailTiles;
  if (tc > g) tc = g;
  if (tc < 1) tc = 1;
  s.tail_ctas = rem > 0 ? (int)tc : 0;
  cp.nsplit = 0;
  int np = 0;
  auto bnd = [&](long long cta) { return (s.tail_iters * cta) / s.tail_ctas; };
  int c = 0;
  for (int ti = 0; ti < rem; ++ti) {
    const long long lo = (long long)ti * s.nkv, hi = lo + s.nkv;
    while (c + 1 < s.tail_ctas && bnd(c + 1) <= lo) ++c;
    int chi = c;
    while (chi + 1 < s.tail_ctas && bnd(chi + 1) < hi) ++chi;
    if (chi == c) continue;
    const int k = cp.nsplit++;
    cp.item[k] = s.rounds * s.grid + ti;
    cp.first[k] = np;
    cp.slot[np++] = 2 * c + (bnd(c) == lo ? 0 : 1);
    for (int cc = c + 1; cc <= chi; ++cc) cp.slot[np++] = 2 * cc;
  }
  cp.first[cp.nsplit] = np;
}

// ----------------------------------------------------------------------------
// Merge of split items: out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p
// ----------------------------------------------------------------------------
// Launched as a programmatic dependent of the attention kernel: it waits until that
// kernel has completed (and its partial results are visible) before reading them.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineParams c) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int E = D / 32;
  const int k = blockIdx.x;
  const int r = blockIdx.y * 8 + (threadIdx.x >> 5);  // row within the item's 256 query rows
  const int lane = threadIdx.x & 31;
  const int item = c.item[k];
  const int head = item / c.nqb;
  const int qrow = (item - head * c.nqb) * kItemRows + r;
  if (qrow >= c.Lq) return;
  const size_t rows_all = (size_t)2 * c.grid * kItemRows;
  const float* pm = c.part + rows_all * D;
  const float* pl = pm + rows_all;
  float M = -INFINITY;
  for (int i = c.first[k]; i < c.first[k + 1]; ++i) M = fmaxf(M, pm[(size_t)c.slot[i] * kItemRows + r]);
  float acc[E], L = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int i = c.first[k]; i < c.first[k + 1]; ++i) {
    const size_t sr = (size_t)c.slot[i] * kItemRows + r;
    const float mi = pm[sr];
    const float wgt = (mi == -INFINITY) ? 0.f : exp2f(mi - M);
    L += wgt * pl[sr];
    const float* o = c.part + sr * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(wgt, o[e], acc[e]);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int64_t ob = ((int64_t)qrow * c.heads + head) * D + lane * E;
  if (c.out_f32) {
    float* out = static_cast<float*>(c.out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = acc[e] * inv;
  } else {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(c.out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = __float2bfloat16_rn(acc[e] * inv);
  }
}

template <int D>
inline cudaError_t launch_combine(CombineParams& cp, const AttendArgs& a, const Sched& s, float* part,
                                  cudaStream_t stream) {
  cp.out = a.out;
  cp.part = part;
  cp.grid = s.grid;
  cp.nqb = s.nqb;
  cp.Lq = a.Lq;
  cp.heads = a.heads;
  cp.out_f32 = a.out_f32;
  const cudaError_t e =
      launch_dependent(combine_kernel<D>, dim3((unsigned)cp.nsplit, kItemRows / 8), dim3(256), 0, stream, cp);
  count_launch();
  return e;
}

// ----------------------------------------------------------------------------
// Tensor maps
// ----------------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

// 3-D tensor map of bf16 (elem_bytes 2), byte-sized e4m3 (elem_bytes 1) or fp32
// (elem_bytes 4) elements, 128-byte swizzle
inline bool encode3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                     uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2, int elem_bytes = 2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// [L][H][D] token tensor, boxes of 128 bytes of d x 1 head x `rows` tokens.
inline bool encode_tokens(CUtensorMap* m, const void* base, int L, int H, int D, int rows, int elem_bytes = 2) {
  return encode3d(m, base, (uint64_t)D, (uint64_t)H, (uint64_t)L, (uint64_t)D * elem_bytes,
                  (uint64_t)H * D * elem_bytes, 128 / elem_bytes, 1, (uint32_t)rows, elem_bytes);
}

// Head-major cache rows of one layer, [H][rows][D] with `head_elems` between heads,
// boxes of 128 bytes of d x `rows_box` rows x 1 head.
inline bool encode_cache(CUtensorMap* m, const void* base, int La, int H, int D, int64_t head_elems,
                         int rows_box, int elem_bytes = 2) {
  const int rows = La > 0 ? La : 1;
  return encode3d(m, base, (uint64_t)D, (uint64_t)rows, (uint64_t)H, (uint64_t)D * elem_bytes,
                  (uint64_t)head_elems * elem_bytes, 128 / elem_bytes, (uint32_t)rows_box, 1, elem_bytes);
}

inline int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  return n;
}

// Shared-memory opt-in of a kernel, once per device (several host threads may launch at once).
template <typename K>
inline cudaError_t smem_opt_in(K kernel, int bytes, std::atomic<int> (&done)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) done[dev].store(1, std::memory_order_release);
  return cudaSuccess;
}

}  // namespace tc
}  // namespace ll
