// Chunk attention on the 5th-generation tensor cores (sm_103a): TMA-staged
// K/V tiles, tcgen05.mma for Q K^T and P V with fp32 accumulators in tensor
// memory, fp32 online softmax.
//
// What it computes ("LongLive: Real-time Interactive Long Video Generation",
// §3.3 Efficient Long Inference, "Short window attention" + "Frame sink"):
// for one head and one block of query rows of the current chunk,
//     O = softmax(Q K^T / sqrt(d)) V
// over the key list [resident sink + window frames of the layer's cache ||
// the chunk's own keys].  Softmax does not depend on the order of the keys,
// so the kernel walks the resident cache rows in slot order (one contiguous
// run per head, see ll_host.cu) and then the chunk's rows.  In prefill mode
// (§3.1 "KV recache") there is one source, the recache window, and query row
// i sees key j iff j / block_tokens <= i / block_tokens.
//
// CTA = one head x 256 query rows, split into two 128-row tiles that share
// every K/V tile.  Warp roles (384 threads):
//   warp 0      TMA producer: Q once, then K0 V0 K1 V1 ... into a 5-stage ring
//   warp 1      TMEM allocator and tcgen05.mma issuer (one thread)
//   warps 4-7   softmax for Q tile 0, warps 8-11 for Q tile 1: thread = row
//   warps 2-3   idle
// Tensor memory (512 columns x 128 lanes): O0 [0,128) O1 [128,256)
// S0 [256,384) S1 [384,512).  P (bf16) overwrites the first 64 columns of S
// and feeds the P V product straight from tensor memory.
// MMA order per key tile j: PV0(j) QK0(j+1) PV1(j) QK1(j+1), so the softmax of
// one tile overlaps the tensor-core work of the other.  A tcgen05.commit
// completes only when every earlier MMA of the issuing thread has completed,
// so when S(j+1) of tile w is ready, PV(j) of tile w is done and the softmax
// threads may rescale O in place.  O is rescaled only when the running row
// maximum grows by more than 2^8; the final 1/l uses the same reference
// maximum, so the result is unchanged.
//
// Every mbarrier wait is bounded (globaltimer).  A wait that runs out sets a
// CTA-wide abort flag and the device error word; all roles then leave their
// loops, the producer waits (bounded) for its copies in flight, the MMA
// thread for its MMAs, and tensor memory is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>

#include "ll_internal.h"

namespace ll {

namespace {

constexpr int BM = 128;        // query rows per tile = TMEM lanes
constexpr int BN = 128;        // keys per K/V tile
constexpr int NQ = 2;          // query tiles per CTA
constexpr int NS = 5;          // stages of the K/V tile ring
constexpr int kThreads = 384;
constexpr int kAtom = 16384;   // one 128-row x 128-byte swizzled TMA box
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kDrainNs = 200000000LL;  // 0.2 s for copies/MMAs already in flight

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;              // 64-element (128-byte) column chunks
  static constexpr int kTileBytes = BN * D * 2;       // one K or V tile
  static constexpr int kQBytes = BM * D * 2;          // one Q tile
  static constexpr int kSmemKV = NQ * kQBytes;
  static constexpr int kSmemBar = kSmemKV + NS * kTileBytes;
  static constexpr int kSmemBytes = kSmemBar + 256 + 1024;  // barriers, then alignment slack
};

struct TcParams {
  CUtensorMap tm_q, tm_kc, tm_vc, tm_kn, tm_vn;
  AttendArgs a;
  int nqb;  // query blocks of NQ * BM rows
};

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

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Ctl& c) {
  const uint64_t t0 = now_ns();
  while (true) {
    if (mbar_try(bar, parity)) return true;
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
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (mbar_try(bar, parity)) return true;
  return wait_slow(bar, parity, c);
}
// Bounded wait that ignores the abort flag (teardown of work in flight).
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = now_ns();
  while (!mbar_try(bar, parity)) {
    if ((long long)(now_ns() - t0) > kDrainNs) return;
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}
// D(tmem) (+)= A(tmem) * B(smem)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc));
}

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
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      LL_W8(0), LL_W8(8), LL_W8(16), LL_W8(24)
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
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start
// address, leading and stride byte offsets in 16-byte units, version 1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M x N, A/B major-ness.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ----------------------------------------------------------------------------
// The kernel
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(const __grid_constant__ TcParams p) {
  using Cf = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sKV = base + Cf::kSmemKV;
  const uint32_t sBar = base + Cf::kSmemBar;
  const uint32_t bQ = sBar;
  const uint32_t bKVfull0 = sBar + 8;
  const uint32_t bKVempty0 = sBar + 8 * (1 + NS);
  const uint32_t bS0 = sBar + 8 * (1 + 2 * NS);
  const uint32_t bP0 = sBar + 8 * (3 + 2 * NS);
  const uint32_t bO = sBar + 8 * (5 + 2 * NS);
  const uint32_t bDrain = sBar + 8 * (6 + 2 * NS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Cf::kSmemBar + 8 * (7 + 2 * NS));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Cf::kSmemBar + 8 * (7 + 2 * NS) + 4);

  const AttendArgs& a = p.a;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: (head, query block).  Prefill schedules the longest rows first.
  int head, qb;
  if (a.mode == 0) {
    head = blockIdx.x / p.nqb;
    qb = blockIdx.x - head * p.nqb;
  } else {
    qb = p.nqb - 1 - (int)(blockIdx.x / a.heads);
    head = blockIdx.x - (blockIdx.x / a.heads) * a.heads;
  }
  const int q0 = qb * NQ * BM;
  const int nA = (a.La + BN - 1) / BN;
  int kv_end = a.Lb;
  if (a.mode == 1) {
    const int qlast = min(q0 + NQ * BM, a.Lq) - 1;
    const long long e = ((long long)qlast / a.block_tokens + 1) * a.block_tokens;
    kv_end = (int)(e < a.Lb ? e : a.Lb);
  }
  const int nkv = nA + (kv_end + BN - 1) / BN;

  if (threadIdx.x == 0) {
    mbar_init(bQ, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bKVfull0 + 8 * s, 1);
      mbar_init(bKVempty0 + 8 * s, 1);
    }
    for (int w = 0; w < NQ; ++w) {
      mbar_init(bS0 + 8 * w, 1);
      mbar_init(bP0 + 8 * w, 128);
    }
    mbar_init(bO, 1);
    mbar_init(bDrain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, a.err, a.timeout_ns};

  int tiles_issued = 0;  // producer: K/V tiles whose copies were started

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer ------------------------------
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_q)) : "memory");
      mbar_expect_tx(bQ, NQ * Cf::kQBytes);
      for (int w = 0; w < NQ; ++w)
        for (int c = 0; c < Cf::kChunks; ++c)
          tma_load_3d(sQ + (w * Cf::kChunks + c) * kAtom, &p.tm_q, bQ, c * 64, head, q0 + w * BM);
      int u = 0;
      for (; u < 2 * nkv; ++u) {
        const int j = u >> 1;
        const bool is_v = (u & 1) != 0;
        const int s = u % NS;
        const int use = u / NS;
        if (use > 0 && !wait(bKVempty0 + 8 * s, (use - 1) & 1, ctl)) break;
        const uint32_t full = bKVfull0 + 8 * s;
        mbar_expect_tx(full, Cf::kTileBytes);
        const uint32_t dst = sKV + s * Cf::kTileBytes;
        if (j < nA) {
          const CUtensorMap* m = is_v ? &p.tm_vc : &p.tm_kc;
          for (int c = 0; c < Cf::kChunks; ++c) tma_load_3d(dst + c * kAtom, m, full, c * 64, j * BN, head);
        } else {
          const CUtensorMap* m = is_v ? &p.tm_vn : &p.tm_kn;
          for (int c = 0; c < Cf::kChunks; ++c) tma_load_3d(dst + c * kAtom, m, full, c * 64, head, (j - nA) * BN);
        }
      }
      tiles_issued = u;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------ MMA issuer --------------------------------
      constexpr uint32_t kIdQK = idesc_bf16(BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t kIdPV = idesc_bf16(BM, D, 0, 1);   // P from TMEM; V is N(=d)-major
      auto issue_qk = [&](int w, int stage) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (uint32_t)((ks >> 2) * kAtom + (ks & 3) * 32);
          const uint64_t ad = sw128_desc(sQ + w * Cf::kQBytes + off, 16, 1024);
          const uint64_t bd = sw128_desc(sKV + stage * Cf::kTileBytes + off, 16, 1024);
          mma_ss(tmem + 256 + 128 * w, ad, bd, kIdQK, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int w, int stage, bool acc) {
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t bd = sw128_desc(sKV + stage * Cf::kTileBytes + ks * 16 * 128, kAtom, 1024);
          mma_ts(tmem + 128 * w, tmem + 256 + 128 * w + ks * 8, bd, kIdPV, (acc || ks > 0) ? 1u : 0u);
        }
      };
      bool ok = wait(bQ, 0, ctl) && wait(bKVfull0, 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
        tc_commit(bS0);
        issue_qk(1, 0);
        tc_commit(bS0 + 8);
        tc_commit(bKVempty0);
        for (int j = 0; j < nkv && ok; ++j) {
          const int uv = 2 * j + 1, sv = uv % NS;
          const int uk = 2 * j + 2, sk = uk % NS;
          const bool more = j + 1 < nkv;
          if (!(ok = wait(bKVfull0 + 8 * sv, (uv / NS) & 1, ctl))) break;
          if (!(ok = wait(bP0, j & 1, ctl))) break;
          tc_fence_after();
          issue_pv(0, sv, j > 0);
          if (more) {
            if (!(ok = wait(bKVfull0 + 8 * sk, (uk / NS) & 1, ctl))) break;
            tc_fence_after();
            issue_qk(0, sk);
            tc_commit(bS0);
          }
          if (!(ok = wait(bP0 + 8, j & 1, ctl))) break;
          tc_fence_after();
          issue_pv(1, sv, j > 0);
          tc_commit(bKVempty0 + 8 * sv);
          if (more) {
            issue_qk(1, sk);
            tc_commit(bS0 + 8);
            tc_commit(bKVempty0 + 8 * sk);
          }
        }
        if (ok) tc_commit(bO);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------ softmax + epilogue ----------------------------
    const int w = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int qrow = q0 + w * BM + row;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + 256 + 128 * w;
    const uint32_t tO = tmem + lane_off + 128 * w;
    const uint32_t bS = bS0 + 8 * w;
    const uint32_t bP = bP0 + 8 * w;
    int row_end = a.Lb;
    if (a.mode == 1) {
      const long long e = ((long long)qrow / a.block_tokens + 1) * a.block_tokens;
      row_end = (int)(e < a.Lb ? e : a.Lb);
    }
    const float sl2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      ok = __all_sync(0xffffffffu, wait(bS, j & 1, ctl));
      if (!ok) break;
      tc_fence_after();
      uint32_t r[128];
      tmem_ld32(tS + 0, r + 0);
      tmem_ld32(tS + 32, r + 32);
      tmem_ld32(tS + 64, r + 64);
      tmem_ld32(tS + 96, r + 96);
      tmem_ld_wait();
      reg_fence(r, 128);
      int valid;
      if (j < nA) {
        valid = a.La - j * BN;
      } else {
        valid = (a.mode == 1 ? row_end : a.Lb) - (j - nA) * BN;
      }
      if (valid < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= valid) r[c] = __float_as_uint(-INFINITY);
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(r[i]);
#pragma unroll
      for (int c = 8; c < BN; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(r[c]));
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m, mt * sl2);
      if (j == 0) {
        m = m_new;
      } else if (__any_sync(0xffffffffu, m_new > m + kRescaleLog2)) {
        const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m - m_new);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * cc, o);
          tmem_ld_wait();
          reg_fence(o, 32);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + 32 * cc, o);
        }
        l *= alpha;
        m = m_new;
      }
      const float mo = (m == -INFINITY) ? 0.f : m;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = half * 64 + 2 * i;
          const float p0 = ex2(fmaf(__uint_as_float(r[c]), sl2, -mo));
          const float p1 = ex2(fmaf(__uint_as_float(r[c + 1]), sl2, -mo));
          ls[i & 3] += p0 + p1;
          pk[i] = pack_bf16(p0, p1);
        }
        tmem_st32(tS + 32 * half, pk);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tmem_st_wait();
      tc_fence_before();
      if (!(a.stall_inject && j == 0 && w == 0)) mbar_arrive(bP);
    }
    if (ok) ok = __all_sync(0xffffffffu, wait(bO, 0, ctl));
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t ob = ((int64_t)qrow * a.heads + head) * D;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ob;
      float* outf = static_cast<float*>(a.out) + ob;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc, o);
        tmem_ld_wait();
        reg_fence(o, 32);
        if (qrow < a.Lq && a.out_f32) {
          float4* dst = reinterpret_cast<float4*>(outf + 32 * cc);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v + 0]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                 __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
        } else if (qrow < a.Lq) {
          uint4* dst = reinterpret_cast<uint4*>(out + 32 * cc);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 x;
            x.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            x.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            x.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            x.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            dst[v] = x;
          }
        }
      }
    }
  }

  // ------------------------------ teardown ------------------------------------
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // copies still in flight land before the shared memory is released
    wait_drain(bQ, 0);
    const int first = tiles_issued > NS ? tiles_issued - NS : 0;
    for (int u = first; u < tiles_issued; ++u) wait_drain(bKVfull0 + 8 * (u % NS), (u / NS) & 1);
  }
  if (warp == 1 && lane == 0) {
    tc_commit(bDrain);
    wait_drain(bDrain, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// ----------------------------------------------------------------------------
// Host side: tensor maps and launch
// ----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool encode3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
              uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [L][H][D] token tensor, boxes of 64 d x 1 head x 128 tokens.
bool encode_tokens(CUtensorMap* m, const void* base, int L, int H, int D) {
  return encode3d(m, base, (uint64_t)D, (uint64_t)H, (uint64_t)L, (uint64_t)D * 2, (uint64_t)H * D * 2, 64, 1, 128);
}

template <int D>
cudaError_t launch_tc(const AttendArgs& a, cudaStream_t stream) {
  TcParams p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  const int La = a.La > 0 ? a.La : 1;
  if (!encode_tokens(&p.tm_q, a.q, a.Lq, a.heads, D) || !encode_tokens(&p.tm_kn, a.kn, a.Lb, a.heads, D) ||
      !encode_tokens(&p.tm_vn, a.vn, a.Lb, a.heads, D) ||
      !encode3d(&p.tm_kc, a.kc, D, (uint64_t)La, (uint64_t)a.heads, (uint64_t)D * 2,
                (uint64_t)a.cache_head_elems * 2, 64, 128, 1) ||
      !encode3d(&p.tm_vc, a.vc, D, (uint64_t)La, (uint64_t)a.heads, (uint64_t)D * 2,
                (uint64_t)a.cache_head_elems * 2, 64, 128, 1))
    return cudaErrorInvalidValue;
  p.nqb = (a.Lq + NQ * BM - 1) / (NQ * BM);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const unsigned grid = (unsigned)(p.nqb * a.heads);
  attend_tc_kernel<D><<<grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend_bf16_tc(const AttendArgs& a, cudaStream_t stream) {
  return a.head_dim == 64 ? launch_tc<64>(a, stream) : launch_tc<128>(a, stream);
}

}  // namespace ll
