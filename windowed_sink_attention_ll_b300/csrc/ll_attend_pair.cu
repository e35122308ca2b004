// Chunk attention on the 5th-generation tensor cores, CTA-pair form (head_dim
// 128): a cluster of two CTAs on two SMs shares every tcgen05.mma of a work
// item (cta_group::2, M = 256).
//
// What it computes ("LongLive: Real-time Interactive Long Video Generation",
// §3.3 Efficient Long Inference, "Short window attention" + "Frame sink"):
// for one head and one block of query rows of the current chunk,
//     O = softmax(Q K^T / sqrt(d)) V
// over the key list [resident sink + window frames of the layer's cache ||
// the chunk's own keys], walked in slot order (softmax does not depend on the
// order of the keys).  Prefill mode (§3.1 "KV recache") and mode 2 (the
// frame-causal chunk) mask the fresh keys block-causally, exactly as in the
// one-CTA kernel (ll_attend_tc.cu); both kernels follow the same work schedule
// (ll_tc_common.cuh) and write the same partial-result layout.
//
// Work item = one head x 256 query rows, taken by a CTA pair: CTA rank r holds
// query rows [128 r, 128 r + 128) of the item, the keys [64 r, 64 r + 64) of
// every 128-key K tile and the d-columns [64 r, 64 r + 64) of every V tile, so
// each SM loads half of every K/V tile.  The leader (rank 0) issues every MMA:
//   S(128 x 128 per CTA) = Q K^T   SS form, M = 256, N = 128 (keys)
//   O(128 x 128 per CTA) += P V    P from tensor memory, M = 256, N = 128 (d)
// Each CTA's tensor memory holds its O (columns [0,128)) and three S buffers
// ([128,256), [256,384), [384,512)); P (bf16) of keys 0-63 overwrites columns
// 0-31 of its S buffer, P of keys 64-127 columns 64-95.  With three S buffers Q K^T runs up to three key tiles ahead
// of the softmax: MMA order QK(0) QK(1) QK(2) PV(0) QK(3) PV(1) QK(4) ..., so
// the softmax threads find the next S ready when they finish a tile and the
// tensor core is fed while they work.
// Warp roles (384 threads per CTA):
//   warp 0      TMA producer: Q per item (two buffers), then K0 V0 K1 V1 ...
//               halves into an 8-stage ring; every copy of both CTAs completes
//               on the leader's barrier, which the leader's producer arms with
//               the bytes of both
//   warp 1      tensor-memory allocation (both CTAs); MMA issue (leader only,
//               the whole warp in step, one lane chosen by elect.sync issues)
//   warps 2-3   idle
//   warps 4-11  softmax + epilogue of this CTA's 128 rows: two warps per 32 rows,
//               warps 4-7 keys 0-63 of every tile, warps 8-11 keys 64-127
// Hand-offs: commits from the leader are multicast to both CTAs (S ready, ring
// stage free, Q buffer free, P V done, O final); each softmax warp reports "P
// stored" and "O read" on the leader's barriers (remote arrive from the peer).
// The reference max of a row moves only when the running max grows by more
// than 2^8 (then O and l are rescaled, after the P V of the previous tile has
// completed); the row sum adds the bf16-rounded P that enters P V.
//
// Every mbarrier wait is bounded (globaltimer); a wait that runs out sets the
// CTA's abort flag and the device error word, every role leaves its loop, the
// leader waits (bounded) for its copies and MMAs in flight, and both CTAs meet
// at a cluster barrier before they free tensor memory and exit.
#include "ll_tc_common.cuh"

namespace ll {

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int BM = 128;       // query rows per CTA = TMEM lanes
constexpr int BN = kKeyTile;  // keys per K/V tile (both CTAs)
constexpr int HK = BN / 2;    // keys of a K tile per CTA
constexpr int HD = D / 2;     // d-columns of a V tile per CTA
constexpr int NS = 8;         // ring stages (one K half or one V half each)
constexpr int NSB = 3;        // S buffers in tensor memory
constexpr int kThreads = 384;
constexpr int kQBytes = BM * D * 2;     // 32 KB: 128 rows x 128 d
constexpr int kStageBytes = 16384;      // K half: 64 keys x 128 d; V half: 128 keys x 64 d
constexpr int kSmemRing = 2 * kQBytes;  // two Q buffers, then the ring
constexpr int kSmemBar = kSmemRing + NS * kStageBytes;
constexpr int kSmemX = kSmemBar + 512;             // max / row-sum exchange of the softmax warp pairs
constexpr int kSmemBytes = kSmemX + 6 * BM * 4 + 1024;  // then alignment slack
static_assert(2 * BM == kItemRows, "a CTA pair takes one work item");
static_assert(HK * D * 2 == kStageBytes && BN * HD * 2 == kStageBytes, "stage size");

struct PairParams {
  CUtensorMap tm_q;   // [Lq][H][D], box 64 d x 1 head x 128 rows
  CUtensorMap tm_kc;  // cache [H][La][D], box 64 d x 64 rows
  CUtensorMap tm_vc;  // cache, box 64 d x 128 rows
  CUtensorMap tm_kn;  // chunk [Lb][H][D], box 64 d x 1 head x 64 rows
  CUtensorMap tm_vn;  // chunk, box 64 d x 1 head x 128 rows
  AttendArgs a;
  Sched s;            // workers = CTA pairs
  float* part;        // scratch: partial O [2*grid][256][D], then m and l [2*grid][256] each
};

// ----------------------------------------------------------------------------
// PTX wrappers of the pair kernel
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// arrive on an mbarrier of either CTA of the pair (shared::cluster address).  The
// default semantics (release at CTA scope) suffice: what the MMA reads after the
// barrier was written by tcgen05.st, which tcgen05.wait::st completed and
// tcgen05.fence::before_thread_sync ordered before this arrive.  A release at
// cluster scope here measured twice as slow over the whole kernel.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
// true in both warps of a softmax warp pair iff `v` is true in both (named barrier
// `id` of their 64 threads)
__device__ __forceinline__ bool pair_all(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 64, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}
// TMA tile load into this CTA's shared memory, completing on an mbarrier of either
// CTA of the pair (cbar: shared::cluster address)
__device__ __forceinline__ void tma_load_pair(uint32_t dst, const CUtensorMap* map, uint32_t cbar, int c0, int c1,
                                              int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cbar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// commit of the pair's MMAs issued so far by this thread, arriving on the barrier at
// offset `bar` of every CTA in `mask`; one elected lane of a converged warp
__device__ __forceinline__ void commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
          bar),
      "h"(mask)
      : "memory");
}
// Eight k-steps of S (+)= Q K^T, M = 256 across the pair, from one asm block.
__device__ __forceinline__ void mma8_ss2(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p0, 0, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %2, %10, %1, p0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %3, %11, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %4, %12, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %5, %13, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %6, %14, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %7, %15, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %8, %16, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %9, %17, %1, p1;\n\t}" ::"r"(d),
      "r"(idesc), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]),
      "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]));
}
// Four k-steps of O (+)= P V, P from tensor memory (columns a, a+8, a+16, a+24).
__device__ __forceinline__ void mma4_ts2(uint32_t d, uint32_t a, const uint64_t (&b)[4], uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\t.reg .b32 t;\n\telect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %7, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%2], %3, %1, p0;\n\t"
      "add.u32 t, %2, 8;\n\t@e tcgen05.mma.cta_group::2.kind::f16 [%0], [t], %4, %1, p1;\n\t"
      "add.u32 t, %2, 16;\n\t@e tcgen05.mma.cta_group::2.kind::f16 [%0], [t], %5, %1, p1;\n\t"
      "add.u32 t, %2, 24;\n\t@e tcgen05.mma.cta_group::2.kind::f16 [%0], [t], %6, %1, p1;\n\t}" ::"r"(d),
      "r"(idesc), "r"(a), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc));
}

// ----------------------------------------------------------------------------
// The kernel
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) attend_pair_kernel(const __grid_constant__ PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;               // two Q buffers of kQBytes
  const uint32_t sKV = base + kSmemRing;  // NS stages of kStageBytes
  const uint32_t sBar = base + kSmemBar;
  const uint32_t bQfull0 = sBar;             // [2]  Q buffer landed (leader; both CTAs' bytes)
  const uint32_t bQempty0 = bQfull0 + 16;    // [2]  Q buffer free (multicast commit)
  const uint32_t bKVfull0 = bQempty0 + 16;   // [NS] stage landed (leader; both CTAs' bytes)
  const uint32_t bKVempty0 = bKVfull0 + 8 * NS;  // [NS] stage free (multicast commit)
  const uint32_t bS0 = bKVempty0 + 8 * NS;   // [3]  S buffer ready (multicast commit)
  const uint32_t bPlo0 = bS0 + 8 * NSB;      // [3]  P of keys 0-63 stored (leader; 4 warps per CTA)
  const uint32_t bPhi0 = bPlo0 + 8 * NSB;    // [3]  P of keys 64-127 stored (leader; 4 warps per CTA)
  const uint32_t bOdone0 = bPhi0 + 8 * NSB;  // [2]  P V of tile g done, by g's parity (multicast commit)
  const uint32_t bOfull = bOdone0 + 16;      // last P V of a piece done (multicast commit)
  const uint32_t bOempty = bOfull + 8;       // O read by the epilogue (leader; 8 warps per CTA)
  const uint32_t bDrain = bOempty + 8;       // leader's MMAs drained at teardown
  constexpr int kBarBytes = 16 + 16 + 16 * NS + 24 * NSB + 16 + 24;
  static_assert(kBarBytes + 8 <= 512, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kSmemBar + kBarBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kSmemBar + kBarBytes + 4);

  const AttendArgs& a = p.a;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int worker = (int)cluster_id();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bQfull0 + 8 * b, 1);
      mbar_init(bQempty0 + 8 * b, 1);
      mbar_init(bOdone0 + 8 * b, 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(bKVfull0 + 8 * s, 1);
      mbar_init(bKVempty0 + 8 * s, 1);
    }
    for (int b = 0; b < NSB; ++b) {
      mbar_init(bS0 + 8 * b, 1);
      mbar_init(bPlo0 + 8 * b, 8);
      mbar_init(bPhi0 + 8 * b, 8);
    }
    mbar_init(bOfull, 1);
    mbar_init(bOempty, 16);
    mbar_init(bDrain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  // both CTAs' barriers are initialised before any copy, commit or arrive reaches them
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, a.err, a.timeout_ns};

  int tiles_issued = 0;  // producer: ring uses started
  int q_issued = 0;      // producer: Q loads started

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer ------------------------------
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_q)) : "memory");
      Walker wk;
      walker_init(wk, a, p.s, worker);
      Piece pc;
      int u = 0;
      bool ok = true;
      while (ok && walker_next(wk, a, p.s, pc, worker)) {
        int head, q0, nA;
        item_geom(a, p.s, pc.item, head, q0, nA);
        const int qb = q_issued & 1;
        // the Q K^T products of the piece before last are done with this Q buffer
        if (q_issued >= 2 && !(ok = wait(bQempty0 + 8 * qb, ((q_issued >> 1) - 1) & 1, ctl))) break;
        const uint32_t qfull = bQfull0 + 8 * qb;
        if (leader) mbar_expect_tx(qfull, 2 * kQBytes);
        const uint32_t cq = peer_addr(qfull, 0);
        for (int c = 0; c < D / 64; ++c)
          tma_load_pair(sQ + qb * kQBytes + c * kAtom, &p.tm_q, cq, c * 64, head, q0 + (int)rank * BM);
        ++q_issued;
        for (int j = pc.j0; ok && j < pc.j1; ++j) {
          for (int is_v = 0; is_v < 2; ++is_v) {
            const int s = u % NS;
            const int use = u / NS;
            if (use > 0 && !(ok = wait(bKVempty0 + 8 * s, (use - 1) & 1, ctl))) break;
            const uint32_t full = bKVfull0 + 8 * s;
            if (leader) mbar_expect_tx(full, 2 * kStageBytes);
            const uint32_t cf = peer_addr(full, 0);
            const uint32_t dst = sKV + s * kStageBytes;
            if (!is_v) {
              // keys [64 rank, 64 rank + 64) of the tile, all d: two 64 x 64 boxes
              if (j < nA) {
                for (int c = 0; c < D / 64; ++c)
                  tma_load_pair(dst + c * (HK * 128), &p.tm_kc, cf, c * 64, j * BN + (int)rank * HK, head);
              } else {
                for (int c = 0; c < D / 64; ++c)
                  tma_load_pair(dst + c * (HK * 128), &p.tm_kn, cf, c * 64, head, (j - nA) * BN + (int)rank * HK);
              }
            } else {
              // all 128 keys of the tile, d-columns [64 rank, 64 rank + 64): one box
              if (j < nA)
                tma_load_pair(dst, &p.tm_vc, cf, (int)rank * HD, j * BN, head);
              else
                tma_load_pair(dst, &p.tm_vn, cf, (int)rank * HD, head, (j - nA) * BN);
            }
            tiles_issued = ++u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ------------------------------ MMA issuer (leader, whole warp) ----------
      constexpr uint32_t kIdQK = idesc_bf16(2 * BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t kIdPV = idesc_bf16(2 * BM, D, 0, 1);   // P from TMEM; V is N(=d)-major
      // Q descriptors of both buffers; K and V descriptors differ from the ring's
      // first stage only in the start address field (16-byte units; shared
      // offsets stay below 256 KB, so no carry reaches the high word)
      uint64_t dq[2][D / 16];
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          dq[b][ks] = sw128_desc(sQ + b * kQBytes + (ks >> 2) * kAtom + (ks & 3) * 32, 16, 1024);
      const uint64_t dK0 = sw128_desc(sKV, 16, 1024);
      const uint64_t dV0 = sw128_desc(sKV, kAtom, 1024);
      const uint32_t k_lo0 = (uint32_t)dK0, k_hi = (uint32_t)(dK0 >> 32);
      const uint32_t v_lo0 = (uint32_t)dV0, v_hi = (uint32_t)(dV0 >> 32);
      auto issue_qk = [&](int qb, int stage, int sb) {
        const uint32_t lo = k_lo0 + (((uint32_t)stage * kStageBytes) >> 4);
        uint64_t bd[D / 16];
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) bd[ks] = make_desc(lo + ((ks >> 2) * (HK * 128) + (ks & 3) * 32) / 16, k_hi);
        if (qb == 0)
          mma8_ss2(tmem + 128 + 128 * sb, dq[0], bd, kIdQK);
        else
          mma8_ss2(tmem + 128 + 128 * sb, dq[1], bd, kIdQK);
      };
      // P V in two groups of four k-steps: keys 0-63, then keys 64-127
      auto issue_pv = [&](int stage, int sb, int half, bool acc) {
        const uint32_t lo = v_lo0 + (((uint32_t)stage * kStageBytes) >> 4);
        uint64_t bd[4];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) bd[ks] = make_desc(lo + ((half * 4 + ks) * 16 * 128) / 16, v_hi);
        mma4_ts2(tmem, tmem + 128 + 128 * sb + 64 * half, bd, kIdPV, acc ? 1u : 0u);
      };
      Walker wk;
      walker_init(wk, a, p.s, worker);
      Piece pc;
      int u = 0, qi = 0, g = 0;
      bool ok = true;
      // Q K^T of tile t of the current piece (ring use u + 2t) into S buffer (g + t) % 3
      auto qk = [&](int t, int n, int qb) -> bool {
        const int uk = u + 2 * t, sk = uk % NS;
        if (!__all_sync(0xffffffffu, wait(bKVfull0 + 8 * sk, (uk / NS) & 1, ctl))) return false;
        tc_fence_after();
        issue_qk(qb, sk, (g + t) % NSB);
        commit_mc(bS0 + 8 * ((g + t) % NSB), 3);
        commit_mc(bKVempty0 + 8 * sk, 3);
        if (t == n - 1) commit_mc(bQempty0 + 8 * qb, 3);
        return true;
      };
      while (ok && walker_next(wk, a, p.s, pc, worker)) {
        const int n = pc.j1 - pc.j0;
        const int qb = qi & 1;
        if (!(ok = __all_sync(0xffffffffu, wait(bQfull0 + 8 * qb, (qi >> 1) & 1, ctl)))) break;
        for (int t = 0; ok && t < n && t < NSB; ++t) ok = qk(t, n, qb);
        for (int t = 0; ok && t < n; ++t) {
          const int gg = g + t, sb = gg % NSB, ph = (gg / NSB) & 1;
          const int uv = u + 2 * t + 1, sv = uv % NS;
          if (!(ok = __all_sync(0xffffffffu, wait(bKVfull0 + 8 * sv, (uv / NS) & 1, ctl)))) break;
          if (!(ok = __all_sync(0xffffffffu, wait(bPlo0 + 8 * sb, ph, ctl)))) break;
          // the previous piece's epilogue must have read O out of tensor memory
          if (t == 0 && qi > 0 && !(ok = __all_sync(0xffffffffu, wait(bOempty, (qi - 1) & 1, ctl)))) break;
          tc_fence_after();
          issue_pv(sv, sb, 0, t > 0);
          if (!(ok = __all_sync(0xffffffffu, wait(bPhi0 + 8 * sb, ph, ctl)))) break;
          tc_fence_after();
          issue_pv(sv, sb, 1, true);
          commit_mc(bOdone0 + 8 * (gg & 1), 3);
          commit_mc(bKVempty0 + 8 * sv, 3);
          if (t + NSB < n) ok = qk(t + NSB, n, qb);
        }
        if (!ok) break;
        commit_mc(bOfull, 3);
        u += 2 * n;
        g += n;
        ++qi;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------ softmax + epilogue ----------------------------
    // Two warps per 32 rows: `half` 0 takes keys 0-63 of every tile and O columns
    // 0-63, half 1 keys 64-127 and O columns 64-127.  Both hold the same
    // reference max per row: a per-tile barrier reduction tells both whether any
    // row must move it, and the maxima are exchanged through shared memory only
    // then and at an item's first tile; the row sums are combined at the end of
    // the item.  Each half writes its P over its own S columns (keys 0-63 at
    // columns 0-31, keys 64-127 at columns 64-95), so neither overwrites scores
    // the other has not read yet.
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tO = tmem + lane_off + 64 * half;
    const uint32_t cP0 = peer_addr(half ? bPhi0 : bPlo0, 0), cOempty = peer_addr(bOempty, 0);
    const int pair_bar = 1 + quad;  // named barrier of the two warps of these rows
    const float sl2 = a.scale_log2;
    Walker wk;
    walker_init(wk, a, p.s, worker);
    Piece pc;
    int qi = 0, g = 0, xc = 0;  // xc: max exchanges so far (selects the exchange slot)
    bool ok = true;
    while (ok && walker_next(wk, a, p.s, pc, worker)) {
      int head, q0, nA;
      item_geom(a, p.s, pc.item, head, q0, nA);
      const int qrow = q0 + (int)rank * BM + row;
      int row_end = a.Lb;
      if (a.mode != 0) {
        const long long e = ((long long)qrow / a.block_tokens + 1) * a.block_tokens;
        row_end = (int)(e < a.Lb ? e : a.Lb);
      }
      const int n = pc.j1 - pc.j0;
      float m = -INFINITY, l = 0.f;
      for (int t = 0; t < n; ++t) {
        const int j = pc.j0 + t;
        const int gg = g + t, sb = gg % NSB;
        const uint32_t tS = tmem + lane_off + 128 + 128 * sb + 64 * half;
        const bool got_s = __all_sync(0xffffffffu, wait(bS0 + 8 * sb, (gg / NSB) & 1, ctl));
        uint32_t r[HK];
        float mt = -INFINITY;
        bool grew = false;
        if (got_s) {
          tc_fence_after();
          // S of this half: both loads in flight, one wait
          tmem_ld32(tS + 0, r + 0);
          tmem_ld32(tS + 32, r + 32);
          tmem_ld_wait();
          reg_fence(r, HK);
          const int valid = (j < nA ? a.La - j * BN : (a.mode != 0 ? row_end : a.Lb) - (j - nA) * BN) - HK * half;
          if (valid < HK) {
#pragma unroll
            for (int c = 0; c < HK; ++c)
              if (c >= valid) r[c] = __float_as_uint(-INFINITY);
          }
          float mx[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = __uint_as_float(r[i]);
#pragma unroll
          for (int c = 4; c < HK; c += 2)
            mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
          mt = max3f(max3f(mx[0], mx[1], mx[2]), mx[3], -INFINITY) * sl2;
          grew = __any_sync(0xffffffffu, t > 0 && mt > m + kRescaleLog2);
        }
        // One barrier reduction over the two warps of these rows tells both (a) whether
        // either gave up waiting (lane 0 of each warp votes), so that they leave
        // together and never wait for each other at a later barrier, and (b) whether
        // any row grew by more than 2^8, so that both move the reference max and
        // rescale O (lanes 1-31 vote): count = gave_up + 31 * grew.
        uint32_t cnt;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.popc.u32 %0, %2, 64, p;\n\t}"
            : "=r"(cnt)
            : "r"((uint32_t)(lane == 0 ? !got_s : grew)), "r"(pair_bar)
            : "memory");
        if (cnt % 31 != 0) {
          ok = false;
          break;
        }
        const bool rescale = cnt != 0;
        float alpha = 1.f;
        if (t == 0 || rescale) {
          float* xm = reinterpret_cast<float*>(gbase + kSmemX) + (xc & 1) * 2 * BM;
          xm[half * BM + row] = mt;
          asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
          const float m_new = fmaxf(fmaxf(m, mt), xm[(1 - half) * BM + row]);
          ++xc;
          if (rescale && m_new != -INFINITY) alpha = ex2(m - m_new);
          l *= alpha;
          m = m_new;
        }
        const float mo = (m == -INFINITY) ? 0.f : m;
        // P = 2^(s*log2e/sqrt(d) - m), rounded to bf16 for the P V product; the row
        // sum adds the same rounded values
        const uint64_t sl2x2 = pack_f32x2(sl2, sl2), nmo2 = pack_f32x2(-mo, -mo);
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int gq = 0; gq < HK / 32; ++gq) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = gq * 32 + 2 * i;
            float x0, x1;
            fma_f32x2(x0, x1, __uint_as_float(r[c]), __uint_as_float(r[c + 1]), sl2x2, nmo2);
            pk[i] = pack_bf16(ex2(x0), ex2(x1));
            add_bf16x2(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], pk[i]);
          }
          tmem_st16(tS + 16 * gq, pk);
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        if (rescale) {
          // P V of the previous tile must be complete before O is rescaled in place
          // (both warps agree on the outcome before either goes on)
          ok = pair_all(pair_bar, __all_sync(0xffffffffu, wait(bOdone0 + 8 * ((gg - 1) & 1), ((gg - 1) >> 1) & 1,
                                                                ctl)));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < HD / 16; ++cc) {
            uint32_t o[16];
            tmem_ld16(tO + 16 * cc, o);
            tmem_ld_wait();
            reg_fence(o, 16);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(tO + 16 * cc, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !(a.stall_inject && leader && gg == 0 && quad == 0 && half == 0))
          mbar_arrive_cluster(cP0 + 8 * sb);
      }
      if (!ok) break;
      // the row sum over both halves
      float* xl = reinterpret_cast<float*>(gbase + kSmemX) + 4 * BM;
      xl[half * BM + row] = l;
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      const float lsum = l + xl[(1 - half) * BM + row];
      ok = pair_all(pair_bar, __all_sync(0xffffffffu, wait(bOfull, qi & 1, ctl)));
      if (!ok) break;
      tc_fence_after();
      if (pc.partial) {
        // unnormalised O with its reference max and sum, merged by combine_kernel
        const size_t rows_all = (size_t)2 * p.s.grid * kItemRows;
        const size_t sr = (size_t)pc.slot * kItemRows + rank * BM + row;
        float* po = p.part + sr * D + HD * half;
#pragma unroll 1
        for (int cc = 0; cc < HD / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * cc, o);
          tmem_ld_wait();
          reg_fence(o, 32);
          float4* dst = reinterpret_cast<float4*>(po + 32 * cc);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v + 0]), __uint_as_float(o[4 * v + 1]),
                                 __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
        }
        if (half == 0) {
          p.part[rows_all * D + sr] = m;
          p.part[rows_all * D + rows_all + sr] = lsum;
        }
      } else {
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const int64_t ob = ((int64_t)qrow * a.heads + head) * D + HD * half;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ob;
        float* outf = static_cast<float*>(a.out) + ob;
#pragma unroll 1
        for (int cc = 0; cc < HD / 32; ++cc) {
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cOempty);
      g += n;
      ++qi;
    }
  }

  // ------------------------------ teardown ------------------------------------
  // this CTA's work is issued: the launch that follows may be scheduled; it
  // waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  if (warp == 0 && lane == 0) {
    if (leader) {
      // copies of both CTAs still in flight land before shared memory is released
      // (each completes on one of the leader's barriers)
      if (q_issued > 0) wait_drain(bQfull0 + 8 * ((q_issued - 1) & 1), ((q_issued - 1) >> 1) & 1);
      const int first = tiles_issued > NS ? tiles_issued - NS : 0;
      for (int u = first; u < tiles_issued; ++u) wait_drain(bKVfull0 + 8 * (u % NS), (u / NS) & 1);
    } else if (*abort_flag) {
      // the peer cannot see its copies complete; they were issued long before a
      // wait ran out, but give any still in flight a moment to land
      const uint64_t t0 = now_ns();
      while ((long long)(now_ns() - t0) < 100000LL) {
      }
    }
  }
  if (warp == 1 && leader) {
    // a commit tracks the MMAs of its own thread: the lane elect.sync picks,
    // as for every MMA and commit of the issue loop
    commit_mc(bDrain, 1);
    wait_drain(bDrain, 0);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's MMAs no longer touch either CTA's memory
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
// CTA pairs that fit on the device at once (one pair per two SMs at most)
int pair_workers(int smem_bytes) {
  static std::atomic<int> cached[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_acquire);
    if (c > 0) return c;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (unsigned)(sm_count() / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attend_pair_kernel, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sm_count() / 2;
  }
  if (n > sm_count() / 2) n = sm_count() / 2;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_release);
  return n;
}

}  // namespace

cudaError_t launch_attend_bf16_pair(const AttendArgs& a, cudaStream_t stream) {
  if (a.head_dim != D) return cudaErrorInvalidValue;
  PairParams p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  if (!encode_tokens(&p.tm_q, a.q, a.Lq, a.heads, D, BM) || !encode_tokens(&p.tm_kn, a.kn, a.Lb, a.heads, D, HK) ||
      !encode_tokens(&p.tm_vn, a.vn, a.Lb, a.heads, D, BN) ||
      !encode_cache(&p.tm_kc, a.kc, a.La, a.heads, D, a.cache_head_elems, HK) ||
      !encode_cache(&p.tm_vc, a.vc, a.La, a.heads, D, a.cache_head_elems, BN))
    return cudaErrorInvalidValue;
  static std::atomic<int> attr_done[64];
  if (cudaError_t e = smem_opt_in(attend_pair_kernel, kSmemBytes, attr_done)) return e;
  const int workers = pair_workers(kSmemBytes);
  p.s.nqb = (a.Lq + kItemRows - 1) / kItemRows;
  CombineParams cp;
  cp.nsplit = 0;
  if (a.mode == 1) {
    // persistent: one pair per two SMs, items in zigzag rounds (see walker_next)
    const int items = p.s.nqb * a.heads;
    p.s.grid = items < workers ? items : workers;
  } else {
    // without scratch for two partial results per pair, no item is split
    int w = workers;
    if (2 * w > a.scratch_slots) w = a.scratch_slots / 2;
    plan_attend(a, p.s, cp, w < 1 ? 1 : w);
    if (cp.nsplit > 0 && !a.scratch) return cudaErrorInvalidValue;
    p.part = a.scratch;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (unsigned)p.s.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attend_pair_kernel, p);
  count_launch();
  if (e != cudaSuccess || cp.nsplit == 0) return e;
  return launch_combine<D>(cp, a, p.s, p.part, stream);
}

}  // namespace ll
