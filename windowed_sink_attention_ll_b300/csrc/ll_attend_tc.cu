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
// (§3.1 "KV recache") query row i sees every cached key (the sink rows of a
// keep-sink prefill; none otherwise) and fresh key j iff
// j / block_tokens <= i / block_tokens.  Mode 2 keeps the attend schedule and
// every cached key, and masks the chunk's own keys the same block-causal way
// (the frame-causal chunk).
//
// This is the one-CTA form of the kernel, the one every bf16 attention runs on
// (as do the e4m3 caches, and fp32 attention at head_dim 64 with tf32
// operands); ll_attend_pair.cu holds a CTA-pair form for bf16 at head_dim 128
// (selected on request).
// Work item = one head x 256 query rows (two 128-row tiles that share every
// K/V tile); one CTA per SM walks several items (see "Work schedule" in
// ll_tc_common.cuh):
// attend launches run whole rounds of items, then split the left-over items
// into runs of key tiles merged by combine_kernel; prefill launches hand out
// their unequal items longest first in zigzag rounds.  Warp roles (384 threads):
//   warp 0      TMA producer: Q per item, then K0 V0 K1 V1 ... into a ring of 5
//               stages (3 with fp32 operands, 8 with e4m3 keys and values)
//   warp 1      TMEM allocator and MMA issuer: the whole warp runs the issue
//               loop in step (every wait is a warp vote), and one lane chosen
//               by elect.sync issues each tcgen05.mma and tcgen05.commit; the
//               eight k-steps of a Q K^T product go out from one asm block, a
//               P V product from two blocks of four (one per key half), with
//               every descriptor ready in registers
//   warps 4-7   softmax for Q tile 0, warps 8-11 for Q tile 1: thread = row
//   warps 2-3   fp32 operands: split each K tile into its tf32 part and the
//               tf32 rounding of the remainder, and transpose each V tile
//               into the K-major layout that P V reads (tf32 operands are
//               taken K-major here); e4m3 values: widen each V tile to fp16
//               (exact) for P V; idle otherwise
// Tensor memory (512 columns x 128 lanes): O0 [0,128) O1 [128,256)
// S0 [256,384) S1 [384,512).  P (bf16; fp16 with e4m3 values) overwrites the
// first 64 columns of S (fp32 operands: P rounded to tf32 overwrites all 128)
// and feeds the P V product straight from tensor memory.
// fp32 operands (head_dim 64): Q K^T is kept accurate to fp32 by splitting
// each operand x into hi = tf32(x) and lo = tf32(x - hi) and summing three
// tf32 products, S = Qhi Khi^T + Qlo Khi^T + Qhi Klo^T (the split-operand
// "3xTF32" method; the dropped Qlo Klo^T is below 2^-22 of each product).  The
// softmax threads split their Q rows (hi in place in shared memory, lo into
// the unused columns [64,128) of their tile's O region, read by the MMA as A);
// warps 2-3 split each K tile (hi in place, lo into a separate buffer).  P V
// reads V rounded to tf32 and P rounded to tf32.
// e4m3 keys and values: Q K^T on kind::f8f6f4; V tiles arrive as e4m3 bytes
// and are widened to fp16 into one of two buffers; P is packed to fp16 and
// P V runs on kind::f16 with fp16 A and B.
// MMA order per key tile j: PV0(j) QK0(j+1) PV1(j) QK1(j+1), so the softmax of
// one tile overlaps the tensor-core work of the other.  P of a tile is handed
// over in two halves: once the P of keys 0-63 is in tensor memory the softmax
// threads signal it and the tensor core starts P V on those four k-steps while
// the exponentials of keys 64-127 run (a tile whose O must be rescaled signals
// both halves at the end, after the rescale).  A tcgen05.commit
// completes only when every earlier MMA issued from the warp has completed,
// so when S(j+1) of tile w is ready, PV(j) of tile w is done and the softmax
// threads may rescale O in place.  The reference max of a row moves only when
// the running max grows by more than 2^8 (then O and l are rescaled); every
// P, the row sum l and the final 1/l use that same reference, so the result
// is unchanged.  The row sum adds the rounded P (bf16, fp16 or tf32) that
// enters P V.

// Every mbarrier wait is bounded (globaltimer).  A wait that runs out sets a
// CTA-wide abort flag and the device error word; all roles then leave their
// loops, the producer waits (bounded) for its copies in flight, the MMA
// warp for its MMAs, and tensor memory is freed before the CTA exits.
#include "ll_tc_common.cuh"

namespace ll {

namespace {

using namespace tc;

constexpr int BM = 128;        // query rows per tile = TMEM lanes
constexpr int BN = kKeyTile;   // keys per K/V tile
constexpr int NQ = 2;          // query tiles per CTA
constexpr int kThreads = 384;
static_assert(NQ * BM == kItemRows, "a CTA takes one work item");

// Operand kinds: bf16 Q, K, V (kind::f16); e4m3 Q and K with bf16 V (Q K^T on
// kind::f8f6f4); fp32 Q, K, V read by the tensor core as tf32 (kind::tf32);
// e4m3 Q, K and V (Q K^T on kind::f8f6f4, P V on kind::f16 with fp16 P and V).
enum Kind : int { kBf16 = 0, kE4m3 = 1, kTf32 = 2, kE4m3KV = 3 };

template <int D, int KIND>
struct Cfg {
  static constexpr bool kQK8 = KIND == kE4m3 || KIND == kE4m3KV;              // Q K^T on kind::f8f6f4
  static constexpr int kQKElem = kQK8 ? 1 : KIND == kTf32 ? 4 : 2;            // bytes per Q / K element
  static constexpr int kVElem = KIND == kTf32 ? 4 : KIND == kE4m3KV ? 1 : 2;  // bytes per V element
  static constexpr int kQKChunks = D * kQKElem / 128;       // 128-byte column chunks of Q and K
  static constexpr int kQKBox = 128 / kQKElem;              // elements per such chunk
  static constexpr int kVChunks = D * kVElem / 128;         // 128-byte column chunks of V
  static constexpr int kVBox = 128 / kVElem;
  static constexpr int kKSteps = D * kQKElem / 32;          // 32-byte k-steps of one Q K^T product
  static constexpr int kKBytes = BN * D * kQKElem;          // one K tile
  static constexpr int kVBytes = BN * D * kVElem;           // one V tile
  static constexpr int kTileBytes = kVBytes;                // one ring stage (K or V)
  static constexpr int kQBytes = BM * D * kQKElem;          // one Q tile
  static constexpr int kNS = KIND == kTf32 ? 3 : KIND == kE4m3KV ? 8 : 5;  // stages of the K/V tile ring
  static constexpr int kVTBytes = KIND == kTf32 ? kVBytes : 0;  // one V tile transposed (tf32)
  static constexpr int kKLBytes = KIND == kTf32 ? kKBytes : 0;  // low parts of one K tile (tf32)
  static constexpr int kV16Tile = BN * D * 2;                   // one V tile widened to fp16 (e4m3 V)
  static constexpr int kV16Bytes = KIND == kE4m3KV ? 2 * kV16Tile : 0;
  static constexpr int kSmemKV = NQ * kQBytes;
  static constexpr int kSmemVT = kSmemKV + kNS * kTileBytes;
  static constexpr int kSmemKL = kSmemVT + kVTBytes;
  static constexpr int kSmemV16 = kSmemKL + kKLBytes;
  static constexpr int kSmemBar = kSmemV16 + kV16Bytes;
  static constexpr int kSmemBytes = kSmemBar + 512 + 1024;  // barriers, then alignment slack
  static_assert(KIND != kTf32 || D == 64, "fp32 tiles fit the shared memory at head_dim 64 only");
  static_assert(!kQK8 || D == 128, "e4m3 Q K^T: one 128-byte chunk per row");
  static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
};

struct TcParams {
  CUtensorMap tm_q, tm_kc, tm_vc, tm_kn, tm_vn;
  AttendArgs a;
  Sched s;
  float* part;  // scratch: partial O [2*grid][NQ*BM][D], then m and l [2*grid][NQ*BM] each
};

// ----------------------------------------------------------------------------
// PTX wrappers of the one-CTA kernel
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// commit from one elected lane of a converged warp
__device__ __forceinline__ void tc_commit_e(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}
// Eight (or four) MMAs of one group from a single asm block, issued by the lane
// that elect.sync picks (the whole warp executes the block; operands are the
// same in every lane): k-step 0 accumulates when acc != 0, the others always.
// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma8_ss(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p0, %18, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %1, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %17, %1, p1;\n\t}" ::"r"(d),
      "r"(idesc), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]),
      "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(acc));
}
// Four k-steps of kind::f8f6f4 (e4m3 A and B, 32 elements per k-step), S = Q K^T.
__device__ __forceinline__ void mma4_ss_f8(uint32_t d, const uint64_t (&a)[4], const uint64_t (&b)[4],
                                           uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p0, 0, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %2, %6, %1, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %7, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %4, %8, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %5, %9, %1, p1;\n\t}" ::"r"(d),
      "r"(idesc), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]));
}
__device__ __forceinline__ void mma4_ss(uint32_t d, const uint64_t (&a)[4], const uint64_t (&b)[4], uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p0, %10, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %1, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %9, %1, p1;\n\t}" ::"r"(d),
      "r"(idesc), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc));
}

// Eight k-steps of kind::tf32 (8 fp32 elements per k-step), D (+)= A(smem) * B(smem);
// k-step 0 accumulates when acc != 0.
__device__ __forceinline__ void mma8_ss_tf32(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8],
                                             uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p0, %18, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %2, %10, %1, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %3, %11, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %4, %12, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %5, %13, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %6, %14, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %7, %15, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %8, %16, %1, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %9, %17, %1, p1;\n\t}" ::"r"(d),
      "r"(idesc), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]),
      "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(acc));
}
// D(tmem) (+)= A(tmem: 8 k-steps of 8 tf32 columns from column a) * B(smem), kind::tf32
__device__ __forceinline__ void mma8_ts_tf32(uint32_t d, uint32_t a, const uint64_t (&b)[8], uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\t.reg .b32 t;\n\telect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %11, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%2], %3, %1, p0;\n\t"
      "add.u32 t, %2, 8;\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [t], %4, %1, p1;\n\t"
      "add.u32 t, %2, 16;\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [t], %5, %1, p1;\n\t"
      "add.u32 t, %2, 24;\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [t], %6, %1, p1;\n\t"
      "add.u32 t, %2, 32;\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [t], %7, %1, p1;\n\t"
      "add.u32 t, %2, 40;\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [t], %8, %1, p1;\n\t"
      "add.u32 t, %2, 48;\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [t], %9, %1, p1;\n\t"
      "add.u32 t, %2, 56;\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [t], %10, %1, p1;\n\t}" ::"r"(d),
      "r"(idesc), "r"(a), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
      "r"(acc));
}
// fp32 -> tf32, round to nearest (ties away from zero); the low 13 bits come out zero
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// x = hi + lo + (below 2^-22 |x|): hi = tf32(x), lo = tf32(x - hi) (x - hi is exact in fp32)
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = __uint_as_float(to_tf32(x));
  lo = __uint_as_float(to_tf32(x - hi));
}

// D(tmem) (+)= A(tmem: 4 k-steps of 8 columns from column a) * B(smem), elected lane
__device__ __forceinline__ void mma4_ts(uint32_t d, uint32_t a, const uint64_t (&b)[4], uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\t.reg .b32 t;\n\telect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %7, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %3, %1, p0;\n\t"
      "add.u32 t, %2, 8;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], %4, %1, p1;\n\t"
      "add.u32 t, %2, 16;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], %5, %1, p1;\n\t"
      "add.u32 t, %2, 24;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], %6, %1, p1;\n\t}" ::"r"(d),
      "r"(idesc), "r"(a), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc));
}

// ----------------------------------------------------------------------------
// The kernel
// ----------------------------------------------------------------------------
template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(const __grid_constant__ TcParams p) {
  using Cf = Cfg<D, KIND>;
  constexpr int NS = Cf::kNS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sKV = base + Cf::kSmemKV;
  const uint32_t sVT = base + Cf::kSmemVT;  // fp32 operands: the V tile P V reads, K-major
  const uint32_t sKL = base + Cf::kSmemKL;  // fp32 operands: low parts of the K tile
  const uint32_t sV16 = base + Cf::kSmemV16;  // e4m3 V: two V tiles widened to fp16
  const uint32_t sBar = base + Cf::kSmemBar;
  const uint32_t bQfull = sBar;
  const uint32_t bQempty = sBar + 8;
  const uint32_t bKVfull0 = sBar + 16;
  const uint32_t bKVempty0 = bKVfull0 + 8 * NS;
  const uint32_t bS0 = bKVempty0 + 8 * NS;
  const uint32_t bP0 = bS0 + 16;
  const uint32_t bOfull = bP0 + 32;  // bP0: P of keys 0-63 of tile w at +8w, of keys 64-127 at +16+8w
  const uint32_t bOempty = bOfull + 8;
  const uint32_t bDrain = bOempty + 8;
  const uint32_t bVTfull = bDrain + 8;    // fp32 operands: V tile transposed
  const uint32_t bVTempty = bDrain + 16;  // fp32 operands: P V of both query tiles done with it
  const uint32_t bKsplit = bDrain + 24;   // fp32 operands: K tile split (hi in place, lo in sKL)
  const uint32_t bKLempty = bDrain + 32;  // fp32 operands: Q K^T of both query tiles done with sKL
  const uint32_t bQsplit = bDrain + 40;   // fp32 operands: both Q tiles split
  const uint32_t bWfull0 = bDrain + 48;   // e4m3 V: fp16 buffer b (at +8b) filled
  const uint32_t bWempty0 = bDrain + 64;  // e4m3 V: P V of both query tiles done with buffer b
  constexpr int kBarBytes = 16 + 16 * NS + 16 + 32 + 24 + 40 + 32;
  static_assert(kBarBytes + 8 <= 512, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Cf::kSmemBar + kBarBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Cf::kSmemBar + kBarBytes + 4);

  const AttendArgs& a = p.a;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bQfull, 1);
    mbar_init(bQempty, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bKVfull0 + 8 * s, 1);
      mbar_init(bKVempty0 + 8 * s, 1);
    }
    for (int w = 0; w < NQ; ++w) {
      mbar_init(bS0 + 8 * w, 1);
      mbar_init(bP0 + 8 * w, 128);
      mbar_init(bP0 + 16 + 8 * w, 128);
    }
    mbar_init(bOfull, 1);
    mbar_init(bOempty, NQ * 128);
    mbar_init(bDrain, 1);
    mbar_init(bVTfull, 64);
    mbar_init(bVTempty, 1);
    mbar_init(bKsplit, 64);
    mbar_init(bKLempty, 1);
    mbar_init(bQsplit, NQ * 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bWfull0 + 8 * b, 64);
      mbar_init(bWempty0 + 8 * b, 1);
    }
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
  int q_issued = 0;      // producer: Q loads started

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer ------------------------------
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tm_q)) : "memory");
      Walker wk;
      walker_init(wk, p.a, p.s, blockIdx.x);
      Piece pc;
      int u = 0;
      bool ok = true;
      while (ok && walker_next(wk, p.a, p.s, pc, blockIdx.x)) {
        int head, q0, nA;
        item_geom(p.a, p.s, pc.item, head, q0, nA);
        // the previous item's Q K^T products must be done with the Q tiles
        if (q_issued > 0 && !(ok = wait(bQempty, (q_issued - 1) & 1, ctl))) break;
        mbar_expect_tx(bQfull, NQ * Cf::kQBytes);
        for (int w = 0; w < NQ; ++w)
          for (int c = 0; c < Cf::kQKChunks; ++c)
            tma_load_3d(sQ + w * Cf::kQBytes + c * kAtom, &p.tm_q, bQfull, c * Cf::kQKBox, head, q0 + w * BM);
        ++q_issued;
        for (int j = pc.j0; ok && j < pc.j1; ++j) {
          for (int is_v = 0; is_v < 2; ++is_v) {
            const int s = u % NS;
            const int use = u / NS;
            if (use > 0 && !(ok = wait(bKVempty0 + 8 * s, (use - 1) & 1, ctl))) break;
            const uint32_t full = bKVfull0 + 8 * s;
            mbar_expect_tx(full, is_v ? Cf::kVBytes : Cf::kKBytes);
            const uint32_t dst = sKV + s * Cf::kTileBytes;
            const int nc = is_v ? Cf::kVChunks : Cf::kQKChunks;
            const int cw = is_v ? Cf::kVBox : Cf::kQKBox;  // elements per 128-byte chunk
            if (j < nA) {
              const CUtensorMap* m = is_v ? &p.tm_vc : &p.tm_kc;
              for (int c = 0; c < nc; ++c) tma_load_3d(dst + c * kAtom, m, full, c * cw, j * BN, head);
            } else {
              const CUtensorMap* m = is_v ? &p.tm_vn : &p.tm_kn;
              for (int c = 0; c < nc; ++c) tma_load_3d(dst + c * kAtom, m, full, c * cw, head, (j - nA) * BN);
            }
            tiles_issued = ++u;
          }
        }
      }
    }
  } else if (warp == 1) {
    {
      // ------------------------------ MMA issuer (whole warp) --------------------
      // Q, K both K-major
      constexpr uint32_t kIdQK = Cf::kQK8        ? idesc_e4m3(BM, BN)
                                 : KIND == kTf32 ? idesc_tf32(BM, BN)
                                                 : idesc_bf16(BM, BN, 0, 0);
      // P from TMEM; V is N(=d)-major, or K-major after the transpose (tf32)
      constexpr uint32_t kIdPV = KIND == kTf32     ? idesc_tf32(BM, D)
                                 : KIND == kE4m3KV ? idesc_f16(BM, D, 0, 1)
                                                   : idesc_bf16(BM, D, 0, 1);
      // The tensor core takes one 128x128x16 MMA per 64 clocks, but this warp
      // shares its SMSP's issue slots with two busy softmax warps and gets few of
      // them, so each MMA group must cost it as few instructions as possible.
      // All 32 lanes run this loop in step: every wait is a warp vote and the
      // MMAs and commits go out under an elect.sync predicate, so the control
      // flow and every descriptor are visibly warp-uniform (one lane alone
      // behind a lane test measured 10 % slower over the whole kernel).  All
      // operands are ready in registers and the eight MMAs of a group go out
      // from one asm block.  The Q descriptors of both query tiles and the
      // tensor-memory addresses of P are built once; the descriptors of a K or V
      // tile differ from the ring's first stage only in the start address field
      // of the low word (16-byte units; shared offsets stay below 256 KB, so no
      // carry reaches the high word).
      constexpr int KS = Cf::kKSteps;
      static_assert(KS == 8 || KS == 4, "k-steps per Q K^T group");
      static_assert(BN / 16 == 8, "k-steps per P V group");
      uint64_t dq[NQ][KS];
#pragma unroll
      for (int w = 0; w < NQ; ++w)
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
          dq[w][ks] = sw128_desc(sQ + w * Cf::kQBytes + (ks >> 2) * kAtom + (ks & 3) * 32, 16, 1024);
      const uint64_t dK0 = sw128_desc(sKV, 16, 1024);
      // V tiles: in the ring, or (e4m3 V) in the two fp16 buffers
      const uint64_t dV0 = sw128_desc(KIND == kE4m3KV ? sV16 : sKV, kAtom, 1024);
      constexpr uint32_t kVStride = KIND == kE4m3KV ? Cf::kV16Tile : Cf::kTileBytes;
      const uint32_t k_lo0 = (uint32_t)dK0, k_hi = (uint32_t)(dK0 >> 32);
      const uint32_t v_lo0 = (uint32_t)dV0, v_hi = (uint32_t)(dV0 >> 32);
      // tf32: the transposed V tile sits at one address; k-step ks (8 keys, 32
      // bytes) lies in the 128-byte column chunk ks / 4, whose D rows take D * 128 bytes
      // (the low parts of a K tile sit at one address too, laid out as the K tile)
      uint64_t dvt0[8], dvt1[8], dkl[8];
      if constexpr (KIND == kTf32) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          dvt0[ks] = sw128_desc(sVT + (ks >> 2) * (D * 128) + (ks & 3) * 32, 16, 1024);
          dvt1[ks] = sw128_desc(sVT + ((ks + 8) >> 2) * (D * 128) + (ks & 3) * 32, 16, 1024);
          dkl[ks] = sw128_desc(sKL + (ks >> 2) * kAtom + (ks & 3) * 32, 16, 1024);
        }
      }
      auto issue_qk = [&](int w, int stage) {
        const uint32_t lo = k_lo0 + (((uint32_t)stage * Cf::kTileBytes) >> 4);
        uint64_t bd[KS];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) bd[ks] = make_desc(lo + ((ks >> 2) * kAtom + (ks & 3) * 32) / 16, k_hi);
        if constexpr (Cf::kQK8)
          mma4_ss_f8(tmem + 256 + 128 * w, dq[w], bd, kIdQK);
        else if constexpr (KIND == kTf32) {
          const uint32_t sd = tmem + 256 + 128 * w;
          mma8_ss_tf32(sd, dq[w], bd, kIdQK, 0u);                // Qhi Khi^T
          mma8_ts_tf32(sd, tmem + 64 + 128 * w, bd, kIdQK, 1u);  // Qlo Khi^T, Qlo in tensor memory
          mma8_ss_tf32(sd, dq[w], dkl, kIdQK, 1u);               // Qhi Klo^T
        }
        else if constexpr (KS == 8)
          mma8_ss(tmem + 256 + 128 * w, dq[w], bd, kIdQK, 0u);
        else
          mma4_ss(tmem + 256 + 128 * w, dq[w], bd, kIdQK, 0u);
      };
      // P V in two groups of k-steps: keys 0-63, then keys 64-127; `stage` is the
      // ring stage of the V tile (e4m3 V: its fp16 buffer)
      auto issue_pv = [&](int w, int stage, int half, bool acc) {
        if constexpr (KIND == kTf32) {
          uint64_t bd[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) bd[ks] = half ? dvt1[ks] : dvt0[ks];
          mma8_ts_tf32(tmem + 128 * w, tmem + 256 + 128 * w + 64 * half, bd, kIdPV, acc ? 1u : 0u);
        } else {
          const uint32_t lo = v_lo0 + (((uint32_t)stage * kVStride) >> 4);
          uint64_t bd[4];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) bd[ks] = make_desc(lo + ((half * 4 + ks) * 16 * 128) / 16, v_hi);
          mma4_ts(tmem + 128 * w, tmem + 256 + 128 * w + 32 * half, bd, kIdPV, acc ? 1u : 0u);
        }
      };
      Walker wk;
      walker_init(wk, p.a, p.s, blockIdx.x);
      Piece pc;
      int u = 0, qi = 0, jt = 0;
      bool ok = true;
      while (ok && walker_next(wk, p.a, p.s, pc, blockIdx.x)) {
        const int n = pc.j1 - pc.j0;
        if (!(ok = __all_sync(0xffffffffu, wait(bQfull, qi & 1, ctl)))) break;
        if (!(ok = __all_sync(0xffffffffu, wait(bKVfull0 + 8 * (u % NS), (u / NS) & 1, ctl)))) break;
        if constexpr (KIND == kTf32) {
          if (!(ok = __all_sync(0xffffffffu, wait(bQsplit, qi & 1, ctl)))) break;
          if (!(ok = __all_sync(0xffffffffu, wait(bKsplit, jt & 1, ctl)))) break;
        }
        tc_fence_after();
        issue_qk(0, u % NS);
        tc_commit_e(bS0);
        issue_qk(1, u % NS);
        tc_commit_e(bS0 + 8);
        tc_commit_e(bKVempty0 + 8 * (u % NS));
        if constexpr (KIND == kTf32) tc_commit_e(bKLempty);
        if (n == 1) tc_commit_e(bQempty);
        for (int t = 0; t < n; ++t) {
          const int uv = u + 2 * t + 1, sv = uv % NS;
          const int uk = u + 2 * t + 2, sk = uk % NS;
          const bool more = t + 1 < n;
          if (!(ok = __all_sync(0xffffffffu, wait(bKVfull0 + 8 * sv, (uv / NS) & 1, ctl)))) break;
          if (!(ok = __all_sync(0xffffffffu, wait(bP0, (jt + t) & 1, ctl)))) break;
          if constexpr (KIND == kTf32) {
            if (!(ok = __all_sync(0xffffffffu, wait(bVTfull, (jt + t) & 1, ctl)))) break;
          }
          // e4m3 V: the fp16 buffer of V tile jt + t
          const int pvs = KIND == kE4m3KV ? ((jt + t) & 1) : sv;
          if constexpr (KIND == kE4m3KV) {
            if (!(ok = __all_sync(0xffffffffu, wait(bWfull0 + 8 * pvs, ((jt + t) >> 1) & 1, ctl)))) break;
          }
          // the previous item's epilogue must have read O out of tensor memory
          if (t == 0 && qi > 0 && !(ok = __all_sync(0xffffffffu, wait(bOempty, (qi - 1) & 1, ctl)))) break;
          tc_fence_after();
          issue_pv(0, pvs, 0, t > 0);
          if (!(ok = __all_sync(0xffffffffu, wait(bP0 + 16, (jt + t) & 1, ctl)))) break;
          tc_fence_after();
          issue_pv(0, pvs, 1, true);
          if (more) {
            if (!(ok = __all_sync(0xffffffffu, wait(bKVfull0 + 8 * sk, (uk / NS) & 1, ctl)))) break;
            if constexpr (KIND == kTf32) {
              if (!(ok = __all_sync(0xffffffffu, wait(bKsplit, (jt + t + 1) & 1, ctl)))) break;
            }
            tc_fence_after();
            issue_qk(0, sk);
            tc_commit_e(bS0);
          }
          if (!(ok = __all_sync(0xffffffffu, wait(bP0 + 8, (jt + t) & 1, ctl)))) break;
          tc_fence_after();
          issue_pv(1, pvs, 0, t > 0);
          if (!(ok = __all_sync(0xffffffffu, wait(bP0 + 24, (jt + t) & 1, ctl)))) break;
          tc_fence_after();
          issue_pv(1, pvs, 1, true);
          tc_commit_e(bKVempty0 + 8 * sv);
          if constexpr (KIND == kTf32) tc_commit_e(bVTempty);
          if constexpr (KIND == kE4m3KV) tc_commit_e(bWempty0 + 8 * pvs);
          if (more) {
            issue_qk(1, sk);
            tc_commit_e(bS0 + 8);
            tc_commit_e(bKVempty0 + 8 * sk);
            if constexpr (KIND == kTf32) tc_commit_e(bKLempty);
            if (t + 2 == n) tc_commit_e(bQempty);
          }
        }
        if (!ok) break;
        tc_commit_e(bOfull);
        u += 2 * n;
        jt += n;
        ++qi;
      }
    }
  } else if (warp < 4) {
    if constexpr (KIND == kTf32) {
      // ------------------------------ K split, V transpose (fp32 operands) -------
      // Per key tile, in the order the producer loads them:
      // K: each element x becomes hi = tf32(x) in place and lo = tf32(x - hi) at
      //    the same offset of the low-part buffer (same layout as the K tile).
      // V: TMA leaves a V tile as key rows: column chunk c holds d in [32c, 32c+32)
      //    of every key, 128 bytes per key, its 16-byte units swizzled by key % 8.
      //    P V reads it K-major, rounded to tf32: rows of d, column chunks of 32
      //    keys (D rows x 128 bytes each), 16-byte units swizzled by d % 8.  Each
      //    warp instruction moves one 16-byte unit of 32 consecutive keys, so
      //    neither the loads nor the 4-byte stores meet a bank conflict.
      const int tt = threadIdx.x - 64;
      uint8_t* vt = gbase + Cf::kSmemVT;
      uint8_t* kl = gbase + Cf::kSmemKL;
      constexpr int kUnits = BN * D / 4;  // 16-byte units of a K or V tile
      Walker wk;
      walker_init(wk, p.a, p.s, blockIdx.x);
      Piece pc;
      int u = 0, ti = 0;
      bool ok = true;
      while (ok && walker_next(wk, p.a, p.s, pc, blockIdx.x)) {
        const int n = pc.j1 - pc.j0;
        for (int t = 0; t < n; ++t, ++ti) {
          const int uk = u + 2 * t, sk = uk % NS;
          if (!(ok = wait(bKVfull0 + 8 * sk, (uk / NS) & 1, ctl))) break;
          // Q K^T of the previous tile (both query tiles) is done with the low parts
          if (ti > 0 && !(ok = wait(bKLempty, (ti - 1) & 1, ctl))) break;
          uint8_t* kt = gbase + Cf::kSmemKV + sk * Cf::kTileBytes;
#pragma unroll 4
          for (int x = tt; x < kUnits; x += 64) {
            float4* ph = reinterpret_cast<float4*>(kt + 16 * x);
            float4* pl = reinterpret_cast<float4*>(kl + 16 * x);
            const float4 val = *ph;
            float4 hi, lo;
            split_tf32(val.x, hi.x, lo.x);
            split_tf32(val.y, hi.y, lo.y);
            split_tf32(val.z, hi.z, lo.z);
            split_tf32(val.w, hi.w, lo.w);
            *ph = hi;
            *pl = lo;
          }
          // generic-proxy writes, read by the tensor core (async proxy)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(bKsplit);

          const int uv = uk + 1, sv = uv % NS;
          if (!(ok = wait(bKVfull0 + 8 * sv, (uv / NS) & 1, ctl))) break;
          // P V of the previous tile (both query tiles) is done with the buffer
          if (ti > 0 && !(ok = wait(bVTempty, (ti - 1) & 1, ctl))) break;
          const uint8_t* raw = gbase + Cf::kSmemKV + sv * Cf::kTileBytes;
#pragma unroll 4
          for (int x = tt; x < kUnits; x += 64) {
            const int k = x % BN;
            const int c = (x / BN) >> 3, q4 = (x / BN) & 7;
            const float4 val = *reinterpret_cast<const float4*>(raw + c * kAtom + k * 128 + ((q4 ^ (k & 7)) << 4));
            const float e4[4] = {val.x, val.y, val.z, val.w};
            uint8_t* col = vt + (k >> 5) * (D * 128) + (k & 3) * 4;
            const int ku = (k & 31) >> 2;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int d = c * 32 + q4 * 4 + e;
              *reinterpret_cast<uint32_t*>(col + d * 128 + ((ku ^ (d & 7)) << 4)) = to_tf32(e4[e]);
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(bVTfull);
        }
        if (!ok) break;
        u += 2 * n;
      }
    } else if constexpr (KIND == kE4m3KV) {
      // ------------------------------ V widening (e4m3 values) ---------------------
      // TMA leaves a V tile as 128 key rows of 128 e4m3 bytes (one column chunk),
      // 16-byte units swizzled by key % 8.  P V reads fp16 in the layout of a bf16
      // V tile: column chunk c (d in [64c, 64c+64)) of 128 key rows of 128 bytes,
      // 16-byte units swizzled by key % 8.  A source unit (16 values of d) widens
      // exactly (cvt.rn.f16x2.e4m3x2) into two units of one chunk.  Consecutive
      // threads take consecutive keys: no bank conflicts on either side.
      const int tt = threadIdx.x - 64;
      Walker wk;
      walker_init(wk, p.a, p.s, blockIdx.x);
      Piece pc;
      int u = 0, vt = 0;
      bool ok = true;
      while (ok && walker_next(wk, p.a, p.s, pc, blockIdx.x)) {
        const int n = pc.j1 - pc.j0;
        for (int t = 0; t < n; ++t, ++vt) {
          const int uv = u + 2 * t + 1, sv = uv % NS;
          const int b = vt & 1;
          if (!(ok = wait(bKVfull0 + 8 * sv, (uv / NS) & 1, ctl))) break;
          // P V of V tile vt - 2 (both query tiles) is done with buffer b
          if (vt >= 2 && !(ok = wait(bWempty0 + 8 * b, ((vt >> 1) - 1) & 1, ctl))) break;
          const uint8_t* raw = gbase + Cf::kSmemKV + sv * Cf::kTileBytes;
          uint8_t* dst = gbase + Cf::kSmemV16 + b * Cf::kV16Tile;
#pragma unroll 4
          for (int x = tt; x < BN * 8; x += 64) {
            const int k = x % BN, q = x / BN;  // key, 16-value unit of d
            const uint4 val = *reinterpret_cast<const uint4*>(raw + k * 128 + ((q ^ (k & 7)) << 4));
            const uint32_t w4[4] = {val.x, val.y, val.z, val.w};
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
                  "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
                  : "=r"(h[2 * i]), "=r"(h[2 * i + 1])
                  : "r"(w4[i]));
            }
            uint8_t* row = dst + (q >> 2) * kAtom + k * 128;
            const int u0 = (q & 3) * 2;
            *reinterpret_cast<uint4*>(row + ((u0 ^ (k & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(row + (((u0 + 1) ^ (k & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
          }
          // generic-proxy writes, read by the tensor core (async proxy)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(bWfull0 + 8 * b);
        }
        if (!ok) break;
        u += 2 * n;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------ softmax + epilogue ----------------------------
    const int w = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + 256 + 128 * w;
    const uint32_t tO = tmem + lane_off + 128 * w;
    const uint32_t bS = bS0 + 8 * w;
    const uint32_t bP = bP0 + 8 * w;        // P of keys 0-63 stored
    const uint32_t bP2 = bP0 + 16 + 8 * w;  // P of keys 64-127 stored
    const float sl2 = a.scale_log2;
    Walker wk;
    walker_init(wk, p.a, p.s, blockIdx.x);
    Piece pc;
    int qi = 0, jt = 0;
    bool ok = true;
    while (ok && walker_next(wk, p.a, p.s, pc, blockIdx.x)) {
      int head, q0, nA;
      item_geom(p.a, p.s, pc.item, head, q0, nA);
      const int qrow = q0 + w * BM + row;
      int row_end = a.Lb;
      if (a.mode != 0) {
        const long long e = ((long long)qrow / a.block_tokens + 1) * a.block_tokens;
        row_end = (int)(e < a.Lb ? e : a.Lb);
      }
      const int n = pc.j1 - pc.j0;
      if constexpr (KIND == kTf32) {
        // split this thread's Q row: hi in place (Q K^T reads it from shared
        // memory), lo into columns [64, 128) of the tile's O region (read as A
        // from tensor memory); the previous piece's Q K^T products are done with
        // both, since the producer reloads Q only after they complete
        ok = __all_sync(0xffffffffu, wait(bQfull, qi & 1, ctl));
        if (!ok) break;
        uint8_t* qs = gbase + w * Cf::kQBytes + row * 128;
        uint32_t qlo[D];
#pragma unroll
        for (int c = 0; c < Cf::kQKChunks; ++c)
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float4* ph = reinterpret_cast<float4*>(qs + c * kAtom + ((q4 ^ (row & 7)) << 4));
            const float4 val = *ph;
            float4 hi, lo;
            split_tf32(val.x, hi.x, lo.x);
            split_tf32(val.y, hi.y, lo.y);
            split_tf32(val.z, hi.z, lo.z);
            split_tf32(val.w, hi.w, lo.w);
            *ph = hi;
            const int d = c * 32 + q4 * 4;
            qlo[d] = __float_as_uint(lo.x);
            qlo[d + 1] = __float_as_uint(lo.y);
            qlo[d + 2] = __float_as_uint(lo.z);
            qlo[d + 3] = __float_as_uint(lo.w);
          }
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) tmem_st16(tO + 64 + 16 * cc, qlo + 16 * cc);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bQsplit);
      }
      float m = -INFINITY, l = 0.f;
      for (int t = 0; t < n; ++t) {
        const int j = pc.j0 + t;
        ok = __all_sync(0xffffffffu, wait(bS, (jt + t) & 1, ctl));
        if (!ok) break;
        tc_fence_after();
        // S: all four loads in flight, one wait
        uint32_t r[BN];
        tmem_ld32(tS + 0, r + 0);
        tmem_ld32(tS + 32, r + 32);
        tmem_ld32(tS + 64, r + 64);
        tmem_ld32(tS + 96, r + 96);
        tmem_ld_wait();
        reg_fence(r, BN);
        const int valid = j < nA ? a.La - j * BN : (a.mode != 0 ? row_end : a.Lb) - (j - nA) * BN;
        if (valid < BN) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= valid) r[c] = __float_as_uint(-INFINITY);
        }
        float mx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = __uint_as_float(r[i]);
#pragma unroll
        for (int c = 4; c < BN; c += 2)
          mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
        const float mt = max3f(max3f(mx[0], mx[1], mx[2]), mx[3], -INFINITY);
        const float m_new = fmaxf(m, mt * sl2);
        // the reference max moves (and O is rescaled, after P is written) only
        // when some row of the warp grew by more than 2^8
        const bool rescale = t > 0 && __any_sync(0xffffffffu, m_new > m + kRescaleLog2);
        float alpha = 1.f;
        if (t == 0 || rescale) {
          if (rescale && m_new != -INFINITY) alpha = ex2(m - m_new);
          l *= alpha;
          m = m_new;
        }
        const float mo = (m == -INFINITY) ? 0.f : m;
        // P = 2^(s*log2e/sqrt(d) - m), rounded to bf16 for the P V product.  The
        // row sum adds the same rounded values, so numerator and denominator
        // carry the same rounding and a dominant key keeps its exact weight.
        // two columns per packed fma; the row sum adds the bf16 halves of each
        // packed P word directly (exact widening, fp32 add)
        const uint64_t sl2x2 = pack_f32x2(sl2, sl2), nmo2 = pack_f32x2(-mo, -mo);
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if constexpr (KIND == kTf32) {
          // P rounded to tf32 (what P V reads), one fp32 column per key; the row
          // sum adds the same rounded values
#pragma unroll
          for (int g = 0; g < BN / 16; ++g) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int c = g * 16 + 2 * i;
              float x0, x1;
              fma_f32x2(x0, x1, __uint_as_float(r[c]), __uint_as_float(r[c + 1]), sl2x2, nmo2);
              pk[2 * i] = to_tf32(ex2(x0));
              pk[2 * i + 1] = to_tf32(ex2(x1));
              ls[2 * (i & 3)] += __uint_as_float(pk[2 * i]);
              ls[2 * (i & 3) + 1] += __uint_as_float(pk[2 * i + 1]);
            }
            tmem_st16(tS + 16 * g, pk);
            if (g == 3 && !rescale) {
              tmem_st_wait();
              tc_fence_before();
              if (!(a.stall_inject && jt + t == 0 && w == 0)) mbar_arrive(bP);
            }
          }
        } else {
#pragma unroll
        for (int g = 0; g < BN / 32; ++g) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = g * 32 + 2 * i;
            float x0, x1;
            fma_f32x2(x0, x1, __uint_as_float(r[c]), __uint_as_float(r[c + 1]), sl2x2, nmo2);
            if constexpr (KIND == kE4m3KV) {
              pk[i] = pack_f16(ex2(x0), ex2(x1));
              add_f16x2(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], pk[i]);
            } else {
              pk[i] = pack_bf16(ex2(x0), ex2(x1));
              add_bf16x2(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], pk[i]);
            }
          }
          tmem_st16(tS + 16 * g, pk);
          if (g == 1 && !rescale) {
            // keys 0-63: their P is in tensor memory and O needs no rescale, so
            // the tensor core may start on them (rescale is warp-uniform)
            tmem_st_wait();
            tc_fence_before();
            if (!(a.stall_inject && jt + t == 0 && w == 0)) mbar_arrive(bP);
          }
        }
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        if (rescale) {
          // PV of the previous tile has completed (it was issued before this S)
#pragma unroll 1
          for (int cc = 0; cc < D / 16; ++cc) {
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
        if (!(a.stall_inject && jt + t == 0 && w == 0)) {
          if (rescale) mbar_arrive(bP);
          mbar_arrive(bP2);
        }
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, wait(bOfull, qi & 1, ctl));
      if (!ok) break;
      tc_fence_after();
      if (pc.partial) {
        // unnormalised O with its reference max and sum, merged by combine_kernel
        const size_t rows_all = (size_t)2 * p.s.grid * (NQ * BM);
        const size_t sr = (size_t)pc.slot * (NQ * BM) + w * BM + row;
        float* po = p.part + sr * D;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
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
        p.part[rows_all * D + sr] = m;
        p.part[rows_all * D + rows_all + sr] = l;
      } else {
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
      tc_fence_before();
      mbar_arrive(bOempty);
      jt += n;
      ++qi;
    }
  }

  // ------------------------------ teardown ------------------------------------
  // this CTA's work is issued: the launch that follows (merge of split items or
  // the commit copy) may be scheduled; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // copies still in flight land before the shared memory is released
    if (q_issued > 0) wait_drain(bQfull, (q_issued - 1) & 1);
    const int first = tiles_issued > NS ? tiles_issued - NS : 0;
    for (int u = first; u < tiles_issued; ++u) wait_drain(bKVfull0 + 8 * (u % NS), (u / NS) & 1);
  }
  if (warp == 1) {
    // a commit tracks the MMAs of its own thread: the lane elect.sync picks,
    // as for every MMA and commit of the issue loop
    tc_commit_e(bDrain);
    wait_drain(bDrain, 0);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

template <int D, int KIND>
cudaError_t launch_tc(const AttendArgs& a, cudaStream_t stream) {
  constexpr int qk = Cfg<D, KIND>::kQKElem, ve = Cfg<D, KIND>::kVElem;  // bytes per element
  TcParams p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  if (!encode_tokens(&p.tm_q, a.q, a.Lq, a.heads, D, BM, qk) ||
      !encode_tokens(&p.tm_kn, a.kn, a.Lb, a.heads, D, BN, qk) ||
      !encode_tokens(&p.tm_vn, a.vn, a.Lb, a.heads, D, BN, ve) ||
      !encode_cache(&p.tm_kc, a.kc, a.La, a.heads, D, a.cache_head_elems, BN, qk) ||
      !encode_cache(&p.tm_vc, a.vc, a.La, a.heads, D, a.cache_head_elems, BN, ve))
    return cudaErrorInvalidValue;
  p.s.nqb = (a.Lq + NQ * BM - 1) / (NQ * BM);
  CombineParams cp;
  cp.nsplit = 0;
  if (a.mode == 1) {
    // persistent: one CTA per SM, items in zigzag rounds (see walker_next)
    const int items = p.s.nqb * a.heads;
    const int sms = sm_count();
    p.s.grid = items < sms ? items : sms;
  } else {
    // without scratch for two partial results per CTA, no item is split
    int ctas = sm_count();
    if (2 * ctas > a.scratch_slots) ctas = a.scratch_slots / 2;
    plan_attend(a, p.s, cp, ctas < 1 ? 1 : ctas);
    if (cp.nsplit > 0 && !a.scratch) return cudaErrorInvalidValue;
    p.part = a.scratch;
  }
  static std::atomic<int> attr_done[64];
  if (cudaError_t e = smem_opt_in(attend_tc_kernel<D, KIND>, Cfg<D, KIND>::kSmemBytes, attr_done)) return e;
  attend_tc_kernel<D, KIND><<<(unsigned)p.s.grid, kThreads, Cfg<D, KIND>::kSmemBytes, stream>>>(p);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || cp.nsplit == 0) return e;
  return launch_combine<D>(cp, a, p.s, p.part, stream);
}

}  // namespace

size_t attend_scratch_bytes(int head_dim, int slots) {
  return (size_t)slots * tc::kItemRows * (head_dim + 2) * sizeof(float);
}

int attend_scratch_slots_wanted() {
  int n = tc::sm_count();
  if (n > tc::kMaxSplit) n = tc::kMaxSplit;
  return 2 * n;
}

int attend_schedule_dump(int Lq, int La, int Lb, int heads, int max_ctas, int mode, int block_tokens, int* grid,
                         int* out, int cap, int* splits, int split_cap, int* split_ints) {
  using namespace tc;
  AttendArgs a;
  std::memset(&a, 0, sizeof(a));
  a.Lq = Lq;
  a.La = La;
  a.Lb = Lb;
  a.heads = heads;
  a.mode = mode;
  a.block_tokens = block_tokens;
  Sched sc;
  std::memset(&sc, 0, sizeof(sc));
  sc.nqb = (Lq + kItemRows - 1) / kItemRows;
  CombineParams cp;
  cp.nsplit = 0;
  if (mode == 1) {
    const int items = sc.nqb * heads;
    sc.grid = items < max_ctas ? items : max_ctas;
  } else {
    plan_attend(a, sc, cp, max_ctas);
  }
  *grid = sc.grid;
  int n = 0;
  for (int c = 0; c < sc.grid; ++c) {
    Walker wk;
    walker_init(wk, a, sc, c);
    Piece pc;
    while (walker_next(wk, a, sc, pc, c)) {
      if (n + 6 <= cap) {
        out[n + 0] = c;
        out[n + 1] = pc.item;
        out[n + 2] = pc.j0;
        out[n + 3] = pc.j1;
        out[n + 4] = pc.partial;
        out[n + 5] = pc.slot;
      }
      n += 6;
    }
  }
  // split list: item, number of parts, then the parts' slots
  int m = 0;
  for (int k = 0; k < cp.nsplit; ++k) {
    const int cnt = cp.first[k + 1] - cp.first[k];
    if (m + 2 + cnt <= split_cap) {
      splits[m] = cp.item[k];
      splits[m + 1] = cnt;
      for (int i = 0; i < cnt; ++i) splits[m + 2 + i] = cp.slot[cp.first[k] + i];
    }
    m += 2 + cnt;
  }
  *split_ints = m;
  return n / 6;
}

cudaError_t launch_attend_bf16_tc(const AttendArgs& a, cudaStream_t stream) {
  if (a.qk_fp8 && a.v_fp8) return a.head_dim == 128 ? launch_tc<128, kE4m3KV>(a, stream) : cudaErrorInvalidValue;
  if (a.qk_fp8) return a.head_dim == 128 ? launch_tc<128, kE4m3>(a, stream) : cudaErrorInvalidValue;
  if (a.head_dim == 64) return launch_tc<64, kBf16>(a, stream);
  return a.pair ? launch_attend_bf16_pair(a, stream) : launch_tc<128, kBf16>(a, stream);
}

cudaError_t launch_attend_tf32_tc(const AttendArgs& a, cudaStream_t stream) {
  return a.head_dim == 64 ? launch_tc<64, kTf32>(a, stream) : cudaErrorInvalidValue;
}

}  // namespace ll
