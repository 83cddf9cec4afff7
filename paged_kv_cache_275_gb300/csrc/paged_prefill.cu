// Chunked paged prefill attention on the 5th-generation tensor cores (sm_103a).
//
// What is computed ("从零实现一个 mini vLLM--开篇", section 2: prefill runs the
// prompt at once and keeps every layer's K and V; section 5: chunked prefill;
// section 5, phases 4-5: K and V are found through the block table): for each
// sequence b, C_b new tokens follow P_b cached ones (context_lens[b] = P_b + C_b,
// the chunk already appended); query row i of the chunk attends causally over
// the first P_b + i + 1 tokens: out = softmax(scale * q K^T) V.
//
// How (GB300-first).  One CTA per (pair of 128-row query tiles, kv head, sequence),
// each holding a whole SM (all 512 TMEM columns), launched longest first.  The 128
// MMA rows of a tile pack 128/G chunk tokens x the G q heads
// of the group; the CTA's two tiles cover consecutive tokens and share every K/V
// tile.  Keys advance 128 at a time (8 pages of 16), so S = Q K^T is an N = 128
// MMA and O += P V an N = D one: at N = 64 an MMA is bound by reading its
// operands from shared memory, at N = 128 by the math.
//   * warp 8: TMA producer.  Each page (16 tokens x D of one kv head) is one 4D
//     tensor-map copy with 128-byte swizzle, gathered through the block table into
//     one ring of five K and V tiles (filled in the order the MMAs read them), one
//     copy per lane; mbarrier
//     completion by transaction bytes.  Per-copy cost, not bytes, bounds the copy
//     engine at 16-token pages, so a page travels as one copy: its two 8-row groups,
//     each the two 64-dim halves one after the other, a layout both products read
//     with 8-row groups one descriptor stride apart.  It also zeroes the rows of the
//     last V tile past the end of the keys.
//   * warp 9 (one lane): MMA issuer.  tcgen05.mma kind::f16 (bf16 in, fp32
//     accumulate): S = Q_t K^T into tile t's TMEM S buffer (M 128, N 128); once
//     the softmax has written P over S, O_t += P V (M 128, N = D, P read from
//     TMEM) and at once S of the next step.  The two tiles alternate, so one
//     tile's softmax overlaps the other's MMAs.  Lane 0 runs the loop alone and
//     polls its waits: the softmax warps sharing its SM sub-partition leave it
//     few issue slots, and the pipe idles while the issuer is late at a group
//     boundary.  The warp also allocates and frees the 512 TMEM columns.
//   * warps 0-7 (one row each; warps 4t..4t+3 serve tile t, each warp the TMEM
//     lanes 32 (warp % 4) .. + 31): stage Q (copies issued before the set-up
//     barrier, as is the producer's first K tile), then per key step read S
//     (tcgen05.ld), apply the causal and length mask, run the online softmax in
//     base 2 (lazy rescale: O is rescaled only when a row's max grows by more than
//     2^8), write P as bf16 pairs into TMEM over the S values just read; finally
//     read O, divide by the row sum and store bf16 rows.
// Every mbarrier wait is bounded by a time limit; a wait that runs out sets
// PKV_DEVERR_PIPELINE_TIMEOUT, the warps finish their loops and the TMEM is
// freed before the CTA exits.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "paged_prefill.h"

namespace pkv {
namespace {

constexpr int kRows = 128;    // MMA M: query rows of one tile (chunk tokens x group heads)
constexpr int kTiles = 2;     // query tiles per CTA; every K/V tile feeds both
constexpr int kKeys = 128;    // keys per step (MMA N of S, MMA K of P.V)
#ifndef PKV_PF_RING
#define PKV_PF_RING 5
#endif
// One ring of K and V tiles, filled in the order the MMAs first read them and freed in the
// same order: tile n = 2 j is K of key step j, n = 2 j + 1 its V.  Tile n sits in slot
// n % kRing.  (Separate K and V rings left V a step and a half of lead at most, shorter
// than its copies take once the copies queue; one ring gives either about two steps.)
constexpr int kRing = PKV_PF_RING;
static_assert(kRing >= 3, "the ring must hold a step's K and V and the next K");
constexpr int kProducerWarp = 4 * kTiles;  // warps 0-7 softmax (four per tile)
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kTmemCols = 512;  // per tile t: S at [256 t, 256 t + 128), O at [256 t + 128, 256 t + 128 + D)
__host__ __device__ constexpr int col_s(int t) { return 256 * t; }  // P (bf16 pairs) over the first 64 of S
__host__ __device__ constexpr int col_o(int t) { return 256 * t + 128; }
constexpr int kTmemSlotOffset = 384;  // in the 512-byte barrier area: barriers below, TMEM slot and sequence pick here
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 8.0f;
constexpr unsigned long long kWaitNs = 2000000000ull;

template <int D>
struct Pf {
  static constexpr int kHalves = D / 64;           // 128-byte swizzle atoms across a row
  static constexpr int kQHalf = kRows * 128;       // 16 KB: 128 rows x 64 dims
  static constexpr int kQTile = kHalves * kQHalf;  // one tile's Q
  static constexpr int kKVHalf = kKeys * 128;      // 16 KB: 128 keys x 64 dims
  static constexpr int kTile = kHalves * kKVHalf;  // one K (or V) tile of a step
  // A K or V tile is 8 pages of 16 keys, each page one tensor copy laid out as two 8-row
  // groups, each group the page's 64-dim halves one after the other: [group][half][8 rows][128 B].
  static constexpr int kGroupBytes = kHalves * 1024;  // stride between 8-key groups (descriptor SBO)
  static constexpr int kPageBytes = 2 * kGroupBytes;  // one page of one kv head
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kTiles * kQTile;
  static constexpr int kOffBar = kOffKV + kRing * kTile;
  // The dynamic shared memory is requested 1024-byte aligned (checked at run time),
  // so no alignment slack: 224.5 KB at D = 128.
  static constexpr int kRaw = kOffBar + 512;  // barriers, TMEM slot, sequence pick
  // At least 120 KB so that one CTA holds the SM: it owns all 512 TMEM columns,
  // and a second CTA's allocation would have to wait.
  static constexpr int kSmem = kRaw > 120 * 1024 ? kRaw : 120 * 1024;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t saddr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void bar_init(uint32_t b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t b) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(b), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait; false if the phase did not complete in time.
__device__ __forceinline__ bool bar_wait(uint32_t b, uint32_t parity) {
  if (bar_try(b, parity)) return true;
  const unsigned long long t0 = now_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (bar_try(b, parity)) return true;
    if ((it & 63u) == 0 && now_ns() - t0 > kWaitNs) return false;
  }
  return false;
}
__device__ __forceinline__ bool bar_test(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(b), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait that polls without suspending the thread: a completed phase costs the
// caller one non-blocking test (a suspending try_wait costs a few hundred cycles of
// issue when the tensor pipe is streaming operands out of shared memory).
__device__ __forceinline__ bool bar_poll(uint32_t b, uint32_t parity) {
  if (bar_test(b, parity)) return true;
  const unsigned long long t0 = now_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (bar_test(b, parity)) return true;
    if ((it & 63u) == 0 && now_ns() - t0 > kWaitNs) return false;
  }
  return false;
}
// 4D tensor copy: one page of one kv head (box 64 dims x 8 rows x halves x 2 row groups).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int group, uint32_t b) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %2, %2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(group), "r"(b)
      : "memory");
}
// 16 bytes global -> shared without a register round trip; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// 3D tensor store shared -> global (one half of a tile's output rows), tracked by a bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_store_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: 128-byte swizzle with 8-row groups `sbo` bytes
// apart (the stride byte offset; 1024 when the groups are packed).  K-major operands
// are one swizzle atom (64 elements) wide across the 16-element K of an MMA; an
// MN-major operand (V, read as N = D) may span two atoms along N, `lbo` bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo = 1024, uint32_t sbo = 1024) {
  uint64_t d = (addr & 0x3FFFFu) >> 4;
  d |= uint64_t(lbo >> 4) << 16;     // leading byte offset (MN-major: next 64-wide atom along N)
  d |= uint64_t(sbo >> 4) << 32;     // stride byte offset: between 8-row groups
  d |= uint64_t(1) << 46;            // descriptor version
  d |= uint64_t(2) << 61;            // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M 128, N n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) | ((static_cast<uint32_t>(n) >> 3) << 17) |
         ((128u >> 4) << 24);
}
// Four MMAs in one block, operand i at base + i * step (descriptor units of 16 bytes, or tensor
// memory columns for an A in tensor memory, 128 lanes = rows, K along the columns as bf16 pairs);
// only the first may start a fresh accumulation.  The instruction descriptor is an immediate.
template <uint32_t kIdesc, uint32_t kAStep, uint32_t kBStep>
__device__ __forceinline__ void mma4_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc_first) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 pf, %3, 0;\n\tsetp.eq.b32 pt, %3, %3;\n\t"
      "add.s64 a1, %1, %5;\n\tadd.s64 a2, %1, %6;\n\tadd.s64 a3, %1, %7;\n\t"
      "add.s64 b1, %2, %8;\n\tadd.s64 b2, %2, %9;\n\tadd.s64 b3, %2, %10;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, pf;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %4, pt;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(acc_first), "n"(kIdesc), "n"(kAStep), "n"(2 * kAStep), "n"(3 * kAStep), "n"(kBStep),
      "n"(2 * kBStep), "n"(3 * kBStep)
      : "memory");
}
template <uint32_t kIdesc, uint32_t kAStep, uint32_t kBStep>
__device__ __forceinline__ void mma4_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t acc_first) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 pf, %3, 0;\n\tsetp.eq.b32 pt, %3, %3;\n\t"
      "add.u32 a1, %1, %5;\n\tadd.u32 a2, %1, %6;\n\tadd.u32 a3, %1, %7;\n\t"
      "add.s64 b1, %2, %8;\n\tadd.s64 b2, %2, %9;\n\tadd.s64 b3, %2, %10;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, pf;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %4, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %4, pt;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(acc_first), "n"(kIdesc), "n"(kAStep), "n"(2 * kAStep), "n"(3 * kAStep), "n"(kBStep),
      "n"(2 * kBStep), "n"(3 * kBStep)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(b) : "memory");
}
// 32 lanes x 32 columns of 32-bit values: this thread's row, 32 consecutive columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 64 columns: this thread's row, 64 consecutive columns.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// 2^x on the SFU (approximate, flush-to-zero): the softmax weights.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 32 lanes x 32 columns of raw 32-bit values; the caller waits (tcgen05.wait::st).
__device__ __forceinline__ void tmem_st32_raw(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// Byte offset of 16-byte chunk `chunk` (0..7) of row `r` in a 128-byte-swizzled
// region of 128-byte rows (the layout the TMA writes and the MMA reads).
__device__ __forceinline__ uint32_t swz(int r, int chunk) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4));
}
// Byte offset of chunk `chunk` of key `r` (0..127), dims half `h`, in a K or V tile of pages.
template <int D>
__device__ __forceinline__ uint32_t kv_off(int r, int h, int chunk) {
  return static_cast<uint32_t>((r >> 4) * Pf<D>::kPageBytes + ((r >> 3) & 1) * Pf<D>::kGroupBytes + h * 1024 +
                               (r & 7) * 128 + ((chunk ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int D, int G, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_out) {
  using T = Pf<D>;
  constexpr int kTokens = kRows / G;            // chunk tokens per 128-row tile
  constexpr int kCtaTokens = kTiles * kTokens;  // chunk tokens per CTA
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t s_base = saddr(smem);
  pdl_trigger();
  pdl_wait();

  const int tile = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);  // longest tiles first
  const int kvh = blockIdx.x;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Longest first: CTAs start in blockIdx order (x fastest), so z indexes the sequences by
  // decreasing context length (ties by index), y counts a sequence's tiles from the longest
  // (the last rows of a chunk see the most keys) and x is the kv head: all kv heads of a
  // sequence's longest tile go out before its next tile.  The launch order approximates
  // longest-processing-time-first, and the last wave holds the shortest tiles.  Ranked in shared memory when num_seqs <= kThreads,
  // in the V ring (not yet in use) and a spare word of the barrier area.
  // The sequences' chunk starts are staged beside the lengths in the same pass, so that the
  // picked sequence's q0, C and L need no second round trip to memory.
  // z = (sequence rank) * num_splits + split: a sequence's splits go out together.
  const int split = kSplit ? static_cast<int>(blockIdx.z) % p.num_splits : 0;
  const int zrank = kSplit ? static_cast<int>(blockIdx.z) / p.num_splits : static_cast<int>(blockIdx.z);
  int b = zrank;
  int q0, C, L;
  if (p.num_seqs <= kThreads) {
    int* s_lens = reinterpret_cast<int*>(smem + T::kOffKV + (kRing - 1) * T::kTile);
    int* s_qs = s_lens + kThreads;
    int& s_pick = *reinterpret_cast<int*>(smem + T::kOffBar + kTmemSlotOffset + 4);
    if (tid < p.num_seqs) {
      s_lens[tid] = p.context_lens[tid];
      s_qs[tid] = p.query_start[tid];
    }
    if (tid == 0) s_qs[p.num_seqs] = p.query_start[p.num_seqs];
    __syncthreads();
    if (tid < p.num_seqs) {
      const int mine = s_lens[tid];
      int rank = 0;
      for (int u = 0; u < p.num_seqs; ++u) {
        const int other = s_lens[u];
        rank += (other > mine) || (other == mine && u < tid);
      }
      if (rank == zrank) s_pick = tid;
    }
    __syncthreads();
    b = s_pick;
    q0 = s_qs[b];
    C = s_qs[b + 1] - q0;
    L = s_lens[b];
  } else {
    q0 = p.query_start[b];
    C = p.query_start[b + 1] - q0;
    L = p.context_lens[b];
  }
  const int cap = p.max_blocks_per_seq * kBlockTokens;
  if (C < 0 || L < C || L > cap) {
    if (tid == 0 && tile == 0) atomicOr(p.err, kErrLenTooLong);
    return;
  }
  if (tile == 0 && C > p.max_query_len && tid == 0) atomicOr(p.err, kErrLenTooLong);  // rows past the grid are lost
  const int i0 = tile * kCtaTokens;  // first chunk token of the CTA
  if (i0 >= C) return;               // uniform for the CTA: nothing allocated yet
  if (s_base & 1023u) {              // the swizzled operands need 1024-byte alignment
    if (tid == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  const int prefix = L - C;
  const int i_last = min(C, i0 + kCtaTokens) - 1;
  const int n_tiles = (i0 + kTokens < C) ? 2 : 1;  // the second tile only if it holds chunk rows
  const int kv_end = prefix + i_last + 1;          // keys the CTA's last row sees
  // This CTA's key steps: [j0, j0 + nsteps) of the tile pair's steps_all, split evenly over the
  // num_splits CTAs of the pair (a split with no step only marks its rows empty).
  const int steps_all = (kv_end + kKeys - 1) / kKeys;
  const int j0 = kSplit ? static_cast<int>(static_cast<int64_t>(split) * steps_all / p.num_splits) : 0;
  const int nsteps =
      kSplit ? static_cast<int>(static_cast<int64_t>(split + 1) * steps_all / p.num_splits) - j0 : steps_all;
  const bool tail = j0 + nsteps == steps_all && kv_end < steps_all * kKeys;  // the last step has keys past the end
  constexpr bool partial = kSplit;  // O, m and l go to the workspace for the merge
  if (kSplit && nsteps == 0) {  // uniform for the CTA: nothing allocated yet
    for (int x = tid; x < kCtaTokens * G; x += kThreads) {
      const int i = i0 + x / G;
      if (i < C)
        reinterpret_cast<float2*>(p.ws + static_cast<size_t>(p.num_splits) * p.num_seqs * p.ws_rows * p.num_q_heads *
                                             D)[((static_cast<size_t>(split) * p.num_seqs + b) * p.ws_rows + i) *
                                                    p.num_q_heads + kvh * G + x % G] = make_float2(-INFINITY, 0.f);
    }
    return;
  }

  // Barriers.  K/V ring: a slot frees when every tile's MMA that reads it has
  // retired.  Per tile: S ready, P ready, O final, Q staged, MMAs drained.  Each
  // tile has one S buffer (P is written over it), so S of step j + 1 is issued
  // after P.V of step j by the same thread: the S-ready arrival of a step also
  // proves the previous P.V retired, and no barrier can run two phases ahead
  // of its waiter.
  const uint32_t bar = s_base + T::kOffBar;
  constexpr uint32_t kBarBytes = 8 * (2 * kRing + 1 + 6 * kTiles);
  static_assert(kBarBytes <= kTmemSlotOffset, "the barriers must end below the TMEM slot");
  const uint32_t r_full = bar, r_empty = r_full + 8 * kRing,  // [slot]
      v_tail = r_empty + 8 * kRing, s_full = v_tail + 8,    // s_full: [tile]
      p_full = s_full + 8 * kTiles,                   // [tile]
      o_full = p_full + 8 * kTiles,                   // [tile]
      q_ready = o_full + 8 * kTiles,                  // [tile]
      mma_drained = q_ready + 8 * kTiles,             // [tile]
      o_staged = mma_drained + 8 * kTiles;            // [tile]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + T::kOffBar + kTmemSlotOffset);

  // The producer's first two windows of block ids are requested before the set-up barrier,
  // ahead of the softmax warps' Q loads, which would otherwise queue in front of them.
  constexpr int kPages = kKeys / kBlockTokens;  // pages per step
  const int npages = (kv_end + kBlockTokens - 1) / kBlockTokens;
  const int32_t* table = p.block_tables + static_cast<size_t>(b) * p.max_blocks_per_seq;
  const int w0 = (j0 * kPages) / 32;  // the block-id window holding the CTA's first step
  int raw_cur = 0, raw_next = 0;
  if (warp == kProducerWarp) {
    if (32 * w0 + lane < npages) raw_cur = __ldg(table + 32 * w0 + lane);
    if (32 * (w0 + 1) + lane < npages) raw_next = __ldg(table + 32 * (w0 + 1) + lane);
  }

  // Stage Q (zero rows past the chunk) in the swizzled K-major layout, issued before the set-up
  // so that its latency overlaps the barrier and tensor-memory set-up.  The tile's 128 threads
  // copy it together, consecutive threads taking consecutive 16-byte chunks of a row, so that a
  // warp reads two whole rows (a token's G head rows are contiguous); the copies go global ->
  // shared directly, all sixteen of a thread in flight at once.  The Q area is not used by the
  // sequence ranking above.
  if ((warp >> 2) < n_tiles && warp < kProducerWarp) {
    constexpr int kChunks = D / 8;
    const int t = warp >> 2, r = tid & (kRows - 1);
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q);
    const uint32_t qt = s_base + T::kOffQ + t * T::kQTile;
#pragma unroll
    for (int c = r; c < kRows * kChunks; c += kRows) {
      const int rr = c / kChunks, ch = c % kChunks;
      const int ii = i0 + t * kTokens + rr / G;
      const bool in_chunk = ii < C;
      const __nv_bfloat16* src =
          in_chunk ? qg + (static_cast<size_t>(q0 + ii) * p.num_q_heads + kvh * G + rr % G) * D + ch * 8 : qg;
      cp_async_16(qt + (ch / 8) * T::kQHalf + swz(rr, ch % 8), src, in_chunk ? 16u : 0u);
    }
  }

  // The producer sets up its ring barriers itself and sends K of step 0 (slot 0) before the
  // set-up barrier, so that the first tile's copies also overlap the set-up; everyone else
  // touches the ring barriers only after that barrier.  Step 0's pages are lanes 0..7 of the
  // first block-id window.
  if (warp == kProducerWarp) {
    if (lane == 0) {
      for (int s = 0; s < kRing; ++s) {
        bar_init(r_full + 8 * s, 1);
        bar_init(r_empty + 8 * s, 1);
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const int first0 = j0 * kPages;  // the first step's pages: lanes first0 % 32 .. + 7 of window w0
    const int pages0 = min(kPages, npages - first0);
    const int id0 = __shfl_sync(0xffffffffu, raw_cur, (first0 % 32) + min(lane, kPages - 1));
    if (lane == 0) bar_expect_tx(r_full, static_cast<uint32_t>(pages0 * T::kPageBytes));
    __syncwarp();
    if (lane < pages0) {
      const int id = (id0 < 0 || id0 >= p.num_blocks) ? 0 : id0;  // flagged by the producer below
      tma_load_4d(s_base + T::kOffKV + lane * T::kPageBytes, &map_k, 2 * (id * p.num_kv_heads + kvh), r_full);
    }
  }
  if (tid == 0) {
    bar_init(v_tail, 1);
    for (int t = 0; t < kTiles; ++t) {
      bar_init(s_full + 8 * t, 1);
      bar_init(p_full + 8 * t, 128);
      bar_init(o_full + 8 * t, 1);
      bar_init(q_ready + 8 * t, 128);
      bar_init(mma_drained + 8 * t, 1);
      bar_init(o_staged + 8 * t, kRows);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp == kProducerWarp) {
    // ---------------- TMA producer (whole warp) ----------------
    // Block ids come from a 32-page window held one per lane, with the next
    // window already in flight, so no copy waits on a dependent table load.
    static_assert(32 % kPages == 0, "a step's pages sit in one window, one copy per lane");
    auto check = [&](int page, int id) -> int {
      if (page >= npages) return 0;
      if (id < 0 || id >= p.num_blocks) {
        atomicOr(p.err, kErrBlockId);
        return 0;
      }
      return id;
    };
    auto fetch = [&](int page) -> int { return page < npages ? check(page, __ldg(table + page)) : 0; };
    int win = w0;
    int id_cur = check(32 * w0 + lane, raw_cur), id_next = check(32 * (w0 + 1) + lane, raw_next);
    int issued = 0;  // ring tiles issued
    // One copy per lane, lane = page of the step: a thread's tensor copies issue one
    // after another, slowly, while copies from different lanes go out together.  A
    // copy moves a whole page of the kv head (both dims halves, 4 KB at D = 128).
    const int my_pg = lane;
    auto issue = [&](int j, int my_id, uint32_t dst, const CUtensorMap* map, uint32_t full) {  // j: absolute step
      const int pages = min(kPages, npages - j * kPages);
      if (lane == 0) bar_expect_tx(full, static_cast<uint32_t>(pages * T::kPageBytes));
      __syncwarp();
      if (my_pg < pages) tma_load_4d(dst + my_pg * T::kPageBytes, map, 2 * (my_id * p.num_kv_heads + kvh), full);
    };
    int my_id = 0;  // this lane's page id of the current step (its K and its V)
    for (int n = 0; n < 2 * nsteps && !failed; ++n) {  // tile n: K (even) or V (odd) of step n / 2
      const int jn = n >> 1, slot = n % kRing;
      if (n >= kRing && !__all_sync(0xffffffffu, bar_wait(r_empty + 8 * slot, ((n / kRing) + 1) & 1))) {
        failed = true;
        break;
      }
      if ((n & 1) == 0) {
        const int first_page = (j0 + jn) * kPages;
        if (first_page / 32 != win) {  // slide the window
          ++win;
          id_cur = id_next;
          id_next = fetch(32 * (win + 1) + lane);
        }
        my_id = __shfl_sync(0xffffffffu, id_cur, (first_page % 32) + min(my_pg, kPages - 1));
      }
      if (n > 0)  // K of the first step went out before the set-up barrier
        issue(j0 + jn, my_id, s_base + T::kOffKV + slot * T::kTile, (n & 1) ? &map_v : &map_k, r_full + 8 * slot);
      issued = n + 1;
    }
    if (!failed && tail) {
      // Keys past the CTA's end in the last V tile (a page's tail, or pages not
      // copied): zero their rows once the copy has landed, so that stale or NaN
      // data never meets p = 0, then release the tile to the MMA warps.
      const int jv = nsteps - 1, nv = 2 * jv + 1;
      if (__all_sync(0xffffffffu, bar_wait(r_full + 8 * (nv % kRing), (nv / kRing) & 1))) {
        unsigned char* vt = smem + T::kOffKV + (nv % kRing) * T::kTile;
        const int first = kv_end - (j0 + jv) * kKeys;
        for (int idx = lane; idx < (kKeys - first) * T::kHalves * 8; idx += 32) {
          const int r = first + idx / (T::kHalves * 8);
          const int rem = idx % (T::kHalves * 8);
          *reinterpret_cast<uint4*>(vt + kv_off<D>(r, rem / 8, rem % 8)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) bar_arrive(v_tail);
      } else {
        failed = true;
      }
    }
    if (failed && lane == 0) {  // let the copies still in flight land before the CTA exits
      atomicOr(p.err, kErrTimeout);
      for (int n = issued > kRing ? issued - kRing : 0; n < issued; ++n)
        bar_wait(r_full + 8 * (n % kRing), (n / kRing) & 1);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (lane 0 alone) ----------------
    // Ping-pong over the two tiles: S of both for step 0, then per step j and tile
    // t: O_t += P_t V_j as soon as P_t is ready, followed at once by S_t of step
    // j + 1.  The tensor pipe runs one tile's MMAs while the other tile's softmax
    // runs.  S = Q K^T is N = 128 keys, P V is N = D.
    // The issuer shares its SM sub-partition with two softmax warps whose dense
    // floating-point runs leave it few issue slots, and the pipe idles whenever the
    // issuer is late at a group boundary.  So lane 0 runs the loop alone (no warp
    // collectives), waits by polling without suspending, and does a step's copy waits
    // (V of the step and K of the next) before the tiles' groups, so that a tile's
    // P.V and next S issue back to back.
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kKeys, false);
      constexpr uint32_t kIdPV = idesc_bf16(D, true);
      const uint32_t kv_base = s_base + T::kOffKV;
      // A descriptor's address field is (address >> 4) in 14 bits and every address here is below
      // 256 KB, so the descriptor of base + offset is the base's descriptor + (offset >> 4): one add
      // of a constant per MMA operand.
      const uint64_t d_q = sdesc(s_base + T::kOffQ), d_kv = sdesc(kv_base, 1024, T::kGroupBytes);
      auto issue_s = [&](int t, int j) {
        const uint64_t q = d_q + static_cast<uint32_t>((t * T::kQTile) >> 4);
        const uint64_t k = d_kv + static_cast<uint32_t>((((2 * j) % kRing) * T::kTile) >> 4);
#pragma unroll
        for (int h = 0; h < T::kHalves; ++h)  // four K steps of 16 dims (32 bytes) per 64-dim half
          mma4_ss<kIdS, 2, 2>(tmem + col_s(t), q + static_cast<uint32_t>((h * T::kQHalf) >> 4),
                              k + static_cast<uint32_t>((h * 1024) >> 4), h != 0);
        mma_commit(s_full + 8 * t);
      };
      for (int t = 0; t < n_tiles; ++t)
        if (!bar_poll(q_ready + 8 * t, 0)) failed = true;
      if (!failed && !bar_poll(r_full, 0)) failed = true;  // K of step 0: tile 0, slot 0
      if (!failed) {
        tc_after_sync();
        for (int t = 0; t < n_tiles; ++t) issue_s(t, 0);
        mma_commit(r_empty);
      }
      for (int j = 0; j < nsteps && !failed; ++j) {
        const int nv = 2 * j + 1, sv = nv % kRing;  // V of step j
        const int nk = 2 * j + 2, sk = nk % kRing;  // K of step j + 1
        const bool last = j == nsteps - 1;
        if (!(last && tail ? bar_poll(v_tail, 0) : bar_poll(r_full + 8 * sv, (nv / kRing) & 1)) ||
            (!last && !bar_poll(r_full + 8 * sk, (nk / kRing) & 1))) {
          failed = true;
          break;
        }
        const uint64_t v = d_kv + static_cast<uint32_t>((sv * T::kTile) >> 4);
        for (int t = 0; t < n_tiles; ++t) {
          if (!bar_poll(p_full + 8 * t, j & 1)) {
            failed = true;
            break;
          }
          tc_after_sync();
          const uint32_t d_s = tmem + col_s(t);
#pragma unroll
          for (int g = 0; g < kKeys / 64; ++g)  // four pages of 16 keys each: P columns 8 apart
            mma4_ts<kIdPV, 8, T::kPageBytes / 16>(tmem + col_o(t), d_s + g * 32,
                                                  v + static_cast<uint32_t>((g * 4 * T::kPageBytes) >> 4), (j | g) != 0);
          if (last) mma_commit(o_full + 8 * t);
          // The last reader of this V slot is issued: release it as soon as that P.V retires, not
          // after the S of the next step, so that the producer can refill it sooner.
          if (t == n_tiles - 1) mma_commit(r_empty + 8 * sv);
          if (!last) issue_s(t, j + 1);  // overwrites P only after the P.V above (same issuer, in order)
        }
        if (failed) break;
        if (!last) mma_commit(r_empty + 8 * sk);  // both tiles' S of step j + 1 are in
      }
      if (failed) atomicOr(p.err, kErrTimeout);
      // Every MMA this lane issued must have completed before the TMEM is freed.
      mma_commit(mma_drained);
      bar_poll(mma_drained, 0);
    }
    __syncwarp();
  } else if ((warp >> 2) < n_tiles) {
    // ---------------- softmax / epilogue (warps 0-7, thread = row of tile warp / 4) ----------------
    const int t = warp >> 2;
    const int r = tid & (kRows - 1);
    const int i = i0 + t * kTokens + r / G;  // chunk token of this row
    const bool row_ok = i < C;
    // Q's copies were issued before the set-up barrier (see there).
    constexpr int kChunks = D / 8;  // 16-byte chunks of a row
    cp_async_wait_all();
    fence_async_smem();
    bar_arrive(q_ready + 8 * t);
    const float qk = p.scale * kLog2e;
    const int limit = row_ok ? prefix + i + 1 : 0;  // keys this row may see
    // A row sees a key of this CTA's steps unless a split's range starts past its causal limit;
    // a row that sees none keeps m = -inf, l = 0 (all its p are 0).
    const bool sees = kSplit ? limit > j0 * kKeys : row_ok;
    float m_used = -INFINITY, l = 0.f;
    // A warp reaches the TMEM lanes 32 * (warp % 4) .. + 31: rows r of either tile.
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_cols = lane_base + col_s(t), o_cols = lane_base + col_o(t);
    for (int j = 0; j < nsteps && !failed; ++j) {
      // S of step j has landed, and with it the tile's P.V of step j - 1 (same issuer, issued before).
      if (!__all_sync(0xffffffffu, bar_wait(s_full + 8 * t, j & 1))) {
        failed = true;
        break;
      }
      tc_after_sync();
      float s[kKeys];
      tmem_ld64(s_cols, *reinterpret_cast<float(*)[64]>(&s[0]));
      tmem_ld64(s_cols + 64, *reinterpret_cast<float(*)[64]>(&s[64]));
      // Causal / length mask, only on steps that some row of the warp does not see whole.
      const int ja = j0 + j;  // absolute key step
      if (__any_sync(0xffffffffu, (ja + 1) * kKeys > limit)) {
#pragma unroll
        for (int x = 0; x < kKeys; ++x) s[x] = (ja * kKeys + x) < limit ? s[x] : -INFINITY;
      }
      // Row max: eight chains of three-input maxima, then their maximum.
      static_assert(kKeys % 8 == 0 && kKeys >= 24, "row max layout");
      float mc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mc[k] = fmax3(s[k], s[k + 8], s[k + 16]);
      constexpr int kPairsEnd = 24 + ((kKeys - 24) / 16) * 16;
#pragma unroll
      for (int x = 24; x < kPairsEnd; x += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) mc[k] = fmax3(mc[k], s[x + k], s[x + 8 + k]);
      if constexpr (kPairsEnd < kKeys) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mc[k] = fmaxf(mc[k], s[kPairsEnd + k]);
      }
      const float row_max = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
      const float bm = row_max * qk;  // the scale is positive: the max of the scaled scores
      const bool raise = sees && bm > m_used + kSlack;
      const float m_new = raise ? bm : m_used;
      const float alpha = raise ? ex2_approx(m_used - m_new) : 1.f;  // 0 on the first raise
      const float neg_m = sees ? -m_new : 0.f;                        // rows seeing no key: all p = 0
      float2 acc4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
      uint32_t packed[kKeys / 2];
      const float2 qk2 = make_float2(qk, qk), neg_m2 = make_float2(neg_m, neg_m);
#pragma unroll
      for (int x = 0; x < kKeys; x += 2) {
        // Paired fp32 arithmetic (one FFMA2 / FADD2 per two keys); the denominator
        // sums the fp32 weights, within 2^-9 relative of the bf16 ones P carries.
        const float2 e = __ffma2_rn(make_float2(s[x], s[x + 1]), qk2, neg_m2);
        const float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
        packed[x / 2] = pack_bf16(p0, p1);
        acc4[(x / 2) & 3] = __fadd2_rn(acc4[(x / 2) & 3], make_float2(p0, p1));
      }
      const float2 a01 = __fadd2_rn(acc4[0], acc4[1]), a23 = __fadd2_rn(acc4[2], acc4[3]);
      const float2 a = __fadd2_rn(a01, a23);
      l = l * alpha + (a.x + a.y);
      m_used = m_new;
      // O is rescaled in place (its previous P.V has retired: see the wait above).
      if (j >= 1 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(o_cols + c0, o);
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] *= alpha;
          tmem_st32(o_cols + c0, o);
        }
      }
      // P over the first kKeys / 2 columns of the S buffer, already read: the
      // tensor-memory A operand of O += P V.
      tmem_st32_raw(s_cols, *reinterpret_cast<const uint32_t(*)[32]>(&packed[0]));
      tmem_st32_raw(s_cols + 32, *reinterpret_cast<const uint32_t(*)[32]>(&packed[32]));
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_before_sync();
      bar_arrive(p_full + 8 * t);
    }
    // Epilogue: O / l in bf16, staged in the tile's Q buffer (every S that read it has retired:
    // the O-final commit follows them) in Q's own layout, the 128-byte-swizzled dims halves of
    // rows ordered token-major, head-minor, which is a tensor box of the output.  A tile whose
    // rows all lie in the chunk then leaves as one tensor store per half; the last, partial tile
    // of a chunk is stored by the tile's 128 threads together, a warp two whole rows at a time.
    if constexpr (partial) {
      // Split call: the tile's rows leave as fp32 partial states, O unnormalised with the running
      // max m (base 2) and sum l they were formed against, for the merge kernel.
      // A thread holds one row; the warp's 32 rows go out through its own 4 KB of the tile's Q buffer
      // (free: every S that read it has retired), 32 columns at a time: written a row per lane with
      // the 16-byte chunks rotated by the row (no bank conflict), read back a quarter-row per lane,
      // so that each store instruction writes four 128-byte row segments.
      if (!failed && __all_sync(0xffffffffu, bar_wait(o_full + 8 * t, 0))) {
        tc_after_sync();
        const size_t row =
            ((static_cast<size_t>(split) * p.num_seqs + b) * p.ws_rows + i) * p.num_q_heads + kvh * G + r % G;
        float* scratch = reinterpret_cast<float*>(smem + T::kOffQ + t * T::kQTile) + (warp & 3) * 32 * 32;
        const size_t seq_row0 = (static_cast<size_t>(split) * p.num_seqs + b) * p.ws_rows;  // chunk row 0
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(o_cols + c0, o);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            *reinterpret_cast<float4*>(scratch + lane * 32 + ((q4 + lane) & 7) * 4) =
                make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + (lane >> 3), q4 = lane & 7;  // the warp's row rr, its chunk q4
            const float4 v = *reinterpret_cast<const float4*>(scratch + rr * 32 + ((q4 + rr) & 7) * 4);
            const int tr = (warp & 3) * 32 + rr;        // tile row
            const int ii = i0 + t * kTokens + tr / G;  // its chunk token
            if (ii < C)
              *reinterpret_cast<float4*>(p.ws + ((seq_row0 + ii) * p.num_q_heads + kvh * G + tr % G) * D + c0 +
                                         q4 * 4) = v;
          }
          __syncwarp();
        }
        if (row_ok)
          reinterpret_cast<float2*>(p.ws + static_cast<size_t>(p.num_splits) * p.num_seqs * p.ws_rows *
                                               p.num_q_heads * D)[row] = make_float2(m_used, l);
      } else {
        failed = true;
      }
    } else {
      bool staged = false;
      unsigned char* ot = smem + T::kOffQ + t * T::kQTile;
      if (!failed && __all_sync(0xffffffffu, bar_wait(o_full + 8 * t, 0))) {
        tc_after_sync();
        const float inv = l > 0.f ? 1.f / l : 0.f;
  #pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(o_cols + c0, o);
  #pragma unroll
          for (int x = 0; x < 32; x += 8) {
            const int ch = (c0 + x) / 8;
            *reinterpret_cast<uint4*>(ot + (ch / 8) * T::kQHalf + swz(r, ch % 8)) =
                make_uint4(pack_bf16(o[x] * inv, o[x + 1] * inv), pack_bf16(o[x + 2] * inv, o[x + 3] * inv),
                           pack_bf16(o[x + 4] * inv, o[x + 5] * inv), pack_bf16(o[x + 6] * inv, o[x + 7] * inv));
          }
        }
        fence_async_smem();  // the tensor store reads the rows through the async proxy
        staged = true;
      } else {
        failed = true;
      }
      // Every thread of the tile arrives, staged or not, so that the bounded wait below ends.
      bar_arrive(o_staged + 8 * t);
      if (__all_sync(0xffffffffu, staged && bar_wait(o_staged + 8 * t, 0))) {
        const int tok0 = i0 + t * kTokens;
        // The tensor map spans num_seqs * max_query_len tokens; a chunk longer than max_query_len (an
        // error the device flags) can put rows past that, which the threads store instead.
        const int64_t map_tokens = static_cast<int64_t>(p.num_seqs) * p.max_query_len;
        if (tok0 + kTokens <= C && static_cast<int64_t>(q0) + tok0 + kTokens <= (map_tokens < INT32_MAX ? map_tokens : INT32_MAX)) {
          if (r == 0) {
  #pragma unroll
            for (int h = 0; h < T::kHalves; ++h)
              tma_store_3d(&map_out, 64 * h, kvh * G, q0 + tok0, s_base + T::kOffQ + t * T::kQTile + h * T::kQHalf);
            tma_store_commit_and_wait_read();  // the buffer is read before the CTA may leave
          }
        } else {
          __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.out);
  #pragma unroll 4
          for (int c = r; c < kRows * kChunks; c += kRows) {
            const int rr = c / kChunks, ch = c % kChunks;
            const int ii = tok0 + rr / G;
            if (ii < C)
              reinterpret_cast<uint4*>(og + (static_cast<size_t>(q0 + ii) * p.num_q_heads + kvh * G + rr % G) * D)[ch] =
                  *reinterpret_cast<const uint4*>(ot + (ch / 8) * T::kQHalf + swz(rr, ch % 8));
          }
        }
      } else {
        failed = true;
      }
    }
    if (failed && lane == 0) atomicOr(p.err, kErrTimeout);
  }

  // Everyone done with TMEM (the MMA warp drained its MMAs).
  tc_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}


// Merge of a split call (the split-K reduction, as in decode): for every chunk row, over the splits
// whose m is finite, M = max m_s and out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, rounded to
// bf16.  A warp takes four (chunk token, q head) rows at a time; lane s reads split s's (m, l).  Rows of a sequence
// the attention kernel rejected are left untouched, as the unsplit call leaves them.
template <int D>
__global__ void __launch_bounds__(256) paged_prefill_merge_kernel(const PrefillParams p) {
  pdl_trigger();
  pdl_wait();
  static_assert(D % 64 == 0, "a lane takes D / 32 contiguous columns, an even count");
  constexpr int kCols = D / 32;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = p.query_start[b];
  const int C = p.query_start[b + 1] - q0;
  const int L = p.context_lens[b];
  if (C < 0 || L < C || L > p.max_blocks_per_seq * kBlockTokens) return;  // flagged by the attention kernel
  const int rows = min(C, p.ws_rows) * p.num_q_heads;
  const size_t split_stride = static_cast<size_t>(p.num_seqs) * p.ws_rows * p.num_q_heads;  // rows per split
  const float2* ml =
      reinterpret_cast<const float2*>(p.ws + static_cast<size_t>(p.num_splits) * split_stride * D);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  constexpr int kRowsPerWarp = 4;  // loads of four rows in flight at once
  for (int row4 = (blockIdx.x * 8 + warp) * kRowsPerWarp; row4 < rows; row4 += gridDim.x * 8 * kRowsPerWarp) {
    const size_t r0 = static_cast<size_t>(b) * p.ws_rows * p.num_q_heads + row4;  // the first row in split 0
    float m[kRowsPerWarp], l[kRowsPerWarp];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      m[k] = -INFINITY;
      l[k] = 0.f;
      if (lane < p.num_splits && row4 + k < rows) {
        const float2 v = ml[lane * split_stride + r0 + k];
        m[k] = v.x;
        l[k] = v.y;
      }
    }
    float w[kRowsPerWarp], inv[kRowsPerWarp];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      float mx = m[k];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      w[k] = m[k] == -INFINITY ? 0.f : exp2f(m[k] - mx);
      float den = w[k] * l[k];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
      inv[k] = den > 0.f ? 1.f / den : 0.f;
    }
    float acc[kRowsPerWarp][kCols];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k)
#pragma unroll
      for (int c = 0; c < kCols; ++c) acc[k][c] = 0.f;
    for (int sp = 0; sp < p.num_splits; ++sp) {
#pragma unroll
      for (int k = 0; k < kRowsPerWarp; ++k) {
        const float wsp = __shfl_sync(0xffffffffu, w[k], sp);
        if (wsp == 0.f) continue;  // the same for the whole warp
        const float* o = p.ws + (sp * split_stride + r0 + k) * D + lane * kCols;
#pragma unroll
        for (int c = 0; c < kCols; c += 2) {
          const float2 v = *reinterpret_cast<const float2*>(o + c);
          acc[k][c] += wsp * v.x;
          acc[k][c + 1] += wsp * v.y;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      if (row4 + k >= rows) break;
      const int i = (row4 + k) / p.num_q_heads, h = (row4 + k) % p.num_q_heads;
      __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(
          out + (static_cast<size_t>(q0 + i) * p.num_q_heads + h) * D + lane * kCols);
#pragma unroll
      for (int c = 0; c < kCols; c += 2)
        dst[c / 2] = __floats2bfloat162_rn(acc[k][c] * inv[k], acc[k][c + 1] * inv[k]);
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t encoder(EncodeTiled* out) {
  static std::mutex mu;
  static EncodeTiled fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !ptr) return cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiled>(ptr);
  }
  *out = fn;
  return cudaSuccess;
}

// The cache viewed as [num_blocks * num_kv_heads * 16 rows][head_dim] bf16; box 16 rows x 64 dims.
cudaError_t cache_map(CUtensorMap* map, const void* cache, int64_t rows, int head_dim) {
  EncodeTiled enc = nullptr;
  cudaError_t e = encoder(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlockTokens)};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The cache as pages for the prefill kernel: 4D [row groups][halves][8 rows][64 dims] bf16
// (rows = num_blocks * num_kv_heads * 16, two 8-row groups a page), box 64 x 8 x halves x 2:
// one copy moves a whole page of one kv head into [group][half][8 rows][128 B], 128-byte
// swizzle (each half's 8 rows one swizzle atom).
cudaError_t page_map(CUtensorMap* map, const void* cache, int64_t rows, int head_dim) {
  EncodeTiled enc = nullptr;
  cudaError_t e = encoder(&enc);
  if (e != cudaSuccess) return e;
  const cuuint32_t halves = static_cast<cuuint32_t>(head_dim / 64);
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(head_dim) * 2;
  const cuuint64_t dims[4] = {64, 8, halves, static_cast<cuuint64_t>(rows / 8)};
  const cuuint64_t strides[3] = {row_bytes, 128, 8 * row_bytes};
  const cuuint32_t box[4] = {64, 8, halves, 2};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The output as [tokens][num_q_heads][head_dim] bf16 for tensor stores: box 64 dims x G heads x kTokens
// tokens, 128-byte swizzle.  `tokens` bounds the box coordinates only (stores land in whole tiles of rows
// that lie in a chunk, below the call's total token count).
cudaError_t out_map(CUtensorMap* map, void* out, int64_t tokens, int num_q_heads, int head_dim, int group,
                    int tile_tokens) {
  EncodeTiled enc = nullptr;
  cudaError_t e = encoder(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                              static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(num_q_heads) * head_dim * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tile_tokens)};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int G, bool kSplit>
cudaError_t launch_t(const PrefillParams& p, int max_query_len, cudaStream_t stream) {
  constexpr int kCtaTokens = kTiles * kRows / G;
  static std::mutex mu;
  static uint64_t ready = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!(dev < 64 && ((ready >> dev) & 1u))) {
      e = cudaFuncSetAttribute(&paged_prefill_kernel<D, G, kSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Pf<D>::kSmem);
      if (e != cudaSuccess) return e;
      if (dev < 64) ready |= uint64_t{1} << dev;
    }
  }
  CUtensorMap mk, mv;
  const int64_t rows = p.num_blocks * p.num_kv_heads * kBlockTokens;
  if ((e = page_map(&mk, p.k_cache, rows, D)) != cudaSuccess) return e;
  if ((e = page_map(&mv, p.v_cache, rows, D)) != cudaSuccess) return e;
  CUtensorMap mo;
  int64_t tokens = static_cast<int64_t>(p.num_seqs) * max_query_len;
  if (tokens > INT32_MAX) tokens = INT32_MAX;
  if ((e = out_map(&mo, p.out, tokens, p.num_q_heads, D, G, kRows / G)) != cudaSuccess) return e;
  const int tiles = (max_query_len + kCtaTokens - 1) / kCtaTokens;
  if constexpr (!kSplit) {
    const dim3 grid(p.num_kv_heads, tiles, p.num_seqs);
    return launch_pdl(paged_prefill_kernel<D, G, false>, grid, dim3(kThreads), Pf<D>::kSmem, stream, p, mk, mv, mo);
  } else {
    PrefillParams q = p;
    q.ws_rows = tiles * kCtaTokens;
    const dim3 grid(p.num_kv_heads, tiles, p.num_seqs * p.num_splits);
    e = launch_pdl(paged_prefill_kernel<D, G, true>, grid, dim3(kThreads), Pf<D>::kSmem, stream, q, mk, mv, mo);
    if (e != cudaSuccess) return e;
    const int64_t row_blocks = (static_cast<int64_t>(q.ws_rows) * p.num_q_heads + 31) / 32;  // 8 warps x 4 rows
    const dim3 mgrid(static_cast<unsigned>(row_blocks < 65535 ? row_blocks : 65535), p.num_seqs);
    return launch_pdl(paged_prefill_merge_kernel<D>, mgrid, dim3(256), 0, stream, q);
  }
}

}  // namespace

cudaError_t encode_cache_map(CUtensorMap_st* map, const void* cache, int64_t rows, int head_dim) {
  return cache_map(map, cache, rows, head_dim);
}

cudaError_t launch_paged_prefill(const PrefillParams& p, int head_dim, int group, int max_query_len,
                                 cudaStream_t stream) {
  const bool split = p.num_splits > 1;
  switch (head_dim * 16 + group) {
#define PKV_PREFILL_CASE(d, g) \
  case d * 16 + g: return split ? launch_t<d, g, true>(p, max_query_len, stream) : launch_t<d, g, false>(p, max_query_len, stream);
    PKV_PREFILL_CASE(64, 1)
    PKV_PREFILL_CASE(64, 2)
    PKV_PREFILL_CASE(64, 4)
    PKV_PREFILL_CASE(64, 8)
    PKV_PREFILL_CASE(128, 1)
    PKV_PREFILL_CASE(128, 2)
    PKV_PREFILL_CASE(128, 4)
    PKV_PREFILL_CASE(128, 8)
#undef PKV_PREFILL_CASE
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
