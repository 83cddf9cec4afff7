// Paged decode attention for GB300 (sm_103a).
//
// What is computed ("从零实现一个 mini vLLM--开篇", sections 2 and 5):
// for each sequence b and q head h, out = softmax(scale * q K^T) V over the
// context_lens[b] cached tokens, whose K/V rows are found through the
// sequence's block table (token t lives in block block_tables[b][t / 16] at
// offset t % 16).  GQA: q head h reads kv head h / G.
//
// How (GB300-first; the pages give no kernel, only the PyTorch definition):
//
// * Decomposition.  The batch is one flat stream of (sequence, kv head,
//   block) items, ordered sequence-major.  It is cut into num_partitions
//   contiguous pieces of equal block count, one per warp, so every warp moves
//   the same number of bytes whatever the length mix (a 131072-token sequence
//   is spread over many warps; a 5-token one shares a warp with others).  A
//   warp that covers a whole (sequence, kv head) pair writes its output rows
//   directly; a pair cut by a piece boundary leaves a partial softmax state
//   (m, l, acc) per piece, and the merge kernel combines them (split-K).
// * Memory pipeline.  Each warp owns a ring of S shared-memory stages.  One
//   lane issues cp.async.bulk (TMA bulk) copies of the block's K tile and V
//   tile (each one contiguous 16 x head_dim bf16 run in the
//   [block][kv head][16][head_dim] layout; 128-byte-swizzled 2D tensor copies
//   on the tensor-core path) plus, at the first block of a pair, the group's G
//   q rows, completing on an mbarrier.  Block ids are fetched one refill
//   ahead.  Every mbarrier wait has a time limit.
// * Compute, G <= 4.  CUDA cores (a GEMV with four or fewer rows per kv head
//   is bound by HBM).  Groups of eight heads run their two small products on
//   the tensor cores instead (process_block_mma).  A lane owns 8 consecutive dims
//   (one 16-byte shared-memory load per row).  Partial dot products of all
//   tokens of a block and all G heads are reduced across the lanes of a row
//   with a transpose-reduction; the lanes' token order and q-head order are
//   XOR-swizzled so every reduction level is a plain shuffle + add.  Packed
//   fp32x2 FMAs (FFMA2) do the q.K and p.V products.  Online softmax in base
//   2 with a lazy rescale: the running max is only raised when a block's max
//   exceeds it by more than 2^8, which keeps the exp2 arguments bounded and
//   skips the rescale of the accumulators on almost every block.
#include <cuda.h>  // CUtensorMap (maps are encoded on the host through the runtime's driver entry point)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kRescaleSlack = 8.0f;                       // base-2 units
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // a healthy wait is microseconds
constexpr unsigned long long kDrainTimeoutNs = 200000000ull;

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }
constexpr int cmin(int a, int b) { return a < b ? a : b; }

// Geometry of one (head_dim D, group G) instance.
template <int D, int G>
struct Geo {
  static constexpr int kLanesPerToken = D / 8;                 // lanes sharing one K/V row
  static constexpr int kTokensPerStep = 32 / kLanesPerToken;   // rows one warp-wide load covers
  static constexpr int kSteps = kBlockTokens / kTokensPerStep; // loads per 16-token tile
  static constexpr int kSlots = kSteps * G;                    // partial scores per lane per block
  static constexpr int kLevels = ilog2(kLanesPerToken);        // reduction levels across a row
  static constexpr int kHalvings = cmin(kLevels, ilog2(kSlots));
  static constexpr int kFinal = kSlots >> kHalvings;           // scores a lane holds after reduction
  static constexpr int kTokenLevels = cmin(ilog2(kSteps), kHalvings);
  static constexpr int kTileBytes = kBlockTokens * D * 2;
  static constexpr int kQBytes = G * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes + kQBytes;
  static constexpr int kPTileBytes = kBlockTokens * G * 8;     // {p, p} per (token, head)
  static constexpr int kPieceFloats = G * D + ((2 * G + 3) / 4) * 4;

  // Swizzle of lane c: physical slot k holds logical item k ^ mask_of(c),
  // item = token_step * G + head.  Level l of the reduction pairs lanes that
  // differ in bit (kLanesPerToken >> l) and halves the slots.
  __host__ __device__ static constexpr int mask_of(int c) {
    int m = 0;
    for (int l = 1; l <= kHalvings; ++l)
      if (c & (kLanesPerToken >> l)) m |= (kSlots >> l);
    return m;
  }
  // Lane bits whose value selects which heads a lane ends up holding.
  __host__ __device__ static constexpr int head_bits() {
    int bits = 0;
    for (int l = kTokenLevels + 1; l <= kHalvings; ++l) bits |= (kLanesPerToken >> l);
    return bits;
  }
  // Lane bits of the plain butterfly levels (lanes differing there hold copies).
  __host__ __device__ static constexpr int copy_bits() {
    int bits = 0;
    for (int l = kHalvings + 1; l <= kLevels; ++l) bits |= (kLanesPerToken >> l);
    return bits;
  }
  __host__ __device__ static constexpr int max_bits() { return 31 & ~head_bits(); }
  __host__ __device__ static constexpr int sum_bits() { return 31 & ~head_bits() & ~copy_bits(); }
  // A lane that holds head g (in slot g % kFinal).
  __host__ __device__ static constexpr int src_lane(int g) {
    for (int c = 0; c < kLanesPerToken; ++c) {
      const int m = mask_of(c);
      if (m / G == 0 && (m % G) == g - g % kFinal) return c;
    }
    return -1;
  }
  __host__ __device__ static constexpr bool valid() {
    for (int g = 0; g < G; ++g)
      if (src_lane(g) < 0) return false;
    return kFinal <= G && (G % kFinal) == 0 && kSteps >= 1;
  }
};

// Groups of PKV_MMA_MIN_G (4 or 8) or more q heads run q.K and p.V on the tensor
// cores (warp-level mma.sync, the group's heads as the N = 8 columns): at eight heads
// the CUDA cores are held back by the arithmetic (8 flop per byte), while for four or
// fewer they are bound by HBM and the tensor cores gain nothing (LLaMA-3-8B shape: 206
// against 204 us).  Either way one warp owns a ring and all the group's heads.
#ifndef PKV_MMA_MIN_G
#define PKV_MMA_MIN_G 8
#endif
static_assert(PKV_MMA_MIN_G == 4 || PKV_MMA_MIN_G == 8,
              "groups of eight always take the tensor cores; four may (their p tile holds the two 256-byte P tiles)");
template <int G>
struct Split {
  static constexpr bool kMma = G >= PKV_MMA_MIN_G;
};
// One ring stage: K tile | V tile | q rows.  The tensor-core path copies K and V as
// 128-byte-swizzled tensor tiles, whose stages start on 1024-byte boundaries.
template <int D, int G>
constexpr int stage_bytes() {
  return Split<G>::kMma ? (Geo<D, G>::kStageBytes + 1023) / 1024 * 1024 : Geo<D, G>::kStageBytes;
}

// Launch shape per (head_dim, group): warps per CTA and stages per warp's ring.  At
// D = 128, four q heads per kv head run best with four warps of three stages
// (LLaMA-3 shape: 201.6 against 209.6 us with eight warps of two); one or two heads
// with eight warps of two stages, since they do little arithmetic per byte and more
// warps keep more copies moving (Qwen3-shape trace: 6.20 against 5.76 TB/s); eight
// heads, on the tensor cores, with eight warps of two as well (LLaMA-3-70B shape:
// 201-202 us; 4 x 2 the same, 4 x 4 226).  The macros override the D = 128 shape
// for every group, for sweeps.
#ifndef PKV_D64_WARPS
#define PKV_D64_WARPS 4
#endif
#ifndef PKV_D64_STAGES
#define PKV_D64_STAGES 4
#endif
template <int D, int G>
struct Shape;
template <int G>
struct Shape<128, G> {
#ifdef PKV_D128_WARPS
  static constexpr int kWarps = PKV_D128_WARPS;
#else
  static constexpr int kWarps = G == 4 ? 4 : 8;
#endif
#ifdef PKV_D128_STAGES
  static constexpr int kStages = PKV_D128_STAGES;
#else
  static constexpr int kStages = G == 4 ? 3 : 2;
#endif
};
template <int G>
struct Shape<64, G> {
  static constexpr int kWarps = PKV_D64_WARPS;
  static constexpr int kStages = PKV_D64_STAGES;
};

// Shared memory of one CTA: a ring and a p tile per warp, a barrier per stage (and, on
// the tensor-core path, up to 1024 bytes to align the first stage).
template <int D, int G, int NW, int S>
constexpr size_t ring_smem_bytes() {
  return (Split<G>::kMma ? 1024 : 0) + size_t(NW) * S * stage_bytes<D, G>() + size_t(NW) * Geo<D, G>::kPTileBytes +
         size_t(NW) * S * 8;
}
template <int D, int G>
constexpr size_t static_smem_bytes() {
  return ring_smem_bytes<D, G, Shape<D, G>::kWarps, Shape<D, G>::kStages>();
}
template <int D, int G>
size_t partition_smem_bytes(int num_seqs) {
  return (static_smem_bytes<D, G>() + size_t(2 * num_seqs + 1) * 4 + 15) & ~size_t(15);
}
// Every instance fits the 227 KB a CTA may opt in to, with the largest batch's lengths and prefix.
template <int D, int G>
constexpr bool fits_largest_batch() {
  return static_smem_bytes<D, G>() + size_t(2 * PKV_MAX_SEQS + 1) * 4 + 16 <= 227u * 1024u;
}
static_assert(fits_largest_batch<64, 1>() && fits_largest_batch<64, 2>() && fits_largest_batch<64, 4>() &&
                  fits_largest_batch<64, 8>() && fits_largest_batch<128, 1>() && fits_largest_batch<128, 2>() &&
                  fits_largest_batch<128, 4>() && fits_largest_batch<128, 8>(),
              "partition kernel shared memory");

// ---------------------------------------------------------------------------
// PTX wrappers (mbarrier, bulk copy, timers).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// 2D tensor copy (box 64 dims x 16 rows of the cache, 128-byte swizzle) into shared memory.
__device__ __forceinline__ void tensor_load(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Warp-level tensor-core operand loads and the m16n8k16 bf16 MMA (fp32 accumulate).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}
__device__ __forceinline__ uint4 lds128(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }
// Two bf16 in one 32-bit word -> two fp32 (exact: bf16 is the top half of fp32).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// One 16-token block: scores, online-softmax update, p.V accumulation.
// ---------------------------------------------------------------------------
template <int D, int G, bool kMasked>
__device__ __forceinline__ void process_block(const unsigned char* sK, const unsigned char* sV, float2* ptile, const float2 (&q)[G][4],
                                              float2 (&acc)[G][4], float (&m_ref)[G],
                                              float (&m_mine)[Geo<D, G>::kFinal],
                                              float (&l_mine)[Geo<D, G>::kFinal], int c, int half, int mask,
                                              int valid) {
  using T = Geo<D, G>;
  constexpr int kFinal = T::kFinal;
  const int mj = mask / G;  // token-step part of the swizzle
  constexpr int kRowBytes = D * 2;

  // q . K_t partial sums over this lane's 8 dims, swizzled slots.
  float part[T::kSlots];
#pragma unroll
  for (int jp = 0; jp < T::kSteps; ++jp) {
    const int tok = T::kTokensPerStep * (jp ^ mj) + half;
    const uint4 w = lds128(sK + tok * kRowBytes + c * 16);
    const float2 k0 = bf16x2_to_float2(w.x), k1 = bf16x2_to_float2(w.y);
    const float2 k2 = bf16x2_to_float2(w.z), k3 = bf16x2_to_float2(w.w);
#pragma unroll
    for (int gp = 0; gp < G; ++gp) {
      float2 s2 = __fmul2_rn(q[gp][0], k0);
      s2 = __ffma2_rn(q[gp][1], k1, s2);
      s2 = __ffma2_rn(q[gp][2], k2, s2);
      s2 = __ffma2_rn(q[gp][3], k3, s2);
      part[jp * G + gp] = s2.x + s2.y;
    }
  }
  // Transpose-reduction across the lanes of a row: each level halves the slots.
#pragma unroll
  for (int l = 1; l <= T::kHalvings; ++l) {
    const int n = T::kSlots >> l;
#pragma unroll
    for (int i = 0; i < n; ++i) part[i] += __shfl_xor_sync(kFull, part[i + n], T::kLanesPerToken >> l);
  }
#pragma unroll
  for (int l = T::kHalvings + 1; l <= T::kLevels; ++l) part[0] += __shfl_xor_sync(kFull, part[0], T::kLanesPerToken >> l);

  // This lane now holds the full scores of logical items mask + k, k < kFinal.
  float s[kFinal];
  int tok_of[kFinal];
#pragma unroll
  for (int k = 0; k < kFinal; ++k) {
    const int item = mask + k;
    tok_of[k] = T::kTokensPerStep * (item / G) + half;
    s[k] = part[k];
    if (kMasked) s[k] = tok_of[k] < valid ? s[k] : -INFINITY;
  }
  // The running max of a head is raised only when some score of the block beats it by more
  // than the slack; one vote decides, and the per-head block max is formed only then.
  bool beats = false;
#pragma unroll
  for (int k = 0; k < kFinal; ++k) beats |= s[k] > m_mine[k] + kRescaleSlack;
  if (__any_sync(kFull, beats)) {  // warp-uniform
    float bm[kFinal];
#pragma unroll
    for (int k = 0; k < kFinal; ++k) {
      bm[k] = s[k];
#pragma unroll
      for (int bit = 1; bit < 32; bit <<= 1)
        if (T::max_bits() & bit) bm[k] = fmaxf(bm[k], __shfl_xor_sync(kFull, bm[k], bit));
    }
    float bm_all[G];
#pragma unroll
    for (int g = 0; g < G; ++g) bm_all[g] = __shfl_sync(kFull, bm[g % kFinal], T::src_lane(g));
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mn = fmaxf(m_ref[g], bm_all[g]);
      const float a = exp2f(m_ref[g] - mn);
      m_ref[g] = mn;
      const float2 a2 = make_float2(a, a);
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[g][i] = __fmul2_rn(acc[g][i], a2);
    }
#pragma unroll
    for (int k = 0; k < kFinal; ++k) {
      const float mn = fmaxf(m_mine[k], bm[k]);
      l_mine[k] *= exp2f(m_mine[k] - mn);
      m_mine[k] = mn;
    }
  }
#pragma unroll
  for (int k = 0; k < kFinal; ++k) {
    const float p = exp2f(s[k] - m_mine[k]);
    l_mine[k] += p;
    ptile[tok_of[k] * G + (mask + k) % G] = make_float2(p, p);
  }
  __syncwarp();

  // acc[g] += p_t,g * V_t over the block's tokens (this lane: its token parity, its 8 dims).
#pragma unroll
  for (int j = 0; j < T::kSteps; ++j) {
    const int tok = T::kTokensPerStep * j + half;
    uint4 w = lds128(sV + tok * kRowBytes + c * 16);
    if (kMasked && tok >= valid) w = make_uint4(0u, 0u, 0u, 0u);  // never multiply a stale row
    const float2 v0 = bf16x2_to_float2(w.x), v1 = bf16x2_to_float2(w.y);
    const float2 v2 = bf16x2_to_float2(w.z), v3 = bf16x2_to_float2(w.w);
    const float2* pp = ptile + tok * G;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float2 p2 = pp[g];
      acc[g][0] = __ffma2_rn(p2, v0, acc[g][0]);
      acc[g][1] = __ffma2_rn(p2, v1, acc[g][1]);
      acc[g][2] = __ffma2_rn(p2, v2, acc[g][2]);
      acc[g][3] = __ffma2_rn(p2, v3, acc[g][3]);
    }
  }
}

// ---------------------------------------------------------------------------
// One block on the tensor cores (groups of up to eight q heads, one warp).
//
// The stage holds K and V as 128-byte-swizzled tensor tiles: D / 64 halves of 16
// rows x 128 bytes (2 KB, 1024-byte aligned), the 16-byte chunk c of row r stored
// at chunk c ^ (r % 8), so every 8-row ldmatrix touches all 32 banks once.
//
//   S^T [16 tokens x 8 heads] = K [16 x D] . q^T [D x 8]       D / 16 MMAs m16n8k16
//   O^T [D x 8 heads]        += V^T [D x 16] . P^T [16 x 8]    2 D / 16 MMAs (P = hi + lo)
//
// Fragments (g = lane / 4, t = lane % 4): the S^T accumulator holds tokens g and
// g + 8 of heads 2t and 2t + 1, so a lane owns the running max and sum of its two
// heads; P goes through two 256-byte shared tiles ([token][head] bf16: the high
// part of each weight and its remainder) and comes back transposed by
// ldmatrix.trans as the B operands of two MMAs; the O^T accumulator o[mt] holds
// dims 16 mt + g and 16 mt + g + 8 of the same two heads.  Scores are scaled after
// the MMA (fp32); the weights reach P.V to within 2^-16 and the sum l adds them in fp32.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t swz_addr(uint32_t tile, int row, int chunk) {
  return tile + (chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

template <int D, bool kMasked>
__device__ __forceinline__ void process_block_mma(uint32_t sK, unsigned char* sV_ptr, uint32_t sV, uint32_t sP,
                                                  const uint32_t (&qf)[D / 16][2], float (&o)[D / 16][4],
                                                  float (&m)[2], float (&l)[2], float qscale, int lane, int valid) {
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3;  // which 8x8 matrix of an x4 load this lane addresses
  // Scores: K rows are the M dimension, the heads the N dimension.
  float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t a[4];
    ldsm_x4(swz_addr(sK, ((mi & 1) << 3) | (lane & 7), 2 * kk + (mi >> 1)), a);
    mma_16816(c, a, qf[kk][0], qf[kk][1]);
  }
  float s0 = c[0] * qscale, s1 = c[1] * qscale, s2 = c[2] * qscale, s3 = c[3] * qscale;
  if (kMasked) {
    if (g >= valid) s0 = s1 = -INFINITY;
    if (g + 8 >= valid) s2 = s3 = -INFINITY;
    // Stale rows past the sequence must not reach the MMA (0 * NaN): zero them.
    for (int x = lane; x < (kBlockTokens - valid) * (D / 8); x += 32) {
      const int row = valid + x / (D / 8), chunk = x % (D / 8);
      *reinterpret_cast<uint4*>(sV_ptr + (swz_addr(0, row, chunk))) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // Block max of each of this lane's two heads over the 16 tokens (lanes of equal t).
  float b0 = fmaxf(s0, s2), b1 = fmaxf(s1, s3);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    b0 = fmaxf(b0, __shfl_xor_sync(kFull, b0, off));
    b1 = fmaxf(b1, __shfl_xor_sync(kFull, b1, off));
  }
  // Lazy rescale: the running max moves only when a block beats it by more than the slack.
  if (__any_sync(kFull, b0 > m[0] + kRescaleSlack || b1 > m[1] + kRescaleSlack)) {
    const float n0 = fmaxf(m[0], b0), n1 = fmaxf(m[1], b1);
    const float a0 = exp2f(m[0] - n0), a1 = exp2f(m[1] - n1);
    m[0] = n0;
    m[1] = n1;
    l[0] *= a0;
    l[1] *= a1;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      o[mt][0] *= a0;
      o[mt][1] *= a1;
      o[mt][2] *= a0;
      o[mt][3] *= a1;
    }
  }
  const float p0 = exp2f(s0 - m[0]), p1 = exp2f(s1 - m[1]);  // token g: heads 2t, 2t + 1
  const float p2 = exp2f(s2 - m[0]), p3 = exp2f(s3 - m[1]);  // token g + 8
  l[0] += p0 + p2;
  l[1] += p1 + p3;
  // Each weight as bf16 hi + bf16 lo (the rounded-off rest): about 16 significant bits,
  // so P.V carries the fp32 weights to within 2^-16 and the result does not depend on
  // which running max a weight was taken against (how the stream was cut).
  const uint32_t h01 = float2_to_bf16x2(p0, p1), h23 = float2_to_bf16x2(p2, p3);
  const float2 r01 = bf16x2_to_float2(h01), r23 = bf16x2_to_float2(h23);
  const uint32_t l01 = float2_to_bf16x2(p0 - r01.x, p1 - r01.y), l23 = float2_to_bf16x2(p2 - r23.x, p3 - r23.y);
  __syncwarp();  // the previous block's P tiles have been read
  unsigned char* pt = reinterpret_cast<unsigned char*>(__cvta_shared_to_generic(sP));
  *reinterpret_cast<uint32_t*>(pt + g * 16 + t * 4) = h01;
  *reinterpret_cast<uint32_t*>(pt + (g + 8) * 16 + t * 4) = h23;
  *reinterpret_cast<uint32_t*>(pt + 256 + g * 16 + t * 4) = l01;
  *reinterpret_cast<uint32_t*>(pt + 256 + (g + 8) * 16 + t * 4) = l23;
  __syncwarp();
  uint32_t ph0, ph1, pl0, pl1;
  ldsm_x2_t(sP + (lane & 15) * 16, ph0, ph1);
  ldsm_x2_t(sP + 256 + (lane & 15) * 16, pl0, pl1);
  // O^T += V^T P^T: V rows are the K dimension, dims the M dimension.
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    uint32_t a[4];
    ldsm_x4_t(swz_addr(sV, ((mi >> 1) << 3) | (lane & 7), 2 * mt + (mi & 1)), a);
    mma_16816(o[mt], a, ph0, ph1);
    mma_16816(o[mt], a, pl0, pl1);
  }
}

// ---------------------------------------------------------------------------
// Fused decode step helpers: rotate-half RoPE of one lane's 8 dims.
// ---------------------------------------------------------------------------
// x: this lane's 8 values (dims 8c .. 8c+7 of a head row), y: the 8 values D/2
// away (the rotation partner).  Lanes of the first half rotate x*cos - y*sin,
// lanes of the second half x*cos + y*sin, with the frequencies of dims
// (8c + e) mod D/2.  Every product and sum is one fp32 operation rounded to
// nearest, then the result is rounded to bf16 -- the same steps as the oracle.
template <int D>
__device__ __forceinline__ uint4 rope_chunk(uint4 x, uint4 y, const float* cs_row, int c) {
  const int fbase = (8 * c) % (D / 2);
  const bool second = (8 * c) >= (D / 2);
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
  const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
  uint32_t ow[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float2 xv = bf16x2_to_float2(xw[w]);
    const float2 yv = bf16x2_to_float2(yw[w]);
    float r[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float xe = h ? xv.y : xv.x;
      const float ye = h ? yv.y : yv.x;
      const int f = fbase + 2 * w + h;
      const float cosv = __ldg(cs_row + f);
      const float sinv = __ldg(cs_row + D / 2 + f);
      const float a = __fmul_rn(xe, cosv);
      const float b = __fmul_rn(ye, sinv);
      r[h] = second ? __fadd_rn(a, b) : __fsub_rn(a, b);
    }
    ow[w] = float2_to_bf16x2(r[0], r[1]);
  }
  return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// Walk of the flat (sequence, kv head, block) stream.
struct Cursor {
  int b, kvh, blk, nblk;
};
__device__ __forceinline__ void advance(Cursor& cur, const int* s_prefix, int num_seqs, int hkv) {
  if (++cur.blk < cur.nblk) return;
  cur.blk = 0;
  if (++cur.kvh < hkv) return;
  cur.kvh = 0;
  do {
    ++cur.b;
    cur.nblk = s_prefix[cur.b + 1] - s_prefix[cur.b];
  } while (cur.nblk == 0 && cur.b + 1 < num_seqs);
}

template <int D, int G, int NW, int S>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_partition_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap map_k,
                                  const __grid_constant__ CUtensorMap map_v) {
  using T = Geo<D, G>;
  constexpr bool kMma = Split<G>::kMma;  // q.K and p.V on the tensor cores
  constexpr int kStage = stage_bytes<D, G>();
  static_assert(kMma || T::valid(), "unsupported (head_dim, group) geometry");
  static_assert(!kMma || T::kPTileBytes >= 512, "the tensor-core path keeps two 256-byte P tiles per warp");
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_wsum[32];

  const int B = p.num_seqs;
  const int hkv = p.num_kv_heads;
  unsigned char* stages = smem;
  if constexpr (kMma) {  // swizzled tensor tiles: the first stage on a 1024-byte boundary
    const uint32_t a = smem_addr(smem);
    stages = smem + (((a + 1023u) & ~1023u) - a);
  }
  float2* ptiles = reinterpret_cast<float2*>(stages + size_t(NW) * S * kStage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(ptiles) + NW * T::kPTileBytes);
  int* s_prefix = reinterpret_cast<int*>(bars + NW * S);
  int* s_len = s_prefix + (B + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool producer = lane == 0;  // issues this warp's copies
  pdl_trigger();
  pdl_wait();

  // --- CTA prologue: clamp lengths, block prefix over sequences -------------
  if (tid == 0) s_prefix[0] = 0;
  const int cap = p.max_blocks_per_seq * kBlockTokens;
  int running = 0;
  for (int base = 0; base < B; base += NW * 32) {
    const int idx = base + tid;
    int L = 0;
    if (idx < B) {
      L = __ldg(p.context_lens + idx);
      if (L < 0) {
        if (blockIdx.x == 0) atomicOr(p.err, kErrLenNegative);
        L = 0;
      }
      if (L > cap) {
        if (blockIdx.x == 0) atomicOr(p.err, kErrLenTooLong);
        L = cap;
      }
      s_len[idx] = L;
    }
    int x = (L + kBlockTokens - 1) / kBlockTokens;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < NW ? s_wsum[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFull, w, off);
        if (lane >= off) w += y;
      }
      if (lane < NW) s_wsum[lane] = w;
    }
    __syncthreads();
    if (idx < B) s_prefix[idx + 1] = running + (warp > 0 ? s_wsum[warp - 1] : 0) + x;
    running += s_wsum[NW - 1];
    __syncthreads();
  }
  if (blockIdx.x == 0)
    for (int i = tid; i <= B; i += NW * 32) p.ws_prefix[i] = s_prefix[i];

  // --- per-warp ring ----------------------------------------------------------
  unsigned char* ring_ptr = stages + size_t(warp) * S * kStage;
  const uint32_t ring = smem_addr(ring_ptr);
  const uint32_t bar0 = smem_addr(bars + warp * S);
  float2* ptile = ptiles + warp * (T::kPTileBytes / 8);
  if (producer) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const long long total = static_cast<long long>(hkv) * s_prefix[B];
  const int gw = blockIdx.x * NW + warp;  // this warp's piece
  if (gw >= p.num_partitions || total == 0) return;
  const long long begin = gw * total / p.num_partitions;
  const long long end = (gw + 1) * total / p.num_partitions;
  if (begin == end) return;
  const int n = static_cast<int>(end - begin);

  // Locate the first item: largest b with hkv * prefix[b] <= begin.
  Cursor cc;
  {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<long long>(hkv) * s_prefix[mid] <= begin) lo = mid;
      else hi = mid - 1;
    }
    cc.b = lo;
    cc.nblk = s_prefix[lo + 1] - s_prefix[lo];
    const int off = static_cast<int>(begin - static_cast<long long>(hkv) * s_prefix[lo]);
    cc.kvh = off / cc.nblk;
    cc.blk = off - cc.kvh * cc.nblk;
  }
  Cursor pc = cc;  // producer cursor (used by lane 0)

  const __nv_bfloat16* kbase = static_cast<const __nv_bfloat16*>(p.k_cache);
  const __nv_bfloat16* vbase = static_cast<const __nv_bfloat16*>(p.v_cache);
  const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(p.q);

  auto block_id = [&](const Cursor& cur) -> int {
    int id = __ldg(p.block_tables + static_cast<size_t>(cur.b) * p.max_blocks_per_seq + cur.blk);
    if (id < 0 || id >= p.num_blocks) {
      atomicOr(p.err, kErrBlockId);
      id = 0;
    }
    return id;
  };
  auto issue = [&](int stage, const Cursor& cur, int id, bool with_q) {
    const uint32_t dst = ring + stage * kStage;
    const uint32_t bar = bar0 + 8 * stage;
    mbar_arrive_expect_tx(bar, 2 * T::kTileBytes + (with_q ? T::kQBytes : 0));
    if constexpr (kMma) {
      const int row = (id * hkv + cur.kvh) * kBlockTokens;  // < 2^31: checked on the host
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tensor_load(dst + h * 2048, &map_k, 64 * h, row, bar);
        tensor_load(dst + T::kTileBytes + h * 2048, &map_v, 64 * h, row, bar);
      }
    } else {
      const size_t tile = (static_cast<size_t>(id) * hkv + cur.kvh) * (kBlockTokens * D);
      bulk_load(dst, kbase + tile, T::kTileBytes, bar);
      bulk_load(dst + T::kTileBytes, vbase + tile, T::kTileBytes, bar);
    }
    if (with_q)
      bulk_load(dst + 2 * T::kTileBytes, qbase + (static_cast<size_t>(cur.b) * p.num_q_heads + cur.kvh * G) * D,
                T::kQBytes, bar);
  };

  // Prologue: fetch the first S + 1 block ids together, fill the ring.
  int next_id = 0;
  if (producer) {
    int ids[S + 1];
    Cursor cur = pc;
#pragma unroll
    for (int s = 0; s <= S; ++s) {
      ids[s] = s < n ? block_id(cur) : 0;
      if (s + 1 < n) advance(cur, s_prefix, B, hkv);
    }
#pragma unroll
    for (int s = 0; s < S; ++s) {
      if (s < n) {
        issue(s, pc, ids[s], s == 0 || pc.blk == 0);
        if (s + 1 < n) advance(pc, s_prefix, B, hkv);
      }
    }
    next_id = ids[S];
  }

  const int c = lane & (T::kLanesPerToken - 1);
  const int half = lane / T::kLanesPerToken;
  const int mask = T::mask_of(c);
  const int mg = mask % G;
  const float qscale = p.qscale;

  // Tensor-core path: q^T fragments (bf16), the O^T accumulator, two heads' max and sum.
  uint32_t qf[D / 16][2];
  float o_t[D / 16][4];
  float m2[2], l2[2];
  // CUDA-core path: q and the accumulators per head (swizzled per lane), the maxima and sums.
  float2 q[G][4];  // q[gp]: head gp ^ mg
  float2 acc[G][4];
  float m_ref[G];
  float m_mine[T::kFinal], l_mine[T::kFinal];
  bool pair_from_start = false;
  bool first_pair = true;

  int stage = 0;
  uint32_t phase = 0;
  for (int i = 0; i < n; ++i) {
    const unsigned char* st_ptr = ring_ptr + stage * kStage;
    const bool landed = mbar_wait(bar0 + 8 * stage, phase, kWaitTimeoutNs);
    if (!__all_sync(kFull, landed)) {
      // Give up on this piece: flag it, let the copies already in flight land, leave.
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      for (int x = i; x < n && x < i + S; ++x) mbar_wait(bar0 + 8 * (x % S), (x / S) & 1, kDrainTimeoutNs);
      return;
    }
    const int seq_len = s_len[cc.b];
    if (i == 0 || cc.blk == 0) {
      // First block of a pair in this piece: load the group's q rows from the stage
      // (rotated to position len - 1 first when the step is fused with RoPE).
      const unsigned char* sq = st_ptr + 2 * T::kTileBytes;
      const float* cs_row = nullptr;
      if (p.cos_sin != nullptr) {
        int64_t pos = seq_len - 1;
        if (pos >= p.max_position) {
          if (lane == 0) atomicOr(p.err, kErrPosition);
          pos = p.max_position - 1;
        }
        cs_row = p.cos_sin + pos * D;
      }
      if constexpr (kMma) {
        if (cs_row != nullptr) {
          // Rotate the group's q rows in place; the result is rounded to bf16, as the
          // oracle rounds it, and enters the MMA unchanged.
          constexpr int kChunks = G * D / 8;
          constexpr int kPer = (kChunks + 31) / 32;
          unsigned char* sqw = ring_ptr + stage * kStage + 2 * T::kTileBytes;
          uint4 rot[kPer];
#pragma unroll
          for (int x = 0; x < kPer; ++x) {
            const int idx = lane + 32 * x;
            if (idx < kChunks) {
              const int head = idx / (D / 8), ch = idx % (D / 8);
              rot[x] = rope_chunk<D>(lds128(sq + head * (D * 2) + ch * 16),
                                     lds128(sq + head * (D * 2) + ((ch * 16 + D) % (D * 2))), cs_row, ch);
            }
          }
          __syncwarp();
#pragma unroll
          for (int x = 0; x < kPer; ++x) {
            const int idx = lane + 32 * x;
            if (idx < kChunks)
              *reinterpret_cast<uint4*>(sqw + (idx / (D / 8)) * (D * 2) + (idx % (D / 8)) * 16) = rot[x];
          }
          __syncwarp();
        }
        // q^T B fragments: head g (a zero column past the group), dims 16 kk + 2t (+1) and + 8.
        const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const unsigned char* qrow = sq + gq * (D * 2) + (16 * kk + 2 * tq) * 2;
          qf[kk][0] = gq < G ? *reinterpret_cast<const uint32_t*>(qrow) : 0u;
          qf[kk][1] = gq < G ? *reinterpret_cast<const uint32_t*>(qrow + 16) : 0u;
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) o_t[mt][0] = o_t[mt][1] = o_t[mt][2] = o_t[mt][3] = 0.f;
        m2[0] = m2[1] = -INFINITY;
        l2[0] = l2[1] = 0.f;
      } else {
#pragma unroll
        for (int gp = 0; gp < G; ++gp) {
          const int head = gp ^ mg;
          uint4 w = lds128(sq + head * (D * 2) + c * 16);
          if (cs_row != nullptr)
            w = rope_chunk<D>(w, lds128(sq + head * (D * 2) + ((c * 16 + D) % (D * 2))), cs_row, c);
          const float2 s2 = make_float2(qscale, qscale);
          q[gp][0] = __fmul2_rn(bf16x2_to_float2(w.x), s2);
          q[gp][1] = __fmul2_rn(bf16x2_to_float2(w.y), s2);
          q[gp][2] = __fmul2_rn(bf16x2_to_float2(w.z), s2);
          q[gp][3] = __fmul2_rn(bf16x2_to_float2(w.w), s2);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[gp][e] = make_float2(0.f, 0.f);
          m_ref[gp] = -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < T::kFinal; ++k) {
          m_mine[k] = -INFINITY;
          l_mine[k] = 0.f;
        }
      }
      pair_from_start = (cc.blk == 0);
      // Record where the pair starts for the merge: this piece, and the slot its state goes to
      // if the pair is cut (the piece's first pair, or a later one).
      if (pair_from_start && lane == 0)
        p.ws_pairs[2 * (static_cast<size_t>(cc.b) * hkv + cc.kvh)] = gw * 2 + (first_pair ? 0 : 1);
    }
    const int valid = seq_len - cc.blk * kBlockTokens;
    if (p.k_new != nullptr && cc.blk == cc.nblk - 1) {
      // Fused step: this block holds position len - 1, the step's new token.  Put its
      // (rotated) K row and its V row into the staged tiles and append them to the cache.
      const int row = (seq_len - 1) % kBlockTokens;
      if (half == 0) {
        const size_t src = (static_cast<size_t>(cc.b) * hkv + cc.kvh) * D;
        const uint4* kn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.k_new) + src);
        const uint4* vn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.v_new) + src);
        uint4 kw = __ldg(kn + c);
        const uint4 vw = __ldg(vn + c);
        if (p.cos_sin != nullptr) {
          int64_t pos = seq_len - 1;
          if (pos >= p.max_position) pos = p.max_position - 1;
          kw = rope_chunk<D>(kw, __ldg(kn + (c + D / 16) % (D / 8)), p.cos_sin + pos * D, c);
        }
        unsigned char* st_w = ring_ptr + stage * kStage;
        const uint32_t at = kMma ? swz_addr(0, row, c) : static_cast<uint32_t>(row * (D * 2) + c * 16);
        *reinterpret_cast<uint4*>(st_w + at) = kw;
        *reinterpret_cast<uint4*>(st_w + T::kTileBytes + at) = vw;
        int id = __ldg(p.block_tables + static_cast<size_t>(cc.b) * p.max_blocks_per_seq + cc.blk);
        if (id >= 0 && id < p.num_blocks) {
          const size_t dst = ((static_cast<size_t>(id) * hkv + cc.kvh) * kBlockTokens + row) * D;
          reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(const_cast<void*>(p.k_cache)) + dst)[c] = kw;
          reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(const_cast<void*>(p.v_cache)) + dst)[c] = vw;
        }
      }
      __syncwarp();
    }
    if constexpr (kMma) {
      const uint32_t sk = ring + stage * kStage;
      unsigned char* sv_ptr = ring_ptr + stage * kStage + T::kTileBytes;
      if (valid >= kBlockTokens)
        process_block_mma<D, false>(sk, sv_ptr, sk + T::kTileBytes, smem_addr(ptile), qf, o_t, m2, l2, qscale, lane,
                                    kBlockTokens);
      else
        process_block_mma<D, true>(sk, sv_ptr, sk + T::kTileBytes, smem_addr(ptile), qf, o_t, m2, l2, qscale, lane,
                                   valid);
    } else {
      if (valid >= kBlockTokens)
        process_block<D, G, false>(st_ptr, st_ptr + T::kTileBytes, ptile, q, acc, m_ref, m_mine, l_mine, c, half,
                                    mask, kBlockTokens);
      else
        process_block<D, G, true>(st_ptr, st_ptr + T::kTileBytes, ptile, q, acc, m_ref, m_mine, l_mine, c, half,
                                   mask, valid);
    }
    __syncwarp();

    // Refill the stage just consumed with block i + S.
    if (producer && i + S < n) {
      fence_proxy_async_smem();
      issue(stage, pc, next_id, pc.blk == 0);
      if (i + S + 1 < n) {
        advance(pc, s_prefix, B, hkv);
        next_id = block_id(pc);
      }
    }

    const bool last_of_pair = (cc.blk == cc.nblk - 1);
    if (last_of_pair && lane == 0) p.ws_pairs[2 * (static_cast<size_t>(cc.b) * hkv + cc.kvh) + 1] = gw;
    if (last_of_pair || i == n - 1) {
      if constexpr (kMma) {
        // Sum each head's l over the eight lanes that share it, then finish the pair
        // (O / l in bf16) or park its partial state (O, m, l in fp32).
        float la = l2[0], lb = l2[1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          la += __shfl_xor_sync(kFull, la, off);
          lb += __shfl_xor_sync(kFull, lb, off);
        }
        const int go = lane >> 2, ha = 2 * (lane & 3), hb = ha + 1;
        if (pair_from_start && last_of_pair) {
          __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                                (static_cast<size_t>(cc.b) * p.num_q_heads + cc.kvh * G) * D;
          const float ia = 1.0f / la, ib = 1.0f / lb;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = 16 * mt + go, d1 = d0 + 8;
            if (ha < G) {
              orow[ha * D + d0] = __float2bfloat16_rn(o_t[mt][0] * ia);
              orow[ha * D + d1] = __float2bfloat16_rn(o_t[mt][2] * ia);
            }
            if (hb < G) {
              orow[hb * D + d0] = __float2bfloat16_rn(o_t[mt][1] * ib);
              orow[hb * D + d1] = __float2bfloat16_rn(o_t[mt][3] * ib);
            }
          }
        } else {
          float* piece = p.ws_pieces + (static_cast<size_t>(gw) * 2 + (first_pair ? 0 : 1)) * T::kPieceFloats;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = 16 * mt + go, d1 = d0 + 8;
            if (ha < G) {
              piece[ha * D + d0] = o_t[mt][0];
              piece[ha * D + d1] = o_t[mt][2];
            }
            if (hb < G) {
              piece[hb * D + d0] = o_t[mt][1];
              piece[hb * D + d1] = o_t[mt][3];
            }
          }
          if (go == 0) {
            if (ha < G) {
              piece[G * D + ha] = m2[0];
              piece[G * D + G + ha] = la;
            }
            if (hb < G) {
              piece[G * D + hb] = m2[1];
              piece[G * D + G + hb] = lb;
            }
          }
        }
      } else {
      // Combine the token-parity lanes, then finish the pair or park its partial state.
#pragma unroll
      for (int off = T::kLanesPerToken; off < 32; off <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[g][e].x += __shfl_xor_sync(kFull, acc[g][e].x, off);
            acc[g][e].y += __shfl_xor_sync(kFull, acc[g][e].y, off);
          }
#pragma unroll
      for (int k = 0; k < T::kFinal; ++k)
#pragma unroll
        for (int bit = 1; bit < 32; bit <<= 1)
          if (T::sum_bits() & bit) l_mine[k] += __shfl_xor_sync(kFull, l_mine[k], bit);
      float l_all[G];
#pragma unroll
      for (int g = 0; g < G; ++g) l_all[g] = __shfl_sync(kFull, l_mine[g % T::kFinal], T::src_lane(g));

      if (pair_from_start && last_of_pair) {
        if (half == 0) {
          uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                 (static_cast<size_t>(cc.b) * p.num_q_heads + cc.kvh * G) * D) +
                        c;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float inv = 1.0f / l_all[g];
            uint4 o;
            o.x = float2_to_bf16x2(acc[g][0].x * inv, acc[g][0].y * inv);
            o.y = float2_to_bf16x2(acc[g][1].x * inv, acc[g][1].y * inv);
            o.z = float2_to_bf16x2(acc[g][2].x * inv, acc[g][2].y * inv);
            o.w = float2_to_bf16x2(acc[g][3].x * inv, acc[g][3].y * inv);
            orow[g * (D / 8)] = o;
          }
        }
      } else {
        float* piece = p.ws_pieces + (static_cast<size_t>(gw) * 2 + (first_pair ? 0 : 1)) * T::kPieceFloats;
        if (half == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float4* dst = reinterpret_cast<float4*>(piece + g * D + c * 8);
            dst[0] = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
            dst[1] = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            piece[G * D + g] = m_ref[g];
            piece[G * D + G + g] = l_all[g];
          }
        }
      }
      }
      first_pair = false;
    }
    if (i + 1 < n) advance(cc, s_prefix, B, hkv);
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

// ---------------------------------------------------------------------------
// Merge: combine the partial states of every pair cut by a piece boundary,
// write zeros for empty sequences.  One CTA per (sequence, kv head), one warp
// per q head of the group.
// ---------------------------------------------------------------------------
#ifndef PKV_MERGE_AHEAD
#define PKV_MERGE_AHEAD 8
#endif
template <int D, int G>
__global__ void __launch_bounds__(G * 32) paged_decode_merge_kernel(const DecodeParams p) {
  using T = Geo<D, G>;
  constexpr int kPer = D / 32;  // dims per lane
  const int hkv = p.num_kv_heads;
  const int b = blockIdx.x / hkv;
  const int kvh = blockIdx.x - b * hkv;
  const int g = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  // One round trip finds the pair's pieces: the partition kernel recorded the piece holding the
  // pair's first block (and the state slot there) and the piece holding its last block.
  const int len = p.context_lens[b];
  const int rec_a = p.ws_pairs[2 * static_cast<size_t>(blockIdx.x)];
  const int wb = p.ws_pairs[2 * static_cast<size_t>(blockIdx.x) + 1];
  const int total_blocks = p.ws_prefix[p.num_seqs];
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                        (static_cast<size_t>(b) * p.num_q_heads + kvh * G + g) * D + lane * kPer;
  if (len <= 0) {  // an empty sequence (a negative length reads as empty): zeros
#pragma unroll
    for (int e = 0; e < kPer; ++e) orow[e] = __float2bfloat16_rn(0.f);
    return;
  }
  const int wa = rec_a >> 1;
  if (wa == wb) return;  // whole pair in one piece: already written
  // With more pieces than items some pieces are empty and hold no state: only then are piece
  // bounds needed (piece w covers items [w N / P, (w + 1) N / P)).
  const long long total = static_cast<long long>(hkv) * total_blocks;
  const long long W = p.num_partitions;
  const bool may_be_empty = W > total;

  float M = -INFINITY, l = 0.f;
  float acc[kPer];
#pragma unroll
  for (int x = 0; x < kPer; ++x) acc[x] = 0.f;
  // Pieces PKV_MERGE_AHEAD at a time: their states are all fetched before any is combined
  // (a pair spans two or three pieces at the LLaMA-3 shape, five or six at the Qwen3 one).
  constexpr int kAhead = PKV_MERGE_AHEAD;
  for (int w0 = wa; w0 <= wb; w0 += kAhead) {
    float mw[kAhead], lw[kAhead], a[kAhead][kPer];
    bool use[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int w = w0 + u;
      use[u] = false;
      if (w <= wb) {
        if (!may_be_empty || w * total / W < (w + 1) * total / W) {  // an empty piece covers nothing
          use[u] = true;
          const int slot = w == wa ? (rec_a & 1) : 0;
          const float* piece = p.ws_pieces + (static_cast<size_t>(w) * 2 + slot) * T::kPieceFloats;
          mw[u] = piece[G * D + g];
          lw[u] = piece[G * D + G + g];
          if constexpr (kPer == 4) {
            const float4 v = *reinterpret_cast<const float4*>(piece + g * D + lane * 4);
            a[u][0] = v.x; a[u][1] = v.y; a[u][2] = v.z; a[u][3] = v.w;
          } else {
            const float2 v = *reinterpret_cast<const float2*>(piece + g * D + lane * 2);
            a[u][0] = v.x; a[u][1] = v.y;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      if (!use[u]) continue;
      const float mn = fmaxf(M, mw[u]);
      const float alpha = exp2f(M - mn);
      const float beta = exp2f(mw[u] - mn);
      l = l * alpha + lw[u] * beta;
#pragma unroll
      for (int x = 0; x < kPer; ++x) acc[x] = acc[x] * alpha + a[u][x] * beta;
      M = mn;
    }
  }
  const float inv = 1.0f / l;
  if constexpr (kPer == 4) {
    uint2 o;
    o.x = float2_to_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = float2_to_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(orow) = o;
  } else {
    *reinterpret_cast<uint32_t*>(orow) = float2_to_bf16x2(acc[0] * inv, acc[1] * inv);
  }
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait: one warp waits, with the given limit, on a
// shared-memory barrier that nothing completes.  The wait must give up and the
// warp report it in the error word, as a partition warp whose copy never lands
// does, and the kernel returns; nothing faults and the context stays usable.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool landed = mbar_wait(b, 0, limit_ns);
  if (!__all_sync(kFull, landed) && threadIdx.x == 0) atomicOr(err, kErrTimeout);
}

// ---------------------------------------------------------------------------
// Host side: per-instance launch helpers.
// ---------------------------------------------------------------------------
template <int D, int G>
struct Instance {
  static constexpr int NW = Shape<D, G>::kWarps;
  static constexpr int S = Shape<D, G>::kStages;
  static void* partition_fn() { return reinterpret_cast<void*>(&paged_decode_partition_kernel<D, G, NW, S>); }

  static cudaError_t prepare(int dev) {
    // Opt in to the largest dynamic shared memory this instance can ask for, once per device.
    static std::mutex mu;
    static uint64_t done_mask = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && (done_mask >> dev) & 1u) return cudaSuccess;
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    int max_bytes = static_cast<int>(partition_smem_bytes<D, G>(4096));
    if (max_bytes > optin) max_bytes = optin;
    e = cudaFuncSetAttribute(&paged_decode_partition_kernel<D, G, NW, S>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(&paged_decode_partition_kernel<D, G, NW, S>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (dev < 64) done_mask |= (uint64_t{1} << dev);
    return cudaSuccess;
  }

  static cudaError_t resident_pieces(int num_seqs, int* pieces) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare(dev)) != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, &paged_decode_partition_kernel<D, G, NW, S>,
                                                      NW * 32, partition_smem_bytes<D, G>(num_seqs));
    if (e != cudaSuccess) return e;
    *pieces = sms * (per_sm > 0 ? per_sm : 1) * NW;
    return cudaSuccess;
  }

  static cudaError_t partition(const DecodeParams& p, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare(dev)) != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>((p.num_partitions + NW - 1) / NW);
    CUtensorMap mk{}, mv{};
    if constexpr (Split<G>::kMma) {  // the caches as swizzled tensor tiles
      const int64_t rows = p.num_blocks * p.num_kv_heads * kBlockTokens;
      if (rows > INT32_MAX) return cudaErrorInvalidValue;  // tensor-copy row coordinates are 32-bit
      if ((e = encode_cache_map(&mk, p.k_cache, rows, D)) != cudaSuccess) return e;
      if ((e = encode_cache_map(&mv, p.v_cache, rows, D)) != cudaSuccess) return e;
    }
    return launch_pdl(paged_decode_partition_kernel<D, G, NW, S>, dim3(grid), dim3(NW * 32),
                      partition_smem_bytes<D, G>(p.num_seqs), stream, p, mk, mv);
  }

  static cudaError_t merge(const DecodeParams& p, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(p.num_seqs) * static_cast<unsigned>(p.num_kv_heads);
    return launch_pdl(paged_decode_merge_kernel<D, G>, dim3(grid), dim3(G * 32), 0, stream, p);
  }
};

template <typename F>
cudaError_t dispatch(int head_dim, int group, F&& f) {
  switch (head_dim * 16 + group) {
    case 64 * 16 + 1: return f(Instance<64, 1>{});
    case 64 * 16 + 2: return f(Instance<64, 2>{});
    case 64 * 16 + 4: return f(Instance<64, 4>{});
    case 64 * 16 + 8: return f(Instance<64, 8>{});
    case 128 * 16 + 1: return f(Instance<128, 1>{});
    case 128 * 16 + 2: return f(Instance<128, 2>{});
    case 128 * 16 + 4: return f(Instance<128, 4>{});
    case 128 * 16 + 8: return f(Instance<128, 8>{});
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int piece_floats(int head_dim, int group) { return group * head_dim + ((2 * group + 3) / 4) * 4; }

size_t workspace_prefix_bytes(int num_seqs) { return (static_cast<size_t>(num_seqs + 1) * 4 + 255) & ~size_t(255); }

size_t workspace_header_bytes(int num_seqs, int num_kv_heads) {
  return workspace_prefix_bytes(num_seqs) +
         ((static_cast<size_t>(num_seqs) * num_kv_heads * 8 + 255) & ~size_t(255));
}

cudaError_t resident_partition_pieces(int head_dim, int group, int num_seqs, int* pieces) {
  return dispatch(head_dim, group, [&](auto inst) { return decltype(inst)::resident_pieces(num_seqs, pieces); });
}

cudaError_t launch_decode_partition(const DecodeParams& p, int head_dim, int group, cudaStream_t stream) {
  return dispatch(head_dim, group, [&](auto inst) { return decltype(inst)::partition(p, stream); });
}

cudaError_t launch_bounded_wait_selftest(unsigned* err, unsigned long long limit_ns, cudaStream_t stream) {
  return launch_pdl(bounded_wait_selftest_kernel, dim3(1), dim3(32), 0, stream, err, limit_ns);
}

cudaError_t launch_decode_merge(const DecodeParams& p, int head_dim, int group, cudaStream_t stream) {
  return dispatch(head_dim, group, [&](auto inst) { return decltype(inst)::merge(p, stream); });
}

}  // namespace pkv
