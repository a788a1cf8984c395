// attention.cuh -- ExpCast FP8 attention forward for sm_103a.
//
// Method ("Open-VC attention" news item, "Solution: ExpCast" and
// "Architectural optimisations"; "Open VC Attention" catalogue entry;
// VC-Attention summary, "ExpCast-FP8"):
//   S = Q^ K^T on E4M3 tensor cores; online softmax with a running reference
//   m8 (1/8-log2 units) and row sum l; the probabilities are written as E4M3
//   bytes by one FMA on the log2-domain score,
//       code = clamp(rint(Z - m8 + c0 + beta), 0, 126),  Z = 8 log2(e) sm sq sk S,
//   with no exponent instruction and no FP32->FP8 conversion; O += P V^ on
//   E4M3 tensor cores; key blocks are visited cyclically from the middle one.
//
// Kernel design (one CTA per SM, persistent over tiles):
//   * a tile is two 128-row query blocks of one head (Q0, Q1);
//   * warp 8 (one lane) streams Q tiles and K/V^T blocks with TMA into a
//     kStages-deep ring of 128x128-byte tiles (128-byte swizzle);
//   * warp 9 (one lane) issues tcgen05.mma: S_t = Q_t K_j^T into TMEM
//     (kind::f8f6f4, M = N = 128, K = 32 per instruction), then
//     O_t += P_t V_j^T with P_t read from TMEM (it overwrites S_t's first 32
//     columns);
//   * warps 10-11 idle; warps 8-11 give registers to warps 0-7 (setmaxnreg);
//   * warps 0-3 and 4-7 are the softmax/ExpCast groups of Q0 and Q1: one
//     thread per query row reads its 128 scores with the max-reducing form of
//     tcgen05.ld (sm_103a), so the block max costs no instruction; applies the
//     lazy rescale; computes each code with one saturating FMA (clamp at 0)
//     and one FMA that adds 1.5*2^23 so that its rounding yields the integer
//     code in the low byte; packs bytes and writes them back with
//     tcgen05.st; only after handing P to the MMA warp does it add the
//     decoded bytes to l (f16x2 pairs), so the row sum runs while the tensor
//     core computes P.V and the next S instead of delaying them;
//   * TMEM: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512) columns.
// Every mbarrier wait is bounded (wall-clock limit); on expiry the CTA
// records a timeout, drains its own async copies and MMAs, frees TMEM and
// exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <cstdint>

#include "ptx.cuh"

namespace ovc {

constexpr int kStages = 4;
constexpr int kAttnThreads = 384;                          // 3 warpgroups
// Register split: 168 per thread at launch (384 x 168 = 64512 <= 65536);
// the producer/MMA warpgroup drops to 104 so that the two softmax warpgroups
// can hold 200 each: 256 x 200 + 128 x 104 = 64512.  (ptxas spills a few
// values at 216/64; 200 is enough for the 128 scores and 32 code words.)
constexpr int kSoftmaxRegs = 200;
constexpr int kControlRegs = 104;
static_assert(256 * kSoftmaxRegs + 128 * kControlRegs <= kAttnThreads * 168, "register split");
// V-Smooth's MMA warp keeps the run bookkeeping as well: 192 / 120 (its
// ExpCast warps fit in 192 with no spill).
constexpr int kSoftmaxRegsVSmooth = 192;
constexpr int kControlRegsVSmooth = 120;
static_assert(256 * kSoftmaxRegsVSmooth + 128 * kControlRegsVSmooth <= kAttnThreads * 168, "register split");
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTile = 128 * 128;                       // bytes of one E4M3 tile
constexpr uint32_t kIdesc = idesc_e4m3_f32(128, 128);
constexpr uint32_t kIdescBf16 = idesc_bf16_f32(128, 128);
constexpr uint32_t kMeanTile = 128 * 16 * 2;               // bytes of one M' tile: 128 channels x 16 blocks BF16
constexpr uint32_t kBiasTile = 128 * 16 * 2;               // bytes of one Q-smoothing operand tile: 128 rows x 16 BF16
// ExpCast constants: c0 = 120 (stored value 2^8 p), beta = -0.35, tau = 0.75.
constexpr float kCodeBase = 119.0f;                         // floor(c0 + beta)
constexpr float kFrac = 0.65f;                              // frac(c0 + beta)
constexpr float kLazy = 6.0f;                               // 8 * tau
constexpr uint64_t kDrainNs = 4000000000ull;

// Status bits recorded by kernels.
constexpr unsigned kStatusTimeout = 1u;

struct AttnParams {
  int32_t B, S, H, nb, S_pad, npairs, ntiles;
  // Split key ranges (short sequences): unit u = tile * nsplit + s covers key
  // blocks [s nb / nsplit, (s+1) nb / nsplit); with nsplit > 1 the epilogue
  // writes partial results for merge_kernel instead of O.
  int32_t nsplit, nunits;
  uint16_t* part_o;       // [nunits][256][128] FP16: O_acc / l of each row
  float2* part_ml;        // [nunits][256]: (m8, l) of each row
  const float* sq;
  const float* sk;
  const float* sv;
  uint16_t* o;
  int64_t os[3];          // output element strides (b, s, h)
  float c8;               // 8 * log2(e) * softmax_scale
  // repair set (rep_blocks == 0: none)
  int32_t n_rep, n_rep_pad, rep_blocks;
  const float* sk_sel;
  const float* sr;
  // Always 1.  The ExpCast threads branch on it before adding up a block's
  // row sum: the compiler cannot drop the branch, so it cannot lift the sum
  // above the P store's wait and the hand-over to fill their latency.
  int32_t rowsum_gate;

  // probe
  int64_t dump_bh, dump_qb, dump_kb;
  uint8_t* dump_codes;
  float* dump_m8;
  uint64_t timeout_ns;
  int32_t skip_mma;
  unsigned int* status;
  // timeline trace (test hook, builds with -DOVC_TRACE=1 only): CTA 0 records clock64() stamps of the first
  // kTraceBlocks blocks: [role][block][event], roles 0 = softmax warp 0,
  // 1 = softmax warp 4, 2 = MMA lane, 3 = producer lane.
  long long* trace;
};

constexpr int kTraceBlocks = 64, kTraceEvents = 8;

// Compiled in only with -DOVC_TRACE=1: clock reads are scheduling barriers,
// so the stamps would slow the loop they measure.
__device__ __forceinline__ void trace_mark(const AttnParams& P, int role, uint32_t blk, int ev) {
#if defined(OVC_TRACE) && OVC_TRACE
  if (P.trace != nullptr && blockIdx.x == 0 && blk < static_cast<uint32_t>(kTraceBlocks) &&
      (threadIdx.x & 31) == 0)
    P.trace[(role * kTraceBlocks + blk) * kTraceEvents + ev] = clock64();
#else
  (void)P, (void)role, (void)blk, (void)ev;
#endif
}

struct AttnSmem {
  uint8_t q[2][kTile];
  uint8_t k[kStages][kTile];
  uint8_t v[kStages][kTile];
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int zero;               // always 0: the "never abort" flag of drain waits
  // V-Smooth only (the other variants are launched without this tail):
  uint64_t m_full[2], m_empty[2];
  alignas(1024) uint8_t mv[2][kMeanTile];   // M' tiles of two runs, 32-byte swizzle
  float lbuf[2][16][128];                   // pending block row sums [tile][block mod 16][row]
  // Q smoothing only (never with V-Smooth; launched with the whole struct):
  uint64_t a_full[2];                        // the tiles' A operands are written
  alignas(1024) uint8_t kb[kStages][kBiasTile];   // key bias rows of each stage's keys (32-byte swizzle)
  alignas(1024) uint8_t ab[2][kBiasTile];         // per query tile: 128 rows of (hi, lo) parts of 1/s_q
};

// Repair variants only: the per-column multipliers of the repair blocks
// (8 log2e sm s_q s_k of each selected key, scaled as the byte step takes
// them), written by the tile's own 128 threads one block ahead into one of
// two buffers, each with a barrier of 128 arrivals.  It takes the place of
// the V-Smooth tail, which the repair variants never use, from the first
// 16-byte boundary there (the multipliers are read as float4).
struct alignas(16) RepairTail {
  float ksc[2][2][128];      // [tile][buffer][column]
  uint64_t ksc_full[2][2];   // [tile][buffer]
};
constexpr size_t kRepairTailOffset = (offsetof(AttnSmem, m_full) + 15) / 16 * 16;

// Dynamic shared memory of a launch, + 1024 bytes of alignment slack.
constexpr size_t kAttnSmemBytes = offsetof(AttnSmem, m_full) + 1024;
constexpr size_t kAttnSmemBytesRepair = kRepairTailOffset + sizeof(RepairTail) + 1024;
static_assert(kRepairTailOffset + sizeof(RepairTail) <= offsetof(AttnSmem, a_full),
              "the repair tail fits in the V-Smooth tail");
constexpr size_t kAttnSmemBytesVSmooth = offsetof(AttnSmem, a_full) + 1024;
constexpr size_t kAttnSmemBytesQBias = sizeof(AttnSmem) + 1024;
static_assert(kAttnSmemBytesQBias <= 232448, "shared memory per CTA");

__device__ __forceinline__ void record_abort(AttnSmem& sm, const AttnParams& P) {
  if (!*reinterpret_cast<volatile int*>(&sm.abort)) atomicOr(P.status, kStatusTimeout);
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
}

struct TileCoord {
  int bh, qb0, qb1, has1;
};

__device__ __forceinline__ TileCoord tile_coord(const AttnParams& P, int tile) {
  TileCoord c;
  c.bh = tile / P.npairs;
  const int pair = tile - c.bh * P.npairs;
  c.qb0 = 2 * pair;
  c.has1 = (2 * pair + 1 < P.nb);
  c.qb1 = c.has1 ? 2 * pair + 1 : c.qb0;
  return c;
}

// Kernel variants (template argument of attention_kernel): ExpCast with the
// mid-window order is the method; the exp-then-cast byte path and the natural
// key order together form the standard FP8 kernel that the two techniques
// improve on, measured in this same pipeline.
constexpr int kVarExpThenCast = 1;   // p byte = E4M3(ex2(...)) on the MUFU
constexpr int kVarNaturalOrder = 2;  // key blocks 0, 1, ..., nb-1
constexpr int kVarSplit = 4;         // split key ranges (nsplit > 1): partial results for merge_kernel
constexpr int kVarVSmooth = 8;       // V-Smooth: block means restored through the block row sums
constexpr int kVarQBias = 16;        // Q smoothing: the key bias added to the scores by one BF16 MMA
constexpr int kVarRepair = 32;       // V residual repair: the selected keys' blocks follow each unit's own
constexpr int kVarDump = 64;         // the probe's P-byte dump (test hook; kept out of the other kernels,
                                     // whose block loop runs faster without its code)
// Instantiated: 0-7, 8 (V-Smooth with ExpCast, mid-window, no split), 16-23
// (Q smoothing with each of 0-7), 32-35 and 48-51 (repair with 0-3 and
// 16-19: never split, never V-Smooth), and dump variants of 0-3, 16 and 32.

// Key block visited at step i of a range of n blocks starting at b0 (the
// whole sequence, or one split range): cyclic from the range's middle block,
// or in order.
template <int kVar>
__device__ __forceinline__ int key_block(int i, int b0, int n) {
  if (kVar & kVarNaturalOrder) return b0 + i;
  const int j = n / 2 + i;
  return b0 + (j >= n ? j - n : j);
}

struct UnitCoord {
  TileCoord tc;
  int b0, nbu;            // key blocks [b0, b0 + nbu)
};

template <int kVar>
__device__ __forceinline__ UnitCoord unit_coord(const AttnParams& P, int u) {
  UnitCoord c;
  if (kVar & kVarSplit) {
    const int tile = u / P.nsplit, sp = u - tile * P.nsplit;
    c.tc = tile_coord(P, tile);
    c.b0 = sp * P.nb / P.nsplit;
    c.nbu = (sp + 1) * P.nb / P.nsplit - c.b0;
  } else {
    c.tc = tile_coord(P, u);
    c.b0 = 0;
    c.nbu = P.nb;
  }
  return c;
}

// ---------------------------------------------------------------------------
// The ExpCast step for one row and one block of 128 scores.
//   s[c]  raw FP32 accumulator bits (masked columns already -inf)
//   a     per-block multiplier (8 log2e sm sq sk)
//   c     c0 + beta - m8, an integer (the reference sits on its grid)
// It produces 32 packed words of codes (bytes in key order); codes_sum adds
// up their decoded values for the row sum.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float expcast_scale_a(float a) { return a * (1.0f / 256.0f); }
__device__ __forceinline__ float expcast_scale_c(float c) {   // c = c0 + beta - m8 (an integer)
  return c * (1.0f / 256.0f);
}

// Two ExpCast codes, each in the low byte of its result.  The inputs are
// scaled by 1/256 (as = a/256, cs = (c0+beta-m8)/256): a saturating FMA per
// score clamps the code at 0, and an FMA by 256 adding 1.5*2^23 rounds it to
// the integer in the low mantissa bits (the code's upper end, 126, is kept
// by the lazy rescale threshold).  The rounding FMA of the two runs as one
// packed FP32-pair FMA: two independently rounded results, the same bits as
// two scalar FMAs, in one instruction (the saturating FMA has no packed
// form).  as0, as1: the two scores' multipliers, equal except in the repair
// blocks.
__device__ __forceinline__ void expcast_code2(uint32_t s0, uint32_t s1, float as0, float as1, float cs,
                                              uint32_t& u0, uint32_t& u1) {
  constexpr uint64_t k256x2 = 0x4380000043800000ull;     // (256, 256)
  constexpr uint64_t kMagicx2 = 0x4B4000004B400000ull;   // (1.5 * 2^23, 1.5 * 2^23)
  const float t0 = fma_sat(__uint_as_float(s0), as0, cs);
  const float t1 = fma_sat(__uint_as_float(s1), as1, cs);
  uint64_t t, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(t) : "f"(t0), "f"(t1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(t), "l"(k256x2), "l"(kMagicx2));
  asm("mov.b64 {%0, %1}, %2;" : "=r"(u0), "=r"(u1) : "l"(r));
}

// Codes of the scores s[4 G0 .. 4 (G0 + NG)) into the words w[G0 .. G0 + NG).
template <int G0, int NG>
__device__ __forceinline__ void expcast_words(const uint32_t* s, float as, float cs, uint32_t* w) {
#pragma unroll
  for (int g = G0; g < G0 + NG; ++g) {
    uint32_t u0, u1, u2, u3;
    expcast_code2(s[4 * g + 0], s[4 * g + 1], as, as, cs, u0, u1);
    expcast_code2(s[4 * g + 2], s[4 * g + 3], as, as, cs, u2, u3);
    w[g] = __byte_perm(__byte_perm(u0, u1, 0x0040), __byte_perm(u2, u3, 0x0040), 0x5410);
  }
}

// Sum of the decoded E4M3 codes of 32 packed words (f16x2 pairs, then FP32).
__device__ __forceinline__ float codes_sum(const uint32_t* w) {
  uint32_t acc[16];
#pragma unroll
  for (int g = 0; g < 32; ++g) {
    uint32_t h0, h1;
    cvt_e4m3x4_to_f16x2x2(w[g], h0, h1);
    const uint32_t h = hadd2(h0, h1);
    if (g < 16) acc[g] = h;
    else acc[g - 16] = hadd2(acc[g - 16], h);
  }
#pragma unroll
  for (int width = 8; width >= 1; width >>= 1)
#pragma unroll
    for (int g = 0; g < width; ++g) acc[g] = hadd2(acc[g], acc[g + width]);
  return f16x2_sum_to_f32(acc[0]);
}

// Same, with one multiplier per column (repair blocks: each selected key
// keeps the scale of the block it came from, so as_c = a_c / 256 comes from
// shared memory, four columns a load) and no row sum.
__device__ __forceinline__ void expcast_block_cols(const uint32_t* s, const float4* as4, float cs, uint32_t* w) {
#pragma unroll
  for (int g = 0; g < 32; ++g) {
    const float4 a4 = as4[g];
    uint32_t u0, u1, u2, u3;
    expcast_code2(s[4 * g + 0], s[4 * g + 1], a4.x, a4.y, cs, u0, u1);
    expcast_code2(s[4 * g + 2], s[4 * g + 3], a4.z, a4.w, cs, u2, u3);
    w[g] = __byte_perm(__byte_perm(u0, u1, 0x0040), __byte_perm(u2, u3, 0x0040), 0x5410);
  }
}

// Exp-then-cast bytes (the baseline path that ExpCast replaces): the stored
// value v = 2^(s * ac + cc), with ac = a/8 and cc = (c0 - 56 - m8)/8, comes
// from one FMA and one ex2 on the MUFU, and a pair of values becomes two
// E4M3 bytes by one FP32->FP8 conversion (round to nearest even, satfinite).
// A masked score (-inf) gives v = 0, code 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// kGuard: the exponent is first raised to at least -127 (ex2 then flushes to
// 0), which also turns the NaN of a masked padding column (-inf times a zero
// key scale) into code 0; the repair blocks need it, the main blocks (key
// scales > 0) do not.
template <bool kGuard>
__device__ __forceinline__ float cast_exponent(uint32_t s, float a, float cc) {
  const float x = fmaf(__uint_as_float(s), a, cc);
  return kGuard ? fmaxf(x, -127.0f) : x;
}

template <bool kGuard>
__device__ __forceinline__ uint32_t cast_word(uint32_t s0, uint32_t s1, uint32_t s2, uint32_t s3, float a0,
                                              float a1, float a2, float a3, float cc) {
  const float v0 = ex2_approx(cast_exponent<kGuard>(s0, a0, cc));
  const float v1 = ex2_approx(cast_exponent<kGuard>(s1, a1, cc));
  const float v2 = ex2_approx(cast_exponent<kGuard>(s2, a2, cc));
  const float v3 = ex2_approx(cast_exponent<kGuard>(s3, a3, cc));
  return __byte_perm(cvt_e4m3x2(v0, v1), cvt_e4m3x2(v2, v3), 0x5410);
}

__device__ __forceinline__ void cast_words(const uint32_t* s, float ac, float cc, uint32_t* w) {
#pragma unroll
  for (int g = 0; g < 32; ++g) w[g] = cast_word<false>(s[4 * g], s[4 * g + 1], s[4 * g + 2], s[4 * g + 3], ac, ac, ac, ac, cc);
}

// Per-column multipliers ac_c = a_c / 8 from shared memory (repair blocks).
__device__ __forceinline__ void cast_block_cols(const uint32_t* s, const float4* ac4, float cc, uint32_t* w) {
#pragma unroll
  for (int g = 0; g < 32; ++g) {
    const float4 a4 = ac4[g];
    w[g] = cast_word<true>(s[4 * g], s[4 * g + 1], s[4 * g + 2], s[4 * g + 3], a4.x, a4.y, a4.z, a4.w, cc);
  }
}

// Ragged tail block (keys >= S): this row's columns [valid, 128) of S set
// to -inf in tensor memory, by a short loop of stores, before the scores are
// loaded; the max-reducing load then skips them and the byte step gives them
// code 0.  A rolled loop keeps the hot block loop small (it runs at most once
// per tile).
__device__ __forceinline__ void tmem_mask_tail(uint32_t taddr, int valid) {
  constexpr uint32_t kNegInf = 0xFF800000u;
  int c = valid;
#pragma unroll 1
  for (; c < 128 && (c & 31) != 0; ++c) tmem_st1(taddr + static_cast<uint32_t>(c), kNegInf);
#pragma unroll 1
  for (; c < 128; c += 32) tmem_fill32(taddr + static_cast<uint32_t>(c), kNegInf);
  tmem_wait_st();
}

__device__ __forceinline__ float tmem_load_row128_max(uint32_t taddr, uint32_t* s) {
  float m0, m1, m2, m3;
  tmem_ld32_max(taddr + 0, s, m0);
  tmem_ld32_max(taddr + 32, s + 32, m1);
  tmem_ld32_max(taddr + 64, s + 64, m2);
  tmem_ld32_max(taddr + 96, s + 96, m3);
  tmem_wait_ld32_max(s, m0);
  tmem_wait_ld32_max(s + 32, m1);
  tmem_wait_ld32_max(s + 64, m2);
  tmem_wait_ld32_max(s + 96, m3);
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

__device__ __forceinline__ void tmem_load_row128(uint32_t taddr, uint32_t* s) {
  tmem_ld32(taddr + 0, s);
  tmem_ld32(taddr + 32, s + 32);
  tmem_ld32(taddr + 64, s + 64);
  tmem_ld32(taddr + 96, s + 96);
  tmem_wait_ld32(s);
  tmem_wait_ld32(s + 32);
  tmem_wait_ld32(s + 64);
  tmem_wait_ld32(s + 96);
}

// V-Smooth: key blocks are grouped in runs of consecutive visited blocks of
// one 16-block chunk (block index / 16); each run's row sums meet the run's
// M' tile in one BF16 MMA.  Visiting step i starts a run when it is the first
// or its chunk differs from the previous step's.
template <int kVar>
__device__ __forceinline__ bool starts_run(int i, int b0, int n) {
  return i == 0 || (key_block<kVar>(i, b0, n) >> 4) != (key_block<kVar>(i - 1, b0, n) >> 4);
}

// Writes a run's 16 pending row sums of this thread's row as the A operand of
// the mean MMA (BF16, two per column, the lower block first): columns
// [taddr, +8) the rounded values, [taddr + 8, +16) the rounding remainders
// (together about 16 significant bits), and clears them.
__device__ __forceinline__ void flush_row_sums(float* lb, uint32_t taddr) {
  uint32_t r[16];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float a = lb[(2 * m) * 128], b = lb[(2 * m + 1) * 128];
    const __nv_bfloat16 ah = __float2bfloat16_rn(a), bh = __float2bfloat16_rn(b);
    const __nv_bfloat16 al = __float2bfloat16_rn(__fsub_rn(a, __bfloat162float(ah)));
    const __nv_bfloat16 bl = __float2bfloat16_rn(__fsub_rn(b, __bfloat162float(bh)));
    r[m] = static_cast<uint32_t>(__bfloat16_as_ushort(ah)) | (static_cast<uint32_t>(__bfloat16_as_ushort(bh)) << 16);
    r[8 + m] = static_cast<uint32_t>(__bfloat16_as_ushort(al)) | (static_cast<uint32_t>(__bfloat16_as_ushort(bl)) << 16);
    lb[(2 * m) * 128] = 0.0f;
    lb[(2 * m + 1) * 128] = 0.0f;
  }
  tmem_st16(taddr, r);
}

// O row *= f in tensor memory (one 128-column row per thread).  kBatched:
// all four 32-column loads in flight at once (one TMEM round trip), then the
// products stored back; else one chunk at a time.  The two give the same
// values; which is faster depends on the variant's schedule (S = 73397,
// H = 56: the method's kernel 67.6 batched against 68.7 ms, the Q-smoothing
// kernel 67.8 against 69.6; the V-Smooth kernel 82.0 chunked against 84.8;
// the repair kernels 18% slower batched).
template <bool kBatched>
__device__ __forceinline__ void tmem_scale_row128(uint32_t taddr, float f) {
  if constexpr (kBatched) {
    uint32_t r[128];
    tmem_load_row128(taddr, r);
#pragma unroll
    for (int i = 0; i < 128; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
#pragma unroll
    for (int c = 0; c < 128; c += 32) tmem_st32(taddr + c, r + c);
  } else {
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c, r);
      tmem_wait_ld32(r);
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
      tmem_st32(taddr + c, r);
    }
  }
  tmem_wait_st();
}

// MMA issue, by lane 0 alone (W = false) or by the whole converged MMA warp
// with one elected lane (W = true; every wait then becomes a warp vote).
// Issued from a converged warp, a tcgen05.commit costs the tensor pipe
// nothing; issued by one lane of a diverged warp, each costs about as much
// as an MMA.  Warp issue is used by every variant but V-Smooth, whose MMA
// warp also runs the mean MMAs' run bookkeeping.
template <bool W>
__device__ __forceinline__ bool issue_vote(bool ok) {
  if constexpr (W) return __all_sync(0xFFFFFFFFu, ok);
  return ok;
}
template <bool W>
__device__ __forceinline__ void issue_f8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  if constexpr (W) mma_f8_ss_w(d, a, b, id, acc);
  else mma_f8_ss(d, a, b, id, acc);
}
template <bool W>
__device__ __forceinline__ void issue_f8_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
  if constexpr (W) mma_f8_ts_w(d, a, b, id, acc);
  else mma_f8_ts(d, a, b, id, acc);
}
template <bool W>
__device__ __forceinline__ void issue_bf16_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  if constexpr (W) mma_bf16_ss_w(d, a, b, id, acc);
  else mma_bf16_ss(d, a, b, id, acc);
}
template <bool W>
__device__ __forceinline__ void issue_commit(uint32_t bar) {
  if constexpr (W) tc_commit_w(bar);
  else tc_commit(bar);
}

template <int kVar>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_ks,
                     const __grid_constant__ CUtensorMap tm_dv, const __grid_constant__ CUtensorMap tm_vm,
                     const __grid_constant__ CUtensorMap tm_kb, const __grid_constant__ CUtensorMap tm_kbs,
                     const __grid_constant__ AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(
      smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int* abort_flag = &sm.abort;
  const uint64_t tmo = P.timeout_ns;
  constexpr bool kRep = (kVar & kVarRepair) != 0;
  RepairTail& rt = *reinterpret_cast<RepairTail*>(reinterpret_cast<uint8_t*>(&sm) + kRepairTailOffset);

  if (warp == kProducerWarp && lane == 0) {
    mbar_init(smem_addr(&sm.q_full), 1);
    mbar_init(smem_addr(&sm.q_empty), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_addr(&sm.k_full[i]), 1);
      mbar_init(smem_addr(&sm.v_full[i]), 1);
      mbar_init(smem_addr(&sm.kv_empty[i]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_addr(&sm.s_full[t]), 1);
      mbar_init(smem_addr(&sm.p_full[t]), 128);
      mbar_init(smem_addr(&sm.o_full[t]), 1);
    }
    mbar_init(smem_addr(&sm.drain), 1);
    if (kVar & kVarVSmooth)
      for (int r = 0; r < 2; ++r) {
        mbar_init(smem_addr(&sm.m_full[r]), 1);
        mbar_init(smem_addr(&sm.m_empty[r]), 1);
      }
    if (kVar & kVarQBias)
      for (int t = 0; t < 2; ++t) mbar_init(smem_addr(&sm.a_full[t]), 128);
    if (kRep)
      for (int t = 0; t < 2; ++t)
        for (int b = 0; b < 2; ++b) mbar_init(smem_addr(&rt.ksc_full[t][b]), 128);
    sm.abort = 0;
    sm.zero = 0;
    fence_mbar_init();
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (warp >= 8) {
    regs_dec<(kVar & kVarVSmooth) ? kControlRegsVSmooth : kControlRegs>();
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      uint32_t kv_iter = 0, q_iter = 0, run = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.nunits && ok; u += gridDim.x) {
        const UnitCoord uc = unit_coord<kVar>(P, u);
        const TileCoord& tc = uc.tc;
        const int nblk = uc.nbu + (kRep ? P.rep_blocks : 0);
        for (int i = 0; i < nblk; ++i) {
          const uint32_t stage = kv_iter % kStages, round = kv_iter / kStages;
          if (kv_iter >= kStages) {
            ok = mbar_wait(smem_addr(&sm.kv_empty[stage]), (round - 1) & 1, tmo, abort_flag);
            if (!ok) break;
          }
          const uint32_t kbar = smem_addr(&sm.k_full[stage]), vbar = smem_addr(&sm.v_full[stage]);
          constexpr bool qbias = (kVar & kVarQBias) != 0;
          mbar_arrive_expect_tx(kbar, qbias ? kTile + kBiasTile : kTile);
          mbar_arrive_expect_tx(vbar, kTile);
          if (!kRep || i < uc.nbu) {
            const int j = key_block<kVar>(i, uc.b0, uc.nbu);
            tma_load_2d(smem_addr(sm.k[stage]), &tm_k, kbar, 0, tc.bh * P.S_pad + j * 128);
            if (qbias) tma_load_2d(smem_addr(sm.kb[stage]), &tm_kb, kbar, 0, tc.bh * P.S_pad + j * 128);
            tma_load_2d(smem_addr(sm.v[stage]), &tm_v, vbar, j * 128, tc.bh * 128);
            if ((kVar & kVarVSmooth) && starts_run<kVar>(i, uc.b0, uc.nbu)) {
              // The M' tile of the run this block starts: channels of this head, blocks of its chunk.
              const uint32_t slot = run & 1;
              if (run >= 2) {
                ok = mbar_wait(smem_addr(&sm.m_empty[slot]), ((run >> 1) - 1) & 1, tmo, abort_flag);
                if (!ok) break;
              }
              const uint32_t mbar = smem_addr(&sm.m_full[slot]);
              mbar_arrive_expect_tx(mbar, kMeanTile);
              tma_load_2d(smem_addr(sm.mv[slot]), &tm_vm, mbar, (j >> 4) * 16, tc.bh * 128);
              ++run;
            }
          } else {
            const int r = i - uc.nbu;
            tma_load_2d(smem_addr(sm.k[stage]), &tm_ks, kbar, 0, tc.bh * P.n_rep_pad + r * 128);
            if (qbias) tma_load_2d(smem_addr(sm.kb[stage]), &tm_kbs, kbar, 0, tc.bh * P.n_rep_pad + r * 128);
            tma_load_2d(smem_addr(sm.v[stage]), &tm_dv, vbar, r * 128, tc.bh * 128);
          }
          ++kv_iter;
          if (i == 0) {
            // The unit's Q after its first K/V block, whose stage the previous
            // unit frees blocks earlier than its last P.V frees Q; then the
            // next unit's Q is pulled into L2 for its own load.
            if (q_iter > 0) ok = mbar_wait(smem_addr(&sm.q_empty), (q_iter - 1) & 1, tmo, abort_flag);
            if (!ok) break;
            const uint32_t qbar = smem_addr(&sm.q_full);
            mbar_arrive_expect_tx(qbar, 2 * kTile);
            tma_load_2d(smem_addr(sm.q[0]), &tm_q, qbar, 0, tc.bh * P.S_pad + tc.qb0 * 128);
            tma_load_2d(smem_addr(sm.q[1]), &tm_q, qbar, 0, tc.bh * P.S_pad + tc.qb1 * 128);
            ++q_iter;
            if (u + static_cast<int>(gridDim.x) < P.nunits) {
              const TileCoord tn = unit_coord<kVar>(P, u + static_cast<int>(gridDim.x)).tc;
              tma_prefetch_l2_2d(&tm_q, 0, tn.bh * P.S_pad + tn.qb0 * 128);
              tma_prefetch_l2_2d(&tm_q, 0, tn.bh * P.S_pad + tn.qb1 * 128);
            }
          }
        }
      }
      if (!ok) {
        record_abort(sm, P);
        // Drain: wait for the copies already issued (they always complete).
        const volatile int* never = &sm.zero;
        for (uint32_t n = (kv_iter > kStages ? kv_iter - kStages : 0); n < kv_iter; ++n) {
          const uint32_t stage = n % kStages, par = (n / kStages) & 1;
          mbar_wait(smem_addr(&sm.k_full[stage]), par, kDrainNs, never);
          mbar_wait(smem_addr(&sm.v_full[stage]), par, kDrainNs, never);
        }
        if (q_iter > 0) mbar_wait(smem_addr(&sm.q_full), (q_iter - 1) & 1, kDrainNs, never);
        for (uint32_t n = (run > 2 ? run - 2 : 0); n < run; ++n)
          mbar_wait(smem_addr(&sm.m_full[n & 1]), (n >> 1) & 1, kDrainNs, never);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    constexpr bool kW = (kVar & kVarVSmooth) == 0;   // issue style, see issue_vote
    if ((kW || lane == 0) && !P.skip_mma) {
      uint32_t kv_iter = 0, q_iter = 0, sp0 = 0, sp1 = 0, mrun = 0;
      bool ok = true, issued = false;
      // V-Smooth: O_t += L_t M'^T for a run's 16 blocks, L_t the BF16 row
      // sums (rounded values, then remainders) the ExpCast warps left in
      // S_t's columns [a, a + 16).
      auto mean_mma = [&sm](uint32_t tO, uint32_t a, uint32_t slot) {
        const uint64_t md = sw32_desc(smem_addr(sm.mv[slot]));
        mma_bf16_ts(tO, a, md, kIdescBf16, 1u);
        mma_bf16_ts(tO, a + 8, md, kIdescBf16, 1u);
      };
      const uint32_t tS0 = tmem + 0, tS1 = tmem + 128;
      const uint32_t tO0 = tmem + 256, tO1 = tmem + 384;
      const uint64_t qd0 = sw128_desc(smem_addr(sm.q[0])), qd1 = sw128_desc(smem_addr(sm.q[1]));
      // Q smoothing: after S_t = Q_t K^T, one BF16 MMA adds (1/s_q)(beta_j)
      // from the tile's A operand and the stage's key bias rows.
      constexpr bool qbias = (kVar & kVarQBias) != 0;
      uint64_t abd0 = 0, abd1 = 0;
      if (qbias) {
        abd0 = sw32_desc(smem_addr(sm.ab[0]));
        abd1 = sw32_desc(smem_addr(sm.ab[1]));
      }
      for (int u = blockIdx.x; u < P.nunits && ok; u += gridDim.x) {
        const UnitCoord ucm = unit_coord<kVar>(P, u);
        const int nbu = ucm.nbu, b0 = ucm.b0;
        const int nblk = nbu + (kRep ? P.rep_blocks : 0);
        ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.q_full), q_iter & 1, tmo, abort_flag));
        if (!ok) break;
        if (qbias) {
          ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.a_full[0]), q_iter & 1, tmo, abort_flag) &&
                              mbar_wait(smem_addr(&sm.a_full[1]), q_iter & 1, tmo, abort_flag));
          if (!ok) break;
        }
        // Scores of the first block for both query tiles.
        {
          const uint32_t stage = kv_iter % kStages;
          ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.k_full[stage]), (kv_iter / kStages) & 1, tmo, abort_flag));
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd = sw128_desc(smem_addr(sm.k[stage]));
          const uint64_t kbd = qbias ? sw32_desc(smem_addr(sm.kb[stage])) : 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) issue_f8_ss<kW>(tS0, qd0 + 2 * kk, kd + 2 * kk, kIdesc, kk > 0);
          if (qbias) issue_bf16_ss<kW>(tS0, abd0, kbd, kIdescBf16, 1u);
          issue_commit<kW>(smem_addr(&sm.s_full[0]));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) issue_f8_ss<kW>(tS1, qd1 + 2 * kk, kd + 2 * kk, kIdesc, kk > 0);
          if (qbias) issue_bf16_ss<kW>(tS1, abd1, kbd, kIdescBf16, 1u);
          issue_commit<kW>(smem_addr(&sm.s_full[1]));
          issued = true;
        }
        for (int i = 0; i < nblk; ++i) {
          const uint32_t stage = kv_iter % kStages;
          trace_mark(P, 2, kv_iter, 0);
          ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.v_full[stage]), (kv_iter / kStages) & 1, tmo, abort_flag));
          if (!ok) break;
          const uint64_t vd = sw128_desc(smem_addr(sm.v[stage]));
          const bool last = (i + 1 == nblk);
          const uint32_t nstage = (kv_iter + 1) % kStages;
          // V-Smooth: this block flushes the previous run (bit 0: it starts a
          // new one, run mrun - 2 after the count) and, as the unit's last
          // block, its own run (bit 1: run mrun - 1).
          uint32_t fl = 0;
          if ((kVar & kVarVSmooth) && i < nbu) {
            if (starts_run<kVar>(i, b0, nbu)) {
              fl = i > 0 ? 1u : 0u;
              ++mrun;
            }
            if (i + 1 == nbu) fl |= 2u;
          }
          // The next block's K (loaded stages ahead) is waited for here, while
          // the warp would wait for P anyway: a wait on a completed barrier
          // still takes a round trip, which between P.V and QK^T sits on the
          // tiles' chain (68.8 against 70.8 ms at S = 73397, H = 56).  The
          // V-Smooth variant keeps it between them (82.1 against 83.7 ms).
          constexpr bool kEarlyK = (kVar & kVarVSmooth) == 0;
          uint64_t kd_next = 0;
          if (kEarlyK && !last) {
            ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.k_full[nstage]), ((kv_iter + 1) / kStages) & 1, tmo, abort_flag));
            if (!ok) break;
            kd_next = sw128_desc(smem_addr(sm.k[nstage]));
          }
          // ---- query tile 0: O0 += P0 V, then the next block's S0
          ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.p_full[0]), sp0, tmo, abort_flag));
          if (!ok) break;
          trace_mark(P, 2, kv_iter, 1);
          sp0 ^= 1;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            issue_f8_ts<kW>(tO0, tS0 + 8 * kk, vd + 2 * kk, kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
          if (kVar & kVarVSmooth) {
#pragma unroll
            for (uint32_t b = 0; b < 2; ++b)
              if (fl & (1u << b)) {
                const uint32_t r = mrun - 2 + b;
                ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.m_full[r & 1]), (r >> 1) & 1, tmo, abort_flag));
                if (!ok) break;
                tc_fence_after();
                mean_mma(tO0, tS0 + 32 + 16 * b, r & 1);
              }
            if (!ok) break;
          }
          if (!last) {
            if (!kEarlyK) {
              ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.k_full[nstage]), ((kv_iter + 1) / kStages) & 1, tmo, abort_flag));
              if (!ok) break;
              tc_fence_after();
              kd_next = sw128_desc(smem_addr(sm.k[nstage]));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) issue_f8_ss<kW>(tS0, qd0 + 2 * kk, kd_next + 2 * kk, kIdesc, kk > 0);
            if (qbias) issue_bf16_ss<kW>(tS0, abd0, sw32_desc(smem_addr(sm.kb[nstage])), kIdescBf16, 1u);
            issue_commit<kW>(smem_addr(&sm.s_full[0]));
          } else {
            issue_commit<kW>(smem_addr(&sm.o_full[0]));
          }
          // ---- query tile 1
          trace_mark(P, 2, kv_iter, 2);
          ok = issue_vote<kW>(mbar_wait(smem_addr(&sm.p_full[1]), sp1, tmo, abort_flag));
          if (!ok) break;
          trace_mark(P, 2, kv_iter, 3);
          sp1 ^= 1;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            issue_f8_ts<kW>(tO1, tS1 + 8 * kk, vd + 2 * kk, kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
          if (kVar & kVarVSmooth) {
#pragma unroll
            for (uint32_t b = 0; b < 2; ++b)
              if (fl & (1u << b)) {
                const uint32_t r = mrun - 2 + b;
                mean_mma(tO1, tS1 + 32 + 16 * b, r & 1);
                issue_commit<kW>(smem_addr(&sm.m_empty[r & 1]));
              }
          }
          issue_commit<kW>(smem_addr(&sm.kv_empty[stage]));
          if (!last) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) issue_f8_ss<kW>(tS1, qd1 + 2 * kk, kd_next + 2 * kk, kIdesc, kk > 0);
            if (qbias) issue_bf16_ss<kW>(tS1, abd1, sw32_desc(smem_addr(sm.kb[nstage])), kIdescBf16, 1u);
            issue_commit<kW>(smem_addr(&sm.s_full[1]));
          } else {
            issue_commit<kW>(smem_addr(&sm.o_full[1]));
            issue_commit<kW>(smem_addr(&sm.q_empty));
          }
          ++kv_iter;
        }
        ++q_iter;
      }
      if (!ok) record_abort(sm, P);
      if (issued) {
        // Every MMA issued so far has completed once this barrier flips.
        issue_commit<kW>(smem_addr(&sm.drain));
        mbar_wait(smem_addr(&sm.drain), 0, kDrainNs, &sm.zero);
      }
    }
  }
  } else {
    regs_inc<(kVar & kVarVSmooth) ? kSoftmaxRegsVSmooth : kSoftmaxRegs>();
    // ------------------------------------------------------- softmax/ExpCast
    const int t = warp >> 2;                    // query tile 0 or 1
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + 256 + t * 128;
    uint32_t blk_count = 0, tile_count = 0;
    uint32_t rep_count = 0;                     // repair blocks started (all units): buffer and parity
    const int trole = (wq == 0) ? t : -1;
    bool ok = true;
    if (kVar & kVarVSmooth) {
#pragma unroll
      for (int c = 0; c < 16; ++c) sm.lbuf[t][c][row] = 0.0f;
    }
    for (int u = blockIdx.x; u < P.nunits && ok; u += gridDim.x) {
      const UnitCoord uc = unit_coord<kVar>(P, u);
      const TileCoord& tc = uc.tc;
      const int qb = t ? tc.qb1 : tc.qb0;
      const bool store = (t == 0) || tc.has1;
      const float sq = P.sq[tc.bh * P.nb + qb];
      const float c8sq = P.c8 * sq;
      float kf = -INFINITY;                     // reference m8 = kf + frac(c0+beta)
      float l = 0.0f;
      const bool dump_tile = (kVar & kVarDump) && tc.bh == P.dump_bh && qb == P.dump_qb && store;
      if (kVar & kVarQBias) {
        // Q smoothing: this row of the tile's A operand, the BF16 pair
        // (hi, lo) of 1/s_q twice, (hi, hi, lo, lo, 0, 0, 0, 0) in every
        // 16-byte chunk (the same in every row and chunk, so the 32-byte
        // swizzle of the operand changes nothing).  The previous unit's
        // MMAs have completed (its epilogue waited for them).
        const float x = __frcp_rn(sq);
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
        const uint32_t hh = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) * 0x10001u;
        const uint32_t ll = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) * 0x10001u;
        uint4* a = reinterpret_cast<uint4*>(sm.ab[t] + row * 32);
        a[0] = make_uint4(hh, ll, 0u, 0u);
        a[1] = make_uint4(hh, ll, 0u, 0u);
        fence_proxy_async_smem();
        mbar_arrive(smem_addr(&sm.a_full[t]));
      }
      // Repair: a selected key's multiplier is rep_base times its block scale.
      const float rep_base = (kVar & kVarExpThenCast) ? c8sq * 0.125f : expcast_scale_a(c8sq);
      if (kRep) {
        // The first repair block's multipliers are written now, so that the
        // key scale's load waits alongside the unit's first scores instead of
        // after its last main block.  The buffer was last read in the repair
        // block before last, which every thread of the tile finished before
        // arriving for the last one (this thread waited for that).
        rt.ksc[t][rep_count & 1][row] =
            rep_base * __ldg(P.sk_sel + static_cast<int64_t>(tc.bh) * P.n_rep_pad + row);
        mbar_arrive(smem_addr(&rt.ksc_full[t][rep_count & 1]));
      }
      // Key scale of the current block, loaded one block ahead.
      float sk_next = __ldg(P.sk + tc.bh * P.nb + key_block<kVar>(0, uc.b0, uc.nbu));
      for (int i = 0; i < uc.nbu; ++i) {
        const int j = key_block<kVar>(i, uc.b0, uc.nbu);
        const float skj = sk_next;
        if (i + 1 < uc.nbu) sk_next = __ldg(P.sk + tc.bh * P.nb + key_block<kVar>(i + 1, uc.b0, uc.nbu));
        const uint32_t gi = blk_count;
        if (trole >= 0) trace_mark(P, trole, gi, 0);
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&sm.s_full[t]), blk_count & 1, tmo, abort_flag));
        ++blk_count;
        if (!ok) break;
        if (trole >= 0) trace_mark(P, trole, gi, 1);
        tc_fence_after();
        uint32_t s[128];
        uint32_t w[32];
        float f = 1.0f;
        bool rescale = false;
        const int valid = P.S - j * 128;
        const float a = c8sq * skj;
        const float as = expcast_scale_a(a);
        if (valid < 128) tmem_mask_tail(tS, valid);
        const float mx = tmem_load_row128_max(tS, s);
        const float bm8 = mx * a;
        const bool need = bm8 > kf + (kFrac + kLazy);
        if (__any_sync(0xFFFFFFFFu, need)) {
          const float kn = need ? ceilf(bm8 - kFrac) : kf;
          f = need ? exp2f((kf - kn) * 0.125f) : 1.0f;
          l *= f;
          kf = kn;
          rescale = i > 0;
          if ((kVar & kVarVSmooth) && rescale) {
            // Row sums not yet added to O change units with it.
#pragma unroll
            for (int c = 0; c < 16; ++c) sm.lbuf[t][c][row] *= f;
          }
        }
        if (trole >= 0) trace_mark(P, trole, gi, 3);
        if (kVar & kVarExpThenCast)
          cast_words(s, a * 0.125f, (64.0f - kFrac - kf) * 0.125f, w);
        else
          expcast_words<0, 32>(s, as, expcast_scale_c(kCodeBase - kf), w);
        if ((kVar & kVarDump) && dump_tile && j == P.dump_kb) {
          uint4* d = reinterpret_cast<uint4*>(P.dump_codes + row * 128);
#pragma unroll
          for (int g = 0; g < 8; ++g) d[g] = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
          P.dump_m8[row] = kf + kFrac;
        }
        if (trole >= 0) trace_mark(P, trole, gi, 4);
        tmem_st32(tS, w);
        bool lsum_done = false;
        if (kVar & kVarVSmooth) {
          // V-Smooth: a block that starts a run hands the previous run's row
          // sums to the mean MMA (columns 32-47 of S_t); the unit's last block
          // adds its own row sum first and hands its run over too (48-63).
          float* lb = &sm.lbuf[t][0][row];
          if (i > 0 && starts_run<kVar>(i, uc.b0, uc.nbu)) flush_row_sums(lb, tS + 32);
          if (i + 1 == uc.nbu) {
            const float lbi = codes_sum(w);
            l += lbi;
            lb[(j & 15) * 128] = lbi;
            flush_row_sums(lb, tS + 48);
            lsum_done = true;
          }
        }
        // O is stable here (every earlier MMA of this tile has completed) and
        // the next P.V waits for this thread's arrival below.
        if (rescale) tmem_scale_row128<(kVar & (kVarRepair | kVarVSmooth)) == 0>(tO, f);
        tmem_wait_st();
        tc_fence_before();
        // Every thread arrives once its own P stores are done (128 arrivals).
        mbar_arrive(smem_addr(&sm.p_full[t]));
        // The row sum waits until the codes are on their way to the tensor core.
        if (!lsum_done && P.rowsum_gate) {
          const float lbi = codes_sum(w);
          l += lbi;
          if (kVar & kVarVSmooth) sm.lbuf[t][j & 15][row] = lbi;
        }
        if (trole >= 0) trace_mark(P, trole, gi, 6);
      }
      if (kRep && ok) {
        // The repair blocks, after the row's final reference is known: codes
        // against it with each selected key's own multiplier, no max, no row
        // sum; the first one changes O's units from s_v to s_r.  Multiplier
        // r + 1 is written while block r runs, into the other buffer; a buffer
        // is written again only after every thread of the tile has arrived for
        // the block after its last reader, so no thread still reads it.
        // (Block 0's were written at the start of the unit.)
        const float* sk_sel = P.sk_sel + static_cast<int64_t>(tc.bh) * P.n_rep_pad + row;
        float sk_rep = 0.0f;
        for (int r = 0; r < P.rep_blocks; ++r) {
          const uint32_t rc = rep_count++;
          const bool more = r + 1 < P.rep_blocks;
          if (more) sk_rep = __ldg(sk_sel + (r + 1) * 128);
          const uint32_t gi = blk_count;
          if (trole >= 0) trace_mark(P, trole, gi, 0);
          // The multipliers (written a block ahead) first, so that this wait's
          // round trip overlaps the scores' computation.
          ok = __all_sync(0xFFFFFFFFu,
                          mbar_wait(smem_addr(&rt.ksc_full[t][rc & 1]), (rc >> 1) & 1, tmo, abort_flag) &&
                              mbar_wait(smem_addr(&sm.s_full[t]), blk_count & 1, tmo, abort_flag));
          ++blk_count;
          if (!ok) break;
          if (trole >= 0) trace_mark(P, trole, gi, 1);
          tc_fence_after();
          uint32_t s[128];
          uint32_t w[32];
          if (!more) tmem_mask_tail(tS, P.n_rep - r * 128);   // only the set's last block has padding
          tmem_load_row128(tS, s);
          const float4* ks = reinterpret_cast<const float4*>(rt.ksc[t][rc & 1]);
          if (kVar & kVarExpThenCast)
            cast_block_cols(s, ks, (64.0f - kFrac - kf) * 0.125f, w);
          else
            expcast_block_cols(s, ks, expcast_scale_c(kCodeBase - kf), w);
          if (trole >= 0) trace_mark(P, trole, gi, 4);
          tmem_st32(tS, w);
          if (r == 0) tmem_scale_row128<false>(tO, P.sv[tc.bh] / P.sr[tc.bh]);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_addr(&sm.p_full[t]));
          if (more) {
            rt.ksc[t][rep_count & 1][row] = rep_base * sk_rep;
            mbar_arrive(smem_addr(&rt.ksc_full[t][rep_count & 1]));
          }
          if (trole >= 0) trace_mark(P, trole, gi, 6);
        }
      }
      if (!ok) break;
      const float s_out = (kRep ? P.sr : P.sv)[tc.bh];   // loaded while O completes
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&sm.o_full[t]), tile_count & 1, tmo, abort_flag));
      ++tile_count;
      if (!ok) break;
      tc_fence_after();
      const int q_row = qb * 128 + row;
      if (kVar & kVarSplit) {
        // Partial result of this key range: O_acc / l as FP16 and (m8, l);
        // merge_kernel combines the ranges of each row.
        const float inv_l = 1.0f / l;
        const int64_t prow = static_cast<int64_t>(u) * 256 + t * 128 + row;
        uint16_t* po = P.part_o + prow * 128;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t r[32];
          tmem_ld32(tO + c, r);
          tmem_wait_ld32(r);
          if (store && q_row < P.S) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              __half2 h2 = __floats2half2_rn(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
              pk[e] = *reinterpret_cast<uint32_t*>(&h2);
            }
            uint4* dst = reinterpret_cast<uint4*>(po + c);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
        if (store && q_row < P.S) P.part_ml[prow] = make_float2(kf + kFrac, l);
        continue;
      }
      // Epilogue: O = scale * O_acc / l, BF16, one 256-byte row per thread;
      // the row comes out of TMEM in one round trip.
      const float scale = s_out / l;
      const int b = tc.bh / P.H, h = tc.bh - b * P.H;
      uint16_t* orow = P.o + b * P.os[0] + static_cast<int64_t>(q_row) * P.os[1] + h * P.os[2];
      uint32_t r[128];
      tmem_load_row128(tO, r);
      if (store && q_row < P.S) {
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(r[c + 2 * e]) * scale,
                                                      __uint_as_float(r[c + 2 * e + 1]) * scale);
            pk[e] = *reinterpret_cast<uint32_t*>(&v2);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
    if (!ok) record_abort(sm, P);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Merge of split key ranges: for each query row, with M = max_s m8_s and
// w_s = l_s 2^((m8_s - M)/8),  O = s_v * sum_s w_s Ohat_s / sum_s w_s  (Ohat_s
// = O_acc / l of range s, FP16), rounded to BF16.  One warp per row, four
// channels per lane (8-byte loads of each partial, 8-byte stores).
// ---------------------------------------------------------------------------
constexpr int kMergeRowsPerBlock = 8;

__global__ void __launch_bounds__(32 * kMergeRowsPerBlock)
    merge_kernel(const __grid_constant__ AttnParams P) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kMergeRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t nrows = static_cast<int64_t>(P.B) * P.H * P.S;
  if (g >= nrows) return;
  const int bh = static_cast<int>(g / P.S);
  const int q = static_cast<int>(g - static_cast<int64_t>(bh) * P.S);
  const int tile = bh * P.npairs + q / 256;
  const int64_t prow0 = static_cast<int64_t>(tile) * P.nsplit * 256 + (q & 255);
  float M = -INFINITY;
  for (int sp = 0; sp < P.nsplit; ++sp) M = fmaxf(M, P.part_ml[prow0 + sp * 256].x);
  float W = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int sp = 0; sp < P.nsplit; ++sp) {
    const float2 ml = P.part_ml[prow0 + sp * 256];
    const float w = ml.y * exp2f((ml.x - M) * 0.125f);
    W += w;
    const uint2 raw = *reinterpret_cast<const uint2*>(P.part_o + (prow0 + sp * 256) * 128 + 4 * lane);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    acc[0] += w * a.x;
    acc[1] += w * a.y;
    acc[2] += w * b.x;
    acc[3] += w * b.y;
  }
  const float scale = P.sv[bh] / W;
  const int b = bh / P.H, h = bh - b * P.H;
  __nv_bfloat162 o01 = __floats2bfloat162_rn(acc[0] * scale, acc[1] * scale);
  __nv_bfloat162 o23 = __floats2bfloat162_rn(acc[2] * scale, acc[3] * scale);
  uint2 outv;
  outv.x = *reinterpret_cast<uint32_t*>(&o01);
  outv.y = *reinterpret_cast<uint32_t*>(&o23);
  *reinterpret_cast<uint2*>(P.o + b * P.os[0] + static_cast<int64_t>(q) * P.os[1] + h * P.os[2] + 4 * lane) = outv;
}

}  // namespace ovc
