// repair.cuh -- V residual repair preparation.
//
// "Open VC Attention" (catalogue entry): the repair re-adds the quantisation
// residual of the worst-rounded V tokens; it is prepared with
// prepare_v_repair and a budget such as 0.005.  "MachGen opened the sources of
// Open-VC Attention", "What happened": quantised residuals are added only to
// the V tokens worst by energy.
//
// Per (batch, head): select the n tokens with the largest FP32 residual
// energy (ties to the lower index), list them in ascending order, quantise
// their FP32 residuals R = v - s_v dec(code) with one scale per head
// s_r = amax|R_sel| / 448, and gather their keys.  The work is spread over a
// grid of (4096-token chunk, head) CTAs so that every SM takes part:
//   repair_hist_kernel (4 launches)  radix select of the n-th largest energy
//       T, 8 bits a pass from the top (FP32 bits of non-negative values order
//       like the values); each CTA histograms its chunk of the keys that
//       match the digits chosen so far into a global per-head histogram.  The
//       digits chosen so far are re-derived from the earlier passes'
//       histograms by every CTA (a 256-bin walk), so no launch is spent on it;
//   repair_count_kernel              per chunk: keys > T and keys == T;
//   repair_scatter_kernel            ordered compaction: every key > T and
//       the first (n - #greater) keys == T, in index order, each CTA writing
//       its chunk's keys at the offset the earlier chunks' counts give;
//   repair_amax_kernel               a warp per selected token: its residual
//       recomputed in FP32 (the code recomputed exactly as prepare does),
//       amax folded into the head's maximum;
//   repair_write_kernel              a warp per slot of the padded set: the
//       residual codes E4M3(R * 448/amax) transposed (dvt), the selected
//       quantised keys (k_sel), the scale of each key's block (sk_sel) and,
//       with Q smoothing, each key's bias row (kb_sel); zero padding to n_pad.
#pragma once

#include <cstdint>

#include "prepare.cuh"

namespace ovc {

struct RepairParams {
  const uint16_t* v;
  int64_t vs[3];
  int32_t B, S, H, nb, S_pad, fp16;
  const uint8_t* kc;
  const float* sk;
  const float* energy;
  const uint32_t* vamax;
  int32_t n, n_pad;
  int32_t* idx;
  uint8_t* k_sel;
  uint8_t* dvt;
  float* sk_sel;
  float* sr;
  // Q smoothing (both NULL when off): the key bias rows [B*H][S_pad][16] of
  // the preparation, and those of the selected keys [B*H][n_pad][16].
  const uint16_t* kbias;
  uint16_t* kb_sel;
  // Scratch (caller workspace, zeroed before the first pass): hist
  // [B*H][4][256] digit counts of each pass, cnt [B*H][nchunk][2] (keys > T,
  // keys == T) of each chunk, ramax [B*H] residual amax bits.
  uint32_t* hist;
  uint32_t* cnt;
  uint32_t* ramax;
  int32_t nchunk;
};

constexpr int kRepairChunk = 4096;    // tokens per CTA in the selection kernels
constexpr int kRepairThreads = 256;
constexpr int kRepairTokensPerCta = kRepairThreads / 32;   // a warp per selected token

// Selected indices are always in [0, S); the clamp only keeps a corrupted
// workspace from turning into an out-of-bounds read.
__device__ __forceinline__ int clamp_token(int t, int S) { return t < 0 ? 0 : (t >= S ? S - 1 : t); }

// The digits of T chosen by passes 0 .. npass-1: the digit of a pass is the
// highest d at which the keys with a larger digit number fewer than those
// still to take, and those with digit >= d at least as many.  prefix/mask:
// the digits so far; remaining: how many keys with that prefix are still to
// take.  Called by every thread of the CTA (kRepairThreads); each pass's
// histogram is staged in shared memory and warp 0 finds the digit with a
// suffix sum over its lanes (lane l holds bins 255-8l .. 248-8l).
struct RadixState {
  uint32_t prefix, mask, remaining;
};

__device__ __forceinline__ RadixState radix_state(const uint32_t* hist_bh, int npass, uint32_t n) {
  __shared__ uint32_t bins[256];
  __shared__ RadixState st;
  if (threadIdx.x == 0) st = RadixState{0u, 0u, n};
  __syncthreads();
  for (int p = 0; p < npass; ++p) {
    for (int b = threadIdx.x; b < 256; b += kRepairThreads) bins[b] = hist_bh[p * 256 + b];
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const uint32_t remaining = st.remaining;
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        c[k] = bins[255 - 8 * lane - k];
        tot += c[k];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - tot;   // keys in the bins above this lane's
      // the lane whose bins hold the cut; the last lane takes it if none does
      // (its lowest bin, digit 0, then holds the remaining keys)
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, excl < remaining && remaining <= incl);
      const int owner = hit ? __ffs(hit) - 1 : 31;
      if (lane == owner) {
        uint32_t cum = excl;
        int d = 255 - 8 * lane;
        for (int k = 0; k < 8; ++k, --d) {
          if (d == 0 || cum + c[k] >= remaining) break;
          cum += c[k];
        }
        const int shift = 24 - 8 * p;
        st.prefix |= static_cast<uint32_t>(d) << shift;
        st.mask |= 255u << shift;
        st.remaining = remaining - cum;
      }
    }
    __syncthreads();
  }
  const RadixState r = st;
  __syncthreads();
  return r;
}

// One radix pass over a chunk of one head's energies.
template <int kPass>
__global__ void __launch_bounds__(kRepairThreads) repair_hist_kernel(const __grid_constant__ RepairParams P) {
  __shared__ uint32_t h[kRepairThreads / 32][256];
  const int bh = blockIdx.y, chunk = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (kRepairThreads / 32) * 256; i += kRepairThreads) (&h[0][0])[i] = 0u;
  uint32_t* hist_bh = P.hist + static_cast<int64_t>(bh) * 4 * 256;
  const RadixState st = radix_state(hist_bh, kPass, static_cast<uint32_t>(P.n));
  const uint32_t prefix = st.prefix, mask = st.mask;
  constexpr int shift = 24 - 8 * kPass;
  const uint32_t* key = reinterpret_cast<const uint32_t*>(P.energy + static_cast<int64_t>(bh) * P.S);
  const int t0 = chunk * kRepairChunk, t1 = min(P.S, t0 + kRepairChunk);
  for (int tb = t0; tb < t1; tb += kRepairThreads) {
    const int t = tb + threadIdx.x;
    const uint32_t k = t < t1 ? __ldg(key + t) : 0u;
    const bool in = t < t1 && (k & mask) == prefix;
    const uint32_t bin = in ? (k >> shift) & 255u : 256u;
    // warp-aggregated: one shared-memory atomic per distinct bin of the warp
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bin);
    if (in && lane == __ffs(peers) - 1) atomicAdd(&h[warp][bin], static_cast<uint32_t>(__popc(peers)));
  }
  __syncthreads();
  for (int b = threadIdx.x; b < 256; b += kRepairThreads) {
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < kRepairThreads / 32; ++w) c += h[w][b];
    if (c) atomicAdd(hist_bh + kPass * 256 + b, c);
  }
}

// Keys above T and keys equal to T in each chunk.
__global__ void __launch_bounds__(kRepairThreads) repair_count_kernel(const __grid_constant__ RepairParams P) {
  __shared__ uint32_t red[2][kRepairThreads / 32];
  const int bh = blockIdx.y, chunk = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t T = radix_state(P.hist + static_cast<int64_t>(bh) * 4 * 256, 4, static_cast<uint32_t>(P.n)).prefix;
  const uint32_t* key = reinterpret_cast<const uint32_t*>(P.energy + static_cast<int64_t>(bh) * P.S);
  const int t0 = chunk * kRepairChunk, t1 = min(P.S, t0 + kRepairChunk);
  uint32_t gt = 0, eq = 0;
  for (int t = t0 + threadIdx.x; t < t1; t += kRepairThreads) {
    const uint32_t k = __ldg(key + t);
    gt += k > T;
    eq += k == T;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt += __shfl_xor_sync(0xFFFFFFFFu, gt, o);
    eq += __shfl_xor_sync(0xFFFFFFFFu, eq, o);
  }
  if (lane == 0) {
    red[0][warp] = gt;
    red[1][warp] = eq;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t g = 0, e = 0;
    for (int w = 0; w < kRepairThreads / 32; ++w) {
      g += red[0][w];
      e += red[1][w];
    }
    uint32_t* c = P.cnt + (static_cast<int64_t>(bh) * P.nchunk + chunk) * 2;
    c[0] = g;
    c[1] = e;
  }
}

// Exclusive prefix sum over the CTA; returns this thread's offset and writes
// the CTA total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t x, uint32_t* red, uint32_t* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kRepairThreads / 32;
  uint32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t wv = lane < kWarps ? red[lane] : 0u;
    uint32_t winc = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, winc, o);
      if (lane >= o) winc += y;
    }
    if (lane < kWarps) red[lane] = winc - wv;   // exclusive offset of each warp
    if (lane == 31) red[32] = winc;             // CTA total
  }
  __syncthreads();
  const uint32_t off = red[warp] + inc - x;
  *total = red[32];
  __syncthreads();
  return off;
}

// Ordered compaction of one chunk: every key > T, and keys == T while the
// head's count of equal keys taken stays below the number needed.
__global__ void __launch_bounds__(kRepairThreads) repair_scatter_kernel(const __grid_constant__ RepairParams P) {
  __shared__ uint32_t red[33];
  __shared__ uint32_t base[2];
  const int bh = blockIdx.y, chunk = blockIdx.x;
  const RadixState st = radix_state(P.hist + static_cast<int64_t>(bh) * 4 * 256, 4, static_cast<uint32_t>(P.n));
  if (threadIdx.x == 0) {
    // Offsets of this chunk: the keys taken and the keys == T seen before it.
    const uint32_t* c = P.cnt + static_cast<int64_t>(bh) * P.nchunk * 2;
    uint32_t out = 0, eq = 0;
    for (int i = 0; i < chunk; ++i) {
      const uint32_t g = c[2 * i], e = c[2 * i + 1];
      const uint32_t e_taken = eq >= st.remaining ? 0u : min(e, st.remaining - eq);
      out += g + e_taken;
      eq += e;
    }
    base[0] = out;
    base[1] = eq;
  }
  __syncthreads();
  const uint32_t T = st.prefix, need_eq = st.remaining;
  uint32_t base_out = base[0], base_eq = base[1];
  const uint32_t* key = reinterpret_cast<const uint32_t*>(P.energy + static_cast<int64_t>(bh) * P.S);
  int32_t* idx = P.idx + static_cast<int64_t>(bh) * P.n;
  const int t0 = chunk * kRepairChunk, t1 = min(P.S, t0 + kRepairChunk);
  for (int tb = t0; tb < t1; tb += kRepairThreads) {
    const int t = tb + threadIdx.x;
    const uint32_t k = t < t1 ? __ldg(key + t) : 0u;
    const uint32_t gt = (t < t1 && k > T) ? 1u : 0u;
    const uint32_t eq = (t < t1 && k == T) ? 1u : 0u;
    uint32_t tot_eq, tot_take;
    const uint32_t eq_rank = base_eq + block_exclusive_scan(eq, red, &tot_eq);
    const uint32_t take = gt | (eq & (eq_rank < need_eq ? 1u : 0u));
    const uint32_t pos = base_out + block_exclusive_scan(take, red, &tot_take);
    if (take && pos < static_cast<uint32_t>(P.n)) idx[pos] = t;
    base_eq += tot_eq;
    base_out += tot_take;
  }
}

// Residual of four consecutive channels of token t, recomputed in FP32.
__device__ __forceinline__ void residual4(const RepairParams& P, int b, int h, int t, int c0, float sv,
                                          float rv, float* R) {
  const uint2 x2 = __ldg(reinterpret_cast<const uint2*>(P.v + b * P.vs[0] + static_cast<int64_t>(t) * P.vs[1] +
                                                        h * P.vs[2] + c0));
  const float2 a = unpack2(x2.x, P.fp16), c = unpack2(x2.y, P.fp16);
  const float x[4] = {a.x, a.y, c.x, c.y};
  const uint32_t codes = quant4(x[0], x[1], x[2], x[3], rv);
  float dq[4];
  dec4(codes, dq);
#pragma unroll
  for (int i = 0; i < 4; ++i) R[i] = __fsub_rn(x[i], __fmul_rn(sv, dq[i]));
}

// amax |R| over the selected tokens, per head.
__global__ void __launch_bounds__(kRepairThreads) repair_amax_kernel(const __grid_constant__ RepairParams P) {
  const int bh = blockIdx.y;
  const int i = blockIdx.x * kRepairTokensPerCta + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (i >= P.n) return;
  const int b = bh / P.H, h = bh % P.H;
  const QScale vsc = scale_from_amax(__uint_as_float(P.vamax[bh]));
  float R[4];
  residual4(P, b, h, clamp_token(P.idx[static_cast<int64_t>(bh) * P.n + i], P.S), 4 * lane, vsc.s, vsc.r, R);
  float m = fmaxf(fmaxf(fabsf(R[0]), fabsf(R[1])), fmaxf(fabsf(R[2]), fabsf(R[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) atomicMax(P.ramax + bh, __float_as_uint(m));
}

// Residual codes (transposed), gathered keys, their block scales and bias
// rows, for slot i of the padded repair set.
__global__ void __launch_bounds__(kRepairThreads) repair_write_kernel(const __grid_constant__ RepairParams P) {
  const int bh = blockIdx.y;
  const int i = blockIdx.x * kRepairTokensPerCta + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const QScale rsc = scale_from_amax(__uint_as_float(P.ramax[bh]));
  if (blockIdx.x == 0 && threadIdx.x == 0) P.sr[bh] = rsc.s;
  if (i >= P.n_pad) return;
  const int b = bh / P.H, h = bh % P.H;
  uint32_t codes = 0, kw = 0, bw = 0;
  float skv = 0.0f;
  if (i < P.n) {
    const QScale vsc = scale_from_amax(__uint_as_float(P.vamax[bh]));
    const int t = clamp_token(P.idx[static_cast<int64_t>(bh) * P.n + i], P.S);
    float R[4];
    residual4(P, b, h, t, 4 * lane, vsc.s, vsc.r, R);
    codes = quant4(R[0], R[1], R[2], R[3], rsc.r);
    kw = __ldg(reinterpret_cast<const uint32_t*>(P.kc + (static_cast<int64_t>(bh) * P.S_pad + t) * 128) + lane);
    skv = P.sk[bh * P.nb + t / 128];
    if (P.kb_sel != nullptr && lane < 8)
      bw = __ldg(reinterpret_cast<const uint32_t*>(P.kbias + (static_cast<int64_t>(bh) * P.S_pad + t) * 16) + lane);
  }
  uint8_t* dvt = P.dvt + static_cast<int64_t>(bh) * 128 * P.n_pad;
#pragma unroll
  for (int e = 0; e < 4; ++e) dvt[static_cast<int64_t>(4 * lane + e) * P.n_pad + i] = static_cast<uint8_t>(codes >> (8 * e));
  reinterpret_cast<uint32_t*>(P.k_sel + (static_cast<int64_t>(bh) * P.n_pad + i) * 128)[lane] = kw;
  if (lane == 0) P.sk_sel[static_cast<int64_t>(bh) * P.n_pad + i] = skv;
  if (P.kb_sel != nullptr && lane < 8)
    reinterpret_cast<uint32_t*>(P.kb_sel + (static_cast<int64_t>(bh) * P.n_pad + i) * 16)[lane] = bw;
}

}  // namespace ovc
