// repair.cuh -- V residual repair preparation.
//
// "Open VC Attention" (catalogue entry): the repair re-adds the quantisation
// residual of the worst-rounded V tokens; it is prepared with
// prepare_v_repair and a budget such as 0.005.  "MachGen opened the sources of
// Open-VC Attention", "What happened": quantised residuals are added only to
// the V tokens worst by energy.
//
// One CTA (1024 threads) per (batch, head):
//   1. radix-select (4 passes of 8 bits over the FP32 energy bits, which order
//      like the values because energies are >= 0) the n-th largest energy T;
//   2. compact, in index order, every token with energy > T and the first
//      (n - #greater) tokens with energy == T -> idx ascending (ties go to the
//      lower index, exactly as a stable sort by energy would);
//   3. recompute each selected token's FP32 residual R = v - s_v*dec(code)
//      (its code recomputed exactly as prepare does), take amax|R| ->
//      s_r = amax/448;
//   4. write the residual codes E4M3(R * 448/amax) transposed (dvt), gather
//      the selected quantised keys (k_sel), the scale of each key's block
//      (sk_sel) and, with Q smoothing, each key's bias row (kb_sel),
//      zero-padding up to n_pad.
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
};

constexpr int kRepairThreads = 1024;

// Selected indices are always in [0, S); the clamp only keeps a corrupted
// workspace from turning into an out-of-bounds read.
__device__ __forceinline__ int clamp_token(int t, int S) { return t < 0 ? 0 : (t >= S ? S - 1 : t); }

// Exclusive prefix sum over the CTA; returns this thread's offset and writes
// the CTA total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t x, uint32_t* red, uint32_t* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t wv = red[lane];
    uint32_t winc = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, winc, o);
      if (lane >= o) winc += y;
    }
    red[lane] = winc - wv;            // exclusive offset of each warp
    if (lane == 31) red[32] = winc;   // CTA total
  }
  __syncthreads();
  const uint32_t off = red[warp] + inc - x;
  *total = red[32];
  __syncthreads();
  return off;
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

__global__ void __launch_bounds__(kRepairThreads, 1) repair_prepare_kernel(const __grid_constant__ RepairParams P) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t red[33];
  __shared__ uint32_t s_digit, s_remaining;
  const int bh = blockIdx.x;
  const int b = bh / P.H, h = bh % P.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t* key = reinterpret_cast<const uint32_t*>(P.energy + static_cast<int64_t>(bh) * P.S);
  int32_t* idx = P.idx + static_cast<int64_t>(bh) * P.n;

  // 1. radix select of the n-th largest key
  uint32_t prefix = 0, mask = 0, remaining = static_cast<uint32_t>(P.n);
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int t = tid; t < P.S; t += kRepairThreads) {
      const uint32_t k = __ldg(key + t);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t cum = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= remaining) break;
        cum += hist[d];
      }
      s_digit = static_cast<uint32_t>(d);
      s_remaining = remaining - cum;
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    remaining = s_remaining;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const uint32_t need_eq = remaining;   // how many keys equal to T are taken

  // 2. ordered compaction
  uint32_t base_eq = 0, base_out = 0;
  for (int c0 = 0; c0 < P.S; c0 += kRepairThreads) {
    const int t = c0 + tid;
    const uint32_t k = t < P.S ? __ldg(key + t) : 0u;
    const uint32_t gt = (t < P.S && k > T) ? 1u : 0u;
    const uint32_t eq = (t < P.S && k == T) ? 1u : 0u;
    uint32_t tot_eq, tot_take;
    const uint32_t eq_rank = base_eq + block_exclusive_scan(eq, red, &tot_eq);
    const uint32_t take = gt | (eq & (eq_rank < need_eq ? 1u : 0u));
    const uint32_t pos = base_out + block_exclusive_scan(take, red, &tot_take);
    if (take && pos < static_cast<uint32_t>(P.n)) idx[pos] = t;
    base_eq += tot_eq;
    base_out += tot_take;
  }
  __syncthreads();

  // 3. residual scale over the selected tokens
  const QScale vsc = scale_from_amax(__uint_as_float(P.vamax[bh]));
  float amax = 0.0f;
  for (int i = warp; i < P.n; i += kRepairThreads / 32) {
    float R[4];
    residual4(P, b, h, clamp_token(idx[i], P.S), 4 * lane, vsc.s, vsc.r, R);
#pragma unroll
    for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(R[e]));
  }
  const float ramax = __uint_as_float(block_max_u32(__float_as_uint(amax), red));
  const QScale rsc = scale_from_amax(ramax);
  if (tid == 0) P.sr[bh] = rsc.s;

  // 4. residual codes (transposed), gathered keys and their block scales
  uint8_t* dvt = P.dvt + static_cast<int64_t>(bh) * 128 * P.n_pad;
  uint8_t* ksel = P.k_sel + static_cast<int64_t>(bh) * P.n_pad * 128;
  float* sksel = P.sk_sel + static_cast<int64_t>(bh) * P.n_pad;
  for (int i = warp; i < P.n_pad; i += kRepairThreads / 32) {
    uint32_t codes = 0, kw = 0;
    float skv = 0.0f;
    if (i < P.n) {
      const int t = clamp_token(idx[i], P.S);
      float R[4];
      residual4(P, b, h, t, 4 * lane, vsc.s, vsc.r, R);
      codes = quant4(R[0], R[1], R[2], R[3], rsc.r);
      kw = __ldg(reinterpret_cast<const uint32_t*>(P.kc + (static_cast<int64_t>(bh) * P.S_pad + t) * 128) + lane);
      skv = P.sk[bh * P.nb + t / 128];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
      dvt[static_cast<int64_t>(4 * lane + e) * P.n_pad + i] = static_cast<uint8_t>(codes >> (8 * e));
    reinterpret_cast<uint32_t*>(ksel + static_cast<int64_t>(i) * 128)[lane] = kw;
    if (lane == 0) sksel[i] = skv;
    if (P.kb_sel != nullptr && lane < 8) {
      const uint32_t bw = i < P.n ? __ldg(reinterpret_cast<const uint32_t*>(
                                        P.kbias + (static_cast<int64_t>(bh) * P.S_pad + clamp_token(idx[i], P.S)) * 16) + lane)
                                  : 0u;
      reinterpret_cast<uint32_t*>(P.kb_sel + (static_cast<int64_t>(bh) * P.n_pad + i) * 16)[lane] = bw;
    }
  }
}

}  // namespace ovc
