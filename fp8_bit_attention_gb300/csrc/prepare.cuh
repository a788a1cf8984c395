// prepare.cuh -- input preparation: BF16/FP16 Q, K, V -> E4M3 plus scales.
//
// "Open VC Attention" (catalogue entry): Q/K scales per block, V per head.
// "Open-VC attention" (news item), "Architectural optimisations": the Q, K and
// V quantisation is one fused preparation step.
//
// Quantisation is defined in FP32: s = amax/448, r = 448/amax (IEEE single
// divisions; amax = 0 gives s = r = 1), code = E4M3_rn_satfinite(x * r).
//
// K smoothing (optional; the VC-Attention summary, "Why attention is the
// video bottleneck", names Q/K smoothing as the prior art): K's per-channel
// means over the sequence are subtracted (FP32) before K is quantised, which
// leaves non-causal softmax unchanged and takes the channel offset out of
// K's block scales.  The mean is summed in a fixed order -- per 128-token
// block in token order, then the block sums in block order, then / S -- so
// that it is reproducible bit for bit:
//   k_mean_partial_kernel  grid (B*H, nb) x 128: one thread per channel.
//   k_mean_final_kernel    grid (B*H) x 128.
// Q smoothing (optional, same summary): Q's channel means mu_q, summed the
// same way, are subtracted before Q is quantised.  That moves every score of
// key t by mu_q . k_t, which differs from key to key, so it is added back:
// while K is quantised, each key's bias beta_t = mu_q . dec(K^_t) is written
// as a BF16 pair (hi, lo), hi + lo ~ beta_t to 16 bits, laid out as the B
// operand of a BF16 MMA that adds beta_t / s_q to the key's scores.
//
// Two launches, both HBM-bound and coalesced.  The head index runs fastest
// in every grid: CTAs that run together read the same tokens of all heads,
// i.e. whole contiguous token rows of the [B,S,H,128] inputs.
//   prepare_qk_kernel  grid (B*H, nb, 3): z = 0 quantises a 128-token block of
//                      Q, z = 1 of K, z = 2 folds the block's amax|V| into the
//                      head's running maximum.
//   prepare_v_kernel   grid (B*H, nb): quantises a 128-token block of V with
//                      the head scale, writes it transposed (keys contiguous)
//                      and the per-token residual energy.
// V-Smooth (optional): vsmooth_mean_kernel replaces the z = 2 amax pass (it
// writes the block means and folds amax|v - mu| into the head maximum), and
// prepare_v_kernel quantises v - mu and writes the restored means.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace ovc {

struct PrepParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  int64_t qs[3], ks[3], vs[3];   // element strides (b, s, h)
  int32_t B, S, H, nb, S_pad;
  int32_t fp16;                  // 0: BF16 inputs, 1: FP16 inputs
  uint8_t* qc;
  uint8_t* kc;
  uint8_t* vt;
  float* sq;
  float* sk;
  float* sv;
  uint32_t* vamax;
  float* energy;
  // K smoothing (both NULL when off): kpart [B*H][nb][128] block sums,
  // kmean [B*H][128] channel means subtracted from K before quantising.
  float* kpart;
  float* kmean;
  // Q smoothing (all NULL when off): qpart, qmean as kpart, kmean for Q;
  // kbias [B*H][S_pad][16] BF16 bits, key t's row (hi, lo, hi, lo, 0 x 12)
  // of beta_t = mu_q . dec(K^_t) (rows >= S zero).
  float* qpart;
  float* qmean;
  uint16_t* kbias;
  // V-Smooth (both NULL when off): vmu [B*H][nb][128] block means of V (BF16
  // values held as FP32); vmean [B*H][128][nbk] BF16 bits of the restored
  // means M'_b = bf16(mu_b r), channel-major with blocks contiguous (the B
  // operand of the mean-restore MMA), nbk = nb rounded up to 16.
  float* vmu;
  uint16_t* vmean;
  int32_t nbk;
  // Grouping (NULL when off): [B*H][S] token order of K and V -- row t of the
  // prepared K and V is input token perm[t] (Q keeps its order).
  const int32_t* perm;
};

// Input row of prepared K/V row t (the identity without grouping).
template <bool kPerm>
__device__ __forceinline__ int kv_row(const PrepParams& P, int bh, int t) {
  return kPerm ? __ldg(P.perm + static_cast<int64_t>(bh) * P.S + t) : t;
}

// Options of the preparation kernels, as template bits, so that the plain
// preparation carries none of their tests.
constexpr int kPrepSmoothK = 1;
constexpr int kPrepPerm = 2;
constexpr int kPrepSmoothQ = 4;

// |x| of two packed 16-bit floats, as ordered integers (sign bit cleared).
__device__ __forceinline__ uint32_t abs2_bits(uint32_t w) { return w & 0x7FFF7FFFu; }

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16, int fp16) {
  if (!fp16) return __uint_as_float(bits16 << 16);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

__device__ __forceinline__ float2 unpack2(uint32_t w, int fp16) {
  return make_float2(half_bits_to_float(w & 0xFFFFu, fp16), half_bits_to_float(w >> 16, fp16));
}

struct QScale {
  float s, r;
};

__device__ __forceinline__ QScale scale_from_amax(float amax) {
  if (amax == 0.0f) return {1.0f, 1.0f};
  return {__fdiv_rn(amax, 448.0f), __fdiv_rn(448.0f, amax)};
}

// Four values -> four E4M3 bytes in one word (first value in bits 0..7).
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float r) {
  const uint32_t lo = cvt_e4m3x2(__fmul_rn(a, r), __fmul_rn(b, r));
  const uint32_t hi = cvt_e4m3x2(__fmul_rn(c, r), __fmul_rn(d, r));
  return lo | (hi << 16);
}

// E4M3 bytes of a word -> four FP32 values (exact).
__device__ __forceinline__ void dec4(uint32_t codes, float* out) {
  uint32_t lo, hi;
  cvt_e4m3x4_to_f16x2x2(codes, lo, hi);
  const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  out[0] = f0.x;
  out[1] = f0.y;
  out[2] = f1.x;
  out[3] = f1.y;
}

// Maximum of a 32-bit value over the CTA (blockDim.x multiple of 32, <= 1024).
__device__ __forceinline__ uint32_t block_max_u32(uint32_t m, uint32_t* red) {
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = (lane < static_cast<int>(blockDim.x >> 5)) ? red[lane] : 0u;
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red[0] = m;
  }
  __syncthreads();
  const uint32_t r = red[0];
  __syncthreads();
  return r;
}

// Channel sums of one 128-token block of K (kQ: of Q, which keeps its token
// order), in token order.
template <bool kPerm, bool kQ = false>
__global__ void __launch_bounds__(128) k_mean_partial_kernel(const __grid_constant__ PrepParams P) {
  const int bh = blockIdx.x, j = blockIdx.y, d = threadIdx.x;
  const int b = bh / P.H, h = bh % P.H;
  const int t1 = min(P.S, j * 128 + 128);
  const int64_t* st = kQ ? P.qs : P.ks;
  const uint16_t* src = (kQ ? P.q : P.k) + b * st[0] + h * st[2] + d;
  float part = 0.0f;
  // The loads are independent and can be in flight together; the additions
  // stay in token order.
#pragma unroll 16
  for (int t = j * 128; t < t1; ++t) {
    const int tr = kQ ? t : kv_row<kPerm>(P, bh, t);
    part = __fadd_rn(part, half_bits_to_float(__ldg(src + static_cast<int64_t>(tr) * st[1]), P.fp16));
  }
  (kQ ? P.qpart : P.kpart)[(static_cast<int64_t>(bh) * P.nb + j) * 128 + d] = part;
}

// Channel means: the block sums in block order, then one division by S.
template <bool kQ = false>
__global__ void __launch_bounds__(128) k_mean_final_kernel(const __grid_constant__ PrepParams P) {
  const int bh = blockIdx.x, d = threadIdx.x;
  const float* part = (kQ ? P.qpart : P.kpart) + static_cast<int64_t>(bh) * P.nb * 128 + d;
  float total = 0.0f;
  for (int j = 0; j < P.nb; ++j) total = __fadd_rn(total, part[j * 128]);
  (kQ ? P.qmean : P.kmean)[bh * 128 + d] = __fdiv_rn(total, static_cast<float>(P.S));
}

// Q smoothing: key t's bias beta_t = mu_q . dec(code_t) from this thread's
// 64 channels (words w, channels 64 half ..), summed with the other half's
// thread (the neighbouring lane), written as the BF16 row
// (hi, lo, hi, lo, 0, ..., 0), hi = bf16(beta), lo = bf16(beta - hi).
__device__ __forceinline__ void write_key_bias(const PrepParams& P, int bh, int t, int half, const uint32_t* w) {
  const float* mu = P.qmean + bh * 128 + half * 64;
  float acc = 0.0f;
#pragma unroll
  for (int g = 0; g < 16; ++g) {
    float dq[4];
    dec4(w[g], dq);
#pragma unroll
    for (int e = 0; e < 4; ++e) acc = fmaf(__ldg(mu + 4 * g + e), dq[e], acc);
  }
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
  if (half == 0) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
    const __nv_bfloat16 lo = __float2bfloat16_rn(acc - __bfloat162float(hi));
    const uint32_t hl = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
    uint4* dst = reinterpret_cast<uint4*>(P.kbias + (static_cast<int64_t>(bh) * P.S_pad + t) * 16);
    dst[0] = make_uint4(hl, hl, 0u, 0u);
    dst[1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// V-Smooth ("VC-Attention" summary, "V-Smooth"), first pass: per 128-token
// block of V and channel, the mean mu = bf16(fl(sum in token order) / n)
// (n = the block's valid tokens), then the block's amax of fl(v - mu) folded
// into the head's running maximum.  One thread per channel; every token row
// is a coalesced 256-byte read, and the second read of the block hits cache.
template <bool kPerm>
__global__ void __launch_bounds__(128) vsmooth_mean_kernel(const __grid_constant__ PrepParams P) {
  __shared__ uint32_t red[32];
  const int bh = blockIdx.x, j = blockIdx.y, d = threadIdx.x;
  const int b = bh / P.H, h = bh % P.H;
  const int t0 = j * 128, t1 = min(P.S, t0 + 128);
  const uint16_t* src = P.v + b * P.vs[0] + h * P.vs[2] + d;
  float sum = 0.0f;
#pragma unroll 16
  for (int t = t0; t < t1; ++t)
    sum = __fadd_rn(sum, half_bits_to_float(__ldg(src + static_cast<int64_t>(kv_row<kPerm>(P, bh, t)) * P.vs[1]), P.fp16));
  const float mu = __bfloat162float(__float2bfloat16_rn(__fdiv_rn(sum, static_cast<float>(t1 - t0))));
  P.vmu[(static_cast<int64_t>(bh) * P.nb + j) * 128 + d] = mu;
  float m = 0.0f;
#pragma unroll 16
  for (int t = t0; t < t1; ++t)
    m = fmaxf(m, fabsf(__fsub_rn(half_bits_to_float(__ldg(src + static_cast<int64_t>(kv_row<kPerm>(P, bh, t)) * P.vs[1]), P.fp16), mu)));
  const uint32_t mb = block_max_u32(__float_as_uint(m), red);
  if (d == 0) atomicMax(P.vamax + bh, mb);
}

// One 128-token block of Q or K (z = 0, 1), or the amax of one block of V
// (z = 2).  256 threads: two per token row, 64 channels each.
template <int kOpt>
__global__ void __launch_bounds__(256) prepare_qk_kernel(const __grid_constant__ PrepParams P) {
  __shared__ uint32_t red[32];
  const int bh = blockIdx.x;
  const int j = blockIdx.y;
  const int which = blockIdx.z;
  const int b = bh / P.H, h = bh % P.H;
  const int tid = threadIdx.x;
  const int row = tid >> 1, half = tid & 1;
  const int t = j * 128 + row;

  const uint16_t* src = which == 0 ? P.q : (which == 1 ? P.k : P.v);
  const int64_t* st = which == 0 ? P.qs : (which == 1 ? P.ks : P.vs);

  uint4 x[8];
  if (t < P.S) {
    const int tr = which > 0 ? kv_row<(kOpt & kPrepPerm) != 0>(P, bh, t) : t;
    const uint4* p = reinterpret_cast<const uint4*>(src + b * st[0] + static_cast<int64_t>(tr) * st[1] + h * st[2] + half * 64);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __ldg(p + i);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = make_uint4(0, 0, 0, 0);
  }

  if (((kOpt & kPrepSmoothK) && which == 1) || ((kOpt & kPrepSmoothQ) && which == 0)) {
    // Smoothed K (or Q): the centred values fl(x - mean) set the block amax
    // and are quantised; rows past S stay zero (no code, no part of the amax).
    const float* mu = (which == 0 ? P.qmean : P.kmean) + bh * 128 + half * 64;
    float c[64];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t wd[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack2(wd[e], P.fp16);
        c[8 * i + 2 * e] = t < P.S ? __fsub_rn(f.x, __ldg(mu + 8 * i + 2 * e)) : 0.0f;
        c[8 * i + 2 * e + 1] = t < P.S ? __fsub_rn(f.y, __ldg(mu + 8 * i + 2 * e + 1)) : 0.0f;
      }
    }
    float m = 0.0f;
#pragma unroll
    for (int e = 0; e < 64; ++e) m = fmaxf(m, fabsf(c[e]));
    const float amax = __uint_as_float(block_max_u32(__float_as_uint(m), red));
    const QScale sc = scale_from_amax(amax);
    if (tid == 0) (which == 0 ? P.sq : P.sk)[bh * P.nb + j] = sc.s;
    uint32_t w[16];
#pragma unroll
    for (int g = 0; g < 16; ++g) w[g] = quant4(c[4 * g], c[4 * g + 1], c[4 * g + 2], c[4 * g + 3], sc.r);
    uint4* d4 = reinterpret_cast<uint4*>((which == 0 ? P.qc : P.kc) + (static_cast<int64_t>(bh) * P.S_pad + t) * 128 +
                                         half * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    if ((kOpt & kPrepSmoothQ) && which == 1) write_key_bias(P, bh, t, half, w);
    return;
  }

  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    m2 = __vmaxu2(m2, abs2_bits(x[i].x));
    m2 = __vmaxu2(m2, abs2_bits(x[i].y));
    m2 = __vmaxu2(m2, abs2_bits(x[i].z));
    m2 = __vmaxu2(m2, abs2_bits(x[i].w));
  }
  const uint32_t mbits = block_max_u32(max(m2 & 0xFFFFu, m2 >> 16), red);
  const float amax = half_bits_to_float(mbits, P.fp16);

  if (which == 2) {
    if (tid == 0) atomicMax(P.vamax + bh, __float_as_uint(amax));
    return;
  }

  const QScale sc = scale_from_amax(amax);
  if (tid == 0) (which == 0 ? P.sq : P.sk)[bh * P.nb + j] = sc.s;

  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 a = unpack2(x[i].x, P.fp16), b2 = unpack2(x[i].y, P.fp16);
    const float2 c = unpack2(x[i].z, P.fp16), d = unpack2(x[i].w, P.fp16);
    w[2 * i] = quant4(a.x, a.y, b2.x, b2.y, sc.r);
    w[2 * i + 1] = quant4(c.x, c.y, d.x, d.y, sc.r);
  }
  uint8_t* dst = (which == 0 ? P.qc : P.kc) + (static_cast<int64_t>(bh) * P.S_pad + t) * 128 + half * 64;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  if ((kOpt & kPrepSmoothQ) && which == 1) write_key_bias(P, bh, t, half, w);
}

// One 128-token block of V.  512 threads: warp w owns channels 8w..8w+7,
// lane l owns tokens 4l..4l+3 of the block.  Writes V^T (keys contiguous)
// with coalesced 128-byte rows, and the residual energy of each token:
// R = fl(v - fl(s_v * dec(code))), sixteen sequential partial sums over 8
// channels, then the pairwise tree p_g += p_(g+w), w = 8, 4, 2, 1.
template <bool kVSmooth, bool kPerm>
__global__ void __launch_bounds__(512) prepare_v_kernel(const __grid_constant__ PrepParams P) {
  __shared__ float part[16][128];
  const int bh = blockIdx.x;
  const int j = blockIdx.y;
  const int b = bh / P.H, h = bh % P.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const float amax = __uint_as_float(P.vamax[bh]);
  const QScale sc = scale_from_amax(amax);
  if (j == 0 && threadIdx.x == 0) P.sv[bh] = sc.s;
  constexpr bool vs = kVSmooth;
  float mu[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mu[i] = vs ? P.vmu[(static_cast<int64_t>(bh) * P.nb + j) * 128 + 8 * warp + i] : 0.0f;
  if (vs && lane == 0) {
    // Restored means in the scale's units, M'_b = bf16(mu_b r).
#pragma unroll
    for (int i = 0; i < 8; ++i)
      P.vmean[(static_cast<int64_t>(bh) * 128 + 8 * warp + i) * P.nbk + j] =
          __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(mu[i], sc.r)));
  }

  uint32_t lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int t = j * 128 + 4 * lane + k;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (t < P.S)
      x = __ldg(reinterpret_cast<const uint4*>(P.v + b * P.vs[0] + static_cast<int64_t>(kv_row<kPerm>(P, bh, t)) * P.vs[1] +
                                               h * P.vs[2] + 8 * warp));
    const float2 a = unpack2(x.x, P.fp16), c = unpack2(x.y, P.fp16);
    const float2 d = unpack2(x.z, P.fp16), e = unpack2(x.w, P.fp16);
    float xv[8] = {a.x, a.y, c.x, c.y, d.x, d.y, e.x, e.y};
    if (vs) {   // V-Smooth: the residual fl(v - mu_b) is quantised; padding rows stay 0
#pragma unroll
      for (int i = 0; i < 8; ++i) xv[i] = t < P.S ? __fsub_rn(xv[i], mu[i]) : 0.0f;
    }
    lo[k] = quant4(xv[0], xv[1], xv[2], xv[3], sc.r);
    hi[k] = quant4(xv[4], xv[5], xv[6], xv[7], sc.r);
    float dq[8];
    dec4(lo[k], dq);
    dec4(hi[k], dq + 4);
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float r = __fsub_rn(xv[i], __fmul_rn(sc.s, dq[i]));
      const float sq = __fmul_rn(r, r);
      acc = (i == 0) ? sq : __fadd_rn(acc, sq);
    }
    part[warp][k * 32 + lane] = acc;
  }

  // 4 tokens x 8 channels -> 8 words (one per channel) of 4 token bytes.
  uint32_t out[8];
  {
    const uint32_t a01 = __byte_perm(lo[0], lo[1], 0x5140), a23 = __byte_perm(lo[2], lo[3], 0x5140);
    const uint32_t b01 = __byte_perm(lo[0], lo[1], 0x7362), b23 = __byte_perm(lo[2], lo[3], 0x7362);
    out[0] = __byte_perm(a01, a23, 0x5410);
    out[1] = __byte_perm(a01, a23, 0x7632);
    out[2] = __byte_perm(b01, b23, 0x5410);
    out[3] = __byte_perm(b01, b23, 0x7632);
    const uint32_t c01 = __byte_perm(hi[0], hi[1], 0x5140), c23 = __byte_perm(hi[2], hi[3], 0x5140);
    const uint32_t d01 = __byte_perm(hi[0], hi[1], 0x7362), d23 = __byte_perm(hi[2], hi[3], 0x7362);
    out[4] = __byte_perm(c01, c23, 0x5410);
    out[5] = __byte_perm(c01, c23, 0x7632);
    out[6] = __byte_perm(d01, d23, 0x5410);
    out[7] = __byte_perm(d01, d23, 0x7632);
  }
  uint8_t* vt = P.vt + (static_cast<int64_t>(bh) * 128 + 8 * warp) * P.S_pad + j * 128 + 4 * lane;
#pragma unroll
  for (int d = 0; d < 8; ++d) *reinterpret_cast<uint32_t*>(vt + static_cast<int64_t>(d) * P.S_pad) = out[d];

  __syncthreads();
  if (threadIdx.x < 128 && !vs) {   // V-Smooth computes no repair energies
    const int tok = threadIdx.x;
    const int t = j * 128 + tok;
    if (t < P.S) {
      float p[16];
#pragma unroll
      for (int g = 0; g < 16; ++g) p[g] = part[g][(tok & 3) * 32 + (tok >> 2)];
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int g = 0; g < w; ++g) p[g] = __fadd_rn(p[g], p[g + w]);
      P.energy[static_cast<int64_t>(bh) * P.S + t] = p[0];
    }
  }
}

}  // namespace ovc
