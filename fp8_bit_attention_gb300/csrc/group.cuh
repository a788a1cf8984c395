// group.cuh -- V-Smooth's grouping step: k-means over each head's value
// tokens, then the tokens ordered by (cluster, index).
//
// "VC-Attention" summary, "V-Smooth": online k-means clusters the value
// tokens of every batch entry and head, and keys and values are permuted
// together (non-causal attention does not change), so that the 128-token
// blocks whose means V-Smooth subtracts hold similar values.
//
// Lloyd's algorithm in FP32 with every step rounded in a fixed order (so the
// labels and the permutation reproduce bit for bit):
//   start   mu_c = x_(floor(c S / C))
//   assign  n_c = sum_d mu_cd^2 (channel order); dot = 16 partial sums over
//           channels 8k..8k+7 (the first product rounded, then fused
//           multiply-adds left to right), then the pairwise tree
//           p_k += p_(k+w), w = 8..1; d = n_c - 2 dot; smallest d, ties to
//           the lower c
//   update  mu_c = sum / count: sums per 128-token block in token order, then
//           over blocks in block order; an empty cluster keeps its centroid
// Kernels (grid, block; the head index runs fastest, so CTAs that run
// together read whole token rows of V):
//   kmeans_init_kernel     (C, B*H) x 128
//   kmeans_assign_kernel   (B*H, nb) x 128: a thread per token, its values in
//                          registers, the centroids in shared memory
//   kmeans_partial_kernel  (B*H, nb) x 128: the block's tokens staged in shared
//                          memory by 16-byte loads and listed per cluster in
//                          token order; a thread per channel then sums each
//                          cluster's members in a register
//   kmeans_update_kernel   (C, B*H) x 128
//   group_count_kernel / group_offset_kernel / group_scatter_kernel: a
//                          stable counting sort of the labels
#pragma once

#include <cstdint>

#include "prepare.cuh"

namespace ovc {

constexpr int kMaxClusters = 64;

struct GroupParams {
  const uint16_t* v;
  int64_t vs[3];            // element strides (b, s, h)
  int32_t B, S, H, nb, C, fp16;
  float* cent;              // [B*H][C][128]
  int32_t* labels;          // [B*H][S]
  float* part;              // [B*H][nb][C][128] per-block member sums
  int32_t* cnt;             // [B*H][nb][C] per-block member counts
  int32_t* off;             // [B*H][nb][C] first position of each (block, cluster)
  int32_t* perm;            // [B*H][S] grouped order: position -> token
};

__device__ __forceinline__ float group_x(const GroupParams& G, int bh, int t, int d) {
  const int b = bh / G.H, h = bh - b * G.H;
  return half_bits_to_float(__ldg(G.v + b * G.vs[0] + static_cast<int64_t>(t) * G.vs[1] + h * G.vs[2] + d), G.fp16);
}

__global__ void __launch_bounds__(128) kmeans_init_kernel(const __grid_constant__ GroupParams G) {
  const int c = blockIdx.x, bh = blockIdx.y, d = threadIdx.x;
  const int t = static_cast<int>(static_cast<int64_t>(c) * G.S / G.C);
  G.cent[(static_cast<int64_t>(bh) * G.C + c) * 128 + d] = group_x(G, bh, t, d);
}

__global__ void __launch_bounds__(128) kmeans_assign_kernel(const __grid_constant__ GroupParams G) {
  __shared__ __align__(16) float mu[kMaxClusters][128];
  __shared__ float nrm[kMaxClusters];
  const int bh = blockIdx.x, j = blockIdx.y, tid = threadIdx.x;
  const float* cent = G.cent + static_cast<int64_t>(bh) * G.C * 128;
  for (int i = tid; i < G.C * 128; i += blockDim.x) mu[i >> 7][i & 127] = cent[i];
  __syncthreads();
  if (tid < G.C) {
    float n = 0.0f;
    for (int d = 0; d < 128; ++d) n = __fadd_rn(n, __fmul_rn(mu[tid][d], mu[tid][d]));
    nrm[tid] = n;
  }
  __syncthreads();
  // One thread per token: its 128 values in registers, the dot product as
  // 16 partial sums over 8 channels (fused multiply-adds) and then the
  // pairwise tree.  The centroids are read from shared memory as warp-wide
  // broadcasts; their delivery to every lane's registers bounds the kernel.
  const int t = j * 128 + tid;
  if (t >= G.S) return;
  const int b = bh / G.H, h = bh - b * G.H;
  const uint4* row = reinterpret_cast<const uint4*>(G.v + b * G.vs[0] + static_cast<int64_t>(t) * G.vs[1] + h * G.vs[2]);
  float x[128];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint4 w = __ldg(row + i);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack2(ws[e], G.fp16);
      x[8 * i + 2 * e] = f.x;
      x[8 * i + 2 * e + 1] = f.y;
    }
  }
  float best = INFINITY;
  int arg = 0;
  for (int c = 0; c < G.C; ++c) {
    float p[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float4 m0 = *reinterpret_cast<const float4*>(&mu[c][8 * k]);
      const float4 m1 = *reinterpret_cast<const float4*>(&mu[c][8 * k + 4]);
      float a = __fmul_rn(x[8 * k], m0.x);
      a = __fmaf_rn(x[8 * k + 1], m0.y, a);
      a = __fmaf_rn(x[8 * k + 2], m0.z, a);
      a = __fmaf_rn(x[8 * k + 3], m0.w, a);
      a = __fmaf_rn(x[8 * k + 4], m1.x, a);
      a = __fmaf_rn(x[8 * k + 5], m1.y, a);
      a = __fmaf_rn(x[8 * k + 6], m1.z, a);
      p[k] = __fmaf_rn(x[8 * k + 7], m1.w, a);
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
      for (int k = 0; k < w; ++k) p[k] = __fadd_rn(p[k], p[k + w]);
    const float dist = __fsub_rn(nrm[c], 2.0f * p[0]);
    if (dist < best) best = dist, arg = c;
  }
  G.labels[static_cast<int64_t>(bh) * G.S + t] = arg;
}

// Dynamic shared memory of kmeans_partial_kernel: the block's tokens
// (kXsPitch 16-bit values a row, rows 16-byte aligned), their labels, the
// members of each cluster in token order, and per-cluster counts and offsets.
constexpr int kXsPitch = 136;

__host__ __device__ constexpr size_t kmeans_partial_smem() {
  return 128 * kXsPitch * 2 + 3 * 128 * 4 + 2 * kMaxClusters * 4;
}

__global__ void __launch_bounds__(128) kmeans_partial_kernel(const __grid_constant__ GroupParams G) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  int* lab = reinterpret_cast<int*>(smem + 128 * kXsPitch * 2);
  int* rank = lab + 128;
  int* member = rank + 128;
  int* cnt = member + 128;
  int* first = cnt + kMaxClusters;
  const int bh = blockIdx.x, j = blockIdx.y, d = threadIdx.x;
  const int b = bh / G.H, h = bh - b * G.H;
  const int t0 = j * 128, nt = min(128, G.S - t0);
  // The block's tokens in one round of 16-byte loads (all in flight before
  // the first store), and their labels.
  const uint16_t* vb = G.v + b * G.vs[0] + static_cast<int64_t>(t0) * G.vs[1] + h * G.vs[2];
  uint4 w[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int t = (d >> 4) + 8 * q, c = d & 15;
    if (t < nt) w[q] = __ldg(reinterpret_cast<const uint4*>(vb + static_cast<int64_t>(t) * G.vs[1]) + c);
  }
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int t = (d >> 4) + 8 * q, c = d & 15;
    if (t < nt) *reinterpret_cast<uint4*>(xs + t * kXsPitch + 8 * c) = w[q];
  }
  if (d < nt) lab[d] = __ldg(G.labels + static_cast<int64_t>(bh) * G.S + t0 + d);
  if (d < G.C) cnt[d] = 0;
  __syncthreads();
  // Members of each cluster, in token order: a token's place is the number
  // of earlier tokens with its label.
  if (d < nt) {
    const int c = lab[d];
    int r = 0;
    for (int t = 0; t < d; ++t) r += (lab[t] == c);
    rank[d] = r;
    atomicAdd(&cnt[c], 1);
  }
  __syncthreads();
  if (d == 0) {
    int pos = 0;
    for (int c = 0; c < G.C; ++c) {
      first[c] = pos;
      pos += cnt[c];
    }
  }
  __syncthreads();
  if (d < nt) member[first[lab[d]] + rank[d]] = d;
  __syncthreads();
  // A thread per channel: each cluster's sum in token order.
  const int64_t base = (static_cast<int64_t>(bh) * G.nb + j) * G.C;
  for (int c = 0; c < G.C; ++c) {
    float acc = 0.0f;
    const int m1 = first[c] + cnt[c];
    for (int m = first[c]; m < m1; ++m) acc = __fadd_rn(acc, half_bits_to_float(xs[member[m] * kXsPitch + d], G.fp16));
    G.part[(base + c) * 128 + d] = acc;
  }
  if (d < G.C) G.cnt[base + d] = cnt[d];
}

__global__ void __launch_bounds__(128) kmeans_update_kernel(const __grid_constant__ GroupParams G) {
  const int c = blockIdx.x, bh = blockIdx.y, d = threadIdx.x;
  float s = 0.0f;
  int n = 0;
  // Sums in block order; the loads of eight blocks are issued together.
  const int64_t base0 = static_cast<int64_t>(bh) * G.nb * G.C + c;
  int j = 0;
  for (; j + 8 <= G.nb; j += 8) {
    float v[8];
    int k[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int64_t base = base0 + static_cast<int64_t>(j + e) * G.C;
      v[e] = __ldg(G.part + base * 128 + d);
      k[e] = __ldg(G.cnt + base);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      s = __fadd_rn(s, v[e]);
      n += k[e];
    }
  }
  for (; j < G.nb; ++j) {
    const int64_t base = base0 + static_cast<int64_t>(j) * G.C;
    s = __fadd_rn(s, G.part[base * 128 + d]);
    n += G.cnt[base];
  }
  if (n > 0) G.cent[(static_cast<int64_t>(bh) * G.C + c) * 128 + d] = __fdiv_rn(s, static_cast<float>(n));
}

// Members of each cluster in each 128-token block.
__global__ void __launch_bounds__(128) group_count_kernel(const __grid_constant__ GroupParams G) {
  __shared__ int cnt[kMaxClusters];
  const int bh = blockIdx.x, j = blockIdx.y, tid = threadIdx.x;
  if (tid < G.C) cnt[tid] = 0;
  __syncthreads();
  const int t = j * 128 + tid;
  if (t < G.S) atomicAdd(&cnt[G.labels[static_cast<int64_t>(bh) * G.S + t]], 1);
  __syncthreads();
  if (tid < G.C) G.cnt[(static_cast<int64_t>(bh) * G.nb + j) * G.C + tid] = cnt[tid];
}

// First grouped position of each (block, cluster): clusters in order, and
// within a cluster the blocks in order.  One thread per cluster.
__global__ void __launch_bounds__(kMaxClusters) group_offset_kernel(const __grid_constant__ GroupParams G) {
  __shared__ int total[kMaxClusters];
  const int bh = blockIdx.x, c = threadIdx.x;
  const int32_t* cnt = G.cnt + static_cast<int64_t>(bh) * G.nb * G.C;
  int n = 0;
  if (c < G.C)
    for (int j = 0; j < G.nb; ++j) n += cnt[j * G.C + c];
  total[c] = n;
  __syncthreads();
  if (c < G.C) {
    int pos = 0;
    for (int i = 0; i < c; ++i) pos += total[i];
    int32_t* off = G.off + static_cast<int64_t>(bh) * G.nb * G.C;
    for (int j = 0; j < G.nb; ++j) {
      off[j * G.C + c] = pos;
      pos += cnt[j * G.C + c];
    }
  }
}

// perm[position] = token: a token goes after the earlier tokens of its
// cluster (earlier blocks through the offsets, earlier tokens of its own
// block by counting).
__global__ void __launch_bounds__(128) group_scatter_kernel(const __grid_constant__ GroupParams G) {
  __shared__ int lab[128];
  const int bh = blockIdx.x, j = blockIdx.y, tid = threadIdx.x;
  const int t = j * 128 + tid;
  lab[tid] = t < G.S ? G.labels[static_cast<int64_t>(bh) * G.S + t] : -1;
  __syncthreads();
  if (t >= G.S) return;
  const int c = lab[tid];
  int rank = 0;
  for (int i = 0; i < tid; ++i) rank += (lab[i] == c);
  G.perm[static_cast<int64_t>(bh) * G.S + G.off[(static_cast<int64_t>(bh) * G.nb + j) * G.C + c] + rank] = t;
}

}  // namespace ovc
