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
//   assign  n_c = sum_d mu_cd^2 (channel order); dot = 32 partial sums over
//           channels 4k..4k+3 (left to right), then the pairwise tree
//           p_k += p_(k+w), w = 16..1; d = n_c - 2 dot; smallest d, ties to
//           the lower c
//   update  mu_c = sum / count: sums per 128-token block in token order, then
//           over blocks in block order; an empty cluster keeps its centroid
// Kernels (grid, block; the head index runs fastest, so CTAs that run
// together read whole token rows of V):
//   kmeans_init_kernel     (C, B*H) x 128
//   kmeans_assign_kernel   (B*H, nb) x 128: a thread per token, its values in
//                          registers, the centroids in shared memory
//   kmeans_partial_kernel  (B*H, nb) x 128: a thread per channel; per-cluster
//                          sums in shared memory, counts by thread 0
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
  // 32 partial sums over 4 channels and then the pairwise tree.
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
    float p[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float4 m = *reinterpret_cast<const float4*>(&mu[c][4 * k]);
      float a = __fmul_rn(x[4 * k], m.x);
      a = __fadd_rn(a, __fmul_rn(x[4 * k + 1], m.y));
      a = __fadd_rn(a, __fmul_rn(x[4 * k + 2], m.z));
      p[k] = __fadd_rn(a, __fmul_rn(x[4 * k + 3], m.w));
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
      for (int k = 0; k < w; ++k) p[k] = __fadd_rn(p[k], p[k + w]);
    const float dist = __fsub_rn(nrm[c], 2.0f * p[0]);
    if (dist < best) best = dist, arg = c;
  }
  G.labels[static_cast<int64_t>(bh) * G.S + t] = arg;
}

__global__ void __launch_bounds__(128) kmeans_partial_kernel(const __grid_constant__ GroupParams G) {
  __shared__ float part[kMaxClusters][128];
  __shared__ int cnt[kMaxClusters];
  const int bh = blockIdx.x, j = blockIdx.y, d = threadIdx.x;
  for (int c = 0; c < G.C; ++c) part[c][d] = 0.0f;
  if (d < G.C) cnt[d] = 0;
  __syncthreads();
  const int32_t* lab = G.labels + static_cast<int64_t>(bh) * G.S;
  const int t1 = min(G.S, j * 128 + 128);
  for (int t = j * 128; t < t1; ++t) {
    const int c = __ldg(lab + t);
    part[c][d] = __fadd_rn(part[c][d], group_x(G, bh, t, d));
    if (d == 0) ++cnt[c];
  }
  __syncthreads();
  const int64_t base = (static_cast<int64_t>(bh) * G.nb + j) * G.C;
  for (int c = 0; c < G.C; ++c) G.part[(base + c) * 128 + d] = part[c][d];
  if (d < G.C) G.cnt[base + d] = cnt[d];
}

__global__ void __launch_bounds__(128) kmeans_update_kernel(const __grid_constant__ GroupParams G) {
  const int c = blockIdx.x, bh = blockIdx.y, d = threadIdx.x;
  float s = 0.0f;
  int n = 0;
  for (int j = 0; j < G.nb; ++j) {
    const int64_t base = (static_cast<int64_t>(bh) * G.nb + j) * G.C + c;
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
