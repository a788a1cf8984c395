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
//   kmeans_assign_kernel   (B*H, nb) x 256: a warp per token, a lane per 4
//                          channels; the dot tree is the shuffle-down tree
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

__global__ void __launch_bounds__(256) kmeans_assign_kernel(const __grid_constant__ GroupParams G) {
  __shared__ float mu[kMaxClusters][128];
  __shared__ float nrm[kMaxClusters];
  const int bh = blockIdx.x, j = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* cent = G.cent + static_cast<int64_t>(bh) * G.C * 128;
  for (int i = threadIdx.x; i < G.C * 128; i += blockDim.x) mu[i >> 7][i & 127] = cent[i];
  __syncthreads();
  if (threadIdx.x < G.C) {
    float n = 0.0f;
    for (int d = 0; d < 128; ++d) n = __fadd_rn(n, __fmul_rn(mu[threadIdx.x][d], mu[threadIdx.x][d]));
    nrm[threadIdx.x] = n;
  }
  __syncthreads();
  const int t1 = min(G.S, j * 128 + 128);
  for (int t = j * 128 + warp; t < t1; t += 8) {
    float x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = group_x(G, bh, t, 4 * lane + i);
    float best = INFINITY;
    int arg = 0;
    for (int c = 0; c < G.C; ++c) {
      float p = __fmul_rn(x[0], mu[c][4 * lane]);
#pragma unroll
      for (int i = 1; i < 4; ++i) p = __fadd_rn(p, __fmul_rn(x[i], mu[c][4 * lane + i]));
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) p = __fadd_rn(p, __shfl_down_sync(0xFFFFFFFFu, p, w));
      // lane 0 holds the tree's result
      const float dist = __fsub_rn(nrm[c], 2.0f * p);
      if (dist < best) best = dist, arg = c;
    }
    if (lane == 0) G.labels[static_cast<int64_t>(bh) * G.S + t] = arg;
  }
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
