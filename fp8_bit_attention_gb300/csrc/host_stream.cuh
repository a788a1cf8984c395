// host_stream.cuh -- the whole call for inputs and output in host memory
// (ovc_attention_host): head chunks streamed through the device so that the
// host<->device copies of one chunk overlap the computation of its
// neighbours.  Host code only; included by ovc.cu after the device entry
// points, which it calls.
//
// The pages' API takes device tensors; this path exists so that a caller
// whose Q, K, V and O live in host memory gets the same result without
// staging whole tensors on the device.  Every head is computed on its own
// (its V scale, residual ranking and attention involve that head alone), so
// a chunked call equals one call over all heads bit for bit.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "ovc.h"

namespace ovc {
namespace host_stream {

// Bytes of one staging tensor of a chunk of `heads` heads.
inline size_t chunk_bytes(int64_t B, int64_t S, int64_t heads, size_t elem) {
  return static_cast<size_t>(B) * static_cast<size_t>(S) * static_cast<size_t>(heads) * 128u * elem;
}

inline size_t align256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

// Layout of the workspace: two sets (chunk c uses set c % 2), each with the
// staged Q, K, V, the preparation, the repair set and the staged output.
struct HostLayout {
  size_t in[2][3], prep[2], rep[2], out[2];
  size_t prep_bytes, rep_bytes, total;
};

// (BF16 and FP16 inputs both take 2 bytes an element.)
inline bool layout(int64_t B, int64_t S, int64_t hmax, uint32_t prep_flags, float budget, HostLayout* L) {
  const size_t elem = 2;
  L->prep_bytes = ovc_prepare_workspace_bytes_ex(B, S, hmax, 128, prep_flags);
  if (L->prep_bytes == 0) return false;
  L->rep_bytes = 0;
  if (budget > 0.0f) {
    L->rep_bytes = ovc_repair_workspace_bytes(B, S, hmax, budget);
    if (L->rep_bytes == 0) return false;
  }
  size_t off = 0;
  for (int st = 0; st < 2; ++st) {
    for (int i = 0; i < 3; ++i) {
      L->in[st][i] = off;
      off = align256(off + chunk_bytes(B, S, hmax, elem));
    }
    L->prep[st] = off;
    off = align256(off + L->prep_bytes);
    L->rep[st] = off;
    off = align256(off + L->rep_bytes);
    L->out[st] = off;
    off = align256(off + chunk_bytes(B, S, hmax, 2));
  }
  L->total = off;
  return true;
}

// The streams and events of one call: chunks alternate between two compute
// streams (so that a chunk's preparation and first CTAs can start on SMs the
// previous chunk's last, partly filled wave leaves idle), with one stream
// for copies in and one for copies out.  Per staging set: `ready` (its
// inputs are on the device), `in_free` (the preparation has read them),
// `done` (its output is computed), `out_free` (its output is copied out).
struct Streams {
  cudaStream_t comp[2] = {nullptr, nullptr}, in = nullptr, out = nullptr;
  cudaEvent_t ready[2] = {nullptr, nullptr}, in_free[2] = {nullptr, nullptr};
  cudaEvent_t done[2] = {nullptr, nullptr}, out_free[2] = {nullptr, nullptr};

  bool create() {
    for (cudaStream_t* s : {&comp[0], &comp[1], &in, &out})
      if (cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) != cudaSuccess) return false;
    for (int st = 0; st < 2; ++st)
      for (cudaEvent_t* e : {&ready[st], &in_free[st], &done[st], &out_free[st]})
        if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
  // Waits for everything issued on the call's streams, then releases them.
  bool finish() {
    bool ok = true;
    for (cudaStream_t s : {out, in, comp[0], comp[1]})
      if (s && cudaStreamSynchronize(s) != cudaSuccess) ok = false;
    for (int st = 0; st < 2; ++st)
      for (cudaEvent_t e : {ready[st], in_free[st], done[st], out_free[st]})
        if (e) cudaEventDestroy(e);
    for (cudaStream_t s : {comp[0], comp[1], in, out})
      if (s) cudaStreamDestroy(s);
    return ok;
  }
};

inline ovc_tensor chunk_tensor(const void* ptr, int32_t dtype, int64_t B, int64_t S, int64_t hc) {
  ovc_tensor t{};
  t.ptr = ptr;
  t.dtype = dtype;
  t.B = B;
  t.S = S;
  t.H = hc;
  t.D = 128;
  t.stride_b = S * hc * 128;
  t.stride_s = hc * 128;
  t.stride_h = 128;
  return t;
}

inline bool copy_ok(cudaError_t e) { return e == cudaSuccess; }

// Issues every chunk; returns the first error.  The caller synchronises.
inline ovc_status issue(const ovc_host_io* io, float softmax_scale, uint32_t prep_flags, float budget,
                        const int32_t* sizes, int32_t nchunks, uint8_t* ws, const HostLayout& L, Streams& X) {
  const int64_t B = io->B, S = io->S, H = io->H;
  const size_t elem = 2;
  const size_t row_in = static_cast<size_t>(H) * 128u * elem, row_out = static_cast<size_t>(H) * 128u * 2u;
  const void* src[3] = {io->q, io->k, io->v};
  bool in_used[2] = {false, false}, out_used[2] = {false, false};
  int64_t h0 = 0;
  for (int32_t c = 0; c < nchunks; ++c) {
    const int64_t hc = sizes[c];
    const int st = c & 1;
    const size_t w_in = static_cast<size_t>(hc) * 128u * elem, w_out = static_cast<size_t>(hc) * 128u * 2u;
    const size_t height = static_cast<size_t>(B) * static_cast<size_t>(S);
    // Copy in: set st's staging buffers are free once chunk c-2's preparation has read them.
    if (in_used[st] && cudaStreamWaitEvent(X.in, X.in_free[st], 0) != cudaSuccess) return OVC_ERR_CUDA;
    for (int i = 0; i < 3; ++i)
      if (!copy_ok(cudaMemcpy2DAsync(ws + L.in[st][i], w_in, static_cast<const uint8_t*>(src[i]) + h0 * 128 * elem,
                                     row_in, w_in, height, cudaMemcpyHostToDevice, X.in)))
        return OVC_ERR_CUDA;
    if (cudaEventRecord(X.ready[st], X.in) != cudaSuccess) return OVC_ERR_CUDA;
    // Compute on stream st.
    cudaStream_t comp = X.comp[st];
    if (cudaStreamWaitEvent(comp, X.ready[st], 0) != cudaSuccess) return OVC_ERR_CUDA;
    const ovc_tensor tq = chunk_tensor(ws + L.in[st][0], io->dtype, B, S, hc);
    const ovc_tensor tk = chunk_tensor(ws + L.in[st][1], io->dtype, B, S, hc);
    const ovc_tensor tv = chunk_tensor(ws + L.in[st][2], io->dtype, B, S, hc);
    ovc_prepared prep{};
    ovc_status s = ovc_prepare_ex(&tq, &tk, &tv, prep_flags, ws + L.prep[st], L.prep_bytes, &prep, comp);
    if (s != OVC_OK) return s;
    ovc_repair rep{};
    if (budget > 0.0f) {
      s = ovc_prepare_v_repair(&tv, &prep, budget, ws + L.rep[st], L.rep_bytes, &rep, comp);
      if (s != OVC_OK) return s;
    }
    if (cudaEventRecord(X.in_free[st], comp) != cudaSuccess) return OVC_ERR_CUDA;
    in_used[st] = true;
    // The staged output of set st is free once chunk c-2's copy out is done.
    if (out_used[st] && cudaStreamWaitEvent(comp, X.out_free[st], 0) != cudaSuccess) return OVC_ERR_CUDA;
    ovc_output o{};
    o.ptr = ws + L.out[st];
    o.stride_b = S * hc * 128;
    o.stride_s = hc * 128;
    o.stride_h = 128;
    s = ovc_attention_ex(&prep, budget > 0.0f ? &rep : nullptr, softmax_scale, &o, 0u, 1, nullptr, 0, comp);
    if (s != OVC_OK) return s;
    if (cudaEventRecord(X.done[st], comp) != cudaSuccess) return OVC_ERR_CUDA;
    // Copy out.
    if (cudaStreamWaitEvent(X.out, X.done[st], 0) != cudaSuccess) return OVC_ERR_CUDA;
    if (!copy_ok(cudaMemcpy2DAsync(static_cast<uint8_t*>(io->o) + h0 * 128 * 2, row_out, ws + L.out[st], w_out,
                                   w_out, height, cudaMemcpyDeviceToHost, X.out)))
      return OVC_ERR_CUDA;
    if (cudaEventRecord(X.out_free[st], X.out) != cudaSuccess) return OVC_ERR_CUDA;
    out_used[st] = true;
    h0 += hc;
  }
  return OVC_OK;
}

}  // namespace host_stream
}  // namespace ovc

extern "C" {

int32_t ovc_host_chunk_plan(int64_t H, int64_t tiles_per_head, int32_t sms, int32_t* sizes, int32_t max_chunks) {
  if (H < 1 || max_chunks < 1 || sizes == nullptr) return -1;
  int32_t n = 0;
  auto put = [&](int64_t h) {
    if (n >= max_chunks) return false;
    sizes[n++] = static_cast<int32_t>(h);
    return true;
  };
  if (H < 12) {   // equal chunks of ceil(H/4) heads
    const int64_t q = (H + 3) / 4;
    for (int64_t h0 = 0; h0 < H; h0 += q)
      if (!put(h0 + q <= H ? q : H - h0)) return -1;
    return n;
  }
  // e: the ramp unit, H/56 rounded half to even, at least 1.
  const int64_t e = std::max<int64_t>(1, static_cast<int64_t>(std::nearbyint(static_cast<double>(H) / 56.0)));
  const int64_t mid = H - 6 * e;
  int64_t h = (H + 3) / 4;
  if (tiles_per_head > 0 && sms > 0) {
    // at most 10 e heads: the 2e-head chunk before must hide its copy
    const int64_t hi = std::max<int64_t>(2, std::min<int64_t>(H / 4, 10 * e));
    const int64_t lo = std::max<int64_t>(1, std::min<int64_t>(H / 8, hi));
    int64_t best = -1, best_key = 0;
    for (int64_t c = lo; c <= hi; ++c) {
      const int64_t t = c * tiles_per_head;
      const int64_t waves = (t + sms - 1) / sms;
      // waste = filled slots / used slots, compared to 4 decimals; ties go to the larger c
      const int64_t key = static_cast<int64_t>(std::nearbyint(1e4 * static_cast<double>(waves * sms) /
                                                              static_cast<double>(t)));
      if (best < 0 || key <= best_key) {
        best = c;
        best_key = key;
      }
    }
    h = best;
  }
  if (mid < 1) {   // too few heads for the ramp: equal chunks of h
    for (int64_t h0 = 0; h0 < H; h0 += h)
      if (!put(h0 + h <= H ? h : H - h0)) return -1;
    return n;
  }
  if (!put(e) || !put(2 * e)) return -1;
  for (int64_t i = 0; i < mid / h; ++i)
    if (!put(h)) return -1;
  if (mid % h && !put(mid % h)) return -1;
  if (!put(2 * e) || !put(e)) return -1;
  return n;
}

size_t ovc_attention_host_workspace_bytes(int64_t B, int64_t S, int64_t max_chunk_heads, int32_t dtype,
                                          uint32_t prep_flags, float repair_budget) {
  if (dtype != OVC_BF16 && dtype != OVC_FP16) return 0;
  if ((prep_flags & OVC_PREPARE_V_SMOOTH) || !(repair_budget >= 0.0f) || repair_budget > 1.0f) return 0;
  ovc::host_stream::HostLayout L;
  if (!ovc::host_stream::layout(B, S, max_chunk_heads, prep_flags, repair_budget, &L)) return 0;
  return L.total;
}

ovc_status ovc_attention_host(const ovc_host_io* io, float softmax_scale, uint32_t prep_flags,
                              float repair_budget, const int32_t* chunk_sizes, int32_t nchunks, void* workspace,
                              size_t workspace_bytes) {
  if (!io || !io->q || !io->k || !io->v || !io->o || !chunk_sizes || nchunks < 1) return OVC_ERR_INVALID_ARG;
  if (io->dtype != OVC_BF16 && io->dtype != OVC_FP16) return OVC_ERR_UNSUPPORTED;
  if (io->B < 1 || io->S < 1 || io->H < 1) return OVC_ERR_INVALID_ARG;
  if (prep_flags & ~static_cast<uint32_t>(OVC_PREPARE_SMOOTH_K | OVC_PREPARE_SMOOTH_Q)) return OVC_ERR_INVALID_ARG;
  if (!(repair_budget >= 0.0f) || repair_budget > 1.0f) return OVC_ERR_INVALID_ARG;
  int64_t sum = 0, hmax = 0;
  for (int32_t c = 0; c < nchunks; ++c) {
    if (chunk_sizes[c] < 1) return OVC_ERR_INVALID_ARG;
    sum += chunk_sizes[c];
    hmax = std::max<int64_t>(hmax, chunk_sizes[c]);
  }
  if (sum != io->H) return OVC_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return OVC_ERR_INVALID_ARG;
  ovc::host_stream::HostLayout L;
  if (!ovc::host_stream::layout(io->B, io->S, hmax, prep_flags, repair_budget, &L))
    return OVC_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return OVC_ERR_WORKSPACE_TOO_SMALL;
  ovc::host_stream::Streams X;
  ovc_status st = X.create() ? OVC_OK : OVC_ERR_CUDA;
  if (st == OVC_OK)
    st = ovc::host_stream::issue(io, softmax_scale, prep_flags, repair_budget, chunk_sizes, nchunks,
                                 static_cast<uint8_t*>(workspace), L, X);
  // Everything issued so far must finish before the workspace and the host
  // buffers go back to the caller, error or not.
  if (!X.finish() && st == OVC_OK) st = OVC_ERR_CUDA;
  return st;
}

}  // extern "C"
