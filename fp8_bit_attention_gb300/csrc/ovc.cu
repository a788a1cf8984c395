// ovc.cu -- libovc: the C ABI of ExpCast FP8 attention (see include/ovc.h).
//
// One translation unit: the kernels (prepare.cuh, attention.cuh, repair.cuh)
// and the host entry points that validate arguments, carve caller workspace,
// build TMA tensor maps and launch on the caller's stream.  Nothing here
// allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "ovc.h"
#include "attention.cuh"
#include "group.cuh"
#include "prepare.cuh"
#include "repair.cuh"

namespace ovc {

// Device-side status word: kernels OR in kStatusTimeout when a bounded wait
// expires.  Read and cleared by ovc_get_device_status().
__device__ unsigned int g_status;

namespace {

// The instantiations of the attention kernel, by variant bits: 0-7, 8
// (V-Smooth), 16-23 (Q smoothing), 32-35 and 48-51 (repair), and the
// P-byte dump of the probe call with the method, the baseline variants, Q
// smoothing and repair (64-67, 80, 96).
using AttnKernelFn = decltype(&attention_kernel<0>);
constexpr int kAttnVariantIds[] = {0,  1,  2,  3,  4,  5,  6,  7,  8,  16, 17, 18, 19, 20, 21, 22, 23,
                                   32, 33, 34, 35, 48, 49, 50, 51, 64, 65, 66, 67, 80, 96};

AttnKernelFn attention_kernel_for(int variant) {
  switch (variant) {
#define OVC_K(n) \
  case n:        \
    return attention_kernel<n>;
    OVC_K(0) OVC_K(1) OVC_K(2) OVC_K(3) OVC_K(4) OVC_K(5) OVC_K(6) OVC_K(7) OVC_K(8)
    OVC_K(16) OVC_K(17) OVC_K(18) OVC_K(19) OVC_K(20) OVC_K(21) OVC_K(22) OVC_K(23)
    OVC_K(32) OVC_K(33) OVC_K(34) OVC_K(35) OVC_K(48) OVC_K(49) OVC_K(50) OVC_K(51)
    OVC_K(64) OVC_K(65) OVC_K(66) OVC_K(67) OVC_K(80) OVC_K(96)
#undef OVC_K
    default:
      return nullptr;
  }
}

// Dynamic shared memory of each variant's launch.
size_t attn_smem_bytes(int variant) {
  variant &= ~kVarDump;
  if (variant == kVarVSmooth) return kAttnSmemBytesVSmooth;
  if (variant & kVarQBias) return kAttnSmemBytesQBias;
  if (variant & kVarRepair) return kAttnSmemBytesRepair;
  return kAttnSmemBytes;
}

constexpr int kMaxDevices = 64;
constexpr uint32_t kPrepareFlags = OVC_PREPARE_SMOOTH_K | OVC_PREPARE_V_SMOOTH | OVC_PREPARE_SMOOTH_Q;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;   // 4 s per wait

struct DeviceState {
  bool init = false;
  bool supported = false;
  int sms = 0;
  unsigned int* status = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

ovc_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OVC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return OVC_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.sms = sms;
    if (d.supported) {
      for (const int v : kAttnVariantIds)
        if (cudaFuncSetAttribute(attention_kernel_for(v), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(attn_smem_bytes(v))) != cudaSuccess)
          return OVC_ERR_CUDA;
      if (cudaFuncSetAttribute(kmeans_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kmeans_partial_smem())) != cudaSuccess)
        return OVC_ERR_CUDA;
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return OVC_ERR_CUDA;
      d.status = static_cast<unsigned int*>(p);
    }
    d.init = true;
  }
  *out = &d;
  return d.supported ? OVC_OK : OVC_ERR_UNSUPPORTED;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D byte tensor [rows][inner] (row pitch `pitch` bytes), 128x128 boxes,
// 128-byte swizzle (the layout tcgen05 reads as K-major SW128).
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// V-Smooth means [rows][pitch] BF16 (rows = B*H*128 channels, pitch = nbk
// blocks): 16 x 128 boxes with the 32-byte swizzle; the extent stops at nb
// blocks so that the boxes of the last chunk read zeros past it.
bool make_mean_map(CUtensorMap* m, const void* base, uint64_t nb, uint64_t rows, uint64_t pitch_elems) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {nb, rows};
  cuuint64_t strides[1] = {pitch_elems * 2};
  cuuint32_t box[2] = {16, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q smoothing's key bias rows [rows][16] BF16 (32 bytes a key): 16 x 128
// boxes with the 32-byte swizzle, the B operand layout of the bias MMA.
bool make_bias_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {16, rows};
  cuuint64_t strides[1] = {32};
  cuuint32_t box[2] = {16, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_ok(int64_t B, int64_t S, int64_t H) {
  if (B < 1 || S < 1 || H < 1) return false;
  const int64_t nb = (S + 127) / 128;
  const int64_t BH = B * H;
  if (BH > 65535 || nb > 65535) return false;               // grid limits
  if (BH * nb * 128 > (int64_t{1} << 31) - 1) return false;  // 32-bit TMA row coordinates
  return true;
}

struct PrepLayout {
  size_t q, k, vt, sq, sk, sv, vamax, energy, kpart, kmean, vmu, vmean, qpart, qmean, kbias, total;
};

PrepLayout prep_layout(int64_t B, int64_t S, int64_t H, uint32_t flags = 0) {
  const int64_t nb = (S + 127) / 128, S_pad = nb * 128, BH = B * H;
  PrepLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.q = take(static_cast<size_t>(BH) * S_pad * 128);
  L.k = take(static_cast<size_t>(BH) * S_pad * 128);
  L.vt = take(static_cast<size_t>(BH) * S_pad * 128);
  L.sq = take(static_cast<size_t>(BH) * nb * 4);
  L.sk = take(static_cast<size_t>(BH) * nb * 4);
  L.sv = take(static_cast<size_t>(BH) * 4);
  L.vamax = take(static_cast<size_t>(BH) * 4);
  L.energy = take(static_cast<size_t>(BH) * S * 4);
  if (flags & OVC_PREPARE_SMOOTH_K) {
    L.kpart = take(static_cast<size_t>(BH) * nb * 128 * 4);
    L.kmean = take(static_cast<size_t>(BH) * 128 * 4);
  }
  if (flags & OVC_PREPARE_V_SMOOTH) {
    L.vmu = take(static_cast<size_t>(BH) * nb * 128 * 4);
    L.vmean = take(static_cast<size_t>(BH) * 128 * ((nb + 15) / 16 * 16) * 2);
  }
  if (flags & OVC_PREPARE_SMOOTH_Q) {
    L.qpart = take(static_cast<size_t>(BH) * nb * 128 * 4);
    L.qmean = take(static_cast<size_t>(BH) * 128 * 4);
    L.kbias = take(static_cast<size_t>(BH) * S_pad * 32);
  }
  L.total = off;
  return L;
}

int64_t repair_n(int64_t S, float budget) {
  const double n = std::ceil(static_cast<double>(budget) * static_cast<double>(S));
  int64_t k = static_cast<int64_t>(n);
  if (k < 1) k = 1;
  if (k > S) k = S;
  return k;
}

struct GroupLayout {
  size_t cent, labels, part, cnt, off, total;
};

GroupLayout group_layout(int64_t B, int64_t S, int64_t H, int64_t C) {
  const int64_t nb = (S + 127) / 128, BH = B * H;
  GroupLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.cent = take(static_cast<size_t>(BH) * C * 128 * 4);
  L.labels = take(static_cast<size_t>(BH) * S * 4);
  L.part = take(static_cast<size_t>(BH) * nb * C * 128 * 4);
  L.cnt = take(static_cast<size_t>(BH) * nb * C * 4);
  L.off = take(static_cast<size_t>(BH) * nb * C * 4);
  L.total = off;
  return L;
}

struct RepLayout {
  size_t idx, k_sel, dvt, sk_sel, sr, kb_sel, hist, cnt, ramax, total;
};

int64_t repair_chunks(int64_t S) { return (S + kRepairChunk - 1) / kRepairChunk; }

RepLayout rep_layout(int64_t B, int64_t S, int64_t H, int64_t n) {
  const int64_t n_pad = (n + 127) / 128 * 128, BH = B * H;
  RepLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.idx = take(static_cast<size_t>(BH) * n * 4);
  L.k_sel = take(static_cast<size_t>(BH) * n_pad * 128);
  L.dvt = take(static_cast<size_t>(BH) * n_pad * 128);
  L.sk_sel = take(static_cast<size_t>(BH) * n_pad * 4);
  L.sr = take(static_cast<size_t>(BH) * 4);
  L.kb_sel = take(static_cast<size_t>(BH) * n_pad * 32);   // used with Q smoothing only
  // selection scratch: digit histograms, per-chunk counts, residual amax
  L.hist = take(static_cast<size_t>(BH) * 4 * 256 * 4);
  L.cnt = take(static_cast<size_t>(BH) * repair_chunks(S) * 2 * 4);
  L.ramax = take(static_cast<size_t>(BH) * 4);
  L.total = off;
  return L;
}

bool tensor_ok(const ovc_tensor* t) {
  if (!t || !t->ptr) return false;
  if (t->dtype != OVC_BF16 && t->dtype != OVC_FP16) return false;
  if (!aligned16(t->ptr)) return false;
  if (t->stride_b % 8 || t->stride_s % 8 || t->stride_h % 8) return false;
  if (t->stride_b < 0 || t->stride_s < 0 || t->stride_h < 0) return false;
  return dims_ok(t->B, t->S, t->H);
}

bool prepared_ok(const ovc_prepared* p) {
  if (!p || !p->q || !p->k || !p->vt || !p->sq || !p->sk || !p->sv || !p->vamax || !p->energy) return false;
  if (!dims_ok(p->B, p->S, p->H)) return false;
  return p->nb == (p->S + 127) / 128 && p->S_pad == p->nb * 128;
}

bool output_ok(const ovc_output* o) {
  if (!o || !o->ptr || !aligned16(o->ptr)) return false;
  if (o->stride_b % 8 || o->stride_s % 8 || o->stride_h % 8) return false;
  return o->stride_b >= 0 && o->stride_s >= 0 && o->stride_h >= 0;
}

ovc_status launch_status() { return cudaGetLastError() == cudaSuccess ? OVC_OK : OVC_ERR_CUDA; }

// Split key ranges (short sequences, opt-in): each tile's keys are cut into
// n ranges, each its own online softmax, and merge_kernel combines them.  A
// different computation from the unsplit method (each range has its own
// reference), so it runs only when the caller asks for it.
constexpr int kMaxSplit = 16;

struct SplitLayout {
  size_t o, ml, total;
};

SplitLayout split_layout(int64_t units) {
  SplitLayout L{};
  L.o = 0;
  L.ml = align_up(static_cast<size_t>(units) * 256 * 128 * 2, 256);
  L.total = L.ml + align_up(static_cast<size_t>(units) * 256 * sizeof(float2), 256);
  return L;
}

bool persistent_schedule(const ovc_prepared* p, const ovc_probe* probe) {
  const int force = probe ? probe->force_persistent : 0;
  return force > 0 || (force == 0 && p->S >= 32768);
}

int64_t ntiles_of(const ovc_prepared* p) { return p->B * p->H * ((p->nb + 1) / 2); }

ovc_status run_attention(const ovc_prepared* p, const ovc_repair* r, float softmax_scale,
                         const ovc_output* o, const ovc_probe* probe, uint32_t flags, int32_t nsplit,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!prepared_ok(p) || !output_ok(o)) return OVC_ERR_INVALID_ARG;
  if (flags & ~(OVC_ATTN_EXP_THEN_CAST | OVC_ATTN_NATURAL_ORDER)) return OVC_ERR_INVALID_ARG;
  if (nsplit < 0 || nsplit > kMaxSplit || nsplit > p->nb || (nsplit > 1 && r)) return OVC_ERR_INVALID_ARG;
  if (nsplit > 1 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))) return OVC_ERR_INVALID_ARG;
  // V-Smooth runs with the method's own kernel only: no repair, no split, no variant.
  const bool vsmooth = p->vmean != nullptr;
  if (vsmooth && (r || nsplit > 1 || flags != 0 || p->kbias)) return OVC_ERR_INVALID_ARG;
  const bool qbias = p->kbias != nullptr;
  if (r) {
    if (!r->idx || !r->k_sel || !r->dvt || !r->sk_sel || !r->sr) return OVC_ERR_INVALID_ARG;
    if (qbias != (r->kb_sel != nullptr)) return OVC_ERR_INVALID_ARG;   // made from this preparation
    if (r->B != p->B || r->S != p->S || r->H != p->H) return OVC_ERR_INVALID_ARG;
    if (r->n < 1 || r->n > p->S || r->n_pad != (r->n + 127) / 128 * 128) return OVC_ERR_INVALID_ARG;
  }
  if (probe && probe->dump_codes && !probe->dump_m8) return OVC_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  ovc_status st = device_state(&dev);
  if (st != OVC_OK) return st;

  const int64_t BH = p->B * p->H;
  CUtensorMap mq, mk, mv, mks, mdv;
  if (!make_map(&mq, p->q, 128, BH * p->S_pad, 128) || !make_map(&mk, p->k, 128, BH * p->S_pad, 128) ||
      !make_map(&mv, p->vt, p->S_pad, BH * 128, p->S_pad))
    return OVC_ERR_CUDA;
  if (r) {
    if (!make_map(&mks, r->k_sel, 128, BH * r->n_pad, 128) || !make_map(&mdv, r->dvt, r->n_pad, BH * 128, r->n_pad))
      return OVC_ERR_CUDA;
  } else {
    mks = mk;
    mdv = mv;
  }
  CUtensorMap mvm = mk;
  if (vsmooth && !make_mean_map(&mvm, p->vmean, p->nb, BH * 128, (p->nb + 15) / 16 * 16)) return OVC_ERR_CUDA;
  CUtensorMap mkb = mk, mkbs = mk;
  if (qbias) {
    if (!make_bias_map(&mkb, p->kbias, BH * p->S_pad)) return OVC_ERR_CUDA;
    mkbs = mkb;
    if (r && !make_bias_map(&mkbs, r->kb_sel, BH * r->n_pad)) return OVC_ERR_CUDA;
  }

  AttnParams P{};
  P.rowsum_gate = 1;
  P.B = static_cast<int32_t>(p->B);
  P.S = static_cast<int32_t>(p->S);
  P.H = static_cast<int32_t>(p->H);
  P.nb = static_cast<int32_t>(p->nb);
  P.S_pad = static_cast<int32_t>(p->S_pad);
  P.npairs = (P.nb + 1) / 2;
  const int64_t ntiles = BH * P.npairs;   // a tile is a pair of 128-row query blocks
  P.ntiles = static_cast<int32_t>(ntiles);
  const bool persistent = persistent_schedule(p, probe);
  const int64_t ns = nsplit > 1 ? nsplit : 1;   // 0 and 1: no split
  const int64_t nunits = ntiles * ns;
  if (nunits > 0x7FFFFFFF) return OVC_ERR_INVALID_ARG;
  P.nsplit = static_cast<int32_t>(ns);
  P.nunits = static_cast<int32_t>(nunits);
  if (ns > 1) {
    const SplitLayout SL = split_layout(nunits);
    if (workspace_bytes < SL.total) return OVC_ERR_WORKSPACE_TOO_SMALL;
    P.part_o = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + SL.o);
    P.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + SL.ml);
  }
  P.sq = p->sq;
  P.sk = p->sk;
  P.sv = p->sv;
  P.o = static_cast<uint16_t*>(o->ptr);
  P.os[0] = o->stride_b;
  P.os[1] = o->stride_s;
  P.os[2] = o->stride_h;
  const double sm = softmax_scale > 0.0f ? static_cast<double>(softmax_scale) : 1.0 / std::sqrt(128.0);
  P.c8 = static_cast<float>(8.0 * 1.4426950408889634074 * sm);
  if (r) {
    P.n_rep = static_cast<int32_t>(r->n);
    P.n_rep_pad = static_cast<int32_t>(r->n_pad);
    P.rep_blocks = static_cast<int32_t>(r->n_pad / 128);
    P.sk_sel = r->sk_sel;
    P.sr = r->sr;
  }
  P.dump_bh = -1;
  P.timeout_ns = kDefaultTimeoutNs;
  if (probe) {
    P.dump_bh = probe->dump_codes ? probe->dump_bh : -1;
    P.dump_qb = probe->dump_qblock;
    P.dump_kb = probe->dump_kblock;
    P.dump_codes = probe->dump_codes;
    P.dump_m8 = probe->dump_m8;
    if (probe->wait_timeout_ns > 0) P.timeout_ns = probe->wait_timeout_ns;
    P.skip_mma = probe->skip_mma;
    P.trace = reinterpret_cast<long long*>(probe->trace);
  }
  P.status = dev->status;

  // The packed long-sequence path (S >= 32768) is persistent: one CTA per SM
  // looping over tiles.  Shorter sequences launch one CTA per unit (a tile,
  // or one key range of a tile).
  const int64_t grid = persistent ? (nunits < dev->sms ? nunits : dev->sms) : nunits;
  static_assert(OVC_ATTN_EXP_THEN_CAST == kVarExpThenCast && OVC_ATTN_NATURAL_ORDER == kVarNaturalOrder,
                "flag bits select the kernel variant");
  const int variant = (vsmooth ? kVarVSmooth
                                 : static_cast<int>(flags | (ns > 1 ? kVarSplit : 0) | (qbias ? kVarQBias : 0) |
                                                    (r ? kVarRepair : 0))) |
                      (P.dump_codes != nullptr ? kVarDump : 0);
  const AttnKernelFn kernel = attention_kernel_for(variant);
  if (kernel == nullptr) return OVC_ERR_INVALID_ARG;   // a P-byte dump with a variant that has none
  const size_t smem = attn_smem_bytes(variant);
  kernel<<<static_cast<unsigned>(grid), kAttnThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      mq, mk, mv, mks, mdv, mvm, mkb, mkbs, P);
  if (ns > 1) {
    const int64_t rows = BH * p->S;
    merge_kernel<<<static_cast<unsigned>((rows + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock),
                   32 * kMergeRowsPerBlock, 0, static_cast<cudaStream_t>(stream)>>>(P);
  }
  return launch_status();
}

}  // namespace
}  // namespace ovc

using namespace ovc;

extern "C" {

size_t ovc_prepare_workspace_bytes(int64_t B, int64_t S, int64_t H, int64_t D) {
  return ovc_prepare_workspace_bytes_ex(B, S, H, D, 0);
}

size_t ovc_prepare_workspace_bytes_ex(int64_t B, int64_t S, int64_t H, int64_t D, uint32_t flags) {
  if (D != 128 || !dims_ok(B, S, H) || (flags & ~kPrepareFlags)) return 0;
  if ((flags & OVC_PREPARE_SMOOTH_Q) && (flags & OVC_PREPARE_V_SMOOTH)) return 0;
  return prep_layout(B, S, H, flags).total;
}

ovc_status ovc_prepare(const ovc_tensor* q, const ovc_tensor* k, const ovc_tensor* v, void* workspace,
                       size_t workspace_bytes, ovc_prepared* out, void* stream) {
  return ovc_prepare_ex(q, k, v, 0, workspace, workspace_bytes, out, stream);
}

ovc_status ovc_prepare_ex(const ovc_tensor* q, const ovc_tensor* k, const ovc_tensor* v, uint32_t flags,
                          void* workspace, size_t workspace_bytes, ovc_prepared* out, void* stream) {
  return ovc_prepare_grouped(q, k, v, nullptr, flags, workspace, workspace_bytes, out, stream);
}

ovc_status ovc_prepare_grouped(const ovc_tensor* q, const ovc_tensor* k, const ovc_tensor* v, const int32_t* perm,
                               uint32_t flags, void* workspace, size_t workspace_bytes, ovc_prepared* out,
                               void* stream) {
  if (flags & ~kPrepareFlags) return OVC_ERR_INVALID_ARG;
  if ((flags & OVC_PREPARE_SMOOTH_Q) && (flags & OVC_PREPARE_V_SMOOTH)) return OVC_ERR_INVALID_ARG;
  if (perm && (reinterpret_cast<uintptr_t>(perm) & 3u)) return OVC_ERR_INVALID_ARG;
  if (!q || !k || !v || !out) return OVC_ERR_INVALID_ARG;
  if (q->D != 128 || k->D != 128 || v->D != 128) return OVC_ERR_UNSUPPORTED;
  if ((q->dtype != OVC_BF16 && q->dtype != OVC_FP16) || k->dtype != q->dtype || v->dtype != q->dtype)
    return OVC_ERR_UNSUPPORTED;
  if (!tensor_ok(q) || !tensor_ok(k) || !tensor_ok(v)) return OVC_ERR_INVALID_ARG;
  if (k->B != q->B || k->S != q->S || k->H != q->H || v->B != q->B || v->S != q->S || v->H != q->H)
    return OVC_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return OVC_ERR_INVALID_ARG;
  const PrepLayout L = prep_layout(q->B, q->S, q->H, flags);
  if (workspace_bytes < L.total) return OVC_ERR_WORKSPACE_TOO_SMALL;
  DeviceState* dev = nullptr;
  ovc_status st = device_state(&dev);
  if (st != OVC_OK) return st;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ovc_prepared p{};
  p.B = q->B;
  p.S = q->S;
  p.H = q->H;
  p.nb = (q->S + 127) / 128;
  p.S_pad = p.nb * 128;
  p.q = ws + L.q;
  p.k = ws + L.k;
  p.vt = ws + L.vt;
  p.sq = reinterpret_cast<float*>(ws + L.sq);
  p.sk = reinterpret_cast<float*>(ws + L.sk);
  p.sv = reinterpret_cast<float*>(ws + L.sv);
  p.vamax = reinterpret_cast<uint32_t*>(ws + L.vamax);
  p.energy = reinterpret_cast<float*>(ws + L.energy);
  p.vmean = (flags & OVC_PREPARE_V_SMOOTH) ? reinterpret_cast<uint16_t*>(ws + L.vmean) : nullptr;
  p.perm = perm;
  p.kbias = (flags & OVC_PREPARE_SMOOTH_Q) ? reinterpret_cast<uint16_t*>(ws + L.kbias) : nullptr;

  PrepParams P{};
  P.q = static_cast<const uint16_t*>(q->ptr);
  P.k = static_cast<const uint16_t*>(k->ptr);
  P.v = static_cast<const uint16_t*>(v->ptr);
  const ovc_tensor* ts[3] = {q, k, v};
  int64_t* ss[3] = {P.qs, P.ks, P.vs};
  for (int i = 0; i < 3; ++i) {
    ss[i][0] = ts[i]->stride_b;
    ss[i][1] = ts[i]->stride_s;
    ss[i][2] = ts[i]->stride_h;
  }
  P.B = static_cast<int32_t>(p.B);
  P.S = static_cast<int32_t>(p.S);
  P.H = static_cast<int32_t>(p.H);
  P.nb = static_cast<int32_t>(p.nb);
  P.S_pad = static_cast<int32_t>(p.S_pad);
  P.fp16 = q->dtype == OVC_FP16;
  P.qc = p.q;
  P.kc = p.k;
  P.vt = p.vt;
  P.sq = p.sq;
  P.sk = p.sk;
  P.sv = p.sv;
  P.vamax = p.vamax;
  P.energy = p.energy;
  P.perm = perm;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(p.vamax, 0, static_cast<size_t>(p.B * p.H) * 4, s) != cudaSuccess) return OVC_ERR_CUDA;
  if (flags & OVC_PREPARE_SMOOTH_K) {
    P.kpart = reinterpret_cast<float*>(ws + L.kpart);
    P.kmean = reinterpret_cast<float*>(ws + L.kmean);
    if (perm)
      k_mean_partial_kernel<true><<<dim3(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.nb)), 128, 0, s>>>(P);
    else
      k_mean_partial_kernel<false><<<dim3(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.nb)), 128, 0, s>>>(P);
    k_mean_final_kernel<<<static_cast<unsigned>(p.B * p.H), 128, 0, s>>>(P);
  }
  if (flags & OVC_PREPARE_SMOOTH_Q) {
    P.qpart = reinterpret_cast<float*>(ws + L.qpart);
    P.qmean = reinterpret_cast<float*>(ws + L.qmean);
    P.kbias = p.kbias;
    k_mean_partial_kernel<false, true><<<dim3(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.nb)), 128, 0, s>>>(P);
    k_mean_final_kernel<true><<<static_cast<unsigned>(p.B * p.H), 128, 0, s>>>(P);
  }
  if (flags & OVC_PREPARE_V_SMOOTH) {
    P.vmu = reinterpret_cast<float*>(ws + L.vmu);
    P.vmean = p.vmean;
    P.nbk = static_cast<int32_t>((p.nb + 15) / 16 * 16);
    if (perm)
      vsmooth_mean_kernel<true><<<dim3(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.nb)), 128, 0, s>>>(P);
    else
      vsmooth_mean_kernel<false><<<dim3(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.nb)), 128, 0, s>>>(P);
  }
  // z = 2 (the amax of V) only without V-Smooth, whose mean pass folds it in
  const dim3 g1(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.nb), (flags & OVC_PREPARE_V_SMOOTH) ? 2 : 3);
  const int qk_opt = ((flags & OVC_PREPARE_SMOOTH_K) ? kPrepSmoothK : 0) | (perm ? kPrepPerm : 0) |
                     ((flags & OVC_PREPARE_SMOOTH_Q) ? kPrepSmoothQ : 0);
  static const decltype(&prepare_qk_kernel<0>) kQK[8] = {
      prepare_qk_kernel<0>, prepare_qk_kernel<1>, prepare_qk_kernel<2>, prepare_qk_kernel<3>,
      prepare_qk_kernel<4>, prepare_qk_kernel<5>, prepare_qk_kernel<6>, prepare_qk_kernel<7>};
  static_assert(kPrepSmoothK == 1 && kPrepPerm == 2 && kPrepSmoothQ == 4, "option bits index the table");
  kQK[qk_opt]<<<g1, 256, 0, s>>>(P);
  const dim3 g2(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.nb), 1);
  const bool vsm = (flags & OVC_PREPARE_V_SMOOTH) != 0;
  if (vsm && perm)
    prepare_v_kernel<true, true><<<g2, 512, 0, s>>>(P);
  else if (vsm)
    prepare_v_kernel<true, false><<<g2, 512, 0, s>>>(P);
  else if (perm)
    prepare_v_kernel<false, true><<<g2, 512, 0, s>>>(P);
  else
    prepare_v_kernel<false, false><<<g2, 512, 0, s>>>(P);
  st = launch_status();
  if (st == OVC_OK) *out = p;
  return st;
}

ovc_status ovc_attention(const ovc_prepared* p, float softmax_scale, const ovc_output* o, void* stream) {
  return run_attention(p, nullptr, softmax_scale, o, nullptr, 0, 1, nullptr, 0, stream);
}

ovc_status ovc_attention_ex(const ovc_prepared* p, const ovc_repair* r, float softmax_scale, const ovc_output* o,
                            uint32_t flags, int32_t nsplit, void* workspace, size_t workspace_bytes,
                            void* stream) {
  return run_attention(p, r, softmax_scale, o, nullptr, flags, nsplit, workspace, workspace_bytes, stream);
}

size_t ovc_attention_workspace_bytes(const ovc_prepared* p, int32_t nsplit) {
  if (!prepared_ok(p) || nsplit < 0 || nsplit > kMaxSplit || nsplit > p->nb) return 0;
  return nsplit > 1 ? split_layout(ntiles_of(p) * nsplit).total : 0;
}

size_t ovc_repair_workspace_bytes(int64_t B, int64_t S, int64_t H, float budget) {
  if (!dims_ok(B, S, H) || !(budget > 0.0f) || budget > 1.0f) return 0;
  return rep_layout(B, S, H, repair_n(S, budget)).total;
}

ovc_status ovc_prepare_v_repair(const ovc_tensor* v, const ovc_prepared* p, float budget, void* workspace,
                                size_t workspace_bytes, ovc_repair* out, void* stream) {
  if (!v || !p || !out) return OVC_ERR_INVALID_ARG;
  if (v->D != 128) return OVC_ERR_UNSUPPORTED;
  if (v->dtype != OVC_BF16 && v->dtype != OVC_FP16) return OVC_ERR_UNSUPPORTED;
  if (!tensor_ok(v) || !prepared_ok(p)) return OVC_ERR_INVALID_ARG;
  if (p->vmean) return OVC_ERR_INVALID_ARG;   // V-Smooth keeps no residual energies
  if (p->perm) return OVC_ERR_INVALID_ARG;    // energies are in the grouped token order
  if (v->B != p->B || v->S != p->S || v->H != p->H) return OVC_ERR_INVALID_ARG;
  if (!(budget > 0.0f) || budget > 1.0f) return OVC_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return OVC_ERR_INVALID_ARG;
  const int64_t n = repair_n(p->S, budget);
  const RepLayout L = rep_layout(p->B, p->S, p->H, n);
  if (workspace_bytes < L.total) return OVC_ERR_WORKSPACE_TOO_SMALL;
  DeviceState* dev = nullptr;
  ovc_status st = device_state(&dev);
  if (st != OVC_OK) return st;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ovc_repair r{};
  r.B = p->B;
  r.S = p->S;
  r.H = p->H;
  r.n = n;
  r.n_pad = (n + 127) / 128 * 128;
  r.idx = reinterpret_cast<int32_t*>(ws + L.idx);
  r.k_sel = ws + L.k_sel;
  r.dvt = ws + L.dvt;
  r.sk_sel = reinterpret_cast<float*>(ws + L.sk_sel);
  r.sr = reinterpret_cast<float*>(ws + L.sr);
  r.kb_sel = p->kbias ? reinterpret_cast<uint16_t*>(ws + L.kb_sel) : nullptr;

  RepairParams P{};
  P.v = static_cast<const uint16_t*>(v->ptr);
  P.vs[0] = v->stride_b;
  P.vs[1] = v->stride_s;
  P.vs[2] = v->stride_h;
  P.B = static_cast<int32_t>(p->B);
  P.S = static_cast<int32_t>(p->S);
  P.H = static_cast<int32_t>(p->H);
  P.nb = static_cast<int32_t>(p->nb);
  P.S_pad = static_cast<int32_t>(p->S_pad);
  P.fp16 = v->dtype == OVC_FP16;
  P.kc = p->k;
  P.sk = p->sk;
  P.energy = p->energy;
  P.vamax = p->vamax;
  P.n = static_cast<int32_t>(r.n);
  P.n_pad = static_cast<int32_t>(r.n_pad);
  P.idx = r.idx;
  P.k_sel = r.k_sel;
  P.dvt = r.dvt;
  P.sk_sel = r.sk_sel;
  P.sr = r.sr;
  P.kbias = p->kbias;
  P.kb_sel = r.kb_sel;
  P.hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  P.cnt = reinterpret_cast<uint32_t*>(ws + L.cnt);
  P.ramax = reinterpret_cast<uint32_t*>(ws + L.ramax);
  P.nchunk = static_cast<int32_t>(repair_chunks(p->S));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the histograms and the amax accumulate: clear them (the counts are written whole)
  if (cudaMemsetAsync(ws + L.hist, 0, L.cnt - L.hist, s) != cudaSuccess ||
      cudaMemsetAsync(ws + L.ramax, 0, static_cast<size_t>(p->B * p->H) * 4, s) != cudaSuccess)
    return OVC_ERR_CUDA;
  const dim3 gsel(static_cast<unsigned>(P.nchunk), static_cast<unsigned>(p->B * p->H));
  repair_hist_kernel<0><<<gsel, kRepairThreads, 0, s>>>(P);
  repair_hist_kernel<1><<<gsel, kRepairThreads, 0, s>>>(P);
  repair_hist_kernel<2><<<gsel, kRepairThreads, 0, s>>>(P);
  repair_hist_kernel<3><<<gsel, kRepairThreads, 0, s>>>(P);
  repair_count_kernel<<<gsel, kRepairThreads, 0, s>>>(P);
  repair_scatter_kernel<<<gsel, kRepairThreads, 0, s>>>(P);
  const unsigned tok = static_cast<unsigned>((r.n + kRepairTokensPerCta - 1) / kRepairTokensPerCta);
  const unsigned pad = static_cast<unsigned>((r.n_pad + kRepairTokensPerCta - 1) / kRepairTokensPerCta);
  repair_amax_kernel<<<dim3(tok, static_cast<unsigned>(p->B * p->H)), kRepairThreads, 0, s>>>(P);
  repair_write_kernel<<<dim3(pad, static_cast<unsigned>(p->B * p->H)), kRepairThreads, 0, s>>>(P);
  st = launch_status();
  if (st == OVC_OK) *out = r;
  return st;
}

ovc_status ovc_attention_v_repair(const ovc_prepared* p, const ovc_repair* r, float softmax_scale,
                                  const ovc_output* o, void* stream) {
  if (!r) return OVC_ERR_INVALID_ARG;
  return run_attention(p, r, softmax_scale, o, nullptr, 0, 1, nullptr, 0, stream);
}

ovc_status ovc_attention_probe(const ovc_prepared* p, const ovc_repair* r, float softmax_scale,
                               const ovc_output* o, const ovc_probe* probe, void* stream) {
  return run_attention(p, r, softmax_scale, o, probe, probe ? probe->flags : 0u, 1, nullptr, 0, stream);
}

ovc_status ovc_get_device_status(void* stream) {
  DeviceState* dev = nullptr;
  ovc_status st = device_state(&dev);
  if (st != OVC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return OVC_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status, sizeof(word)) != cudaSuccess) return OVC_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return OVC_ERR_CUDA;
    return OVC_ERR_TIMEOUT;
  }
  return OVC_OK;
}

const char* ovc_status_string(ovc_status s) {
  switch (s) {
    case OVC_OK: return "ok";
    case OVC_ERR_INVALID_ARG: return "invalid argument";
    case OVC_ERR_UNSUPPORTED: return "unsupported (needs D = 128, BF16/FP16 inputs and an sm_103 GPU)";
    case OVC_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case OVC_ERR_CUDA: return "CUDA runtime error";
    case OVC_ERR_TIMEOUT: return "a device-side wait timed out";
    case OVC_ERR_SCRATCH_LIMIT: return "B*H exceeds the fixed scratch of ovc_prepare_noalloc (OVC_NOALLOC_MAX_HEADS)";
  }
  return "unknown status";
}

size_t ovc_vsmooth_group_workspace_bytes(int64_t B, int64_t S, int64_t H, int32_t clusters) {
  if (!dims_ok(B, S, H) || clusters < 1 || clusters > kMaxClusters || clusters > S) return 0;
  return group_layout(B, S, H, clusters).total;
}

ovc_status ovc_vsmooth_group(const ovc_tensor* v, int32_t clusters, int32_t iters, void* workspace,
                             size_t workspace_bytes, int32_t* perm, void* stream) {
  if (!v || !perm || (reinterpret_cast<uintptr_t>(perm) & 3u)) return OVC_ERR_INVALID_ARG;
  if (v->D != 128) return OVC_ERR_UNSUPPORTED;
  if (v->dtype != OVC_BF16 && v->dtype != OVC_FP16) return OVC_ERR_UNSUPPORTED;
  if (!tensor_ok(v)) return OVC_ERR_INVALID_ARG;
  if (clusters < 1 || clusters > kMaxClusters || clusters > v->S || iters < 1 || iters > 1000)
    return OVC_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return OVC_ERR_INVALID_ARG;
  const GroupLayout L = group_layout(v->B, v->S, v->H, clusters);
  if (workspace_bytes < L.total) return OVC_ERR_WORKSPACE_TOO_SMALL;
  DeviceState* dev = nullptr;
  ovc_status st = device_state(&dev);
  if (st != OVC_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  GroupParams G{};
  G.v = static_cast<const uint16_t*>(v->ptr);
  G.vs[0] = v->stride_b;
  G.vs[1] = v->stride_s;
  G.vs[2] = v->stride_h;
  G.B = static_cast<int32_t>(v->B);
  G.S = static_cast<int32_t>(v->S);
  G.H = static_cast<int32_t>(v->H);
  G.nb = static_cast<int32_t>((v->S + 127) / 128);
  G.C = clusters;
  G.fp16 = v->dtype == OVC_FP16;
  G.cent = reinterpret_cast<float*>(ws + L.cent);
  G.labels = reinterpret_cast<int32_t*>(ws + L.labels);
  G.part = reinterpret_cast<float*>(ws + L.part);
  G.cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
  G.off = reinterpret_cast<int32_t*>(ws + L.off);
  G.perm = perm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned BH = static_cast<unsigned>(v->B * v->H), nb = static_cast<unsigned>(G.nb);
  kmeans_init_kernel<<<dim3(static_cast<unsigned>(clusters), BH), 128, 0, s>>>(G);
  for (int it = 0; it < iters; ++it) {
    kmeans_assign_kernel<<<dim3(BH, nb), 128, 0, s>>>(G);
    if (it + 1 == iters) break;
    kmeans_partial_kernel<<<dim3(BH, nb), 128, kmeans_partial_smem(), s>>>(G);
    kmeans_update_kernel<<<dim3(static_cast<unsigned>(clusters), BH), 128, 0, s>>>(G);
  }
  group_count_kernel<<<dim3(BH, nb), 128, 0, s>>>(G);
  group_offset_kernel<<<BH, kMaxClusters, 0, s>>>(G);
  group_scatter_kernel<<<dim3(BH, nb), 128, 0, s>>>(G);
  return launch_status();
}

}  // extern "C"

#include "host_stream.cuh"

// ---------------------------------------------------------------------------
// ovc_prepare_noalloc: ovc_prepare for callers that cannot allocate.  The
// one piece of scratch the preparation needs beyond its outputs, the per-head
// running amax of V, lives in a fixed array inside the library instead of in
// caller workspace.
// ---------------------------------------------------------------------------
namespace ovc {
namespace {

// The scratch: one FP32 amax (as ordered bits) per (batch, head).  Every GPU
// that loads the library holds it until the process exits.
static __device__ __align__(256) uint32_t g_noalloc_amax[OVC_NOALLOC_MAX_HEADS];

// Device address of g_noalloc_amax on each device.  In host code the
// symbol's name is only a host-side stand-in for the array, so the address a
// kernel can use is looked up once per device, with that device current.
uint32_t* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

ovc_status noalloc_scratch(uint32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OVC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_amax) != cudaSuccess || p == nullptr) return OVC_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return OVC_OK;
}

__global__ void noalloc_copy_kernel(const uint32_t* scratch, uint32_t* dst, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) dst[i] = scratch[i];
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace ovc

extern "C" ovc_status ovc_prepare_noalloc(const ovc_tensor* q, const ovc_tensor* k, const ovc_tensor* v,
                                          const ovc_prepared* out, void* stream) {
  if (!q || !k || !v || !out) return OVC_ERR_INVALID_ARG;
  if (q->D != 128 || k->D != 128 || v->D != 128) return OVC_ERR_UNSUPPORTED;
  if ((q->dtype != OVC_BF16 && q->dtype != OVC_FP16) || k->dtype != q->dtype || v->dtype != q->dtype)
    return OVC_ERR_UNSUPPORTED;
  if (!tensor_ok(q) || !tensor_ok(k) || !tensor_ok(v)) return OVC_ERR_INVALID_ARG;
  if (k->B != q->B || k->S != q->S || k->H != q->H || v->B != q->B || v->S != q->S || v->H != q->H)
    return OVC_ERR_INVALID_ARG;
  const int64_t nb = (q->S + 127) / 128;
  if (out->B != q->B || out->S != q->S || out->H != q->H || out->nb != nb || out->S_pad != nb * 128)
    return OVC_ERR_INVALID_ARG;
  if (!out->q || !out->k || !out->vt || !out->sq || !out->sk || !out->sv || !out->vamax || !out->energy)
    return OVC_ERR_INVALID_ARG;
  // A plain preparation: no V-Smooth means, no grouping order, no Q smoothing.
  if (out->vmean || out->perm || out->kbias) return OVC_ERR_INVALID_ARG;
  if (!aligned16(out->q) || !aligned16(out->k) || !aligned16(out->vt)) return OVC_ERR_INVALID_ARG;
  if (!aligned4(out->sq) || !aligned4(out->sk) || !aligned4(out->sv) || !aligned4(out->vamax) ||
      !aligned4(out->energy))
    return OVC_ERR_INVALID_ARG;
  const int64_t BH = q->B * q->H;
  if (BH > OVC_NOALLOC_MAX_HEADS) return OVC_ERR_SCRATCH_LIMIT;
  DeviceState* dev = nullptr;
  ovc_status st = device_state(&dev);
  if (st != OVC_OK) return st;
  uint32_t* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != OVC_OK) return st;

  PrepParams P{};
  P.q = static_cast<const uint16_t*>(q->ptr);
  P.k = static_cast<const uint16_t*>(k->ptr);
  P.v = static_cast<const uint16_t*>(v->ptr);
  const ovc_tensor* ts[3] = {q, k, v};
  int64_t* ss[3] = {P.qs, P.ks, P.vs};
  for (int i = 0; i < 3; ++i) {
    ss[i][0] = ts[i]->stride_b;
    ss[i][1] = ts[i]->stride_s;
    ss[i][2] = ts[i]->stride_h;
  }
  P.B = static_cast<int32_t>(q->B);
  P.S = static_cast<int32_t>(q->S);
  P.H = static_cast<int32_t>(q->H);
  P.nb = static_cast<int32_t>(nb);
  P.S_pad = static_cast<int32_t>(nb * 128);
  P.fp16 = q->dtype == OVC_FP16;
  P.qc = out->q;
  P.kc = out->k;
  P.vt = out->vt;
  P.sq = out->sq;
  P.sk = out->sk;
  P.sv = out->sv;
  P.vamax = scratch;          // the fixed array instead of caller workspace
  P.energy = out->energy;

  // The array keeps the previous call's maxima: clear this call's entries.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n = static_cast<int>(BH);
  if (cudaMemsetAsync(scratch, 0, static_cast<size_t>(BH) * 4, s) != cudaSuccess) return OVC_ERR_CUDA;
  const dim3 g1(static_cast<unsigned>(BH), static_cast<unsigned>(nb), 3);
  prepare_qk_kernel<0><<<g1, 256, 0, s>>>(P);
  const dim3 g2(static_cast<unsigned>(BH), static_cast<unsigned>(nb), 1);
  prepare_v_kernel<false, false><<<g2, 512, 0, s>>>(P);
  noalloc_copy_kernel<<<(n + 255) / 256, 256, 0, s>>>(scratch, out->vamax, n);
  return launch_status();
}
