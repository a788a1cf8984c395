/*
 * ovc.h -- C ABI of libovc: ExpCast FP8 attention for GB300 (sm_103a).
 *
 * Non-causal multi-head forward attention, head dim 128, long sequences, with
 * Q/K/V quantised to FP8 E4M3 and the softmax probabilities written straight
 * out as E4M3 bytes by one FMA on the log2-domain score ("ExpCast").
 *
 * What each call computes follows these pages (title, section):
 *   "Open VC Attention" (catalogue entry): the API covers forward MHA with head
 *     dim 128 on FP16/BF16 inputs shaped [S,H,128] or [B,S,H,128] and returns
 *     BF16; per-block Q/K scales and per-head V scales; keys traversed from the
 *     middle of the window; a packed fast path for non-causal S >= 32768;
 *     V residual repair prepared with prepare_v_repair(budget) and applied by
 *     attention_v_repair.
 *   "Open-VC attention" (news item), "Solution: ExpCast": one FMA per score,
 *     no MUFU exponent, no FP32->FP8 conversion; "Architectural
 *     optimisations": mid-window traversal, warp-specialised pipeline, Q/K/V
 *     quantisation fused into one preparation step.
 *   VC-Attention summary, "ExpCast-FP8": an E4M3 byte read as an integer is
 *     about 8*log2(v)+56; beta = -0.35.
 *
 * Conventions for every call:
 *   - All pointers inside ovc_tensor / ovc_output / ovc_prepared / ovc_repair
 *     are DEVICE pointers of the current CUDA device.  The caller owns every
 *     buffer; the library never allocates or frees device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call is asynchronous on it; argument errors are returned synchronously
 *     and nothing is launched.
 *   - Input tensors must be 16-byte aligned with unit channel stride and
 *     element strides that are multiples of 8.
 *   - The library requires an sm_103 device (GB300); others get
 *     OVC_ERR_UNSUPPORTED.
 *   - Device-side waits are bounded: a kernel that waits too long records
 *     OVC_ERR_TIMEOUT, which ovc_get_device_status() reports.
 */
#ifndef OVC_H_
#define OVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OVC_OK = 0,
  OVC_ERR_INVALID_ARG = 1,          /* null pointer, bad shape, stride or alignment */
  OVC_ERR_UNSUPPORTED = 2,          /* D != 128, unknown dtype, device not sm_103 */
  OVC_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below the *_workspace_bytes() figure */
  OVC_ERR_CUDA = 4,                 /* a CUDA runtime call failed */
  OVC_ERR_TIMEOUT = 5,              /* a device-side wait hit its limit */
  OVC_ERR_SCRATCH_LIMIT = 6         /* ovc_prepare_noalloc: B*H above its fixed scratch */
} ovc_status;

enum { OVC_BF16 = 0, OVC_FP16 = 1 };

/* A BF16/FP16 tensor [B,S,H,D] (use B = 1 for [S,H,D]); strides in elements,
 * the channel stride is 1. */
typedef struct {
  const void* ptr;
  int32_t dtype;                    /* OVC_BF16 or OVC_FP16 */
  int64_t B, S, H, D;               /* D must be 128 */
  int64_t stride_b, stride_s, stride_h;
} ovc_tensor;

/* The BF16 output O [B,S,H,128]; strides in elements, channel stride 1. */
typedef struct {
  void* ptr;
  int64_t stride_b, stride_s, stride_h;
} ovc_output;

/* Quantised inputs written by ovc_prepare into caller workspace.  Layouts
 * (nb = ceil(S/128), S_pad = 128*nb, E4M3 bytes, rows >= S are zero):
 *   q, k  [B,H,S_pad,128]  head-major, 128-token blocks contiguous
 *   vt    [B,H,128,S_pad]  V transposed: keys contiguous ("packed transposed V")
 *   sq,sk [B,H,nb]         FP32 scale of each 128-token block, amax/448
 *   sv    [B,H]            FP32 scale of each head of V, amax/448
 *   vamax [B,H]            FP32 bits of each head's amax|V|
 *   energy[B,H,S]          FP32 residual energy ||v_t - sv*dec(code_t)||^2
 *   vmean [B,H,128,nbk]    V-Smooth only (else NULL): BF16 bits of the restored
 *                          block means M'_b = bf16(mu_b / sv), channel-major,
 *                          nbk = nb rounded up to 16 (entries >= nb unused);
 *                          vt then holds the residuals v - mu_b and energy is
 *                          not computed
 *   perm  [B,H,S]          grouping only (else NULL): the token order of k, vt
 *                          and vmean (row t is input token perm[t]); the
 *                          caller's array, which must outlive the struct's use
 *                          (q keeps its order, so O does too)
 *   kbias [B,H,S_pad,16]   Q smoothing only (else NULL): BF16 bits, key t's
 *                          row (hi, lo, hi, lo, 0 x 12) with hi + lo ~ beta_t =
 *                          mu_q . dec(k_t) (rows >= S zero) */
typedef struct {
  int64_t B, S, H, nb, S_pad;
  uint8_t* q;
  uint8_t* k;
  uint8_t* vt;
  float* sq;
  float* sk;
  float* sv;
  uint32_t* vamax;
  float* energy;
  uint16_t* vmean;
  const int32_t* perm;
  uint16_t* kbias;
} ovc_prepared;

/* V residual repair set written by ovc_prepare_v_repair (n_pad = 128*ceil(n/128)):
 *   idx    [B,H,n]         selected token indices, ascending
 *   k_sel  [B,H,n_pad,128] their quantised keys (zero padded)
 *   dvt    [B,H,128,n_pad] their quantised V residuals, transposed
 *   sk_sel [B,H,n_pad]     the key scale of each selected token's block
 *   sr     [B,H]           FP32 residual scale, amax|R_sel|/448
 *   kb_sel [B,H,n_pad,16]  Q smoothing only (else NULL): the selected keys'
 *                          bias rows (as ovc_prepared.kbias, zero padded) */
typedef struct {
  int64_t B, S, H, n, n_pad;
  int32_t* idx;
  uint8_t* k_sel;
  uint8_t* dvt;
  float* sk_sel;
  float* sr;
  uint16_t* kb_sel;
} ovc_repair;

/* Bytes of workspace ovc_prepare needs for these dimensions (0 if invalid). */
size_t ovc_prepare_workspace_bytes(int64_t B, int64_t S, int64_t H, int64_t D);

/* Quantise Q, K (one scale per 128-token block) and V (one scale per head) to
 * E4M3 and lay them out for the attention kernel; also computes the per-token
 * V residual energy used by repair.  q, k, v must have identical shapes and
 * dtypes.  `workspace` (>= ovc_prepare_workspace_bytes, 256-byte aligned)
 * backs every buffer of *out; it must stay alive while *out is used.
 * ("Open VC Attention": per-block Q/K and per-head V scales; "Open-VC
 * attention", "Architectural optimisations": fused input preparation.) */
ovc_status ovc_prepare(const ovc_tensor* q, const ovc_tensor* k, const ovc_tensor* v,
                       void* workspace, size_t workspace_bytes, ovc_prepared* out, void* stream);

/* O = softmax(Q K^T * softmax_scale) V with ExpCast probabilities, written as
 * BF16 to *o.  softmax_scale <= 0 selects 1/sqrt(128).  Non-causal only.
 * S >= 32768 runs the persistent (packed) schedule; shorter sequences run one
 * CTA per pair of 128-row Q blocks.  Both give identical results. */
ovc_status ovc_attention(const ovc_prepared* p, float softmax_scale, const ovc_output* o,
                         void* stream);

/* ovc_attention / ovc_attention_v_repair (r may be NULL) with a kernel
 * variant and, on request, split key ranges.
 *
 * Split key ranges (nsplit > 1; opt-in, never chosen by the library): each
 * pair of 128-row query blocks has its key blocks cut into nsplit contiguous
 * ranges [s nb/nsplit, (s+1) nb/nsplit), each run as its own online softmax
 * (own reference, own row sum, mid-window order within the range), and a
 * merge pass combines them: with M = max m8_s and w_s = l_s 2^((m8_s - M)/8),
 * O = sum w_s O_s / sum w_s.  Because every range takes its ExpCast bytes
 * against its own reference, this is a different computation from the
 * method's single pass: results differ from ovc_attention's (both lie within
 * the ExpCast error of exact attention).  The partial results live in caller
 * workspace (ovc_attention_workspace_bytes).
 *   nsplit     0 or 1: no split (the method; identical to ovc_attention);
 *              2..16 (<= nb): forced split, needs workspace and no repair set.
 *   workspace  device memory, 256-byte aligned, at least
 *              ovc_attention_workspace_bytes(p, nsplit) bytes; may be NULL
 *              when no split is made.  Calls that share it must not overlap.
 * Errors: OVC_ERR_INVALID_ARG (bad nsplit, repair with nsplit > 1, unaligned
 * workspace), OVC_ERR_WORKSPACE_TOO_SMALL.
 *
 * flags (OR of):
 *   OVC_ATTN_EXP_THEN_CAST  each probability byte is produced the way
 *     ExpCast avoids: v = 2^8 p from one FMA and one ex2 on the special
 *     function unit, then an FP32 -> E4M3 conversion (round to nearest even,
 *     saturating).  "Open-VC attention", "Problem": one exponent per score
 *     holds standard FP8 kernels to about half the FP8 peak on B200.
 *   OVC_ATTN_NATURAL_ORDER  key blocks in order 0..nb-1 instead of cyclically
 *     from the middle ("Architectural optimisations": mid-window traversal).
 * Both together (OVC_ATTN_BASELINE) make the standard FP8 kernel that ExpCast
 * and the mid-window order improve on, in this library's own pipeline: the
 * same quantisation, lazy rescale, row sum (decoded bytes) and warp
 * specialisation, so that a timing difference isolates the two techniques.
 * (The pages' baselines.vc_attention is the VC-Attention authors' code, which
 * already uses ExpCast; that implementation is not reproduced here.)
 * flags = 0 is ovc_attention.
 * Unknown flags give OVC_ERR_INVALID_ARG. */
#define OVC_ATTN_EXP_THEN_CAST 1u
#define OVC_ATTN_NATURAL_ORDER 2u
#define OVC_ATTN_BASELINE 3u
ovc_status ovc_attention_ex(const ovc_prepared* p, const ovc_repair* r, float softmax_scale,
                            const ovc_output* o, uint32_t flags, int32_t nsplit, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Workspace bytes ovc_attention_ex needs for nsplit ranges: 0 when no split
 * is made (nsplit 0 or 1) or for invalid arguments. */
size_t ovc_attention_workspace_bytes(const ovc_prepared* p, int32_t nsplit);

/* Bytes of workspace ovc_prepare_v_repair needs (0 if invalid).  budget in (0,1]. */
size_t ovc_repair_workspace_bytes(int64_t B, int64_t S, int64_t H, float budget);

/* Select, per head, the n = ceil(budget*S) V tokens with the largest residual
 * energy (ties to the lower index), quantise their residuals with one scale
 * per head and gather their keys.  `v` is the same tensor given to
 * ovc_prepare for `p`.  ("Open VC Attention": prepare_v_repair with a budget
 * such as 0.005; "MachGen opened the sources...", "What happened".) */
ovc_status ovc_prepare_v_repair(const ovc_tensor* v, const ovc_prepared* p, float budget,
                                void* workspace, size_t workspace_bytes, ovc_repair* out,
                                void* stream);

/* ovc_attention plus one more sparse P*dV term over the repair set: the
 * selected keys are scored again with the row's final reference and their
 * quantised residuals are accumulated into O; the row sum is unchanged. */
ovc_status ovc_attention_v_repair(const ovc_prepared* p, const ovc_repair* r, float softmax_scale,
                                  const ovc_output* o, void* stream);

/* Synchronise `stream`, then report and clear the device-side status word:
 * OVC_ERR_TIMEOUT if any kernel gave up on a wait since the last call. */
ovc_status ovc_get_device_status(void* stream);

/* A static English description of a status code. */
const char* ovc_status_string(ovc_status s);

/* Test hook (not part of the method): ovc_attention / ovc_attention_v_repair
 * with extra controls.  For every row of 128-row query block `dump_qblock` of
 * head `dump_bh` (= b*H + h), the P bytes written for key block `dump_kblock`
 * go to dump_codes [128,128] (device, uint8) and the reference used for them
 * (in 1/8-log2 units) to dump_m8 [128] (device, float).  wait_timeout_ns > 0
 * overrides the device wait limit; skip_mma != 0 makes the MMA warp issue
 * nothing so that every other wait runs into the limit (exercises the timeout
 * path without faulting or hanging).  force_persistent: 1 = persistent
 * schedule, -1 = one CTA per tile, 0 = automatic.  trace, if not NULL and
 * the library was built with -DOVC_TRACE=1, receives per-role SM clock
 * stamps of the first 64 blocks of CTA 0 (pipeline analysis; ignored
 * otherwise).  r may be NULL.  The dump runs in separate kernel builds
 * (the production kernels carry no dump code): it is available with the
 * method's kernel and its OVC_ATTN_* variants, and with Q smoothing or a
 * repair set on the method's kernel.  Other combinations (V-Smooth; Q
 * smoothing or repair together with OVC_ATTN_* flags or with each other)
 * return OVC_ERR_INVALID_ARG. */
typedef struct {
  int64_t dump_bh, dump_qblock, dump_kblock;
  uint8_t* dump_codes;
  float* dump_m8;
  uint64_t wait_timeout_ns;
  int32_t skip_mma;
  int32_t force_persistent;
  int64_t* trace;   /* device [4][64][8] int64 clock64() stamps of CTA 0, or NULL */
  uint32_t flags;   /* OVC_ATTN_* variant flags, as for ovc_attention_ex */
} ovc_probe;

ovc_status ovc_attention_probe(const ovc_prepared* p, const ovc_repair* r, float softmax_scale,
                               const ovc_output* o, const ovc_probe* probe, void* stream);

/* ovc_prepare for callers that cannot allocate device memory -- the paper
 * has no counterpart; it exists for integration only.  Some callers cannot
 * call cudaMalloc or provide the workspace that ovc_prepare asks for: plugin
 * interfaces whose host owns every device allocation and lends a kernel only
 * fixed input and output buffers, or code on a latency-critical or captured
 * path where allocation is not allowed.  This entry point computes exactly
 * what ovc_prepare computes and allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine): the only scratch it needs beyond its outputs,
 * the per-head running amax of V, lives in a fixed device array of
 * OVC_NOALLOC_MAX_HEADS 32-bit entries inside the library, which every GPU
 * that loads the library holds until the process exits.
 *   out: filled in by the caller: B, S, H, nb = ceil(S/128), S_pad = 128*nb,
 *        and the output buffers q, k, vt (16-byte aligned), sq, sk, sv, vamax,
 *        energy (4-byte aligned), in the layouts of ovc_prepared; vmean,
 *        perm and kbias must be NULL.  The struct is then usable with ovc_attention and
 *        ovc_prepare_v_repair like one filled by ovc_prepare.
 * Errors: OVC_ERR_SCRATCH_LIMIT if B*H > OVC_NOALLOC_MAX_HEADS (nothing is
 * launched); OVC_ERR_INVALID_ARG for a NULL or misaligned buffer, a vmean,
 * perm or kbias that is not NULL, or dimensions that do not match the inputs.
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  Every call shares the one array, which keeps the last call's
 * contents (each call clears the entries it uses first), so calls whose
 * kernels could overlap on the GPU race: issue them on one stream or
 * otherwise serialise them. */
#define OVC_NOALLOC_MAX_HEADS 4096
ovc_status ovc_prepare_noalloc(const ovc_tensor* q, const ovc_tensor* k, const ovc_tensor* v,
                               const ovc_prepared* out, void* stream);

/* ovc_prepare with options.  flags (OR of):
 *   OVC_PREPARE_SMOOTH_K  K smoothing -- optional, off in ovc_prepare.  The
 *     VC-Attention summary ("Why attention is the video bottleneck") names
 *     Q/K smoothing as the prior art of low-bit attention.  Per (b,h) the
 *     channel means of K over the sequence are subtracted (FP32) before K is
 *     quantised.  Exact non-causal softmax attention is unchanged (every
 *     score of a row moves by q.mean); K's block scales lose the channel
 *     offset, which lowers the quantisation error when keys carry a common
 *     per-channel bias.  The mean is summed in a fixed order (per 128-token
 *     block in token order, the block sums in block order, then one FP32
 *     division by S) so that it reproduces bit for bit.  The means themselves
 *     are not part of ovc_prepared (attention does not need them).
 *   OVC_PREPARE_V_SMOOTH  V-Smooth ("VC-Attention" summary, "V-Smooth"), the
 *     paper's treatment of V that Open-VC replaced with repair.  Per head and
 *     128-token block b: mu_b = bf16(FP32 mean of the block's valid tokens,
 *     summed in token order); the residuals v - mu_b are quantised with one
 *     scale per head (amax of the residuals / 448) and written to vt; the
 *     restored means M'_b = bf16(mu_b r) go to vmean.  Attention adds M'_b,
 *     weighted by each row's block row sum, back into O.  Not combinable with
 *     repair (no energies) or with split key ranges.
 *   OVC_PREPARE_SMOOTH_Q  Q smoothing -- optional, off in ovc_prepare (same
 *     prior art as K smoothing).  Per (b,h) Q's channel means mu_q over the
 *     sequence (FP32, summed as K's) are subtracted before Q is quantised,
 *     so Q's block scales lose the channel offset.  That moves every score
 *     of key t by mu_q . k_t, which is not the same for all keys, so it is
 *     added back: each key gets the bias beta_t = mu_q . dec(k_t) (its
 *     quantised code, decoded), stored as a BF16 (hi, lo) pair in
 *     ovc_prepared.kbias, and attention adds s_k beta_t to the key's
 *     scores through one BF16 MMA per key block (the score is then the
 *     product of mu_q + s_q dec(q') with s_k dec(k_t)).  Combines with K
 *     smoothing, grouping, repair and split key ranges; not with V-Smooth.
 * ovc_prepare_workspace_bytes_ex gives the workspace for the same flags
 * (0 for unknown flags, SMOOTH_Q with V_SMOOTH, or unsupported shapes);
 * such flags make ovc_prepare_ex return OVC_ERR_INVALID_ARG.  Otherwise as
 * ovc_prepare. */
#define OVC_PREPARE_SMOOTH_K 1u
#define OVC_PREPARE_V_SMOOTH 2u
#define OVC_PREPARE_SMOOTH_Q 4u
size_t ovc_prepare_workspace_bytes_ex(int64_t B, int64_t S, int64_t H, int64_t D, uint32_t flags);

/* V-Smooth's grouping ("VC-Attention" summary, "V-Smooth": online k-means
 * clusters each head's value tokens; keys and values are permuted together,
 * which non-causal attention does not notice).  Per (b,h): Lloyd's k-means
 * with `clusters` (1..64, <= S) centroids started at tokens floor(c S / C)
 * and `iters` (1..1000) assign steps, FP32 with a fixed operation order (see
 * the grouping kernels); then perm [B,H,S] (device, int32, 4-byte aligned)
 * lists the tokens ordered by (cluster, index).  Pass perm to
 * ovc_prepare_grouped so that V-Smooth's 128-token blocks hold similar
 * values.  Workspace: ovc_vsmooth_group_workspace_bytes (256-byte aligned).
 * After the call the workspace begins with the state of the last assignment
 * step, for inspection: the centroids it used, FP32 [B,H,C,128] at offset 0,
 * then its labels, int32 [B,H,S], at the next multiple of 256 bytes.
 * Asynchronous on `stream`. */
size_t ovc_vsmooth_group_workspace_bytes(int64_t B, int64_t S, int64_t H, int32_t clusters);
ovc_status ovc_vsmooth_group(const ovc_tensor* v, int32_t clusters, int32_t iters, void* workspace,
                             size_t workspace_bytes, int32_t* perm, void* stream);

/* ovc_prepare_ex with K and V taken in the token order perm [B,H,S] (device,
 * int32; NULL: the input order), e.g. the grouping of ovc_vsmooth_group.
 * Queries keep their order, so attention's output rows do too.  perm must
 * stay valid while the prepared struct is used; repair is not available on
 * grouped inputs. */
ovc_status ovc_prepare_grouped(const ovc_tensor* q, const ovc_tensor* k, const ovc_tensor* v, const int32_t* perm,
                               uint32_t flags, void* workspace, size_t workspace_bytes, ovc_prepared* out,
                               void* stream);
ovc_status ovc_prepare_ex(const ovc_tensor* q, const ovc_tensor* k, const ovc_tensor* v, uint32_t flags,
                          void* workspace, size_t workspace_bytes, ovc_prepared* out, void* stream);

/* The whole call for inputs and output in HOST memory -- the pages' API takes
 * device tensors; this entry point serves callers whose tensors live on the
 * host (no counterpart in the pages).  Q, K, V and O are streamed through the
 * current device in chunks of whole heads: while one chunk is prepared and
 * attended, the next chunk's inputs are copied in and the previous chunk's
 * output is copied out, so the copies (bound by the host link) hide behind
 * the attention kernels.  Every head is computed on its own (its V scale,
 * residual ranking and attention involve that head alone), so the result
 * equals ovc_prepare_ex + (ovc_prepare_v_repair +) ovc_attention_ex over all
 * heads at once, bit for bit.
 *   io            host pointers q, k, v (contiguous [B,S,H,128] of dtype
 *                 OVC_BF16 or OVC_FP16) and o (contiguous BF16 [B,S,H,128]).
 *                 Pinned (page-locked) memory lets the copies run
 *                 asynchronously at full speed; pageable memory gives the
 *                 same result, more slowly.
 *   softmax_scale <= 0 selects 1/sqrt(128).
 *   prep_flags    OR of OVC_PREPARE_SMOOTH_K and OVC_PREPARE_SMOOTH_Q.
 *   repair_budget 0 for none, else in (0, 1] as for ovc_prepare_v_repair.
 *   chunk_sizes   nchunks head counts, each >= 1, summing to H, in head order
 *                 (ovc_host_chunk_plan gives the default plan).
 *   workspace     device memory, 256-byte aligned, at least
 *                 ovc_attention_host_workspace_bytes(B, S, largest chunk, ...)
 *                 bytes: two sets of staging buffers, preparations and repair
 *                 sets (chunk c uses set c % 2).
 * Synchronous: the call creates its own streams (two for compute, one for
 * each copy direction), and returns once O is complete in host memory and
 * every stream has finished with the workspace, also after an error.
 * Returns OVC_ERR_INVALID_ARG, OVC_ERR_UNSUPPORTED (dtype),
 * OVC_ERR_WORKSPACE_TOO_SMALL, any error of the calls it makes, or
 * OVC_ERR_CUDA if a copy, stream or event call fails.  Device-side timeouts
 * are reported by ovc_get_device_status() as for every other call. */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  int32_t dtype;                    /* OVC_BF16 or OVC_FP16 (q, k, v); o is BF16 */
  int64_t B, S, H;
} ovc_host_io;

ovc_status ovc_attention_host(const ovc_host_io* io, float softmax_scale, uint32_t prep_flags,
                              float repair_budget, const int32_t* chunk_sizes, int32_t nchunks,
                              void* workspace, size_t workspace_bytes);

/* Workspace bytes of ovc_attention_host whose largest chunk has
 * max_chunk_heads heads (0 for invalid arguments). */
size_t ovc_attention_host_workspace_bytes(int64_t B, int64_t S, int64_t max_chunk_heads, int32_t dtype,
                                          uint32_t prep_flags, float repair_budget);

/* The default head-chunk plan of ovc_attention_host, a host-only
 * computation: writes the chunk sizes (in head order) to sizes[0..n) and
 * returns n, or -1 if H < 1 or more than max_chunks sizes would be needed.
 * The first chunk's copy in and the last chunk's copy out are the only
 * copies no computation hides, so the plan ramps: e and 2e heads first, 2e
 * and e last, e = H/56 rounded (half to even, at least 1).  A chunk's
 * attention takes about five times as long as the copy of as many heads
 * (73397 tokens on a GB300), so each chunk still hides the next one's copy;
 * hence also h <= 10 e below.  The chunks between take h heads each, h in
 * [H/8, min(H/4, 10 e)] chosen so that h * tiles_per_head fills whole waves
 * of `sms` CTAs best (filled / used slots compared to four decimals, the
 * larger h on a tie); with tiles_per_head or sms <= 0, h = ceil(H/4).  Fewer
 * than 12 heads: equal chunks of ceil(H/4).  tiles_per_head = B * ceil(nb/2)
 * for the attention kernel's pairs of 128-row query blocks (nb = ceil(S/128));
 * sms = the device's SM count. */
int32_t ovc_host_chunk_plan(int64_t H, int64_t tiles_per_head, int32_t sms, int32_t* sizes, int32_t max_chunks);

#ifdef __cplusplus
}
#endif

#endif /* OVC_H_ */
