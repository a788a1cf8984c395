"""Python binding of libovc (PyTorch supplies device memory and streams).

Every step of the computation runs in libovc's CUDA kernels; this module only
marshals arguments.  There is no CPU fallback: without the built library or a
GB300 every call raises.

Entry points follow the "Open VC Attention" catalogue entry: ``attention(q, k,
v)`` on BF16/FP16 ``[S,H,128]`` or ``[B,S,H,128]`` returning BF16, and V
residual repair via ``prepare_v_repair(..., budget)`` + ``attention_v_repair``.
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _abi
from ._abi import OvcError, check, lib

_DTYPES = {torch.bfloat16: _abi.OVC_BF16, torch.float16: _abi.OVC_FP16}


def _stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _device_of(*xs, stream=None) -> torch.device:
    """The one CUDA device that every tensor in xs (None entries skipped) and
    an explicit stream live on.  libovc launches on the current device, so
    each call below runs under ``torch.cuda.device`` of this device."""
    devs = {x.device for x in xs if x is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one CUDA device, got {sorted(map(str, devs))}")
    dev = devs.pop()
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if stream is not None and stream.device != dev:
        raise ValueError(f"stream is on {stream.device}, tensors on {dev}")
    return dev


def _as4d(x: torch.Tensor) -> torch.Tensor:
    if x.dim() == 3:
        return x.unsqueeze(0)
    if x.dim() != 4:
        raise ValueError(f"expected [S,H,128] or [B,S,H,128], got {tuple(x.shape)}")
    return x


def _tensor_desc(x: torch.Tensor) -> _abi.OvcTensor:
    x = _as4d(x)
    if x.dtype not in _DTYPES:
        raise TypeError(f"inputs must be bfloat16 or float16, got {x.dtype}")
    if not x.is_cuda:
        raise ValueError("inputs must be CUDA tensors")
    if x.stride(3) != 1:
        raise ValueError("channel stride must be 1")
    B, S, H, D = x.shape
    return _abi.OvcTensor(x.data_ptr(), _DTYPES[x.dtype], B, S, H, D, x.stride(0), x.stride(1),
                          x.stride(2))


def _output_desc(o: torch.Tensor, prep: "Prepared") -> _abi.OvcOutput:
    """O's pointer and strides.  The C ABI takes no extent for O, so its
    shape is checked here against the prepared inputs."""
    o = _as4d(o)
    if o.dtype != torch.bfloat16 or not o.is_cuda or o.stride(3) != 1:
        raise ValueError("output must be a CUDA bfloat16 tensor with unit channel stride")
    want = (prep.B, prep.S, prep.H, 128)
    if tuple(o.shape) != want:
        raise ValueError(f"output shape {tuple(o.shape)} does not match the inputs' {want}")
    return _abi.OvcOutput(o.data_ptr(), o.stride(0), o.stride(1), o.stride(2))


def _view(ws: torch.Tensor, ptr: int, nbytes: int) -> torch.Tensor:
    off = ptr - ws.data_ptr()
    return ws[off:off + nbytes]


@dataclasses.dataclass
class Prepared:
    """E4M3 Q/K/V, their scales and the V residual energies, in `workspace`."""
    desc: _abi.OvcPrepared
    workspace: torch.Tensor
    shape: tuple
    dtype: torch.dtype
    perm: torch.Tensor | None = None      # grouping order of K and V, kept alive here

    @property
    def B(self):
        return self.desc.B

    @property
    def S(self):
        return self.desc.S

    @property
    def H(self):
        return self.desc.H

    def q_codes(self):
        d = self.desc
        return _view(self.workspace, d.q, d.B * d.H * d.S_pad * 128).view(d.B, d.H, d.S_pad, 128)

    def k_codes(self):
        d = self.desc
        return _view(self.workspace, d.k, d.B * d.H * d.S_pad * 128).view(d.B, d.H, d.S_pad, 128)

    def vt_codes(self):
        d = self.desc
        return _view(self.workspace, d.vt, d.B * d.H * 128 * d.S_pad).view(d.B, d.H, 128, d.S_pad)

    def q_scales(self):
        d = self.desc
        return _view(self.workspace, d.sq, 4 * d.B * d.H * d.nb).view(torch.float32).view(d.B, d.H, d.nb)

    def k_scales(self):
        d = self.desc
        return _view(self.workspace, d.sk, 4 * d.B * d.H * d.nb).view(torch.float32).view(d.B, d.H, d.nb)

    def v_scales(self):
        d = self.desc
        return _view(self.workspace, d.sv, 4 * d.B * d.H).view(torch.float32).view(d.B, d.H)

    def energy(self):
        d = self.desc
        return _view(self.workspace, d.energy, 4 * d.B * d.H * d.S).view(torch.float32).view(d.B, d.H, d.S)

    def key_bias(self):
        """Q smoothing's key bias rows, BF16 [B,H,S_pad,16] (None without it)."""
        d = self.desc
        if not d.kbias:
            return None
        return _view(self.workspace, d.kbias, 32 * d.B * d.H * d.S_pad).view(torch.bfloat16).view(
            d.B, d.H, d.S_pad, 16)

    def v_means(self):
        """V-Smooth's restored block means M'_b, BF16 [B,H,128,nbk] (None without V-Smooth)."""
        d = self.desc
        if not d.vmean:
            return None
        nbk = -(-d.nb // 16) * 16
        return _view(self.workspace, d.vmean, 2 * d.B * d.H * 128 * nbk).view(torch.bfloat16).view(d.B, d.H, 128, nbk)


@dataclasses.dataclass
class Repair:
    desc: _abi.OvcRepair
    workspace: torch.Tensor

    def idx(self):
        d = self.desc
        return _view(self.workspace, d.idx, 4 * d.B * d.H * d.n).view(torch.int32).view(d.B, d.H, d.n)

    def k_sel(self):
        d = self.desc
        return _view(self.workspace, d.k_sel, d.B * d.H * d.n_pad * 128).view(d.B, d.H, d.n_pad, 128)

    def dvt(self):
        d = self.desc
        return _view(self.workspace, d.dvt, d.B * d.H * 128 * d.n_pad).view(d.B, d.H, 128, d.n_pad)

    def sk_sel(self):
        d = self.desc
        return _view(self.workspace, d.sk_sel, 4 * d.B * d.H * d.n_pad).view(torch.float32).view(d.B, d.H, d.n_pad)

    def sr(self):
        d = self.desc
        return _view(self.workspace, d.sr, 4 * d.B * d.H).view(torch.float32).view(d.B, d.H)


def prepare_workspace_bytes(B: int, S: int, H: int, *, smooth_k: bool = False, v_smooth: bool = False,
                            smooth_q: bool = False) -> int:
    return int(lib().ovc_prepare_workspace_bytes_ex(B, S, H, 128, _prep_flags(smooth_k, v_smooth, smooth_q)))


def _prep_flags(smooth_k: bool, v_smooth: bool = False, smooth_q: bool = False) -> int:
    return ((_abi.OVC_PREPARE_SMOOTH_K if smooth_k else 0) | (_abi.OVC_PREPARE_V_SMOOTH if v_smooth else 0) |
            (_abi.OVC_PREPARE_SMOOTH_Q if smooth_q else 0))


def group_v(v: torch.Tensor, clusters: int = 16, iters: int = 4, *, stream=None, return_state: bool = False):
    """V-Smooth's grouping (ovc_vsmooth_group): k-means over each head's value
    tokens, returned as the token order perm [B,H,S] (int32, CUDA) for
    ``prepare(..., perm=perm)``.  return_state=True also returns the last
    assignment step's labels [B,H,S] (int32) and the centroids it used
    [B,H,C,128] (float32), views of the call's workspace."""
    dev = _device_of(v, stream=stream)
    with torch.cuda.device(dev):
        tv = _tensor_desc(v)
        nbytes = int(lib().ovc_vsmooth_group_workspace_bytes(tv.B, tv.S, tv.H, int(clusters)))
        if nbytes == 0:
            raise ValueError("invalid cluster count or shape")
        ws = torch.empty(nbytes, dtype=torch.uint8, device=v.device)
        perm = torch.empty((tv.B, tv.H, tv.S), dtype=torch.int32, device=v.device)
        check(lib().ovc_vsmooth_group(ctypes.byref(tv), int(clusters), int(iters), ctypes.c_void_p(ws.data_ptr()),
                                      ws.numel(), ctypes.c_void_p(perm.data_ptr()),
                                      ctypes.c_void_p(_stream_handle(stream))), "ovc_vsmooth_group")
        if not return_state:
            return perm
        ncent = tv.B * tv.H * int(clusters) * 128 * 4
        cent = ws[:ncent].view(torch.float32).view(tv.B, tv.H, int(clusters), 128)
        off = -(-ncent // 256) * 256
        labels = ws[off:off + 4 * tv.B * tv.H * tv.S].view(torch.int32).view(tv.B, tv.H, tv.S)
        return perm, labels, cent


def prepare(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, smooth_k: bool = False,
            v_smooth: bool = False, perm: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
            stream=None, smooth_q: bool = False) -> Prepared:
    """Quantise Q/K (per 128-token block) and V (per head) to E4M3
    (ovc_prepare_ex).  smooth_k subtracts K's channel means first (optional
    K smoothing; exact non-causal attention is unchanged by it).  v_smooth
    quantises V's residuals after each 128-token block's mean and keeps the
    means for attention to restore (V-Smooth; no repair with it).  perm
    [B,H,S] int32 (e.g. from :func:`group_v`): K and V are taken in that
    token order (ovc_prepare_grouped); Q and so O keep theirs.  smooth_q
    subtracts Q's channel means and adds each key's bias mu_q . k back in
    attention (Q smoothing; not with v_smooth)."""
    dev = _device_of(q, k, v, perm, workspace, stream=stream)
    with torch.cuda.device(dev):
        tq, tk, tv = _tensor_desc(q), _tensor_desc(k), _tensor_desc(v)
        flags = _prep_flags(smooth_k, v_smooth, smooth_q)
        nbytes = prepare_workspace_bytes(tq.B, tq.S, tq.H, smooth_k=smooth_k, v_smooth=v_smooth, smooth_q=smooth_q)
        if nbytes == 0:
            raise ValueError(f"unsupported shape {tuple(q.shape)}")
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        desc = _abi.OvcPrepared()
        if perm is None:
            st = lib().ovc_prepare_ex(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), flags,
                                      ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                      ctypes.byref(desc), ctypes.c_void_p(_stream_handle(stream)))
            check(st, "ovc_prepare_ex")
        else:
            if perm.dtype != torch.int32 or not perm.is_cuda or tuple(perm.shape) != (tq.B, tq.H, tq.S):
                raise ValueError("perm must be a CUDA int32 tensor [B,H,S]")
            perm = perm.contiguous()
            st = lib().ovc_prepare_grouped(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                           ctypes.c_void_p(perm.data_ptr()), flags,
                                           ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                           ctypes.byref(desc), ctypes.c_void_p(_stream_handle(stream)))
            check(st, "ovc_prepare_grouped")
        return Prepared(desc, workspace, tuple(q.shape), q.dtype, perm)


def _out_for(prep: Prepared, out):
    if out is None:
        out = torch.empty(prep.shape, dtype=torch.bfloat16, device=prep.workspace.device)
    return out


def attn_flags(exp_then_cast: bool = False, natural_order: bool = False) -> int:
    """OVC_ATTN_* bits of a kernel variant (both set: the baseline kernel)."""
    return (_abi.OVC_ATTN_EXP_THEN_CAST if exp_then_cast else 0) | (
        _abi.OVC_ATTN_NATURAL_ORDER if natural_order else 0)


def attention_workspace_bytes(prep: Prepared, nsplit: int = 1) -> int:
    """Workspace of split key ranges (0 when nsplit is 0 or 1: no split)."""
    return int(lib().ovc_attention_workspace_bytes(ctypes.byref(prep.desc), int(nsplit)))


def attention_prepared(prep: Prepared, *, softmax_scale: float | None = None,
                       out: torch.Tensor | None = None, stream=None, flags: int = 0,
                       rep: "Repair | None" = None, nsplit: int | None = None,
                       workspace: torch.Tensor | None = None) -> torch.Tensor:
    """O from prepared inputs (ovc_attention_ex): kernel variant ``flags`` (see
    :func:`attn_flags`), optional repair set.  ``nsplit`` > 1 asks for split
    key ranges, a different computation from the method's single pass (each
    range takes its bytes against its own reference) that only the caller
    chooses; ``None``, 0 and 1 never split, and the result is then
    ovc_attention's bit for bit."""
    dev = _device_of(prep.workspace, out, workspace, None if rep is None else rep.workspace, stream=stream)
    with torch.cuda.device(dev):
        out = _out_for(prep, out)
        od = _output_desc(out, prep)
        h = ctypes.c_void_p(_stream_handle(stream))
        ns = 1 if nsplit is None else int(nsplit)
        need = attention_workspace_bytes(prep, ns) if ns > 1 else 0
        if need and (workspace is None or workspace.numel() < need):
            workspace = torch.empty(need, dtype=torch.uint8, device=prep.workspace.device)
        wp = workspace.data_ptr() if (need and workspace is not None) else None
        if ns <= 1 and flags == 0 and rep is None:
            check(lib().ovc_attention(ctypes.byref(prep.desc), float(softmax_scale or 0.0), ctypes.byref(od), h),
                  "ovc_attention")
            return out
        st = lib().ovc_attention_ex(ctypes.byref(prep.desc), ctypes.byref(rep.desc) if rep is not None else None,
                                    float(softmax_scale or 0.0), ctypes.byref(od), int(flags), ns,
                                    ctypes.c_void_p(wp), need, h)
        check(st, "ovc_attention_ex")
        return out


def baseline_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *,
                       softmax_scale: float | None = None, out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """The exp-then-cast baseline on CUDA tensors: the same preparation, then
    probability bytes from an exponent and an FP8 conversion ("Open-VC
    attention", "Problem") and the natural key order, in the same kernel
    pipeline as :func:`attention` so that the two differ only there."""
    prep = prepare(q, k, v, stream=stream)
    return attention_prepared(prep, softmax_scale=softmax_scale, out=out, stream=stream,
                              flags=_abi.OVC_ATTN_BASELINE)


def repair_workspace_bytes(B: int, S: int, H: int, budget: float) -> int:
    return int(lib().ovc_repair_workspace_bytes(B, S, H, budget))


def prepare_v_repair(v: torch.Tensor, prep: Prepared, budget: float = 0.005, *,
                     workspace: torch.Tensor | None = None, stream=None) -> Repair:
    """Select and quantise the V residuals of the worst tokens (ovc_prepare_v_repair)."""
    dev = _device_of(v, prep.workspace, workspace, stream=stream)
    with torch.cuda.device(dev):
        tv = _tensor_desc(v)
        nbytes = repair_workspace_bytes(tv.B, tv.S, tv.H, budget)
        if nbytes == 0:
            raise ValueError("invalid repair budget or shape")
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=v.device)
        desc = _abi.OvcRepair()
        st = lib().ovc_prepare_v_repair(ctypes.byref(tv), ctypes.byref(prep.desc), float(budget),
                                        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                        ctypes.byref(desc), ctypes.c_void_p(_stream_handle(stream)))
        check(st, "ovc_prepare_v_repair")
        return Repair(desc, workspace)


def attention_v_repair(prep: Prepared, rep: Repair, *, softmax_scale: float | None = None,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """O with the repair term (ovc_attention_v_repair)."""
    dev = _device_of(prep.workspace, rep.workspace, out, stream=stream)
    with torch.cuda.device(dev):
        out = _out_for(prep, out)
        od = _output_desc(out, prep)
        st = lib().ovc_attention_v_repair(ctypes.byref(prep.desc), ctypes.byref(rep.desc),
                                          float(softmax_scale or 0.0), ctypes.byref(od),
                                          ctypes.c_void_p(_stream_handle(stream)))
        check(st, "ovc_attention_v_repair")
        return out


def attention_probe(prep: Prepared, rep: Repair | None = None, *, softmax_scale=None, out=None,
                    dump=None, wait_timeout_ns: int = 0, skip_mma: bool = False,
                    force_persistent: int = 0, trace: torch.Tensor | None = None, stream=None,
                    flags: int = 0):
    """Test hook: attention with P-byte dumps / wait-limit controls.

    dump = (bh, qblock, kblock) returns (out, codes [128,128] uint8, m8 [128])."""
    dev = _device_of(prep.workspace, None if rep is None else rep.workspace, out, trace, stream=stream)
    with torch.cuda.device(dev):
        out = _out_for(prep, out)
        od = _output_desc(out, prep)
        probe = _abi.OvcProbe()
        probe.dump_bh = -1
        probe.wait_timeout_ns = int(wait_timeout_ns)
        probe.skip_mma = int(skip_mma)
        probe.force_persistent = int(force_persistent)
        probe.flags = int(flags)
        if trace is not None:
            if trace.dtype != torch.int64 or not trace.is_cuda or trace.numel() < 4 * 64 * 8:
                raise ValueError("trace must be a CUDA int64 tensor of at least 4 * 64 * 8 entries")
            probe.trace = trace.data_ptr()
        codes = m8 = None
        if dump is not None:
            dev = prep.workspace.device
            codes = torch.zeros((128, 128), dtype=torch.uint8, device=dev)
            m8 = torch.full((128,), float("nan"), dtype=torch.float32, device=dev)
            probe.dump_bh, probe.dump_qblock, probe.dump_kblock = (int(x) for x in dump)
            probe.dump_codes = codes.data_ptr()
            probe.dump_m8 = m8.data_ptr()
        st = lib().ovc_attention_probe(ctypes.byref(prep.desc),
                                       ctypes.byref(rep.desc) if rep is not None else None,
                                       float(softmax_scale or 0.0), ctypes.byref(od), ctypes.byref(probe),
                                       ctypes.c_void_p(_stream_handle(stream)))
        check(st, "ovc_attention_probe")
        return out, codes, m8


def device_status(stream=None) -> int:
    """Synchronise and return (and clear) the device-side status (0 = ok)."""
    return int(lib().ovc_get_device_status(ctypes.c_void_p(_stream_handle(stream))))


def head_chunks(H: int, chunk_heads=None, tiles_per_head: int | None = None,
                sms: int | None = None) -> list[tuple[int, int]]:
    """Head ranges [h0, h1) of the host-buffer path.

    chunk_heads: an int (equal chunks of that many heads), a sequence of chunk
    sizes summing to H, or None for the library's default plan
    (``ovc_host_chunk_plan``: a ramp of small chunks at both ends, and chunks
    between whose tile pairs fill whole waves of `sms` CTAs best)."""
    if chunk_heads is None:
        buf = (ctypes.c_int32 * 64)()
        n = lib().ovc_host_chunk_plan(int(H), int(tiles_per_head or 0), int(sms or 0), buf, 64)
        if n < 1:
            raise ValueError(f"no chunk plan for H = {H}")
        return head_chunks(H, list(buf[:n]))
    if isinstance(chunk_heads, int):
        n = max(1, chunk_heads)
        return [(h0, min(H, h0 + n)) for h0 in range(0, H, n)]
    sizes = [int(x) for x in chunk_heads]
    if sum(sizes) != H or min(sizes) < 1:
        raise ValueError(f"chunk sizes {sizes} do not cover {H} heads")
    bounds = [0]
    for n in sizes:
        bounds.append(bounds[-1] + n)
    return list(zip(bounds[:-1], bounds[1:]))


def _attention_device(q, k, v, softmax_scale, repair_budget, out, smooth_k=False, smooth_q=False):
    prep = prepare(q, k, v, smooth_k=smooth_k, smooth_q=smooth_q)
    if repair_budget:
        rep = prepare_v_repair(v, prep, repair_budget)
        return attention_v_repair(prep, rep, softmax_scale=softmax_scale, out=out)
    return attention_prepared(prep, softmax_scale=softmax_scale, out=out)


def _attention_host(q, k, v, softmax_scale, repair_budget, out, dev, chunk_heads, smooth_k=False, smooth_q=False):
    """Host-resident inputs and output: ``ovc_attention_host`` streams them
    through `dev` in head chunks (copies overlapping the neighbouring chunks'
    computation) and returns once O is in `out`.  This function only checks
    the tensors, computes the chunk plan and provides the device workspace."""
    q4, k4, v4 = (_as4d(x) for x in (q, k, v))
    if k4.shape != q4.shape or v4.shape != q4.shape:
        raise ValueError("q, k and v must have the same shape")
    if q4.dtype not in _DTYPES or k4.dtype != q4.dtype or v4.dtype != q4.dtype:
        raise TypeError("inputs must all be bfloat16 or all float16")
    for x in (q4, k4, v4):
        if x.is_cuda or not x.is_contiguous():
            raise ValueError("host inputs must be contiguous CPU tensors (pinned for speed)")
    B, S, H, D = q4.shape
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    o4 = _as4d(out)
    if o4.shape != q4.shape or o4.dtype != torch.bfloat16 or o4.is_cuda or not o4.is_contiguous():
        raise ValueError("out must be a contiguous CPU bfloat16 tensor shaped like q")
    nb = -(-S // 128)
    chunks = head_chunks(H, chunk_heads, tiles_per_head=B * (-(-nb // 2)),
                         sms=torch.cuda.get_device_properties(dev).multi_processor_count)
    sizes = [h1 - h0 for h0, h1 in chunks]
    flags = _prep_flags(smooth_k, False, smooth_q)
    budget = float(repair_budget or 0.0)
    nbytes = lib().ovc_attention_host_workspace_bytes(B, S, max(sizes), _DTYPES[q4.dtype], flags, budget)
    if nbytes == 0:
        raise ValueError("unsupported arguments for the host-buffer path")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    io = _abi.OvcHostIO(q4.data_ptr(), k4.data_ptr(), v4.data_ptr(), o4.data_ptr(), _DTYPES[q4.dtype], B, S, H)
    arr = (ctypes.c_int32 * len(sizes))(*sizes)
    # The workspace comes from the caching allocator on the current stream;
    # the call's own streams must not start before work pending there is done.
    torch.cuda.current_stream(dev).synchronize()
    check(lib().ovc_attention_host(ctypes.byref(io), float(softmax_scale or 0.0), flags, budget, arr, len(sizes),
                                   ctypes.c_void_p(ws.data_ptr()), nbytes), "ovc_attention_host")
    return out


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, softmax_scale: float | None = None,
              repair_budget: float | None = None, out: torch.Tensor | None = None,
              device=None, chunk_heads: int | None = None, smooth_k: bool = False,
              smooth_q: bool = False) -> torch.Tensor:
    """Full call: prepare + ExpCast attention (+ optional V residual repair).

    CUDA inputs give a CUDA output (asynchronous on the current stream).  CPU
    inputs (pinned for speed) are streamed through `device` (default: the
    current CUDA device) in head chunks (`chunk_heads`: a size, a list of
    sizes, or None for the default plan of :func:`head_chunks`), so that
    host<->device copies overlap the computation; O
    lands in `out` (or a new pinned tensor), complete when the call returns.
    smooth_k, smooth_q: optional K and Q smoothing in prepare (see `prepare`).

    Empty inputs (B, S or H of 0: no query rows) give an empty output
    without a launch; the C ABI itself rejects zero sizes."""
    if q.numel() == 0 or k.numel() == 0 or v.numel() == 0:
        q4, k4, v4 = (_as4d(x) for x in (q, k, v))
        if k4.shape != q4.shape or v4.shape != q4.shape or q4.shape[3] != 128:
            raise ValueError("q, k and v must have the same [B,S,H,128] shape")
        if out is None:
            out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
        if tuple(out.shape) != tuple(q.shape) or out.dtype != torch.bfloat16:
            raise ValueError("out must be a bfloat16 tensor shaped like q")
        return out
    if q.is_cuda:
        return _attention_device(q, k, v, softmax_scale, repair_budget, out, smooth_k, smooth_q)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        return _attention_host(q, k, v, softmax_scale, repair_budget, out, dev, chunk_heads, smooth_k, smooth_q)


class CapturedAttention:
    """The full call on CUDA tensors of fixed shape -- prepare, then attention
    (with V residual repair when ``repair_budget`` is set) -- captured once as
    a CUDA graph and replayed.

    Every libovc call is asynchronous on the current stream, allocates no
    memory and never synchronises, so the sequence captures as it stands; a
    replay then costs one graph launch instead of one host call per kernel,
    which is what bounds short sequences.  The inputs are copied into the
    graph's own buffers on each call (``q``, ``k``, ``v`` of the captured
    shape, dtype and device), or, called without arguments, the replay reads
    whatever those buffers (``self.q``, ``self.k``, ``self.v``) hold.  The
    result is written to ``self.out`` and returned; it is the eager call's
    output bit for bit."""

    def __init__(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, softmax_scale: float | None = None,
                 repair_budget: float | None = None, smooth_k: bool = False):
        dev = _device_of(q, k, v)
        with torch.cuda.device(dev):
            self.q, self.k, self.v = (x.clone() for x in (q, k, v))
            self._args = dict(softmax_scale=softmax_scale, repair_budget=repair_budget, smooth_k=smooth_k)
            # One eager call first: it loads the library and sets its
            # per-device state, which must not happen during the capture.
            _attention_device(self.q, self.k, self.v, softmax_scale, repair_budget, None, smooth_k)
            torch.cuda.synchronize(dev)
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph):
                self.out = _attention_device(self.q, self.k, self.v, softmax_scale, repair_budget, None, smooth_k)
            self.device = dev

    def __call__(self, q: torch.Tensor | None = None, k: torch.Tensor | None = None,
                 v: torch.Tensor | None = None) -> torch.Tensor:
        with torch.cuda.device(self.device):
            for src, dst in ((q, self.q), (k, self.k), (v, self.v)):
                if src is not None:
                    if src.shape != dst.shape or src.dtype != dst.dtype or src.device != dst.device:
                        raise ValueError("inputs must match the captured shape, dtype and device")
                    dst.copy_(src)
            self.graph.replay()
            return self.out


def flops(B: int, S: int, H: int, D: int = 128) -> float:
    """Attention FLOPs counted as 4 * B * H * S^2 * D."""
    return 4.0 * B * H * float(S) ** 2 * D


__all__ = ["Prepared", "Repair", "OvcError", "CapturedAttention", "prepare", "attention_prepared", "attention_workspace_bytes",
           "group_v", "prepare_v_repair",
           "attention_v_repair", "attention_probe", "device_status", "attention",
           "head_chunks", "prepare_workspace_bytes", "repair_workspace_bytes", "flops"]
