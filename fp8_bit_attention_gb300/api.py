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


def _output_desc(o: torch.Tensor) -> _abi.OvcOutput:
    o = _as4d(o)
    if o.dtype != torch.bfloat16 or not o.is_cuda or o.stride(3) != 1:
        raise ValueError("output must be a CUDA bfloat16 tensor with unit channel stride")
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


def prepare_workspace_bytes(B: int, S: int, H: int) -> int:
    return int(lib().ovc_prepare_workspace_bytes(B, S, H, 128))


def prepare(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, workspace: torch.Tensor | None = None,
            stream=None) -> Prepared:
    """Quantise Q/K (per 128-token block) and V (per head) to E4M3 (ovc_prepare)."""
    tq, tk, tv = _tensor_desc(q), _tensor_desc(k), _tensor_desc(v)
    nbytes = prepare_workspace_bytes(tq.B, tq.S, tq.H)
    if nbytes == 0:
        raise ValueError(f"unsupported shape {tuple(q.shape)}")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    desc = _abi.OvcPrepared()
    st = lib().ovc_prepare(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                           ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                           ctypes.byref(desc), ctypes.c_void_p(_stream_handle(stream)))
    check(st, "ovc_prepare")
    return Prepared(desc, workspace, tuple(q.shape), q.dtype)


def _out_for(prep: Prepared, out):
    if out is None:
        out = torch.empty(prep.shape, dtype=torch.bfloat16, device=prep.workspace.device)
    return out


def attention_prepared(prep: Prepared, *, softmax_scale: float | None = None,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """O from prepared inputs (ovc_attention)."""
    out = _out_for(prep, out)
    od = _output_desc(out)
    st = lib().ovc_attention(ctypes.byref(prep.desc), float(softmax_scale or 0.0), ctypes.byref(od),
                             ctypes.c_void_p(_stream_handle(stream)))
    check(st, "ovc_attention")
    return out


def repair_workspace_bytes(B: int, S: int, H: int, budget: float) -> int:
    return int(lib().ovc_repair_workspace_bytes(B, S, H, budget))


def prepare_v_repair(v: torch.Tensor, prep: Prepared, budget: float = 0.005, *,
                     workspace: torch.Tensor | None = None, stream=None) -> Repair:
    """Select and quantise the V residuals of the worst tokens (ovc_prepare_v_repair)."""
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
    out = _out_for(prep, out)
    od = _output_desc(out)
    st = lib().ovc_attention_v_repair(ctypes.byref(prep.desc), ctypes.byref(rep.desc),
                                      float(softmax_scale or 0.0), ctypes.byref(od),
                                      ctypes.c_void_p(_stream_handle(stream)))
    check(st, "ovc_attention_v_repair")
    return out


def attention_probe(prep: Prepared, rep: Repair | None = None, *, softmax_scale=None, out=None,
                    dump=None, wait_timeout_ns: int = 0, skip_mma: bool = False,
                    force_persistent: int = 0, trace: torch.Tensor | None = None, stream=None):
    """Test hook: attention with P-byte dumps / wait-limit controls.

    dump = (bh, qblock, kblock) returns (out, codes [128,128] uint8, m8 [128])."""
    out = _out_for(prep, out)
    od = _output_desc(out)
    probe = _abi.OvcProbe()
    probe.dump_bh = -1
    probe.wait_timeout_ns = int(wait_timeout_ns)
    probe.skip_mma = int(skip_mma)
    probe.force_persistent = int(force_persistent)
    if trace is not None:
        assert trace.dtype == torch.int64 and trace.is_cuda and trace.numel() >= 4 * 64 * 8
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


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, softmax_scale: float | None = None,
              repair_budget: float | None = None, out: torch.Tensor | None = None,
              device=None) -> torch.Tensor:
    """Full call: prepare + ExpCast attention (+ optional V residual repair).

    CUDA inputs give a CUDA output.  CPU inputs (pinned for speed) are copied
    to `device` (default: the current CUDA device), computed there, and O is
    copied back into `out` (or a new pinned tensor)."""
    host = not q.is_cuda
    if host:
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        q, k, v = (x.to(dev, non_blocking=True) for x in (q, k, v))
    prep = prepare(q, k, v)
    o = None if host else out
    if repair_budget:
        rep = prepare_v_repair(v, prep, repair_budget)
        o = attention_v_repair(prep, rep, softmax_scale=softmax_scale, out=o)
    else:
        o = attention_prepared(prep, softmax_scale=softmax_scale, out=o)
    if host:
        if out is None:
            out = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        out.copy_(o, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return out
    return o


def flops(B: int, S: int, H: int, D: int = 128) -> float:
    """Attention FLOPs counted as 4 * B * H * S^2 * D."""
    return 4.0 * B * H * float(S) ** 2 * D


__all__ = ["Prepared", "Repair", "OvcError", "prepare", "attention_prepared", "prepare_v_repair",
           "attention_v_repair", "attention_probe", "device_status", "attention",
           "prepare_workspace_bytes", "repair_workspace_bytes", "flops"]
