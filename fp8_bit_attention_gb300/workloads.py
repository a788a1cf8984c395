"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no arithmetic of the method: it only draws random BF16
Q/K/V tensors.  Both the CUDA path and the CPU oracle are fed from the same
host buffers it returns.

The pages measure on a BF16 capture of one MiniMax-H3 video denoising step
(S = 73397, 56 heads, head dim 128; "Open-VC attention" news item, "Results";
"Open VC Attention" catalogue entry).  That capture is not available, so these
seeded draws stand in for it with the same shapes:

* ``small``      B=1 H=2  S=1024   Q,K,V ~ N(0,1)
* ``h7_s8k``     B=1 H=7  S=8192   Q,K ~ N(0,1) + per-(head,channel) bias N(0, var 2);
                                   V ~ N(0,1), 0.5 % of tokens x20 on 8 channels
* ``h14_s32k``   B=1 H=14 S=32768  as h7_s8k
* ``h56_s73397`` B=1 H=56 S=73397  Q,K as h7_s8k; V ~ Student-t(3), outliers as h7_s8k
* ``b2_h56_s36864`` B=2 H=56 S=36864, distributions of h56_s73397

Outlier tokens are one set of positions per batch entry, shared by all heads,
and so are the 8 outlier channels.  Every (tensor, batch, head) slice has its
own child stream of ``numpy.random.SeedSequence(seed)``, so the draw does not
depend on the number of worker threads.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

SEED_BASE = 20260000


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    qk_bias: bool          # per-(head, channel) bias N(0, var 2) on Q and K
    v_dist: str            # "normal" or "student_t3"
    v_outliers: bool       # 0.5 % of tokens scaled x20 on 8 channels
    seed: int

    @property
    def flops(self) -> float:
        """4 * B * H * S^2 * D with D = 128."""
        return 4.0 * self.B * self.H * float(self.S) ** 2 * 128


WORKLOADS = {
    "small": Workload("small", 1, 2, 1024, False, "normal", False, SEED_BASE + 0),
    "h7_s8k": Workload("h7_s8k", 1, 7, 8192, True, "normal", True, SEED_BASE + 1),
    "h14_s32k": Workload("h14_s32k", 1, 14, 32768, True, "normal", True, SEED_BASE + 2),
    "h56_s73397": Workload("h56_s73397", 1, 56, 73397, True, "student_t3", True, SEED_BASE + 3),
    "b2_h56_s36864": Workload("b2_h56_s36864", 2, 56, 36864, True, "student_t3", True,
                              SEED_BASE + 4),
}


def custom(B: int, H: int, S: int, *, qk_bias=True, v_dist="student_t3", v_outliers=True,
           seed=SEED_BASE + 99, name=None) -> Workload:
    """A workload of any shape with the distributions of the named ones."""
    return Workload(name or f"b{B}_h{H}_s{S}", B, H, S, qk_bias, v_dist, v_outliers, seed)


def _workers() -> int:
    return max(1, min(32, len(os.sched_getaffinity(0))))


def generate(w: Workload, *, pin: bool = False):
    """Return (q, k, v): CPU BF16 tensors [B, S, H, 128] (pinned if asked)."""
    B, H, S, D = w.B, w.H, w.S, 128
    root = np.random.SeedSequence(w.seed)
    s_bias, s_q, s_k, s_v, s_out = root.spawn(5)
    g = np.random.Generator(np.random.PCG64(s_bias))
    if w.qk_bias:
        bias_q = (g.standard_normal((H, D)) * np.sqrt(2.0)).astype(np.float32)
        bias_k = (g.standard_normal((H, D)) * np.sqrt(2.0)).astype(np.float32)
    else:
        bias_q = bias_k = None
    go = np.random.Generator(np.random.PCG64(s_out))
    outliers = []
    for _ in range(B):
        if w.v_outliers:
            n_tok = int(round(0.005 * S))
            toks = np.sort(go.choice(S, size=n_tok, replace=False))
            chans = np.sort(go.choice(D, size=8, replace=False))
        else:
            toks = chans = np.zeros(0, np.int64)
        outliers.append((toks, chans))

    tensors = [torch.empty((B, S, H, D), dtype=torch.bfloat16, pin_memory=pin) for _ in range(3)]
    streams = [s_q.spawn(B * H), s_k.spawn(B * H), s_v.spawn(B * H)]

    def fill(task):
        which, b, h = task
        gg = np.random.Generator(np.random.PCG64(streams[which][b * H + h]))
        if which == 2 and w.v_dist == "student_t3":
            x = gg.standard_t(3, size=(S, D)).astype(np.float32)
        else:
            x = np.empty((S, D), np.float32)
            gg.standard_normal(out=x, dtype=np.float32)
        if which == 0 and bias_q is not None:
            x += bias_q[h]
        if which == 1 and bias_k is not None:
            x += bias_k[h]
        if which == 2 and w.v_outliers:
            toks, chans = outliers[b]
            x[np.ix_(toks, chans)] *= np.float32(20.0)
        tensors[which][b, :, h, :] = torch.from_numpy(x).to(torch.bfloat16)

    tasks = [(t, b, h) for t in range(3) for b in range(B) for h in range(H)]
    with ThreadPoolExecutor(_workers()) as ex:
        list(ex.map(fill, tasks))
    return tuple(tensors)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """View a CPU BF16 tensor as a numpy uint16 array of its bits (no copy)."""
    if t.dtype != torch.bfloat16 or t.device.type != "cpu":
        raise ValueError("expected a CPU bfloat16 tensor")
    return t.view(torch.int16).numpy().view(np.uint16)
