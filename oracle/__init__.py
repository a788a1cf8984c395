"""CPU oracle for ExpCast FP8 attention -- TEST INFRASTRUCTURE ONLY.

A plain, slow restatement of the method in C++ (``ovc_oracle.cpp``: FP32-defined
quantisation, double-precision attention), wrapped here with ctypes and numpy.
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and never imports it.

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
against facts the pages or mathematics fix (format definition of E4M3, the
byte/log2 relation, the 79.6 % exp-then-cast agreement, the 3.64 % total
variation bound, brute-force softmax attention, brute-force top-n).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ovc_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Readings of the pages shared by name with the CUDA library's compile-time
# constants (the values are restated, not imported).
C0 = 120.0          # code of p = 1 before beta: stored value v = 2^8 p
BETA = -0.35        # centring constant of the byte relation
TAU = 0.75          # lazy-rescale threshold, log2 units


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no FMA contraction) and return the path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            d = ctypes.c_double
            L.ovc_oracle_e4m3_value.restype = d
            L.ovc_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.ovc_oracle_e4m3_from_float.restype = ctypes.c_uint8
            L.ovc_oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            L.ovc_oracle_bf16_from_double.restype = ctypes.c_uint16
            L.ovc_oracle_bf16_from_double.argtypes = [d]
            L.ovc_oracle_residual_energy.restype = ctypes.c_float
            L.ovc_oracle_residual_energy.argtypes = [P]
            L.ovc_oracle_half_bits_to_float.restype = ctypes.c_float
            L.ovc_oracle_half_bits_to_float.argtypes = [ctypes.c_uint16]
            L.ovc_oracle_expcast_code.restype = ctypes.c_uint8
            L.ovc_oracle_expcast_code.argtypes = [d, d, d, d]
            L.ovc_oracle_exp_cast_code.restype = ctypes.c_uint8
            L.ovc_oracle_exp_cast_code.argtypes = [d, d, d]
            L.ovc_oracle_quantize_blocks.restype = None
            L.ovc_oracle_quantize_blocks.argtypes = [P, ctypes.c_int, i64, i64, i64, i64, i64, i64, P, P, P]
            L.ovc_oracle_k_mean.restype = None
            L.ovc_oracle_k_mean.argtypes = [P, ctypes.c_int, i64, i64, i64, i64, i64, i64, P]
            L.ovc_oracle_vsmooth_v.restype = None
            L.ovc_oracle_vsmooth_v.argtypes = [P, ctypes.c_int, i64, i64, i64, i64, i64, i64, P, P, P]
            L.ovc_oracle_kmeans_group.restype = ctypes.c_int
            L.ovc_oracle_kmeans_group.argtypes = [P, ctypes.c_int, i64, i64, i64, i64, i64, i64, i64, i64, P, P, P]
            L.ovc_oracle_quantize_v.restype = None
            L.ovc_oracle_quantize_v.argtypes = [P, ctypes.c_int, i64, i64, i64, i64, i64, i64, P, P, P]
            L.ovc_oracle_repair_count.restype = i64
            L.ovc_oracle_repair_count.argtypes = [i64, ctypes.c_float]
            L.ovc_oracle_repair_select.restype = None
            L.ovc_oracle_repair_select.argtypes = [P, i64, i64, i64, P]
            L.ovc_oracle_repair_quantize.restype = None
            L.ovc_oracle_repair_quantize.argtypes = [P, ctypes.c_int, i64, i64, i64, i64, i64, i64, P, P, P,
                                                     i64, P, P]
            L.ovc_oracle_block_codes.restype = None
            L.ovc_oracle_block_codes.argtypes = [P, ctypes.c_float, P, P, P, i64, i64, d, d, d, d, ctypes.c_int, P]
            L.ovc_oracle_attention_rows.restype = ctypes.c_int
            L.ovc_oracle_attention_rows.argtypes = (
                [P, P, P, P, P, P, i64, i64, i64, P, P, P, i64, P, P, P, P, i64, d, d, d, d,
                 ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, P, P, P, P, i64, P, P, ctypes.c_int])
            L.ovc_oracle_attention_exact_rows.restype = ctypes.c_int
            L.ovc_oracle_attention_exact_rows.argtypes = (
                [P, P, P, P, i64, i64, P, P, i64, d, d, ctypes.c_int, ctypes.c_int, i64, P, P,
                 ctypes.c_int])
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


# --------------------------------------------------------------------------
# Scalar codecs
# --------------------------------------------------------------------------
def e4m3_value(code: int) -> float:
    return lib().ovc_oracle_e4m3_value(int(code) & 0xFF)


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_from_float(x: float) -> int:
    return int(lib().ovc_oracle_e4m3_from_float(float(np.float32(x))))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    f = lib().ovc_oracle_e4m3_from_float
    return np.array([f(float(v)) for v in x], dtype=np.uint8)


def bf16_from_double(x: np.ndarray) -> np.ndarray:
    """double -> BF16 bits with one round to nearest even."""
    x = np.asarray(x, dtype=np.float64)
    f = lib().ovc_oracle_bf16_from_double
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def expcast_code(Z: float, m8: float = 0.0, c0: float = C0, beta: float = BETA) -> int:
    """ExpCast byte of a score Z (code units, 8*log2) under reference m8."""
    return int(lib().ovc_oracle_expcast_code(float(Z), float(m8), float(c0), float(beta)))


def exp_cast_code(Z: float, m8: float = 0.0, c0: float = C0) -> int:
    """Exp-then-cast byte: E4M3(fl32(2^((Z - m8 + c0 - 56)/8)))."""
    return int(lib().ovc_oracle_exp_cast_code(float(Z), float(m8), float(c0)))


def exp_cast_codes(Z: np.ndarray, m8: float = 0.0, c0: float = C0) -> np.ndarray:
    f = lib().ovc_oracle_exp_cast_code
    return np.array([f(float(z), float(m8), float(c0)) for z in np.ravel(Z)],
                    dtype=np.uint8).reshape(np.shape(Z))


def expcast_codes(Z: np.ndarray, m8: float = 0.0, c0: float = C0, beta: float = BETA) -> np.ndarray:
    f = lib().ovc_oracle_expcast_code
    return np.array([f(float(z), float(m8), float(c0), float(beta)) for z in np.ravel(Z)],
                    dtype=np.uint8).reshape(np.shape(Z))


def residual_energy(R: np.ndarray) -> np.float32:
    R = np.ascontiguousarray(R, dtype=np.float32)
    assert R.shape == (128,)
    return np.float32(lib().ovc_oracle_residual_energy(_ptr(R)))


# --------------------------------------------------------------------------
# Quantisation (FP32-defined)
# --------------------------------------------------------------------------
def half_bits_to_float(bits: int) -> float:
    """IEEE binary16 bits -> value (the oracle's own decoder)."""
    return float(lib().ovc_oracle_half_bits_to_float(int(bits)))


def _bf16_view(x: np.ndarray):
    """x: uint16 array of BF16 (or FP16) bits shaped [B,S,H,128] (any strides, unit last)."""
    assert x.dtype == np.uint16 and x.ndim == 4 and x.shape[3] == 128
    assert x.strides[3] == 2
    sb, ss, sh = (s // 2 for s in x.strides[:3])
    return x, sb, ss, sh


def k_mean(x: np.ndarray, fp16: bool = False) -> np.ndarray:
    """Channel means of K (or Q) over the sequence, [B,H,128] float32 (K and
    Q smoothing; FP32 block sums in token order, then over blocks, then / S)."""
    x, sb, ss, sh = _bf16_view(x)
    B, S, H, _ = x.shape
    mean = np.zeros((B, H, 128), np.float32)
    lib().ovc_oracle_k_mean(_ptr(x), int(fp16), B, S, H, sb, ss, sh, _ptr(mean))
    return mean


def quantize_blocks(x: np.ndarray, fp16: bool = False, mean: np.ndarray | None = None):
    """Q or K (BF16 bits, or FP16 bits if fp16; minus `mean` [B,H,128] if given)
    -> (codes [B,H,S_pad,128] uint8, scales [B,H,nb] float32)."""
    x, sb, ss, sh = _bf16_view(x)
    B, S, H, _ = x.shape
    nb = (S + 127) // 128
    codes = np.zeros((B, H, nb * 128, 128), np.uint8)
    scales = np.zeros((B, H, nb), np.float32)
    mp = None
    if mean is not None:
        mean = np.ascontiguousarray(mean, dtype=np.float32)
        assert mean.shape == (B, H, 128)
        mp = _ptr(mean)
    lib().ovc_oracle_quantize_blocks(_ptr(x), int(fp16), B, S, H, sb, ss, sh, mp, _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_v(v: np.ndarray, fp16: bool = False):
    """V -> (codes token-major [B,H,S_pad,128], sv [B,H], energy [B,H,S])."""
    v, sb, ss, sh = _bf16_view(v)
    B, S, H, _ = v.shape
    nb = (S + 127) // 128
    codes = np.zeros((B, H, nb * 128, 128), np.uint8)
    sv = np.zeros((B, H), np.float32)
    energy = np.zeros((B, H, S), np.float32)
    lib().ovc_oracle_quantize_v(_ptr(v), int(fp16), B, S, H, sb, ss, sh, _ptr(codes), _ptr(sv), _ptr(energy))
    return codes, sv, energy


def vsmooth_v(v: np.ndarray, fp16: bool = False):
    """V-Smooth of V -> (codes token-major [B,H,S_pad,128], sv [B,H],
    mu [B,H,nb,128] block means (BF16 values, held as float32)); token t of
    block b is restored as sv * dec(code_t) + mu_b."""
    v, sb, ss, sh = _bf16_view(v)
    B, S, H, _ = v.shape
    nb = (S + 127) // 128
    codes = np.zeros((B, H, nb * 128, 128), np.uint8)
    sv = np.zeros((B, H), np.float32)
    mu = np.zeros((B, H, nb, 128), np.float32)
    lib().ovc_oracle_vsmooth_v(_ptr(v), int(fp16), B, S, H, sb, ss, sh, _ptr(codes), _ptr(sv), _ptr(mu))
    return codes, sv, mu


def kmeans_group(v: np.ndarray, clusters: int, iters: int, fp16: bool = False):
    """V-Smooth grouping of V [B,S,H,128] bits (Lloyd's k-means in double)
    -> (labels [B,H,S] int32, centroids used by the last assignment
    [B,H,C,128] float64, perm [B,H,S] int32: the token at position t' of the
    grouped order is perm[t'])."""
    v, sb, ss, sh = _bf16_view(v)
    B, S, H, _ = v.shape
    labels = np.zeros((B, H, S), np.int32)
    cent = np.zeros((B, H, clusters, 128), np.float64)
    perm = np.zeros((B, H, S), np.int32)
    rc = lib().ovc_oracle_kmeans_group(_ptr(v), int(fp16), B, S, H, sb, ss, sh, int(clusters), int(iters),
                                       _ptr(labels), _ptr(cent), _ptr(perm))
    if rc != 0:
        raise ValueError("invalid k-means arguments")
    return labels, cent, perm


def permute_tokens(x: np.ndarray, perm: np.ndarray) -> np.ndarray:
    """x [B,S,H,D] gathered per (b, h) along S by perm [B,H,S]."""
    B, S, H, D = x.shape
    out = np.empty_like(x)
    for b in range(B):
        for h in range(H):
            out[b, :, h] = x[b, perm[b, h], h]
    return out


def repair_count(S: int, budget: float) -> int:
    return int(lib().ovc_oracle_repair_count(S, float(np.float32(budget))))


def repair_select(energy: np.ndarray, n: int) -> np.ndarray:
    """energy [B,H,S] float32 -> idx [B,H,n] int32 (ascending per head)."""
    energy = np.ascontiguousarray(energy, dtype=np.float32)
    B, H, S = energy.shape
    idx = np.zeros((B, H, n), np.int32)
    lib().ovc_oracle_repair_select(_ptr(energy), B * H, S, n, _ptr(idx))
    return idx


def repair_quantize(v: np.ndarray, vcodes: np.ndarray, sv: np.ndarray, idx: np.ndarray, fp16: bool = False):
    """-> (dcodes [B,H,n,128] uint8, sr [B,H] float32)."""
    v, sb, ss, sh = _bf16_view(v)
    B, S, H, _ = v.shape
    n = idx.shape[2]
    vcodes = np.ascontiguousarray(vcodes)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    dcodes = np.zeros((B, H, n, 128), np.uint8)
    sr = np.zeros((B, H), np.float32)
    lib().ovc_oracle_repair_quantize(_ptr(v), int(fp16), B, S, H, sb, ss, sh, _ptr(vcodes),
                                     _ptr(np.ascontiguousarray(sv, dtype=np.float32)),
                                     _ptr(idx), n, _ptr(dcodes), _ptr(sr))
    return dcodes, sr


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------
class Prepared:
    """The oracle's own quantised tensors for one (Q, K, V) triple."""

    def __init__(self, q, k, v, fp16: bool = False, smooth_k: bool = False, v_smooth: bool = False,
                 perm: np.ndarray | None = None, smooth_q: bool = False):
        """q, k, v: uint16 bits [B,S,H,128] of BF16 inputs, or of FP16 ones if
        fp16.  smooth_k: subtract K's channel means before quantising K.
        v_smooth: V-Smooth (block means subtracted, residual quantised, means
        restored through the row sums); no residual energies then.  perm
        [B,H,S]: V-Smooth's grouping -- keys and values are taken in this
        token order (queries are not).  smooth_q: Q smoothing -- Q's channel
        means mu_q are subtracted before quantising Q, and every score of key
        t gains s_k beta_t with beta_t = mu_q . dec(K^_t) (kbias [B,H,S],
        float64), so that a score is the exact product of mu_q + s_q dec(Q^')
        with s_k dec(K^_t) (VC-Attention summary, "Why attention is the video
        bottleneck": Q/K smoothing of the prior low-bit kernels)."""
        if perm is not None:
            k = permute_tokens(k, perm)
            v = permute_tokens(v, perm)
        self.B, self.S, self.H, _ = q.shape
        self.nb = (self.S + 127) // 128
        self.fp16 = bool(fp16)
        self.kmean = k_mean(k, fp16) if smooth_k else None
        self.qmean = k_mean(q, fp16) if smooth_q else None
        self.qc, self.sq = quantize_blocks(q, fp16, self.qmean)
        self.kc, self.sk = quantize_blocks(k, fp16, self.kmean)
        self.kbias = None
        if smooth_q:
            tab = e4m3_table()
            kdec = tab[self.kc[:, :, :self.S, :]]                       # [B,H,S,128] double
            self.kbias = np.ascontiguousarray(
                np.einsum("bhtd,bhd->bht", kdec, self.qmean.astype(np.float64)))
        self.vmu = None
        if v_smooth:
            self.vc, self.sv, self.vmu = vsmooth_v(v, fp16)
            self.energy = None
        else:
            self.vc, self.sv, self.energy = quantize_v(v, fp16)
        self.v = v


class Repair:
    def __init__(self, prep: Prepared, budget: float):
        self.n = repair_count(prep.S, budget)
        self.idx = repair_select(prep.energy, self.n)
        self.dcodes, self.sr = repair_quantize(prep.v, prep.vc, prep.sv, self.idx, prep.fp16)


def attention_rows(prep: Prepared, rows_bh, rows_s, *, sm=None, repair: Repair | None = None,
                   c0=C0, beta=BETA, tau=TAU, mid_window=True, snap=True, cast=False, nsplit=1,
                   dump_block=-1, nthreads=None):
    """ExpCast attention for query rows (bh = b*H + h, s); cast=True gives the
    exp-then-cast baseline's bytes, mid_window=False the natural key order,
    nsplit > 1 the split key ranges merged at the end (no repair).

    Returns dict(out [n,128] float64, m8 [n], l [n], nres [n,2], and, when
    dump_block >= 0, codes [n,128] uint8 + dump_m8 [n])."""
    rows_bh = np.ascontiguousarray(rows_bh, dtype=np.int64)
    rows_s = np.ascontiguousarray(rows_s, dtype=np.int64)
    n = rows_bh.shape[0]
    sm = 1.0 / np.sqrt(128.0) if sm is None else float(sm)
    out = np.zeros((n, 128), np.float64)
    m8 = np.zeros(n, np.float64)
    l = np.zeros(n, np.float64)
    nres = np.zeros((n, 2), np.int32)
    codes = np.zeros((n, 128), np.uint8) if dump_block >= 0 else None
    dm8 = np.zeros(n, np.float64) if dump_block >= 0 else None
    if repair is not None:
        ridx, rdc, rsr, nrep = repair.idx, repair.dcodes, repair.sr, repair.n
    else:
        ridx = rdc = rsr = None
        nrep = 0
    rc = lib().ovc_oracle_attention_rows(
        _ptr(prep.qc), _ptr(prep.sq), _ptr(prep.kc), _ptr(prep.sk), _ptr(prep.vc), _ptr(prep.sv),
        prep.B, prep.S, prep.H, _ptr(ridx), _ptr(rdc), _ptr(rsr), nrep, _ptr(prep.vmu), _ptr(prep.kbias),
        _ptr(rows_bh), _ptr(rows_s), n, c0, beta, tau, sm, int(mid_window), int(snap), int(cast),
        int(nsplit), _ptr(out), _ptr(m8), _ptr(l), _ptr(nres), dump_block, _ptr(codes), _ptr(dm8),
        nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle attention_rows failed ({rc})")
    res = dict(out=out, m8=m8, l=l, nres=nres)
    if codes is not None:
        res["codes"] = codes
        res["dump_m8"] = dm8
    return res


def attention_full(prep: Prepared, **kw):
    """All rows of all heads -> out [B,S,H,128] float64."""
    B, S, H = prep.B, prep.S, prep.H
    bh, s = np.meshgrid(np.arange(B * H), np.arange(S), indexing="ij")
    r = attention_rows(prep, bh.ravel(), s.ravel(), **kw)
    out = r["out"].reshape(B, H, S, 128).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(out), r


def block_codes(prep: Prepared, bh: int, s: int, j: int, m8: float, *, sm=None,
                c0=C0, beta=BETA, cast=False) -> np.ndarray:
    """Codes of key block j for query row (bh, s) under reference m8
    (cast=True: exp-then-cast bytes)."""
    sm = 1.0 / np.sqrt(128.0) if sm is None else float(sm)
    B, H = prep.B, prep.H
    qrow = np.ascontiguousarray(prep.qc.reshape(B * H, -1, 128)[bh, s])
    kc = np.ascontiguousarray(prep.kc.reshape(B * H, -1, 128)[bh])
    sk = np.ascontiguousarray(prep.sk.reshape(B * H, -1)[bh])
    sq = float(prep.sq.reshape(B * H, -1)[bh, s // 128])
    kb = None if prep.kbias is None else np.ascontiguousarray(prep.kbias.reshape(B * H, -1)[bh])
    codes = np.zeros(128, np.uint8)
    lib().ovc_oracle_block_codes(_ptr(qrow), sq, _ptr(kc), _ptr(sk), _ptr(kb), prep.S, j, float(m8),
                                 c0, beta, sm, int(cast), _ptr(codes))
    return codes


def attention_exact_rows(q, k, v, rows_bh, rows_s, *, sm=None, tau=TAU, mid_window=True,
                         snap=True, nsplit=1, kbias=None, nthreads=None):
    """Online-softmax skeleton with exact exp2 on raw inputs [BH,S,128]
    (double); kbias [BH,S] (optional) is added to every score of its key
    before the softmax scale."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    BH, S, _ = q.shape
    rows_bh = np.ascontiguousarray(rows_bh, dtype=np.int64)
    rows_s = np.ascontiguousarray(rows_s, dtype=np.int64)
    n = rows_bh.shape[0]
    sm = 1.0 / np.sqrt(128.0) if sm is None else float(sm)
    out = np.zeros((n, 128), np.float64)
    nres = np.zeros(n, np.int32)
    if kbias is not None:
        kbias = np.ascontiguousarray(kbias, dtype=np.float64)
        assert kbias.shape == (BH, S)
    rc = lib().ovc_oracle_attention_exact_rows(
        _ptr(q), _ptr(k), _ptr(v), _ptr(kbias), BH, S, _ptr(rows_bh), _ptr(rows_s), n, tau, sm,
        int(mid_window), int(snap), int(nsplit), _ptr(out), _ptr(nres), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle attention_exact_rows failed ({rc})")
    return out, nres
