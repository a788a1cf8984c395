"""CPU checks of the C ABI: the library loads, exports every function that
include/ovc.h declares, sizes workspaces, and rejects bad arguments on the
host before touching a GPU."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp8_bit_attention_gb300 import _abi, build
    build.build()
    return _abi.lib()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^\s*(?:size_t|ovc_status|int32_t|const char\*)\s+(ovc_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("ovc_prepare", "ovc_attention", "ovc_prepare_v_repair", "ovc_attention_v_repair"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from fp8_bit_attention_gb300 import _abi
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in _abi.SIGNATURES, name


def test_workspace_sizes(lib):
    nb, S_pad = 574, 574 * 128
    bh = 56
    got = lib.ovc_prepare_workspace_bytes(1, 73397, 56, 128)
    assert got >= 3 * bh * S_pad * 128 + 2 * bh * nb * 4 + bh * 73397 * 4
    assert got % 256 == 0
    assert lib.ovc_prepare_workspace_bytes(1, 73397, 56, 64) == 0      # D must be 128
    assert lib.ovc_prepare_workspace_bytes(0, 10, 1, 128) == 0
    assert lib.ovc_prepare_workspace_bytes(1, 0, 1, 128) == 0
    r = lib.ovc_repair_workspace_bytes(1, 73397, 56, 0.005)
    assert r >= bh * 367 * 4 + 2 * bh * 384 * 128
    assert lib.ovc_repair_workspace_bytes(1, 73397, 56, 0.0) == 0
    assert lib.ovc_repair_workspace_bytes(1, 73397, 56, 1.5) == 0


def test_host_validation_rejects_bad_arguments(lib):
    from fp8_bit_attention_gb300 import _abi
    t = _abi.OvcTensor(0x1000, _abi.OVC_BF16, 1, 128, 1, 128, 128 * 128, 128, 128)
    out = _abi.OvcPrepared()
    ws = ctypes.c_void_p(0x100000)
    # null output struct / null tensors
    assert lib.ovc_prepare(None, ctypes.byref(t), ctypes.byref(t), ws, 1 << 30, ctypes.byref(out), None) == _abi.OVC_ERR_INVALID_ARG
    # unsupported head dim and dtype
    bad_d = _abi.OvcTensor(0x1000, _abi.OVC_BF16, 1, 128, 1, 64, 64 * 128, 64, 64)
    assert lib.ovc_prepare(ctypes.byref(bad_d), ctypes.byref(bad_d), ctypes.byref(bad_d), ws, 1 << 30,
                           ctypes.byref(out), None) == _abi.OVC_ERR_UNSUPPORTED
    bad_t = _abi.OvcTensor(0x1000, 7, 1, 128, 1, 128, 128 * 128, 128, 128)
    assert lib.ovc_prepare(ctypes.byref(bad_t), ctypes.byref(bad_t), ctypes.byref(bad_t), ws, 1 << 30,
                           ctypes.byref(out), None) == _abi.OVC_ERR_UNSUPPORTED
    # misaligned pointer, bad strides, shape mismatch
    mis = _abi.OvcTensor(0x1002, _abi.OVC_BF16, 1, 128, 1, 128, 128 * 128, 128, 128)
    assert lib.ovc_prepare(ctypes.byref(mis), ctypes.byref(t), ctypes.byref(t), ws, 1 << 30,
                           ctypes.byref(out), None) == _abi.OVC_ERR_INVALID_ARG
    strided = _abi.OvcTensor(0x1000, _abi.OVC_BF16, 1, 128, 1, 128, 128 * 128, 130, 128)
    assert lib.ovc_prepare(ctypes.byref(strided), ctypes.byref(t), ctypes.byref(t), ws, 1 << 30,
                           ctypes.byref(out), None) == _abi.OVC_ERR_INVALID_ARG
    other = _abi.OvcTensor(0x1000, _abi.OVC_BF16, 1, 256, 1, 128, 256 * 128, 128, 128)
    assert lib.ovc_prepare(ctypes.byref(t), ctypes.byref(other), ctypes.byref(t), ws, 1 << 30,
                           ctypes.byref(out), None) == _abi.OVC_ERR_INVALID_ARG
    # workspace: misaligned, too small
    assert lib.ovc_prepare(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), ctypes.c_void_p(0x100010),
                           1 << 30, ctypes.byref(out), None) == _abi.OVC_ERR_INVALID_ARG
    assert lib.ovc_prepare(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), ws, 100, ctypes.byref(out),
                           None) == _abi.OVC_ERR_WORKSPACE_TOO_SMALL
    # attention with an empty prepared struct
    o = _abi.OvcOutput(0x2000, 128 * 128, 128, 128)
    assert lib.ovc_attention(ctypes.byref(_abi.OvcPrepared()), 0.0, ctypes.byref(o), None) == _abi.OVC_ERR_INVALID_ARG
    assert lib.ovc_attention_v_repair(ctypes.byref(_abi.OvcPrepared()), None, 0.0, ctypes.byref(o), None) == _abi.OVC_ERR_INVALID_ARG
    # kernel-variant flags: unknown bits are rejected before any device call;
    # known ones pass validation (and then fail only for want of a GPU)
    p = _abi.OvcPrepared(1, 128, 1, 1, 128, 0x1000, 0x2000, 0x3000, 0x4000, 0x4100, 0x4200, 0x4300, 0x4400)
    def ex(prep, flags, nsplit=0, ws=None, nbytes=0, rep=None):
        return lib.ovc_attention_ex(ctypes.byref(prep), rep, 0.0, ctypes.byref(o), flags, nsplit,
                                    ctypes.c_void_p(ws), nbytes, None)
    assert ex(p, 4) == _abi.OVC_ERR_INVALID_ARG
    assert ex(_abi.OvcPrepared(), 3) == _abi.OVC_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert ex(p, 3) in (_abi.OVC_ERR_CUDA, _abi.OVC_ERR_UNSUPPORTED)
    # split key ranges: nsplit beyond the key blocks, above 16, negative, without workspace,
    # with an unaligned workspace or with a repair set are rejected before any device call
    p8 = _abi.OvcPrepared(1, 1000, 1, 8, 1024, 0x1000, 0x2000, 0x3000, 0x4000, 0x4100, 0x4200, 0x4300, 0x4400)
    assert ex(p8, 0, nsplit=9, ws=0x100000, nbytes=1 << 30) == _abi.OVC_ERR_INVALID_ARG
    assert ex(p8, 0, nsplit=-1) == _abi.OVC_ERR_INVALID_ARG
    assert ex(p8, 0, nsplit=2) == _abi.OVC_ERR_INVALID_ARG
    assert ex(p8, 0, nsplit=2, ws=0x100010, nbytes=1 << 30) == _abi.OVC_ERR_INVALID_ARG
    r = _abi.OvcRepair(1, 1000, 1, 5, 128, 0x5000, 0x5100, 0x5200, 0x5300, 0x5400)
    assert ex(p8, 0, nsplit=2, ws=0x100000, nbytes=1 << 30, rep=ctypes.byref(r)) == _abi.OVC_ERR_INVALID_ARG
    # workspace of a forced split: 4 tiles x n ranges x 256 rows x (128 FP16 + m8, l)
    for n in (2, 3, 8):
        units = 4 * n
        want = -(-units * 256 * 256 // 256) * 256 + -(-units * 256 * 8 // 256) * 256
        assert lib.ovc_attention_workspace_bytes(ctypes.byref(p8), n) == want
    assert lib.ovc_attention_workspace_bytes(ctypes.byref(p8), 1) == 0
    assert lib.ovc_attention_workspace_bytes(ctypes.byref(p8), 9) == 0
    assert lib.ovc_attention_workspace_bytes(ctypes.byref(p8), 0) == 0   # 0: no split, never automatic


def test_status_strings(lib):
    for s in range(6):
        assert lib.ovc_status_string(s)
    assert b"timed out" in lib.ovc_status_string(5)


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    from fp8_bit_attention_gb300 import _abi, build
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _abi.lib()


def _host_io(B=1, S=300, H=4, dtype=0, ptr=0x1000):
    from fp8_bit_attention_gb300 import _abi
    return _abi.OvcHostIO(ptr, ptr, ptr, ptr, dtype, B, S, H)


def test_attention_host_validates_on_the_host(lib):
    """Every argument check of the host-buffer call runs before it touches a device."""
    import ctypes
    from fp8_bit_attention_gb300 import _abi
    sizes = (ctypes.c_int32 * 2)(1, 3)
    need = lib.ovc_attention_host_workspace_bytes(1, 300, 3, 0, 0, 0.0)
    assert need > 0
    ws = 0x10000
    call = lambda io, fl=0, bud=0.0, sz=sizes, n=2, w=ws, nbytes=need: lib.ovc_attention_host(
        ctypes.byref(io) if io is not None else None, 0.0, fl, bud, sz, n, w, nbytes)
    assert call(None) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(ptr=0)) == _abi.OVC_ERR_INVALID_ARG                 # null host pointers
    assert call(_host_io(dtype=7)) == _abi.OVC_ERR_UNSUPPORTED
    assert call(_host_io(S=0)) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(H=5)) == _abi.OVC_ERR_INVALID_ARG                   # sizes sum to 4, not 5
    assert call(_host_io(), sz=(ctypes.c_int32 * 2)(0, 4)) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(), sz=None) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(), n=0) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(), fl=_abi.OVC_PREPARE_V_SMOOTH) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(), fl=8) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(), bud=1.5) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(), bud=-0.1) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(), w=None) == _abi.OVC_ERR_INVALID_ARG
    assert call(_host_io(), w=ws + 16) == _abi.OVC_ERR_INVALID_ARG          # not 256-byte aligned
    assert call(_host_io(), nbytes=need - 1) == _abi.OVC_ERR_WORKSPACE_TOO_SMALL


def test_attention_host_workspace_bytes(lib):
    """Two sets of: Q, K, V staging, a preparation, a repair set, an output staging."""
    from fp8_bit_attention_gb300 import _abi
    al = lambda x: (x + 255) // 256 * 256
    for B, S, hmax, flags, bud in ((1, 73397, 9, 0, 0.0), (2, 300, 3, _abi.OVC_PREPARE_SMOOTH_K, 0.02),
                                   (1, 1, 1, _abi.OVC_PREPARE_SMOOTH_Q, 1.0)):
        chunk = al(B * S * hmax * 128 * 2)
        prep = al(lib.ovc_prepare_workspace_bytes_ex(B, S, hmax, 128, flags))
        rep = al(lib.ovc_repair_workspace_bytes(B, S, hmax, bud)) if bud > 0 else 0
        want = 2 * (3 * chunk + prep + rep + chunk)
        for dtype in (_abi.OVC_BF16, _abi.OVC_FP16):
            assert lib.ovc_attention_host_workspace_bytes(B, S, hmax, dtype, flags, bud) == want
    assert lib.ovc_attention_host_workspace_bytes(1, 300, 3, 5, 0, 0.0) == 0             # dtype
    assert lib.ovc_attention_host_workspace_bytes(1, 300, 3, 0, _abi.OVC_PREPARE_V_SMOOTH, 0.0) == 0
    assert lib.ovc_attention_host_workspace_bytes(1, 300, 3, 0, 0, 2.0) == 0             # budget
    assert lib.ovc_attention_host_workspace_bytes(1, 0, 3, 0, 0, 0.0) == 0


def test_host_chunk_plan_follows_its_rule(lib):
    """ovc_host_chunk_plan against its documented rule, restated here."""
    import ctypes
    for H in list(range(1, 40)) + [56, 57, 84, 112, 200]:
        for tph, sms in ((0, 0), (287, 152), (1, 152), (144, 148), (18, 152)):
            buf = (ctypes.c_int32 * 128)()
            n = lib.ovc_host_chunk_plan(H, tph, sms, buf, 128)
            sizes = list(buf[:n])
            assert n >= 1 and sum(sizes) == H and min(sizes) >= 1
            if H < 12:
                q = -(-H // 4)
                assert sizes == [q] * (H // q) + ([H % q] if H % q else [])
                continue
            e = max(1, round(H / 56))
            if tph and sms:
                hi = max(2, min(H // 4, 10 * e))
                lo = max(1, min(H // 8, hi))
                waste = lambda c: round(-(-c * tph // sms) * sms / (c * tph), 4)
                h = min(range(lo, hi + 1), key=lambda c: (waste(c), -c))
            else:
                h = -(-H // 4)
            mid = H - 6 * e
            assert sizes == [e, 2 * e] + [h] * (mid // h) + ([mid % h] if mid % h else []) + [2 * e, e]
    buf = (ctypes.c_int32 * 3)()
    assert lib.ovc_host_chunk_plan(56, 287, 152, buf, 3) == -1       # needs 10 sizes
    assert lib.ovc_host_chunk_plan(0, 287, 152, buf, 3) == -1


def test_head_chunks_cover_every_head_once():
    from fp8_bit_attention_gb300.api import head_chunks
    for H in (1, 2, 3, 7, 14, 56, 57, 112):
        for n in (None, 1, 3, 64):
            for tph, sms in ((None, None), (287, 152), (1, 152), (144, 148)):
                ch = head_chunks(H, n, tiles_per_head=tph, sms=sms)
                assert ch[0][0] == 0 and ch[-1][1] == H
                assert all(a1 == b0 for (_, a1), (b0, _) in zip(ch, ch[1:]))
                assert all(h1 > h0 for h0, h1 in ch)
    # the default for 56 heads of 73397 tokens on 152 SMs: a 1, 2 ramp at
    # both ends, 9-head chunks between (9 x 287 tile pairs = exactly 17 waves)
    assert [b - a for a, b in head_chunks(56, None, 287, 152)] == [1, 2, 9, 9, 9, 9, 9, 5, 2, 1]
    assert [b - a for a, b in head_chunks(112, None, 287, 152)][:2] == [2, 4]
    assert [b - a for a, b in head_chunks(10, [3, 7])] == [3, 7]
    with pytest.raises(ValueError):
        head_chunks(10, [3, 6])


def test_prepare_options_on_the_host(lib):
    from fp8_bit_attention_gb300 import _abi
    base = lib.ovc_prepare_workspace_bytes(1, 73397, 56, 128)
    assert lib.ovc_prepare_workspace_bytes_ex(1, 73397, 56, 128, 0) == base
    smooth = lib.ovc_prepare_workspace_bytes_ex(1, 73397, 56, 128, _abi.OVC_PREPARE_SMOOTH_K)
    assert smooth >= base + 56 * 574 * 128 * 4 + 56 * 128 * 4
    vsm = lib.ovc_prepare_workspace_bytes_ex(1, 73397, 56, 128, _abi.OVC_PREPARE_V_SMOOTH)
    assert vsm >= base + 56 * 574 * 128 * 4 + 56 * 128 * 576 * 2     # block means + M' tiles
    assert lib.ovc_prepare_workspace_bytes_ex(1, 73397, 56, 128, 8) == 0        # unknown flag
    t = _abi.OvcTensor(0x1000, _abi.OVC_BF16, 1, 128, 1, 128, 128 * 128, 128, 128)
    out = _abi.OvcPrepared()
    st = lib.ovc_prepare_ex(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), 12, ctypes.c_void_p(0x100000),
                            1 << 30, ctypes.byref(out), None)
    assert st == _abi.OVC_ERR_INVALID_ARG


def test_binding_keeps_every_call_on_one_cuda_device():
    """libovc launches on the current device, so the binding finds the one
    device of a call's tensors (and rejects host tensors or a mix) before
    any launch; checked here with host and meta tensors."""
    from fp8_bit_attention_gb300.api import _device_of
    with pytest.raises(ValueError, match="CUDA"):
        _device_of(torch.zeros(4))
    with pytest.raises(ValueError, match="one CUDA device"):
        _device_of(torch.zeros(4), torch.zeros(4, device="meta"))
    with pytest.raises(ValueError, match="one CUDA device"):
        _device_of()


def test_empty_inputs_give_an_empty_output_without_a_launch():
    """No query rows (S, H or B of 0) means nothing to compute: the binding
    returns an empty BF16 output on the inputs' device (checked here on the
    host, where no GPU exists to launch on)."""
    import fp8_bit_attention_gb300 as ovc
    for shape in [(0, 4, 128), (1, 0, 4, 128), (0, 8, 2, 128), (2, 8, 0, 128)]:
        q = torch.zeros(shape, dtype=torch.bfloat16)
        o = ovc.attention(q, q.clone(), q.clone())
        assert o.shape == q.shape and o.dtype == torch.bfloat16 and o.numel() == 0
    with pytest.raises(ValueError):
        ovc.attention(torch.zeros((0, 4, 128)), torch.zeros((0, 5, 128)), torch.zeros((0, 4, 128)))


def test_prepare_flag_workspaces(lib):
    """Q smoothing adds its means and one 32-byte bias row per padded key;
    it does not combine with V-Smooth; unknown flags size to 0."""
    from fp8_bit_attention_gb300 import _abi
    B, S, H = 1, 1000, 2
    plain = lib.ovc_prepare_workspace_bytes_ex(B, S, H, 128, 0)
    qs = lib.ovc_prepare_workspace_bytes_ex(B, S, H, 128, _abi.OVC_PREPARE_SMOOTH_Q)
    assert qs >= plain + B * H * 1024 * 32 + B * H * 128 * 4
    assert lib.ovc_prepare_workspace_bytes_ex(B, S, H, 128, _abi.OVC_PREPARE_SMOOTH_Q | _abi.OVC_PREPARE_V_SMOOTH) == 0
    assert lib.ovc_prepare_workspace_bytes_ex(B, S, H, 128, 8) == 0
    t = _abi.OvcTensor(0x1000, _abi.OVC_BF16, B, S, H, 128, S * H * 128, H * 128, 128)
    out = _abi.OvcPrepared()
    assert lib.ovc_prepare_ex(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t),
                              _abi.OVC_PREPARE_SMOOTH_Q | _abi.OVC_PREPARE_V_SMOOTH, ctypes.c_void_p(0x100000),
                              1 << 30, ctypes.byref(out), None) == _abi.OVC_ERR_INVALID_ARG
