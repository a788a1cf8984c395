"""GPU test of ovc_prepare_noalloc, the preparation entry point for callers
that cannot allocate device memory: plugin hosts that own every device
allocation and lend a kernel only fixed buffers, or code on a path where
cudaMalloc is not allowed.

The entry point keeps the one piece of scratch the preparation needs, the
per-head running amax of V, in a fixed device array inside the library
instead of in a caller workspace.  The test calls it through the C ABI twice
in a row, on two different inputs (so the second call finds the first call's
maxima in the array and must clear them), and checks each result against
ovc_prepare's: the quantised tensors, scales, amax bits and energies must be
identical (the prepare tests compare bit for bit), and so must the attention
output computed from either.  The output buffers are allocated by the test,
not by the entry point.

This file is collected last on purpose (a failure here leaves every other
test already run); it also passes when run alone in a fresh process, where
its first call is the one that looks up the array's device address."""
import ctypes

import pytest
import torch

import fp8_bit_attention_gb300 as ovc
from fp8_bit_attention_gb300 import _abi

from gpu_util import inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _desc(x):
    x = x if x.dim() == 4 else x.unsqueeze(0)
    B, S, H, D = x.shape
    return _abi.OvcTensor(x.data_ptr(), _abi.OVC_BF16, B, S, H, D, x.stride(0), x.stride(1), x.stride(2))


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc_prepare(q, k, v):
    """Output buffers come from the caller; the entry point allocates nothing."""
    B, S, H, _ = q.shape
    nb = (S + 127) // 128
    dev = q.device
    bufs = dict(
        q=torch.empty((B, H, nb * 128, 128), dtype=torch.uint8, device=dev),
        k=torch.empty((B, H, nb * 128, 128), dtype=torch.uint8, device=dev),
        vt=torch.empty((B, H, 128, nb * 128), dtype=torch.uint8, device=dev),
        sq=torch.empty((B, H, nb), dtype=torch.float32, device=dev),
        sk=torch.empty((B, H, nb), dtype=torch.float32, device=dev),
        sv=torch.empty((B, H), dtype=torch.float32, device=dev),
        vamax=torch.empty((B, H), dtype=torch.int32, device=dev),
        energy=torch.empty((B, H, S), dtype=torch.float32, device=dev),
    )
    # poison the outputs so that stale values cannot pass
    for t in bufs.values():
        t.view(torch.uint8).fill_(0xA5)
    desc = _abi.OvcPrepared(B, S, H, nb, nb * 128, *(bufs[n].data_ptr() for n in
                            ("q", "k", "vt", "sq", "sk", "sv", "vamax", "energy")))
    tq, tk, tv = _desc(q), _desc(k), _desc(v)
    st = _abi.lib().ovc_prepare_noalloc(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                        ctypes.byref(desc), _stream())
    assert st == _abi.OVC_OK, _abi.lib().ovc_status_string(st)
    return desc, bufs


def _assert_same_prepare(prep, bufs):
    d = prep.desc
    torch.cuda.synchronize()
    assert torch.equal(bufs["q"], prep.q_codes())
    assert torch.equal(bufs["k"], prep.k_codes())
    assert torch.equal(bufs["vt"], prep.vt_codes())
    assert torch.equal(bufs["sq"], prep.q_scales())
    assert torch.equal(bufs["sk"], prep.k_scales())
    assert torch.equal(bufs["sv"], prep.v_scales())
    assert torch.equal(bufs["energy"].view(torch.int32), prep.energy().view(torch.int32))
    ref_amax = prep.workspace[d.vamax - prep.workspace.data_ptr():][: 4 * d.B * d.H].view(torch.int32)
    assert torch.equal(bufs["vamax"].flatten(), ref_amax)


def test_noalloc_prepare_matches_prepare_on_two_calls_in_a_row():
    # The larger problem first: the second call must clear the maxima the
    # first one left in the shared array (a stale, larger amax would change
    # the second call's V scale).
    shapes = [(2, 3, 1000, 701), (1, 2, 300, 702)]
    for B, H, S, seed in shapes:
        q, k, v = to_dev(*inputs(B, H, S, seed=seed))
        desc, bufs = _noalloc_prepare(q, k, v)
        prep = ovc.prepare(q, k, v)
        _assert_same_prepare(prep, bufs)
        # attention from the no-allocation preparation equals the usual one
        o_ref = ovc.attention_prepared(prep, nsplit=1)
        o = torch.empty_like(o_ref)
        od = _abi.OvcOutput(o.data_ptr(), o.stride(0), o.stride(1), o.stride(2))
        st = _abi.lib().ovc_attention(ctypes.byref(desc), 0.0, ctypes.byref(od), _stream())
        assert st == _abi.OVC_OK
        assert ovc.device_status() == 0
        assert torch.equal(o, o_ref)


def test_noalloc_prepare_rejects_sizes_beyond_its_scratch():
    B, H, S = 1, _abi.OVC_NOALLOC_MAX_HEADS + 1, 1
    x = torch.zeros((B, S, H, 128), dtype=torch.bfloat16, device="cuda")
    desc = _abi.OvcPrepared(B, S, H, 1, 128, *([x.data_ptr()] * 8))
    t = _desc(x)
    st = _abi.lib().ovc_prepare_noalloc(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t),
                                        ctypes.byref(desc), _stream())
    assert st == _abi.OVC_ERR_SCRATCH_LIMIT
    assert "OVC_NOALLOC_MAX_HEADS" in _abi.lib().ovc_status_string(st).decode()
    # a missing amax output is an argument error, not a silent skip
    desc_ok = _abi.OvcPrepared(B, S, 1, 1, 128, *([x.data_ptr()] * 8))
    desc_ok.vamax = None
    t1 = _desc(x[:, :, :1])
    st = _abi.lib().ovc_prepare_noalloc(ctypes.byref(t1), ctypes.byref(t1), ctypes.byref(t1),
                                        ctypes.byref(desc_ok), _stream())
    assert st == _abi.OVC_ERR_INVALID_ARG
    assert ovc.device_status() == 0
