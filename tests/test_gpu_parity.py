"""GPU parity: libovc (through the C ABI) against the CPU oracle.

Bit-exact: quantised Q/K/V codes and scales, residual energies, repair
indices and repair codes.  Floating point: O within relative L2 5e-3 of the
oracle's double result; P bytes within one code of the oracle's recomputation
under the device's own reference."""
import math

import numpy as np
import pytest
import torch

import oracle
import fp8_bit_attention_gb300 as ovc
from fp8_bit_attention_gb300 import workloads as W

from gpu_util import TOL_REL_L2, inputs, oracle_prep, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    yield
    assert ovc.device_status() == 0


SHAPES = [(1, 2, 1024), (1, 1, 1), (1, 1, 127), (1, 2, 129), (2, 3, 300), (1, 2, 1000), (1, 1, 640)]


@pytest.mark.parametrize("B,H,S", SHAPES)
def test_prepare_bit_exact(B, H, S):
    q, k, v = inputs(B, H, S, seed=100 + S)
    ref = oracle_prep(q, k, v)
    prep = ovc.prepare(*to_dev(q, k, v))
    torch.cuda.synchronize()
    assert np.array_equal(prep.q_codes().cpu().numpy(), ref.qc)
    assert np.array_equal(prep.k_codes().cpu().numpy(), ref.kc)
    assert np.array_equal(prep.q_scales().cpu().numpy(), ref.sq)
    assert np.array_equal(prep.k_scales().cpu().numpy(), ref.sk)
    assert np.array_equal(prep.v_scales().cpu().numpy(), ref.sv)
    vt = prep.vt_codes().cpu().numpy()
    assert np.array_equal(vt.transpose(0, 1, 3, 2), ref.vc)
    assert np.array_equal(prep.energy().cpu().numpy().view(np.uint32), ref.energy.view(np.uint32))


@pytest.mark.parametrize("B,H,S", SHAPES)
def test_attention_matches_oracle(B, H, S):
    q, k, v = inputs(B, H, S, seed=200 + S)
    ref, _ = oracle.attention_full(oracle_prep(q, k, v))
    o = ovc.attention(*to_dev(q, k, v))
    assert ovc.device_status() == 0
    got = o.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) <= TOL_REL_L2


def test_attention_3d_layout_and_strided_inputs():
    q, k, v = inputs(1, 2, 700, seed=301)
    ref, _ = oracle.attention_full(oracle_prep(q, k, v))
    qd, kd, vd = to_dev(q, k, v)
    o3 = ovc.attention(qd[0], kd[0], vd[0])                       # [S,H,128]
    assert rel_l2(o3.float().cpu().numpy(), ref[0]) <= TOL_REL_L2
    # inputs embedded in a wider buffer (head stride 256 elements)
    big = torch.zeros((3, 1, 700, 2, 256), dtype=torch.bfloat16, device="cuda")
    big[0, ..., :128], big[1, ..., :128], big[2, ..., :128] = qd, kd, vd
    out = torch.zeros((1, 700, 2, 256), dtype=torch.bfloat16, device="cuda")
    prep = ovc.prepare(big[0, ..., :128], big[1, ..., :128], big[2, ..., :128])
    ovc.attention_prepared(prep, out=out[..., 128:])
    assert rel_l2(out[..., 128:].float().cpu().numpy(), ref) <= TOL_REL_L2
    assert not out[..., :128].any()


def test_persistent_and_plain_schedules_agree_bitwise():
    q, k, v = inputs(1, 3, 1500, seed=302)
    prep = ovc.prepare(*to_dev(q, k, v))
    a, _, _ = ovc.attention_probe(prep, force_persistent=1)
    b, _, _ = ovc.attention_probe(prep, force_persistent=-1)
    assert ovc.device_status() == 0
    assert torch.equal(a, b)


def test_softmax_scale_argument():
    q, k, v = inputs(1, 1, 512, seed=303)
    ref, _ = oracle.attention_full(oracle_prep(q, k, v), sm=0.05)
    o = ovc.attention(*to_dev(q, k, v), softmax_scale=0.05)
    assert rel_l2(o.float().cpu().numpy(), ref) <= TOL_REL_L2


@pytest.mark.parametrize("S,qb,kb", [(1024, 3, 4), (1000, 7, 7), (1000, 0, 3), (300, 2, 1)])
def test_p_codes_within_one_code_under_device_reference(S, qb, kb):
    H = 2
    q, k, v = inputs(1, H, S, seed=400 + S)
    ref = oracle_prep(q, k, v)
    prep = ovc.prepare(*to_dev(q, k, v))
    bh = 1
    _, codes, m8 = ovc.attention_probe(prep, dump=(bh, qb, kb))
    codes = codes.cpu().numpy()
    m8 = m8.cpu().numpy()
    rows = [r for r in range(128) if qb * 128 + r < S]
    diffs = []
    for r in rows:
        assert np.isfinite(m8[r])
        want = oracle.block_codes(ref, bh, qb * 128 + r, kb, float(m8[r]))
        d = np.abs(codes[r].astype(int) - want.astype(int))
        assert d.max() <= 1, (r, d.max())
        diffs.append(d)
    frac_equal = float(np.mean(np.concatenate(diffs) == 0))
    assert frac_equal > 0.99


@pytest.mark.parametrize("budget", [0.005, 0.02, 0.3])
def test_repair_selection_bit_exact_and_output(budget):
    B, H, S = 1, 2, 1100
    q, k, v = inputs(B, H, S, seed=500)
    ref = oracle_prep(q, k, v)
    rep_ref = oracle.Repair(ref, budget)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    rep = ovc.prepare_v_repair(vd, prep, budget)
    torch.cuda.synchronize()
    assert rep.desc.n == rep_ref.n
    assert np.array_equal(rep.idx().cpu().numpy(), rep_ref.idx)
    assert np.array_equal(rep.sr().cpu().numpy(), rep_ref.sr)
    n = rep_ref.n
    dvt = rep.dvt().cpu().numpy()
    assert np.array_equal(dvt[..., :n].transpose(0, 1, 3, 2), rep_ref.dcodes)
    assert not dvt[..., n:].any()
    ksel = rep.k_sel().cpu().numpy()
    for h in range(H):
        assert np.array_equal(ksel[0, h, :n], ref.kc[0, h, rep_ref.idx[0, h]])
        assert np.array_equal(rep.sk_sel().cpu().numpy()[0, h, :n], ref.sk[0, h, rep_ref.idx[0, h] // 128])
    want, _ = oracle.attention_full(ref, repair=rep_ref)
    o = ovc.attention_v_repair(prep, rep)
    assert ovc.device_status() == 0
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2


def test_timeout_path_reports_and_recovers():
    q, k, v = inputs(1, 1, 512, seed=600)
    prep = ovc.prepare(*to_dev(q, k, v))
    ovc.attention_probe(prep, skip_mma=True, wait_timeout_ns=20_000_000)
    assert ovc.device_status() == 5          # OVC_ERR_TIMEOUT, context still usable
    ref, _ = oracle.attention_full(oracle_prep(q, k, v))
    o = ovc.attention_prepared(prep)
    assert ovc.device_status() == 0
    assert rel_l2(o.float().cpu().numpy(), ref) <= TOL_REL_L2


def test_repair_persistent_and_plain_schedules_agree_bitwise():
    q, k, v = inputs(1, 3, 1300, seed=303)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    rep = ovc.prepare_v_repair(vd, prep, 0.05)
    a, _, _ = ovc.attention_probe(prep, rep, force_persistent=1)
    b, _, _ = ovc.attention_probe(prep, rep, force_persistent=-1)
    assert ovc.device_status() == 0
    assert torch.equal(a, b)
    want, _ = oracle.attention_full(oracle_prep(q, k, v), repair=oracle.Repair(oracle_prep(q, k, v), 0.05))
    assert rel_l2(a.float().cpu().numpy(), want) <= TOL_REL_L2


@pytest.mark.parametrize("B,H,S,chunk,budget", [(1, 7, 1000, 3, None), (2, 5, 700, 2, 0.02),
                                                 (1, 4, 300, None, None)])
def test_host_buffer_path_streams_head_chunks_bit_exactly(B, H, S, chunk, budget):
    """CPU inputs go through the GPU in head chunks (copies overlapping the
    previous chunk's attention); every head is independent, so the result
    must equal the whole-tensor device call bit for bit."""
    q, k, v = inputs(B, H, S, seed=31 + H)
    qd, kd, vd = to_dev(q, k, v)
    want = ovc.attention(qd, kd, vd, repair_budget=budget).cpu()
    qp, kp, vp = (x.pin_memory() for x in (q, k, v))
    got = ovc.attention(qp, kp, vp, repair_budget=budget, chunk_heads=chunk)
    assert not got.is_cuda
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    # [S,H,128] host inputs, pageable memory (synchronous copies), caller's out
    if B == 1:
        out = torch.empty(q[0].shape, dtype=torch.bfloat16)
        got3 = ovc.attention(q[0].contiguous(), k[0].contiguous(), v[0].contiguous(),
                             repair_budget=budget, chunk_heads=chunk, out=out)
        assert got3 is out
        assert torch.equal(got3.view(torch.int16), want[0].view(torch.int16))
    assert ovc.device_status() == 0


@pytest.mark.parametrize("B,H,S,dtype,smooth,budget,sizes", [
    (1, 5, 900, torch.bfloat16, (False, False), None, [1, 3, 1]),
    (2, 4, 333, torch.float16, (True, True), 0.03, [4]),
    (1, 6, 129, torch.bfloat16, (True, False), 1.0, [2, 2, 1, 1]),
])
def test_c_abi_host_call_matches_device_call(B, H, S, dtype, smooth, budget, sizes):
    """ovc_attention_host called directly through the C ABI (host pointers,
    caller workspace, explicit chunk sizes) against the device call with the
    same options, bit for bit."""
    import ctypes
    from fp8_bit_attention_gb300 import _abi
    q, k, v = (x.to(dtype) for x in inputs(B, H, S, seed=71 + S))
    qd, kd, vd = to_dev(q, k, v)
    want = ovc.attention(qd, kd, vd, repair_budget=budget, smooth_k=smooth[0], smooth_q=smooth[1]).cpu()
    qp, kp, vp = (x.contiguous().pin_memory() for x in (q, k, v))
    o = torch.full((B, S, H, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
    flags = (_abi.OVC_PREPARE_SMOOTH_K if smooth[0] else 0) | (_abi.OVC_PREPARE_SMOOTH_Q if smooth[1] else 0)
    dt = _abi.OVC_FP16 if dtype == torch.float16 else _abi.OVC_BF16
    lib = _abi.lib()
    nbytes = lib.ovc_attention_host_workspace_bytes(B, S, max(sizes), dt, flags, float(budget or 0.0))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    io = _abi.OvcHostIO(qp.data_ptr(), kp.data_ptr(), vp.data_ptr(), o.data_ptr(), dt, B, S, H)
    arr = (ctypes.c_int32 * len(sizes))(*sizes)
    st = lib.ovc_attention_host(ctypes.byref(io), 0.0, flags, float(budget or 0.0), arr, len(sizes),
                                ctypes.c_void_p(ws.data_ptr()), nbytes)
    assert st == _abi.OVC_OK
    assert ovc.device_status() == 0
    assert torch.equal(o.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("B,H,S", [(1, 2, 1000), (2, 1, 300)])
def test_fp16_inputs_match_oracle(B, H, S):
    """FP16 inputs ("Open VC Attention" catalogue entry: FP16 or BF16):
    quantised codes, scales, energies and repair indices bit-exact against
    the oracle's FP16 path; O within relative L2 5e-3."""
    q, k, v = (x.to(torch.float16) for x in inputs(B, H, S, seed=57 + S))
    bits = [x.contiguous().view(torch.int16).numpy().view(np.uint16) for x in (q, k, v)]
    ref = oracle.Prepared(*bits, fp16=True)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    assert np.array_equal(prep.q_codes().cpu().numpy(), ref.qc[:, :, :, :])
    assert np.array_equal(prep.k_codes().cpu().numpy(), ref.kc)
    assert np.array_equal(prep.vt_codes().cpu().numpy().transpose(0, 1, 3, 2), ref.vc)
    assert np.array_equal(prep.q_scales().cpu().numpy(), ref.sq)
    assert np.array_equal(prep.k_scales().cpu().numpy(), ref.sk)
    assert np.array_equal(prep.v_scales().cpu().numpy(), ref.sv)
    assert np.array_equal(prep.energy().cpu().numpy().view(np.uint32), ref.energy.view(np.uint32))
    o = ovc.attention_prepared(prep).float().cpu().numpy()
    bh = np.repeat(np.arange(B * H), S)
    ss = np.tile(np.arange(S), B * H)
    r = oracle.attention_rows(ref, bh, ss)["out"].reshape(B, H, S, 128).transpose(0, 2, 1, 3)
    assert rel_l2(o, r) <= TOL_REL_L2
    rep = ovc.prepare_v_repair(vd, prep, 0.02)
    rr = oracle.Repair(ref, 0.02)
    assert np.array_equal(rep.idx().cpu().numpy(), rr.idx)
    assert np.array_equal(rep.sr().cpu().numpy(), rr.sr)
    orep = ovc.attention_v_repair(prep, rep).float().cpu().numpy()
    rrep = oracle.attention_rows(ref, bh, ss, repair=rr)["out"].reshape(B, H, S, 128).transpose(0, 2, 1, 3)
    assert rel_l2(orep, rrep) <= TOL_REL_L2


@pytest.mark.parametrize("B,H,S,fp16", [(1, 2, 1000, False), (2, 1, 300, True), (1, 1, 1, False)])
def test_k_smoothing_matches_oracle(B, H, S, fp16):
    """prepare(smooth_k=True): K codes and scales bit-exact against the
    oracle's smoothed quantisation (which pins the channel means' FP32 sums);
    O within 5e-3; the host-buffer path agrees bit for bit."""
    q, k, v = inputs(B, H, S, seed=71 + S)
    if fp16:
        q, k, v = (x.to(torch.float16) for x in (q, k, v))
    bits = [x.contiguous().view(torch.int16).numpy().view(np.uint16) for x in (q, k, v)]
    ref = oracle.Prepared(*bits, fp16=fp16, smooth_k=True)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd, smooth_k=True)
    assert np.array_equal(prep.k_codes().cpu().numpy(), ref.kc)
    assert np.array_equal(prep.k_scales().cpu().numpy(), ref.sk)
    assert np.array_equal(prep.q_codes().cpu().numpy(), ref.qc)
    assert np.array_equal(prep.vt_codes().cpu().numpy().transpose(0, 1, 3, 2), ref.vc)
    o = ovc.attention_prepared(prep).float().cpu().numpy()
    bh = np.repeat(np.arange(B * H), S)
    ss = np.tile(np.arange(S), B * H)
    r = oracle.attention_rows(ref, bh, ss)["out"].reshape(B, H, S, 128).transpose(0, 2, 1, 3)
    assert rel_l2(o, r) <= TOL_REL_L2
    dev = ovc.attention(qd, kd, vd, smooth_k=True).cpu()
    host = ovc.attention(q.pin_memory(), k.pin_memory(), v.pin_memory(), smooth_k=True)
    assert torch.equal(host.view(torch.int16), dev.view(torch.int16))
    assert ovc.device_status() == 0


def test_k_smoothing_lowers_error_on_biased_keys():
    """On the workloads' per-channel key bias, smoothing lowers the GPU
    output's error against exact softmax attention."""
    B, H, S = 1, 2, 1024
    q, k, v = inputs(B, H, S, seed=77)
    qf, kf, vf = (x.to(torch.float64).numpy() for x in (q, k, v))
    errs = []
    for smooth in (False, True):
        o = ovc.attention(*to_dev(q, k, v), smooth_k=smooth).double().cpu().numpy()
        num = den = 0.0
        for h in range(H):
            s = (qf[0, :, h] @ kf[0, :, h].T) / math.sqrt(128.0)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            ref = (p @ vf[0, :, h]) / p.sum(axis=1, keepdims=True)
            num += np.sum((o[0, :, h] - ref) ** 2)
            den += np.sum(ref ** 2)
        errs.append(math.sqrt(num / den))
    assert errs[1] < errs[0]


# ---- kernel variants: exp-then-cast bytes and the natural key order -------
VARIANTS = [(1, True, False), (2, False, True), (3, True, True)]


@pytest.mark.parametrize("flags,cast,natural", VARIANTS)
@pytest.mark.parametrize("B,H,S", [(1, 2, 1024), (1, 1, 127), (2, 3, 300), (1, 2, 1000)])
def test_attention_variants_match_oracle(flags, cast, natural, B, H, S):
    q, k, v = inputs(B, H, S, seed=600 + S)
    ref, _ = oracle.attention_full(oracle_prep(q, k, v), cast=cast, mid_window=not natural)
    prep = ovc.prepare(*to_dev(q, k, v))
    o = ovc.attention_prepared(prep, flags=flags)
    assert ovc.device_status() == 0
    got = o.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) <= TOL_REL_L2
    if cast or (S + 127) // 128 > 1:              # one key block: both orders coincide
        base = ovc.attention_prepared(prep).float().cpu().numpy()
        assert not np.array_equal(got, base)      # the variant really ran


@pytest.mark.parametrize("S,qb,kb", [(1024, 3, 0), (1000, 7, 7), (300, 2, 1)])
def test_baseline_p_codes_within_one_code_under_device_reference(S, qb, kb):
    H = 2
    q, k, v = inputs(1, H, S, seed=700 + S)
    ref = oracle_prep(q, k, v)
    prep = ovc.prepare(*to_dev(q, k, v))
    bh = 1
    _, codes, m8 = ovc.attention_probe(prep, dump=(bh, qb, kb), flags=3)
    codes = codes.cpu().numpy()
    m8 = m8.cpu().numpy()
    diffs = []
    for r in [r for r in range(128) if qb * 128 + r < S]:
        assert np.isfinite(m8[r])
        want = oracle.block_codes(ref, bh, qb * 128 + r, kb, float(m8[r]), cast=True)
        d = np.abs(codes[r].astype(int) - want.astype(int))
        assert d.max() <= 1, (r, d.max())
        diffs.append(d)
    assert float(np.mean(np.concatenate(diffs) == 0)) > 0.99


def test_baseline_with_repair_and_schedules():
    B, H, S, budget = 1, 2, 1100, 0.02
    q, k, v = inputs(B, H, S, seed=800)
    ref = oracle_prep(q, k, v)
    want, _ = oracle.attention_full(ref, repair=oracle.Repair(ref, budget), cast=True, mid_window=False)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    rep = ovc.prepare_v_repair(vd, prep, budget)
    o = ovc.attention_prepared(prep, rep=rep, flags=3)
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2
    a, _, _ = ovc.attention_probe(prep, rep, force_persistent=1, flags=3)
    b, _, _ = ovc.attention_probe(prep, rep, force_persistent=-1, flags=3)
    assert ovc.device_status() == 0
    assert torch.equal(a, b) and torch.equal(a, o)


def test_baseline_attention_entry_point():
    q, k, v = inputs(1, 2, 700, seed=801)
    want, _ = oracle.attention_full(oracle_prep(q, k, v), cast=True, mid_window=False)
    o = ovc.baseline_attention(*to_dev(q, k, v))
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2


# ---- split key ranges (short sequences) ------------------------------------
@pytest.mark.parametrize("B,H,S,n", [(1, 2, 1024, 2), (1, 2, 1000, 3), (2, 3, 300, 3), (1, 1, 640, 5),
                                     (1, 2, 1024, 8), (1, 3, 129, 2)])
def test_split_key_ranges_match_oracle(B, H, S, n):
    q, k, v = inputs(B, H, S, seed=900 + S + n)
    ref = oracle_prep(q, k, v)
    want, _ = oracle.attention_full(ref, nsplit=n)
    prep = ovc.prepare(*to_dev(q, k, v))
    assert ovc.attention_workspace_bytes(prep, n) > 0
    o = ovc.attention_prepared(prep, nsplit=n)
    assert ovc.device_status() == 0
    got = o.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_l2(got, want) <= TOL_REL_L2
    # the split is a different computation from the unsplit one (each range
    # has its own reference); where the two differ clearly, the output follows
    # the split one
    unsplit, _ = oracle.attention_full(ref)
    if rel_l2(want, unsplit) > 4 * TOL_REL_L2:
        assert rel_l2(got, unsplit) > TOL_REL_L2


@pytest.mark.parametrize("flags,cast,natural", VARIANTS)
def test_split_key_ranges_with_variants(flags, cast, natural):
    q, k, v = inputs(1, 2, 1000, seed=950 + flags)
    want, _ = oracle.attention_full(oracle_prep(q, k, v), nsplit=4, cast=cast, mid_window=not natural)
    prep = ovc.prepare(*to_dev(q, k, v))
    o = ovc.attention_prepared(prep, nsplit=4, flags=flags)
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2


def test_default_entry_points_give_the_c_call_result_bit_for_bit():
    """No entry point splits by itself: attention(), attention_prepared()
    and the host-buffer path give ovc_attention's result bit for bit on
    seven heads of 8192 tokens (224 tile pairs, too few for two full waves
    of a GB300), whatever the GPU, and that result is the method's."""
    import ctypes

    from fp8_bit_attention_gb300 import _abi
    B, H, S = 1, 7, 8192
    q, k, v = inputs(B, H, S, seed=960)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    o_c = torch.empty_like(qd)
    od = _abi.OvcOutput(o_c.data_ptr(), o_c.stride(0), o_c.stride(1), o_c.stride(2))
    assert _abi.lib().ovc_attention(ctypes.byref(prep.desc), 0.0, ctypes.byref(od),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == _abi.OVC_OK
    assert torch.equal(ovc.attention_prepared(prep), o_c)
    assert torch.equal(ovc.attention(qd, kd, vd), o_c)
    host = ovc.attention(q.pin_memory(), k.pin_memory(), v.pin_memory())
    assert torch.equal(host.view(torch.int16), o_c.cpu().view(torch.int16))
    assert ovc.attention_workspace_bytes(prep, 0) == 0 and ovc.attention_workspace_bytes(prep, 1) == 0
    assert ovc.device_status() == 0
    ref = oracle_prep(q, k, v)
    rng = np.random.default_rng(961)
    rows = np.unique(np.concatenate([rng.integers(0, S, 40), [0, S - 1, 4096]]))
    got = o_c.float().cpu().numpy()
    for h in (0, H - 1):
        r = oracle.attention_rows(ref, np.full_like(rows, h), rows)["out"]
        assert rel_l2(got[0, rows, h], r) <= TOL_REL_L2


def test_forced_split_into_a_strided_output():
    """A split the caller asks for (n = 2 on seven heads of 8192 tokens)
    matches the oracle run with the same split on sampled rows; the merge
    pass honours the output strides."""
    B, H, S, n = 1, 7, 8192, 2
    q, k, v = inputs(B, H, S, seed=962)
    ref = oracle_prep(q, k, v)
    prep = ovc.prepare(*to_dev(q, k, v))
    big = torch.zeros((B, S, H, 256), dtype=torch.bfloat16, device="cuda")
    ovc.attention_prepared(prep, out=big[..., 64:192], nsplit=n)
    assert ovc.device_status() == 0
    rng = np.random.default_rng(963)
    rows = np.unique(np.concatenate([rng.integers(0, S, 40), [0, S - 1, 4096]]))
    got = big.float().cpu().numpy()
    for h in (0, H - 1):
        r = oracle.attention_rows(ref, np.full_like(rows, h), rows, nsplit=n)["out"]
        assert rel_l2(got[0, rows, h, 64:192], r) <= TOL_REL_L2
    assert not big[..., :64].any() and not big[..., 192:].any()


def test_split_rejected_with_repair_and_without_workspace():
    q, k, v = inputs(1, 1, 1000, seed=970)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    rep = ovc.prepare_v_repair(vd, prep, 0.02)
    with pytest.raises(ovc.OvcError):
        ovc.attention_prepared(prep, rep=rep, nsplit=2)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    from fp8_bit_attention_gb300 import _abi
    out = torch.empty_like(qd)
    od = _abi.OvcOutput(out.data_ptr(), out.stride(0), out.stride(1), out.stride(2))
    import ctypes
    st = _abi.lib().ovc_attention_ex(ctypes.byref(prep.desc), None, 0.0, ctypes.byref(od), 0, 2,
                                     ctypes.c_void_p(small.data_ptr()), 16, None)
    assert st == _abi.OVC_ERR_WORKSPACE_TOO_SMALL
    assert ovc.device_status() == 0


# ---- V-Smooth ---------------------------------------------------------------
def _vsmooth_inputs(B, H, S, seed, offset=20.0):
    """Values with large per-block, per-channel offsets (the case V-Smooth is for)."""
    q, k, v = inputs(B, H, S, seed=seed)
    rng = np.random.default_rng(seed)
    nb = (S + 127) // 128
    offs = offset * rng.standard_normal((B, nb, H, 128)).astype(np.float32)
    v = (v.float() + torch.from_numpy(np.repeat(offs, 128, axis=1)[:, :S])).to(torch.bfloat16)
    return q, k, v


def _check_restored_means(prep, ref):
    """The kernel restores the block means through a BF16 MMA operand, the
    mean in V-scale units M' = bf16(mu_b / s_v) (as the product fl(mu_b r)).
    The oracle keeps mu_b exact; M' must be that value within one BF16
    rounding (2^-8 relative: 7 stored mantissa bits) plus the rounding of the
    product."""
    nb = ref.nb
    mp = prep.v_means().float().cpu().numpy()[..., :nb].transpose(0, 1, 3, 2).astype(np.float64)
    want = ref.vmu.astype(np.float64) / ref.sv.astype(np.float64)[:, :, None, None]
    assert np.all(np.abs(mp - want) <= 2.0 ** -8 * np.abs(want) * (1 + 2.0 ** -20) + 1e-30)


@pytest.mark.parametrize("B,H,S", [(1, 2, 1024), (1, 1, 1), (1, 2, 129), (2, 3, 300), (1, 2, 1000), (1, 1, 2300)])
def test_v_smooth_prepare_bit_exact_and_attention(B, H, S):
    q, k, v = _vsmooth_inputs(B, H, S, seed=1100 + S)
    ref = oracle.Prepared(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), v_smooth=True)
    prep = ovc.prepare(*to_dev(q, k, v), v_smooth=True)
    torch.cuda.synchronize()
    assert np.array_equal(prep.vt_codes().cpu().numpy().transpose(0, 1, 3, 2), ref.vc)
    assert np.array_equal(prep.v_scales().cpu().numpy(), ref.sv)
    assert np.array_equal(prep.q_codes().cpu().numpy(), ref.qc) and np.array_equal(prep.k_codes().cpu().numpy(), ref.kc)
    _check_restored_means(prep, ref)
    want, _ = oracle.attention_full(ref)
    o = ovc.attention_prepared(prep)
    assert ovc.device_status() == 0
    got = o.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_l2(got, want) <= TOL_REL_L2
    # the restore matters here: without it the output is far off
    plain_ref = oracle.Prepared(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v))
    if S > 1:
        base, _ = oracle.attention_full(plain_ref)
        assert rel_l2(got, base) < 0.05


def test_v_smooth_persistent_schedule_and_rejections():
    q, k, v = _vsmooth_inputs(1, 2, 3000, seed=1200)
    ref = oracle.Prepared(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), v_smooth=True)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd, v_smooth=True)
    a, _, _ = ovc.attention_probe(prep, force_persistent=1)
    b, _, _ = ovc.attention_probe(prep, force_persistent=-1)
    assert ovc.device_status() == 0
    assert torch.equal(a, b)
    want, _ = oracle.attention_full(ref)
    assert rel_l2(a.float().cpu().numpy(), want) <= TOL_REL_L2
    with pytest.raises(ovc.OvcError):
        ovc.prepare_v_repair(vd, prep, 0.01)
    with pytest.raises(ovc.OvcError):
        ovc.attention_prepared(prep, nsplit=2)
    with pytest.raises(ovc.OvcError):
        ovc.attention_prepared(prep, flags=1)
    with pytest.raises(ovc.OvcError):          # no P-byte dump build of the V-Smooth kernel
        ovc.attention_probe(prep, dump=(0, 1, 2))
    assert ovc.device_status() == 0


def test_p_byte_dump_builds_give_the_production_output():
    """The probe's P-byte dump runs in separate kernel builds; with the dump
    on, the output must still be the production kernel's, within the
    tolerance (the same arithmetic, compiled separately)."""
    q, k, v = inputs(1, 2, 1000, seed=3100)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    o = ovc.attention_prepared(prep).float()
    od, codes, m8 = ovc.attention_probe(prep, dump=(1, 3, 5))
    assert ovc.device_status() == 0
    assert rel_l2(od.float().cpu().numpy(), o.cpu().numpy()) <= 1e-3
    assert int(codes.max()) <= 126 and bool(torch.isfinite(m8).all())


# ---- V-Smooth grouping --------------------------------------------------------
def _clustered_inputs(B, H, S, seed, centres=6):
    q, k, _ = inputs(B, H, S, seed=seed)
    rng = np.random.default_rng(seed)
    c = rng.standard_normal((B, H, centres, 128)).astype(np.float32) * 4.0
    lab = rng.integers(0, centres, (B, S, H))
    v = c[np.arange(B)[:, None, None], np.arange(H)[None, None, :], lab]
    v = v + 0.3 * rng.standard_normal(v.shape).astype(np.float32)
    return q, k, torch.from_numpy(v).to(torch.bfloat16)


def _kmeans_dist(x, mu):
    """Squared distances [S, C] in double, and the size of the FP32 error the
    kernel's evaluation n_c - 2 x.mu may make in each (it sums 128 products
    and 128 squares in FP32: below 128 ulps of the magnitudes involved)."""
    d = ((x[:, None, :] - mu[None, :, :]) ** 2).sum(-1)
    err = 2.0 ** -24 * 160 * ((mu ** 2).sum(-1)[None, :] + 2.0 * np.abs(x) @ np.abs(mu).T)
    return d, err


def _check_kmeans_step(x, labels, mu):
    """labels: a nearest centroid of mu for every token, within the FP32
    error bound of the two distances compared."""
    d, err = _kmeans_dist(x, mu)
    best = d.argmin(axis=1)
    idx = np.arange(len(x))
    assert np.all(d[idx, labels] - d[idx, best] <= err[idx, labels] + err[idx, best])


@pytest.mark.parametrize("B,H,S,C,iters", [(1, 1, 1, 1, 1), (1, 2, 200, 7, 3), (2, 3, 300, 16, 4),
                                           (1, 2, 1000, 16, 4), (1, 1, 2300, 64, 2)])
def test_grouping_is_lloyds_algorithm(B, H, S, C, iters):
    """k-means labels have several correct answers at near ties, so the
    GPU's grouping is checked for what Lloyd's algorithm fixes, step by step
    on its own state (each run of i steps is the first i steps of a longer
    one): the first centroids are the tokens floor(c S / C) exactly; every
    assignment is a nearest centroid within the FP32 rounding bound; every
    update is the members' mean within the FP32 summation bound (an empty
    cluster keeps its centroid); the permutation is ordered by (label,
    index).  The first assignment, made from the same centroids as the
    oracle's, must agree with the oracle's wherever the choice is clear by
    more than that bound."""
    q, k, v = _clustered_inputs(B, H, S, seed=1300 + S)
    vd = v.cuda()
    x_all = v.float().numpy().astype(np.float64)              # [B,S,H,128]
    states = []
    for i in range(1, iters + 1):
        perm, labels, cent = ovc.group_v(vd, clusters=C, iters=i, return_state=True)
        torch.cuda.synchronize()
        states.append((perm.cpu().numpy(), labels.cpu().numpy().copy(), cent.cpu().numpy().astype(np.float64)))
    lab1_ref, _, _ = oracle.kmeans_group(W.bf16_bits(v), C, 1)
    nb = (S + 127) // 128
    for b in range(B):
        for h in range(H):
            x = x_all[b, :, h, :]
            start = x[(np.arange(C) * S) // C]
            assert np.array_equal(states[0][2][b, h], start)
            for i, (perm, labels, cent) in enumerate(states):
                lab, mu = labels[b, h], cent[b, h]
                _check_kmeans_step(x, lab, mu)
                p = perm[b, h]
                assert np.array_equal(np.sort(p), np.arange(S))
                key = lab[p].astype(np.int64) * S + p
                assert np.all(np.diff(key) > 0)
                if i + 1 < len(states):
                    nxt = states[i + 1][2][b, h]
                    for c in range(C):
                        m = lab == c
                        if not m.any():
                            assert np.array_equal(nxt[c], mu[c])
                            continue
                        mean = x[m].mean(axis=0)
                        bound = 2.0 ** -24 * (m.sum() + nb + 4) * np.abs(x[m]).mean(axis=0) + 1e-30
                        assert np.all(np.abs(nxt[c] - mean) <= bound), (i, c)
            # the first step against the oracle's, where the choice is clear
            d, err = _kmeans_dist(x, start)
            srt = np.sort(d, axis=1)
            margin = srt[:, 1] - srt[:, 0] if C > 1 else np.full(S, np.inf)
            clear = margin > 2 * err.max(axis=1)
            assert clear.mean() > 0.5
            assert np.array_equal(states[0][1][b, h][clear], lab1_ref[b, h][clear])


@pytest.mark.parametrize("B,H,S,C,iters", [(1, 2, 200, 7, 3), (2, 3, 300, 16, 4), (1, 1, 2300, 64, 2)])
def test_grouped_v_smooth_prepare_bit_exact(B, H, S, C, iters):
    """Preparation in a grouping order -- the oracle's own k-means order,
    handed to the GPU -- gives the oracle's grouped V-Smooth tensors bit for
    bit and its attention output within 5e-3."""
    q, k, v = _clustered_inputs(B, H, S, seed=1300 + S)
    _, _, perm_ref = oracle.kmeans_group(W.bf16_bits(v), C, iters)
    ref = oracle.Prepared(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), v_smooth=True, perm=perm_ref)
    qd, kd, vd = to_dev(q, k, v)
    perm = torch.from_numpy(perm_ref).cuda()
    prep = ovc.prepare(qd, kd, vd, v_smooth=True, perm=perm)
    torch.cuda.synchronize()
    assert np.array_equal(prep.k_codes().cpu().numpy(), ref.kc) and np.array_equal(prep.k_scales().cpu().numpy(), ref.sk)
    assert np.array_equal(prep.vt_codes().cpu().numpy().transpose(0, 1, 3, 2), ref.vc)
    assert np.array_equal(prep.v_scales().cpu().numpy(), ref.sv)
    _check_restored_means(prep, ref)
    want, _ = oracle.attention_full(ref)
    o = ovc.attention_prepared(prep)
    assert ovc.device_status() == 0
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2
    with pytest.raises(ovc.OvcError):
        ovc.prepare_v_repair(vd, ovc.prepare(qd, kd, vd, perm=perm), 0.01)


def test_grouping_keeps_attention_and_lowers_v_smooth_error():
    """Grouped keys/values give the same exact attention; on clustered values
    grouped V-Smooth is closer to exact attention than ungrouped V-Smooth."""
    B, H, S = 1, 2, 2048
    q, k, v = _clustered_inputs(B, H, S, seed=1400, centres=12)
    qd, kd, vd = to_dev(q, k, v)
    rows = np.arange(0, S, 37)
    perm = ovc.group_v(vd, clusters=16, iters=4)
    o_g = ovc.attention_prepared(ovc.prepare(qd, kd, vd, v_smooth=True, perm=perm)).float().cpu().numpy()
    o_u = ovc.attention_prepared(ovc.prepare(qd, kd, vd, v_smooth=True)).float().cpu().numpy()
    qq, kk, vv = (x.double().numpy() for x in (q, k, v))
    e_g, e_u = [], []
    for h in range(H):
        s = qq[0, rows, h] @ kk[0, :, h].T / math.sqrt(128.0)
        p = np.exp(s - s.max(1, keepdims=True))
        ex = (p @ vv[0, :, h]) / p.sum(1, keepdims=True)
        e_g.append(rel_l2(o_g[0, rows, h], ex))
        e_u.append(rel_l2(o_u[0, rows, h], ex))
    assert np.mean(e_g) < np.mean(e_u), (e_g, e_u)


def test_fp16_3d_inputs_through_grouping_v_smooth_and_split():
    """FP16 [S,H,128] inputs: the grouping is Lloyd's algorithm on the FP16
    values (first step checked), grouped V-Smooth preparation in the
    oracle's order bit-exact, O within 5e-3; split key ranges on FP16
    inputs."""
    B, H, S = 1, 2, 1100
    q, k, v = _clustered_inputs(B, H, S, seed=1500)
    q, k, v = (x.to(torch.float16) for x in (q, k, v))
    bits = [x.contiguous().view(torch.int16).numpy().view(np.uint16) for x in (q, k, v)]
    _, _, perm_ref = oracle.kmeans_group(bits[2], 8, 3, fp16=True)
    ref = oracle.Prepared(*bits, fp16=True, v_smooth=True, perm=perm_ref)
    qd, kd, vd = (x[0].cuda() for x in (q, k, v))               # [S,H,128]
    _, lab, cent = ovc.group_v(vd, clusters=8, iters=1, return_state=True)
    xv = v.float().numpy().astype(np.float64)
    for h in range(H):
        _check_kmeans_step(xv[0, :, h], lab[0, h].cpu().numpy(), cent[0, h].cpu().numpy().astype(np.float64))
    prep = ovc.prepare(qd, kd, vd, v_smooth=True, perm=torch.from_numpy(perm_ref).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(prep.vt_codes().cpu().numpy().transpose(0, 1, 3, 2), ref.vc)
    assert np.array_equal(prep.k_codes().cpu().numpy(), ref.kc)
    want, _ = oracle.attention_full(ref)
    o = ovc.attention_prepared(prep)
    assert o.shape == (S, H, 128)
    assert rel_l2(o.float().cpu().numpy(), want[0]) <= TOL_REL_L2
    plain = oracle.Prepared(*bits, fp16=True)
    want3, _ = oracle.attention_full(plain, nsplit=3)
    o3 = ovc.attention_prepared(ovc.prepare(qd, kd, vd), nsplit=3)
    assert rel_l2(o3.float().cpu().numpy(), want3[0]) <= TOL_REL_L2
    assert ovc.device_status() == 0


def test_no_write_outside_the_output_view():
    """Canaries: O is a view inside a larger buffer filled with a sentinel
    (extra tokens after S, an extra head, channels on both sides); every
    attention path writes its rows of the view and nothing else."""
    B, H, S = 1, 2, 1000                      # ragged: the last key/query block has 104 rows
    q, k, v = inputs(B, H, S, seed=1600)
    qd, kd, vd = to_dev(q, k, v)
    sentinel = torch.tensor(12345, dtype=torch.int16).view(torch.bfloat16).item()
    paths = {
        "plain": lambda prep, out: ovc.attention_prepared(prep, out=out, nsplit=1),
        "split": lambda prep, out: ovc.attention_prepared(prep, out=out, nsplit=4),
        "baseline": lambda prep, out: ovc.attention_prepared(prep, out=out, flags=3, nsplit=1),
        "repair": lambda prep, out: ovc.attention_v_repair(prep, ovc.prepare_v_repair(vd, prep, 0.02), out=out),
        "v_smooth": None,
    }
    for name, run in paths.items():
        big = torch.full((B, S + 37, H + 1, 192), sentinel, dtype=torch.bfloat16, device="cuda")
        view = big[:, :S, :H, 32:160]
        if name == "v_smooth":
            ovc.attention_prepared(ovc.prepare(qd, kd, vd, v_smooth=True), out=view)
        else:
            run(ovc.prepare(qd, kd, vd), view)
        assert ovc.device_status() == 0, name
        bits = big.view(torch.int16)
        mask = torch.ones_like(bits, dtype=torch.bool)
        mask[:, :S, :H, 32:160] = False
        assert bool((bits[mask] == 12345).all()), name
        assert bool((bits[:, :S, :H, 32:160] != 12345).all()), name


def test_output_and_device_checks_of_the_binding():
    """The C ABI takes O as a pointer and strides only, so the binding checks
    O's shape, dtype and device against the prepared inputs before launching."""
    B, H, S = 1, 2, 300
    q, k, v = inputs(B, H, S, seed=1700)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    rep = ovc.prepare_v_repair(vd, prep, 0.02)
    bad = [torch.empty((B, S - 1, H, 128), dtype=torch.bfloat16, device="cuda"),     # too few rows
           torch.empty((B, S, H + 1, 128), dtype=torch.bfloat16, device="cuda"),     # an extra head
           torch.empty((B, S, H, 128), dtype=torch.float16, device="cuda"),          # dtype
           torch.empty((B, S, H, 128), dtype=torch.bfloat16)]                         # host memory
    for out in bad:
        with pytest.raises(ValueError):
            ovc.attention_prepared(prep, out=out)
        with pytest.raises(ValueError):
            ovc.attention_v_repair(prep, rep, out=out)
    with pytest.raises(ValueError):
        ovc.prepare(qd, kd, vd.cpu())
    o = ovc.attention_prepared(prep, out=torch.empty((S, H, 128), dtype=torch.bfloat16, device="cuda"))
    assert o.shape == (S, H, 128)
    assert ovc.device_status() == 0


@pytest.mark.parametrize("B,H,S,budget", [(1, 2, 1024, None), (1, 3, 1000, 0.02), (2, 2, 300, None)])
def test_captured_full_call_replays_the_eager_result(B, H, S, budget):
    """The CUDA-graph capture of prepare + attention (+ repair) gives the
    eager call's output bit for bit, also after new inputs are copied in."""
    q, k, v = to_dev(*inputs(B, H, S, seed=1800 + S))
    cap = ovc.CapturedAttention(q, k, v, repair_budget=budget)
    assert torch.equal(cap(), ovc.attention(q, k, v, repair_budget=budget))
    q2, k2, v2 = to_dev(*inputs(B, H, S, seed=1801 + S))
    got = cap(q2, k2, v2).clone()
    assert torch.equal(got, ovc.attention(q2, k2, v2, repair_budget=budget))
    assert not torch.equal(got, cap(q, k, v))
    with pytest.raises(ValueError):
        cap(q2[:, :-1])
    assert ovc.device_status() == 0


@pytest.mark.parametrize("B,H,S,budget", [(1, 2, 300, 1.0), (1, 1, 1, 1.0), (1, 3, 129, 0.5), (2, 1, 640, 1.0)])
def test_repair_edge_budgets(B, H, S, budget):
    """Budget 1 repairs every token (n = S, the largest repair set: as many
    repair blocks as key blocks); S = 1 and a ragged S = 129 cover the
    degenerate sizes.  Selection bit-exact, output within the tolerance."""
    q, k, v = inputs(B, H, S, seed=2100 + S)
    ref = oracle_prep(q, k, v)
    rep_ref = oracle.Repair(ref, budget)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    rep = ovc.prepare_v_repair(vd, prep, budget)
    torch.cuda.synchronize()
    assert rep.desc.n == rep_ref.n == (S if budget == 1.0 else rep_ref.n)
    assert np.array_equal(rep.idx().cpu().numpy(), rep_ref.idx)
    assert np.array_equal(rep.sr().cpu().numpy(), rep_ref.sr)
    want, _ = oracle.attention_full(ref, repair=rep_ref)
    for force in (0, 1):
        o = ovc.attention_probe(prep, rep, force_persistent=force)[0]
        assert ovc.device_status() == 0
        assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2


def test_many_heads_ragged_sequence():
    """2000 heads of 130 tokens (two key blocks, the second with 2 keys):
    large head grids and the head-fastest preparation.  The quantised tensors
    are compared in full, O on every row of a sample of heads (first, last
    and spread between)."""
    B, H, S = 1, 2000, 130
    q, k, v = inputs(B, H, S, seed=2200)
    ref = oracle_prep(q, k, v)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    o = ovc.attention_prepared(prep, nsplit=1)
    assert ovc.device_status() == 0
    assert np.array_equal(prep.q_codes().cpu().numpy()[..., :S, :], ref.qc[..., :S, :])
    assert np.array_equal(prep.vt_codes().cpu().numpy()[..., :S], ref.vc.transpose(0, 1, 3, 2)[..., :S])
    assert np.array_equal(prep.v_scales().cpu().numpy(), ref.sv)
    heads = np.array([0, 1, 777, 1234, 1998, 1999])
    rows_bh = np.repeat(heads, S)
    rows_s = np.tile(np.arange(S), heads.size)
    want = oracle.attention_rows(ref, rows_bh, rows_s)["out"]
    got = o.float().cpu().numpy()[0][:, heads, :].transpose(1, 0, 2).reshape(-1, 128)
    assert rel_l2(got, want) <= TOL_REL_L2


@pytest.mark.parametrize("B,H,S,budget", [(1, 2, 1000, 0.02), (2, 1, 300, 0.3)])
def test_k_smoothing_with_repair(B, H, S, budget):
    """K smoothing and V residual repair together: the repair set's keys are
    gathered from the smoothed K codes with their block scales; selection
    bit-exact and O within 5e-3 of the oracle doing the same."""
    q, k, v = inputs(B, H, S, seed=2300 + S)
    bits = [x.contiguous().view(torch.int16).numpy().view(np.uint16) for x in (q, k, v)]
    ref = oracle.Prepared(*bits, smooth_k=True)
    rep_ref = oracle.Repair(ref, budget)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd, smooth_k=True)
    rep = ovc.prepare_v_repair(vd, prep, budget)
    torch.cuda.synchronize()
    assert np.array_equal(rep.idx().cpu().numpy(), rep_ref.idx)
    n = rep_ref.n
    ksel = rep.k_sel().cpu().numpy()
    for b in range(B):
        for h in range(H):
            assert np.array_equal(ksel[b, h, :n], ref.kc[b, h, rep_ref.idx[b, h]])
    want, _ = oracle.attention_full(ref, repair=rep_ref)
    o = ovc.attention_v_repair(prep, rep)
    assert ovc.device_status() == 0
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2


# ---- degenerate inputs and sharp rows ---------------------------------------
def test_all_zero_blocks_and_heads():
    """All-zero data takes the scale-1 path of the quantiser: a zero V head
    (its output must be exactly 0), a zero K block (its scores are all 0), a
    zero Q block (all its scores are 0: a uniform row), and a zero tail
    block.  Prepared tensors bit-exact, O within 5e-3, the zero head's O
    exactly 0."""
    B, H, S = 1, 3, 700                      # nb = 6, tail block of 60 tokens
    q, k, v = inputs(B, H, S, seed=2400)
    v[0, :, 0] = 0                           # head 0: V all zero
    k[0, 256:384, 1] = 0                     # head 1: K block 2 zero
    q[0, 128:256, 1] = 0                     # head 1: Q block 1 zero
    q[0, 640:, 2] = 0                        # head 2: the ragged tail block of Q, K and V zero
    k[0, 640:, 2] = 0
    v[0, 640:, 2] = 0
    ref = oracle_prep(q, k, v)
    prep = ovc.prepare(*to_dev(q, k, v))
    torch.cuda.synchronize()
    assert np.array_equal(prep.q_codes().cpu().numpy(), ref.qc)
    assert np.array_equal(prep.k_codes().cpu().numpy(), ref.kc)
    assert np.array_equal(prep.q_scales().cpu().numpy(), ref.sq)
    assert np.array_equal(prep.k_scales().cpu().numpy(), ref.sk)
    assert np.array_equal(prep.v_scales().cpu().numpy(), ref.sv)
    assert np.array_equal(prep.vt_codes().cpu().numpy().transpose(0, 1, 3, 2), ref.vc)
    assert np.array_equal(prep.energy().cpu().numpy().view(np.uint32), ref.energy.view(np.uint32))
    assert ref.sv[0, 0] == 1.0 and ref.sk[0, 1, 2] == 1.0 and ref.sq[0, 1, 1] == 1.0 and ref.sq[0, 2, 5] == 1.0
    want, _ = oracle.attention_full(ref)
    o = ovc.attention_prepared(prep)
    assert ovc.device_status() == 0
    got = o.float().cpu().numpy()
    assert not got[0, :, 0].any()
    assert rel_l2(got, want) <= TOL_REL_L2
    # the zero Q block's rows: every score is 0, so each row is the mean of V's rows
    assert rel_l2(got[0, 128:256, 1], want[0, 128:256, 1]) <= TOL_REL_L2


@pytest.mark.parametrize("sm,qb,kb", [(1.0, 2, 3), (2.5, 0, 4), (1.0, 5, 5)])
def test_sharp_rows_p_codes_and_output(sm, qb, kb):
    """A large softmax scale makes rows sharp: most codes are 0 or
    subnormal and the reference moves late in the traversal.  P bytes are
    within one code of the oracle's under the device's reference, and O is
    within 5e-3."""
    B, H, S = 1, 2, 700
    q, k, v = inputs(B, H, S, seed=2500)
    ref = oracle_prep(q, k, v)
    prep = ovc.prepare(*to_dev(q, k, v))
    bh = 1
    o, codes, m8 = ovc.attention_probe(prep, softmax_scale=sm, dump=(bh, qb, kb))
    assert ovc.device_status() == 0
    codes, m8 = codes.cpu().numpy(), m8.cpu().numpy()
    small = 0
    for r in [r for r in range(128) if qb * 128 + r < S]:
        want = oracle.block_codes(ref, bh, qb * 128 + r, kb, float(m8[r]), sm=sm)
        assert np.abs(codes[r].astype(int) - want.astype(int)).max() <= 1
        small += int((want < 8).sum())
    assert small > 0.5 * 128 * min(128, S - qb * 128)       # the rows are sharp
    want, res = oracle.attention_full(ref, sm=sm)
    assert res["nres"][:, 0].max() >= 2                     # some rows rescale after the first block
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2


def test_tail_block_codes_with_a_repair_set():
    """The ragged last key block's P bytes, dumped from a call with a repair
    set: within one code of the oracle's under the device reference, and 0
    past the last key; the repaired output within 5e-3."""
    B, H, S, budget = 1, 2, 1000, 0.02        # nb = 8, last block 104 keys
    q, k, v = inputs(B, H, S, seed=2600)
    ref = oracle_prep(q, k, v)
    rr = oracle.Repair(ref, budget)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd)
    rep = ovc.prepare_v_repair(vd, prep, budget)
    nb = (S + 127) // 128
    for bh, qb in ((0, nb - 1), (1, 3)):
        o, codes, m8 = ovc.attention_probe(prep, rep, dump=(bh, qb, nb - 1))
        assert ovc.device_status() == 0
        codes, m8 = codes.cpu().numpy(), m8.cpu().numpy()
        rows = [r for r in range(128) if qb * 128 + r < S]
        for r in rows:
            want = oracle.block_codes(ref, bh, qb * 128 + r, nb - 1, float(m8[r]))
            assert np.abs(codes[r].astype(int) - want.astype(int)).max() <= 1
            assert not codes[r, S - (nb - 1) * 128:].any()
    want, _ = oracle.attention_full(ref, repair=rr)
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2


# ---- Q smoothing ---------------------------------------------------------------
def _check_key_bias(prep, ref):
    """The prepared key bias rows: (hi, lo, hi, lo, 0, ...) per key, zero
    past S, and hi + lo the oracle's beta_t = mu_q . dec(k_t) within the FP32
    rounding of a 128-term dot product plus the BF16 split (2^-16)."""
    kb = prep.key_bias().float().cpu().numpy().astype(np.float64)       # [B,H,S_pad,16]
    S = ref.S
    assert np.array_equal(kb[..., 2], kb[..., 0]) and np.array_equal(kb[..., 3], kb[..., 1])
    assert not kb[..., 4:].any() and not kb[:, :, S:].any()
    beta = kb[:, :, :S, 0] + kb[:, :, :S, 1]
    tab = oracle.e4m3_table()
    mag = np.einsum("bhtd,bhd->bht", np.abs(tab[ref.kc[:, :, :S]]), np.abs(ref.qmean.astype(np.float64)))
    assert np.all(np.abs(beta - ref.kbias) <= 2.0 ** -16 * np.abs(ref.kbias) + 2.0 ** -15 * mag + 1e-30)


@pytest.mark.parametrize("B,H,S,fp16,smooth_k", [(1, 2, 1000, False, True), (2, 1, 300, True, False),
                                                  (1, 1, 1, False, False), (1, 3, 129, False, True),
                                                  (1, 2, 1024, False, False)])
def test_q_smoothing_matches_oracle(B, H, S, fp16, smooth_k):
    """prepare(smooth_q=True): Q codes and scales bit-exact (the channel means
    are FP32 sums in a fixed order), the key bias rows within their rounding
    bound, O within 5e-3 of the oracle's Q-smoothed attention, and both
    schedules bit for bit."""
    q, k, v = inputs(B, H, S, seed=2700 + S)
    if fp16:
        q, k, v = (x.to(torch.float16) for x in (q, k, v))
    bits = [x.contiguous().view(torch.int16).numpy().view(np.uint16) for x in (q, k, v)]
    ref = oracle.Prepared(*bits, fp16=fp16, smooth_k=smooth_k, smooth_q=True)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd, smooth_k=smooth_k, smooth_q=True)
    torch.cuda.synchronize()
    assert np.array_equal(prep.q_codes().cpu().numpy(), ref.qc)
    assert np.array_equal(prep.q_scales().cpu().numpy(), ref.sq)
    assert np.array_equal(prep.k_codes().cpu().numpy(), ref.kc)
    assert np.array_equal(prep.k_scales().cpu().numpy(), ref.sk)
    assert np.array_equal(prep.vt_codes().cpu().numpy().transpose(0, 1, 3, 2), ref.vc)
    _check_key_bias(prep, ref)
    want, _ = oracle.attention_full(ref)
    o = ovc.attention_prepared(prep)
    assert ovc.device_status() == 0
    got = o.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_l2(got, want) <= TOL_REL_L2
    a, _, _ = ovc.attention_probe(prep, force_persistent=1)
    b, _, _ = ovc.attention_probe(prep, force_persistent=-1)
    assert torch.equal(a, b) and torch.equal(a, o)
    if S > 1:                                   # without the bias the output is clearly another one
        plain_q = oracle.Prepared(*bits, fp16=fp16, smooth_k=smooth_k)
        assert rel_l2(got, oracle.attention_full(plain_q)[0]) < 0.5


@pytest.mark.parametrize("S,qb,kb", [(1000, 3, 5), (1000, 7, 7), (300, 0, 2)])
def test_q_smoothing_p_codes_under_device_reference(S, qb, kb):
    q, k, v = inputs(1, 2, S, seed=2800 + S)
    ref = oracle.Prepared(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), smooth_q=True)
    prep = ovc.prepare(*to_dev(q, k, v), smooth_q=True)
    _, codes, m8 = ovc.attention_probe(prep, dump=(1, qb, kb))
    codes, m8 = codes.cpu().numpy(), m8.cpu().numpy()
    diffs = []
    for r in [r for r in range(128) if qb * 128 + r < S]:
        want = oracle.block_codes(ref, 1, qb * 128 + r, kb, float(m8[r]))
        d = np.abs(codes[r].astype(int) - want.astype(int))
        assert d.max() <= 1, (r, d.max())
        diffs.append(d)
    assert float(np.mean(np.concatenate(diffs) == 0)) > 0.99
    assert ovc.device_status() == 0


@pytest.mark.parametrize("budget", [0.02, 1.0])
def test_q_smoothing_with_repair_split_and_variants(budget):
    """Q smoothing with V residual repair (the selected keys carry their
    bias rows), with split key ranges and with the exp-then-cast baseline."""
    B, H, S = 1, 2, 1100
    q, k, v = inputs(B, H, S, seed=2900)
    ref = oracle.Prepared(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), smooth_q=True, smooth_k=True)
    rr = oracle.Repair(ref, budget)
    qd, kd, vd = to_dev(q, k, v)
    prep = ovc.prepare(qd, kd, vd, smooth_q=True, smooth_k=True)
    rep = ovc.prepare_v_repair(vd, prep, budget)
    torch.cuda.synchronize()
    assert np.array_equal(rep.idx().cpu().numpy(), rr.idx)
    n = rr.n
    kbs = _abi_view_kb_sel(rep)
    kbp = prep.key_bias()
    for h in range(H):
        assert torch.equal(kbs[0, h, :n], kbp[0, h, torch.from_numpy(rr.idx[0, h]).long().cuda()])
    assert not kbs[0, :, n:].float().any()
    want, _ = oracle.attention_full(ref, repair=rr)
    o = ovc.attention_v_repair(prep, rep)
    assert ovc.device_status() == 0
    assert rel_l2(o.float().cpu().numpy(), want) <= TOL_REL_L2
    if budget < 1.0:
        want3, _ = oracle.attention_full(ref, nsplit=3)
        assert rel_l2(ovc.attention_prepared(prep, nsplit=3).float().cpu().numpy(), want3) <= TOL_REL_L2
        wantb, _ = oracle.attention_full(ref, cast=True, mid_window=False)
        assert rel_l2(ovc.attention_prepared(prep, flags=3).float().cpu().numpy(), wantb) <= TOL_REL_L2
    with pytest.raises(ValueError):
        ovc.prepare(qd, kd, vd, smooth_q=True, v_smooth=True)
    assert ovc.device_status() == 0


def _abi_view_kb_sel(rep):
    d = rep.desc
    off = d.kb_sel - rep.workspace.data_ptr()
    return rep.workspace[off:off + 32 * d.B * d.H * d.n_pad].view(torch.bfloat16).view(d.B, d.H, d.n_pad, 16)


def test_q_smoothing_lowers_error_on_biased_queries():
    """On the workloads' per-channel Q/K bias, smoothing Q as well as K
    brings the GPU output closer to exact softmax attention."""
    B, H, S = 1, 2, 2048
    q, k, v = inputs(B, H, S, seed=3000)
    qf, kf, vf = (x.to(torch.float64).numpy() for x in (q, k, v))
    rows = np.arange(0, S, 13)
    errs = []
    for sq in (False, True):
        o = ovc.attention(*to_dev(q, k, v), smooth_k=True, smooth_q=sq).double().cpu().numpy()
        num = den = 0.0
        for h in range(H):
            s = (qf[0, rows, h] @ kf[0, :, h].T) / math.sqrt(128.0)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            ex = (p @ vf[0, :, h]) / p.sum(axis=1, keepdims=True)
            num += np.sum((o[0, rows, h] - ex) ** 2)
            den += np.sum(ex ** 2)
        errs.append(math.sqrt(num / den))
    assert errs[1] < 0.95 * errs[0], errs
