"""GPU parity at the full workload sizes, in the launch configuration bench.py
times (persistent schedule for S >= 32768): sampled heads and query rows are
checked against the CPU oracle one by one.

Per sampled head: quantised Q/K/V codes, scales and energies bit-exact; output
rows within relative L2 5e-3; P bytes of one tile within one code under the
device's reference; repair indices (budgets 0.005 / 0.01 / 0.02) bit-exact and
the repaired rows within 5e-3."""
import zlib

import numpy as np
import pytest
import torch

import fp8_bit_attention_gb300 as ovc
import oracle
from fp8_bit_attention_gb300 import workloads as W

from gpu_util import TOL_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _head_view(x, b, h):
    """[1, S, 1, 128] BF16-bits view of one (batch, head) of a CPU tensor."""
    return W.bf16_bits(x)[b:b + 1, :, h:h + 1, :]


def _sample_rows(S, nb, rng, k=24):
    rows = {0, S - 1, (nb // 2) * 128, (nb - 1) * 128}
    rows |= set(rng.integers(0, S, k).tolist())
    return np.array(sorted(r for r in rows if r < S), dtype=np.int64)


@pytest.mark.parametrize("name", ["h7_s8k", "h14_s32k", "h56_s73397", "b2_h56_s36864"])
def test_full_size_sampled_parity(name):
    w = W.WORKLOADS[name]
    q, k, v = W.generate(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    prep = ovc.prepare(qd, kd, vd)
    o = ovc.attention_prepared(prep)
    reps = {bud: ovc.prepare_v_repair(vd, prep, bud) for bud in (0.005, 0.01, 0.02)}
    o_rep = ovc.attention_v_repair(prep, reps[0.005])
    assert ovc.device_status() == 0
    torch.cuda.synchronize()
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    B, H, S = w.B, w.H, w.S
    nb = (S + 127) // 128
    heads = sorted({(0, 0), (B - 1, H - 1), (int(rng.integers(B)), int(rng.integers(H)))})
    o_cpu = o.float().cpu().numpy()
    orep_cpu = o_rep.float().cpu().numpy()
    for b, h in heads:
        ref = oracle.Prepared(_head_view(q, b, h), _head_view(k, b, h), _head_view(v, b, h))
        # quantised tensors of this head, bit-exact
        assert np.array_equal(prep.q_codes()[b, h].cpu().numpy(), ref.qc[0, 0])
        assert np.array_equal(prep.k_codes()[b, h].cpu().numpy(), ref.kc[0, 0])
        assert np.array_equal(prep.vt_codes()[b, h].cpu().numpy().T, ref.vc[0, 0])
        assert np.array_equal(prep.q_scales()[b, h].cpu().numpy(), ref.sq[0, 0])
        assert np.array_equal(prep.k_scales()[b, h].cpu().numpy(), ref.sk[0, 0])
        assert prep.v_scales()[b, h].item() == ref.sv[0, 0]
        assert np.array_equal(prep.energy()[b, h].cpu().numpy().view(np.uint32),
                              ref.energy[0, 0].view(np.uint32))
        # sampled output rows
        rows = _sample_rows(S, nb, rng)
        r = oracle.attention_rows(ref, np.zeros_like(rows), rows)
        got = o_cpu[b, rows, h, :]
        assert np.isfinite(got).all()
        assert rel_l2(got, r["out"]) <= TOL_REL_L2, (name, b, h)
        # P bytes of one tile under the device reference
        qb, kb = int(rng.integers(nb)), int(rng.integers(nb))
        _, codes, m8 = ovc.attention_probe(prep, dump=(b * H + h, qb, kb))
        codes, m8 = codes.cpu().numpy(), m8.cpu().numpy()
        for row in range(0, 128, 9):
            if qb * 128 + row >= S:
                continue
            want = oracle.block_codes(ref, 0, qb * 128 + row, kb, float(m8[row]))
            assert np.abs(codes[row].astype(int) - want.astype(int)).max() <= 1
        # repair: indices bit-exact for every budget, repaired rows at 0.005
        for bud, rep in reps.items():
            rr = oracle.Repair(ref, bud)
            assert np.array_equal(rep.idx()[b, h].cpu().numpy(), rr.idx[0, 0]), (name, bud)
            assert rep.sr()[b, h].item() == rr.sr[0, 0]
            if bud == 0.005:
                want = oracle.attention_rows(ref, np.zeros_like(rows), rows, repair=rr)["out"]
                assert rel_l2(orep_cpu[b, rows, h, :], want) <= TOL_REL_L2
    del qd, kd, vd, prep, o, o_rep, reps
    torch.cuda.empty_cache()
