"""The host-built per-SM schedule (ll_plan, no GPU needed): every matrix row and
every (KV head, split) attention item is assigned exactly once per layer, every
wait names a counter that exactly that many completions bump, and the lists run
to completion when executed in order against those counters (no deadlock)."""
import numpy as np
import pytest

from decode_megakernel_persistent_gb300 import build as llbuild
from decode_megakernel_persistent_gb300 import ll, synth

QKV, ATTN, OPROJ, GATEUP, DOWN, LMHEAD = range(6)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    llbuild.build()


def coverage(intervals, total):
    cover = np.zeros(total, dtype=np.int32)
    for a, b in intervals:
        assert 0 <= a <= b <= total
        cover[a:b] += 1
    return cover


@pytest.mark.parametrize("key", sorted(synth.WORKLOADS))
@pytest.mark.parametrize("nsm", [148, 152, 160])
def test_rows_and_items_assigned_once(key, nsm):
    shape = synth.WORKLOADS[key].shape
    max_seq = synth.WORKLOADS[key].context + 200
    plan = ll.ll_plan(ll.make_config(shape, max_seq), nsm)
    qd, kd = shape.q_dim, shape.kv_dim
    S = max(1, min(-(-max_seq // 128), nsm // shape.n_kv_heads))
    rows = {QKV: qd + 2 * kd, OPROJ: shape.hidden, GATEUP: shape.inter, DOWN: shape.hidden}
    for l in range(shape.n_layers):
        for op, total in rows.items():
            m = (plan[:, :, 0] == op) & (plan[:, :, 1] == l)
            assert m.sum() == nsm
            assert np.all(coverage(zip(plan[:, :, 2][m], plan[:, :, 3][m]), total) == 1)
        m = (plan[:, :, 0] == ATTN) & (plan[:, :, 1] == l)
        items = sorted(zip(plan[:, :, 2][m].tolist(), plan[:, :, 3][m].tolist()))
        assert items == [(g, c) for g in range(shape.n_kv_heads) for c in range(S)]
    m = plan[:, :, 0] == LMHEAD
    assert np.all(coverage(zip(plan[:, :, 2][m], plan[:, :, 3][m]), shape.vocab) == 1)


@pytest.mark.parametrize("key", sorted(synth.WORKLOADS))
def test_waits_match_signals_and_lists_complete(key):
    shape = synth.WORKLOADS[key].shape
    nsm = 152
    plan = ll.ll_plan(ll.make_config(shape, synth.WORKLOADS[key].context + 200), nsm)
    # completions that bump each counter per step
    bumps = {}
    for sm in range(nsm):
        for ins in plan[sm]:
            if ins[0] < 0 or ins[6] < 0:
                continue
            bumps[ins[6]] = bumps.get(ins[6], 0) + 1
    for sm in range(nsm):
        for ins in plan[sm]:
            if ins[0] >= 0 and ins[4] >= 0:
                assert bumps[ins[4]] == ins[5], (key, ins.tolist())
    # run every list in order; an instruction runs once its counter has its count
    ctr = {}
    pc = [0] * nsm
    progress = True
    while progress:
        progress = False
        for sm in range(nsm):
            while pc[sm] < plan.shape[1] and plan[sm, pc[sm], 0] >= 0:
                ins = plan[sm, pc[sm]]
                if ins[4] >= 0 and ctr.get(ins[4], 0) < ins[5]:
                    break
                if ins[6] >= 0:
                    ctr[ins[6]] = ctr.get(ins[6], 0) + 1
                pc[sm] += 1
                progress = True
    for sm in range(nsm):
        assert pc[sm] == plan.shape[1] or plan[sm, pc[sm], 0] < 0, f"SM {sm} stuck at {pc[sm]}"


def test_plan_rejects_bad_arguments():
    cfg = ll.make_config(synth.TINY, 16)
    with pytest.raises(ll.LLError):
        ll.ll_plan(cfg, 0)
