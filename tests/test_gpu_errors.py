"""Error handling on the GPU without faulting it: host-side argument checks, a
token rejected on the device, a dependency wait that runs out because the
schedule was built without one completion signal (nothing sets the counter the
wait is for), and logits with no orderable value (no greedy token). After each
error the handle keeps working."""
import pytest

from decode_megakernel_persistent_gb300 import ll, synth
from helpers import Pair

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_megakernel_persistent_gb300 import build
    build.build()


def test_host_rejects_bad_token_and_pos():
    pr = Pair(synth.TINY, 8)
    with pytest.raises(ll.LLError) as e:
        pr.dec.step(synth.TINY.vocab, 0)
    assert e.value.code == ll.LL_ERR_ARG
    with pytest.raises(ll.LLError) as e:
        pr.dec.step(0, 8)
    assert e.value.code == ll.LL_ERR_ARG
    with pytest.raises(ll.LLError) as e:
        pr.dec.step(-1, 0)
    assert e.value.code == ll.LL_ERR_ARG
    pr.step(3, 0)
    pr.close()


@pytest.mark.parametrize("backend", [ll.LL_BACKEND_MEGAKERNEL, ll.LL_BACKEND_CHAIN])
def test_device_rejects_bad_token_then_recovers(backend):
    pr = Pair(synth.TINY, 8, backend)
    bad = torch.tensor([synth.TINY.vocab + 5], dtype=torch.int32, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    pr.dec.step_async(bad, 0, pr.logits, out)
    pr.dec.step_async(bad, 1, pr.logits, out)  # sticky: returns at once
    with pytest.raises(ll.LLError) as e:
        pr.dec.synchronize()
    assert e.value.code == ll.LL_ERR_ARG
    pr.dec.synchronize()  # cleared
    pr.step(9, 0)
    pr.step(4, 1)
    pr.close()


@pytest.mark.parametrize("op", [ll.OP_QKV, ll.OP_ATTN, ll.OP_OPROJ, ll.OP_GATEUP, ll.OP_DOWN])
def test_dropped_signal_times_out_and_recovers(op):
    pr = Pair(synth.TINY, 8)
    pr.step(1, 0)
    ll.ll_set_timeout_ns(pr.dec.handle, 20_000_000)  # 20 ms
    ll.ll_debug_inject(pr.dec.handle, ll.LL_FAULT_DROP_SIGNAL, 1, op)
    with pytest.raises(ll.LLError) as e:
        pr.dec.step(2, 1, pr.logits)
    assert e.value.code == ll.LL_ERR_DEP_TIMEOUT
    ll.ll_debug_inject(pr.dec.handle, ll.LL_FAULT_NONE)
    ll.ll_set_timeout_ns(pr.dec.handle, 1_000_000_000)
    pr.step(2, 1)  # same position again, now complete and matching the oracle
    pr.step(5, 2)
    pr.close()


@pytest.mark.parametrize("backend", [ll.LL_BACKEND_MEGAKERNEL, ll.LL_BACKEND_CHAIN])
def test_logits_without_an_orderable_value(backend):
    # a NaN final-norm gain makes every logit NaN: there is no greedy token. A
    # single step reports LL_ERR_NUMERIC; a multi-step launch stops at the hand-off
    # of its first step's (missing) token with the same code; with the gain
    # finite again the handle decodes and matches the oracle
    pr = Pair(synth.TINY, 16, backend)
    pr.step(3, 0)
    pr.w["final_norm"].fill_(float("nan"))
    with pytest.raises(ll.LLError) as e:
        pr.dec.step(4, 1, pr.logits)
    assert e.value.code == ll.LL_ERR_NUMERIC
    toks = torch.zeros(4, dtype=torch.int32, device="cuda")
    pr.dec.steps(torch.tensor([4], dtype=torch.int32, device="cuda"), 1, 4, None, toks)
    with pytest.raises(ll.LLError) as e:
        pr.dec.synchronize()
    assert e.value.code == ll.LL_ERR_NUMERIC
    pr.w["final_norm"].fill_(1.0)
    pr.step(4, 1)
    pr.step(6, 2)
    pr.close()


@pytest.mark.parametrize("n", [2, 4])
def test_batch_logits_without_an_orderable_value(n):
    # the same in a batched launch, on CUDA-core (2) and tensor-core (4) pages
    shape = synth.ModelShape("h1024i2048", 2, 1024, 16, 4, 64, 2048, 4096, True)
    w = synth.make_weights(shape, seed=0, device="cuda")
    w["final_norm"].fill_(float("nan"))
    caches = [synth.make_kv(shape, 16, 0, seed=10 + b, device="cuda") for b in range(n)]
    dec = ll.BatchDecoder(shape, w, [c[0] for c in caches], [c[1] for c in caches], 16)
    toks = torch.zeros((3, n), dtype=torch.int32, device="cuda")
    dec.steps_batch(torch.arange(1, n + 1, dtype=torch.int32, device="cuda"), [0] * n, 3, None, toks)
    with pytest.raises(ll.LLError) as e:
        dec.synchronize()
    assert e.value.code == ll.LL_ERR_NUMERIC
    dec.close()


def test_query_reports_schedule():
    pr = Pair(synth.TINY, 8)
    h = pr.dec.handle
    nsm = ll.ll_query(h, ll.LL_Q_NUM_SMS)
    assert nsm == torch.cuda.get_device_properties(0).multi_processor_count
    assert ll.ll_query(h, ll.LL_Q_ATTN_SPLITS) == max(1, min(1, nsm // synth.TINY.n_kv_heads))  # max_seq 8
    assert ll.ll_query(h, ll.LL_Q_LAUNCHES_PER_STEP) == 1
    assert ll.ll_query(h, ll.LL_Q_PAGE_BYTES) * ll.ll_query(h, ll.LL_Q_NUM_PAGES) <= ll.ll_query(h, ll.LL_Q_SMEM_BYTES)
    pr.close()
