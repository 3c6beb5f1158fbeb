"""The library's failure paths, made to run without faulting the GPU.

* A bounded wait that gives up: with rl_kv_set_wait_limit(kv, 1) the
  persistent step kernel's grid-wide phase barrier (batch 1) and the
  tensor-core GEMM's first accumulator wait (batch 16, generic path) give up
  at once; the step must end (the kernels drain their own copies and tensor
  memory), rl_sync must report RL_ERR_DEVICE with the timeout bit, and after
  the limit is restored and the position rewound the same step must match
  the oracle again, and so must the next one.
* An allocation that fails: rl_debug_fail_allocations(n) lets n library
  allocations succeed and fails the next; every allocating entry point must
  return RL_ERR_OOM at every such point, free what it had taken (device free
  memory returns to where it was) and leave earlier objects usable.
"""
import numpy as np
import pytest

import synth
from oracle.model import KVState, Policy as OPolicy
from tests.harness import build_pair, check_step, to_cuda

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TINY = synth.TINY


@pytest.fixture(scope="module")
def river():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import early_exit_decoding_gb300 as r
    yield r
    r.rl_debug_fail_allocations(-1)


@pytest.fixture(scope="module")
def stream(river):
    return torch.cuda.Stream()


@pytest.fixture(scope="module")
def tiny(river, stream):
    with torch.cuda.stream(stream):
        m, om, w = build_pair(TINY, seed=0, gains="random", stream=stream)
    stream.synchronize()
    return m, om, w


@pytest.mark.parametrize("B,path", [(1, 1), (16, 3)])
def test_wait_that_gives_up_is_reported_and_the_step_can_be_redone(river, tiny, stream, B, path):
    m, om, _ = tiny
    S = TINY
    kv = m.kv_cache_alloc(B, 64)
    kv.set_decode_path(path)
    assert kv.decode_path(B) == path
    st = KVState(S, B, 64)
    toks = synth.gen_tokens(S.vocab, (B, 20), seed=1)
    sched = torch.tensor([2], dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        river.prefill(m, kv, torch.from_numpy(toks).cuda(), river.Policy.tau_(1.01), stream=stream)
        kv.sync(stream)
        ref = om.prefill(toks, st, OPolicy.tau_(1.01))
        nxt = ref.logits.argmax(-1).astype(np.int32)
        tin = torch.from_numpy(nxt.copy()).cuda()
        p, s_idx = kv.position()
        river.rl_kv_set_wait_limit(kv.handle, 1)
        status = None
        for _ in range(3):  # the first try practically always gives up; a few for certainty
            kv.set_position(p, s_idx, stream)
            river.decode_step(m, kv, tin, river.Policy.forced(sched), stream=stream)
            try:
                kv.sync(stream)
            except river.RiverError as ex:
                status = ex
                break
        assert status is not None, "no wait gave up"
        assert status.status == river.RL_ERR_DEVICE and "timed out" in str(status)
        # the context is usable: restore the limit, rewind, redo the step
        river.rl_kv_set_wait_limit(kv.handle, 0)
        kv.set_position(p, s_idx, stream)
        for i in range(2):
            out = river.decode_step(m, kv, torch.from_numpy(nxt.copy()).cuda(),
                                    river.Policy.forced(sched), stream=stream)
            kv.sync(stream)
            ref = om.decode_step(nxt, st, OPolicy.forced(2))
            assert int(out["exit_layer"].item()) == 2
            check_step(out, ref, None, B, f"after the timeout, step {i}")
            nxt = ref.logits.argmax(-1).astype(np.int32)


def _free():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def _sweep(river, call, limit=200):
    """Fail allocation n for n = 0, 1, ... until the call succeeds; every
    failing call must raise RL_ERR_OOM.  Returns the successful result and
    how many allocations it made."""
    for n in range(limit):
        river.rl_debug_fail_allocations(n)
        try:
            r = call()
        except river.RiverError as ex:
            assert ex.status == river.RL_ERR_OOM, ex
            assert "injected" in str(ex)
            continue
        finally:
            river.rl_debug_fail_allocations(-1)
        return r, n
    raise AssertionError("the call never succeeded")


def test_injected_allocation_failures_leak_nothing(river, stream):
    w = synth.gen_weights(TINY, seed=0, device="cpu", gains="random")
    wd = to_cuda(w)
    base = _free()
    m, n_model = _sweep(river, lambda: river.Model(TINY, wd, stream))
    assert n_model > 3
    assert river.rl_quantize_exit_layers is not None
    _, n_q = _sweep(river, lambda: m.quantize_exit_layers(stream))
    after_model = _free()
    for _ in range(2):  # twice: a leak per failed call would grow
        kv, n_kv = _sweep(river, lambda: m.kv_cache_alloc(4, 64))
        assert n_kv > 10
        kv.close()
        assert _free() == after_model, "a failed rl_kv_cache_alloc leaked device memory"
    # prefill's workspace: the call fails cleanly and the cache stays usable
    kv = m.kv_cache_alloc(2, 64)
    toks = torch.from_numpy(synth.gen_tokens(TINY.vocab, (2, 16), seed=1)).cuda()
    river.rl_debug_fail_allocations(0)
    try:
        with pytest.raises(river.RiverError) as ei:
            river.prefill(m, kv, toks, river.Policy.tau_(1.01), stream=stream)
        assert ei.value.status == river.RL_ERR_OOM
    finally:
        river.rl_debug_fail_allocations(-1)
    with torch.cuda.stream(stream):
        out = river.prefill(m, kv, toks, river.Policy.tau_(1.01), stream=stream)
        kv.sync(stream)
    assert np.isfinite(out["logits"].cpu().numpy()).all()
    kv.close()
    m.close()
    del wd
    torch.cuda.empty_cache()
    assert _free() >= base - (4 << 20), "model and caches did not give their memory back"
