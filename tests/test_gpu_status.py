"""GPU error paths: every failure is reported through a return code or the
device status word, the context stays usable, and later runs are correct.
No test here faults, traps or hangs the GPU: the timeout tests make a
bounded wait run out, either on a flag that nothing sets (a test switch of
the library) or by a zero wait limit, and the kernels return after draining
their own copies in flight."""
import numpy as np
import pytest
import torch

import spec_inputs as si
import speculative_decoding_verification_22_gb300 as sv
from gpu_common import compare_tokens, flagged, gpu_verify, oracle_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    # V = 9000: three residual chunks per sequence, so that the selection's
    # wait for the other chunks' masses is a wait that a zero limit ends
    wl = si.workload("tiny", dtype="bf16", B=3, K=4, V=9000, d=512, w_std=1 / 22.6)
    W = si.make_weights(wl, seed=5, device=dev)
    inp = si.make_round(wl, W, seed=6)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    yield dev, wl, W, si.to_oracle(W), inp, eng
    eng.close()


def _check_ok(eng, W, W_np, inp, T=1.0):
    got = gpu_verify(eng, W, inp, T)
    assert got["status"] == sv.SV_OK
    ref = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"], inp["uniforms"], T)
    assert compare_tokens(got, ref, T)[0] == 0


def test_out_of_range_draft_token(setup):
    dev, wl, W, W_np, inp, eng = setup
    bad = dict(inp)
    bad["draft"] = inp["draft"].clone()
    bad["draft"][1, 2] = wl.V          # sequence 1 invalid
    got = gpu_verify(eng, W, bad, 1.0)
    assert got["status"] == sv.SV_ERR_TOKEN
    assert got["n_accepted"][1] == -1 and np.all(got["tokens"][1] == -1)
    ref = oracle_verify(bad["hidden"], W_np, bad["draft"], bad["q_logits"], bad["uniforms"], 1.0)
    assert ref["n_accepted"][1] == -1
    for b in (0, 2):
        assert np.array_equal(got["tokens"][b], ref["tokens"][b])
    _check_ok(eng, W, W_np, inp)


def test_misaligned_and_bad_arguments_are_rejected_on_the_host(setup):
    dev, wl, W, W_np, inp, eng = setup
    out_t = torch.empty((wl.B, wl.K + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((wl.B,), dtype=torch.int32, device=dev)
    q_off = torch.empty(inp["q_logits"].numel() + 1, device=dev)[1:].view_as(inp["q_logits"])
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_run(eng.h, inp["hidden"], W, inp["draft"], q_off, inp["uniforms"],
                           1.0, out_t, out_n)
    assert e.value.code == sv.SV_ERR_ALIGN
    for T in (float("nan"), -1.0, float("inf")):
        with pytest.raises(sv.SpecVerifyError) as e:
            sv.spec_verify_run(eng.h, inp["hidden"], W, inp["draft"], inp["q_logits"],
                               inp["uniforms"], T, out_t, out_n)
        assert e.value.code == sv.SV_ERR_ARG
    # sampling needs the uniforms (q_logits may be NULL: point-mass drafts)
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_run(eng.h, inp["hidden"], W, inp["draft"], inp["q_logits"], None,
                           1.0, out_t, out_n)
    assert e.value.code == sv.SV_ERR_ARG
    assert eng.status() == sv.SV_OK
    _check_ok(eng, W, W_np, inp)


def test_non_finite_weights_are_reported(setup):
    dev, wl, W, W_np, inp, eng = setup
    Wbad = W.clone()
    Wbad[17, 3] = float("inf")
    for T in (1.0, 0.0):
        got = gpu_verify(eng, Wbad, inp, T)
        assert got["status"] == sv.SV_ERR_NONFINITE
        assert np.all(got["n_accepted"] == -1)
    _check_ok(eng, W, W_np, inp)


def test_a_wait_that_runs_out_is_reported_and_recovers(setup):
    """A bounded device-side wait that runs out.  With the test stall on,
    each run's decision/selection kernel first waits for a flag that nothing
    sets; after the wait limit (1 ms here) the run reports SV_ERR_TIMEOUT
    and withdraws sequence 0, the others come out as the oracle has them,
    and once the stall is off and the limit restored every run is right."""
    dev, wl, W, W_np, inp, eng = setup
    ref = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"], inp["uniforms"], 1.0)
    fl = flagged(ref, 1.0)
    sv.spec_verify_set_wait_limit(eng.h, 1_000_000)
    sv.spec_verify_debug_stall(eng.h, True)
    try:
        for _ in range(3):
            got = gpu_verify(eng, W, inp, 1.0)
            assert got["status"] == sv.SV_ERR_TIMEOUT
            assert got["n_accepted"][0] == -1 and np.all(got["tokens"][0] == -1)
            for b in range(1, wl.B):
                same = np.array_equal(got["tokens"][b], ref["tokens"][b]) and \
                    got["n_accepted"][b] == ref["n_accepted"][b]
                assert same or fl[b]
    finally:
        sv.spec_verify_debug_stall(eng.h, False)
        sv.spec_verify_set_wait_limit(eng.h, 1_000_000_000)
    for _ in range(3):
        _check_ok(eng, W, W_np, inp)


def test_wait_limit_zero_never_draws_from_partial_results(setup):
    """With a zero limit the first wait that is not already satisfied gives
    up.  Which waits that hits depends on timing (a wait satisfied at its
    first poll does not time out, and the run may then succeed), so each
    sequence must come out either withdrawn (-1 throughout, with the status
    SV_ERR_TIMEOUT) or exactly as the oracle has it; never a token drawn
    from partial results.  Runs after it are right again."""
    dev, wl, W, W_np, inp, eng = setup
    ref = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"], inp["uniforms"], 1.0)
    fl = flagged(ref, 1.0)
    sv.spec_verify_set_wait_limit(eng.h, 0)
    try:
        for _ in range(5):
            got = gpu_verify(eng, W, inp, 1.0)
            assert got["status"] in (sv.SV_OK, sv.SV_ERR_TIMEOUT)
            for b in range(wl.B):
                if got["n_accepted"][b] == -1:
                    assert np.all(got["tokens"][b] == -1)
                    assert got["status"] == sv.SV_ERR_TIMEOUT
                else:
                    same = np.array_equal(got["tokens"][b], ref["tokens"][b]) and \
                        got["n_accepted"][b] == ref["n_accepted"][b]
                    assert same or fl[b]
    finally:
        sv.spec_verify_set_wait_limit(eng.h, 1_000_000_000)
    for _ in range(3):
        _check_ok(eng, W, W_np, inp)


def test_run_host_matches_device_run(setup):
    dev, wl, W, W_np, inp, eng = setup
    tok_d, n_d = eng.run(inp["hidden"], W, inp["draft"], inp["q_logits"], inp["uniforms"], 1.0)
    host = {k: inp[k].cpu().pin_memory() for k in ("hidden", "draft", "q_logits", "uniforms")}
    ht = torch.empty((wl.B, wl.K + 1), dtype=torch.int32).pin_memory()
    hn = torch.empty((wl.B,), dtype=torch.int32).pin_memory()
    sv.spec_verify_run_host(eng.h, host["hidden"], W, host["draft"], host["q_logits"],
                            host["uniforms"], 1.0, ht, hn)
    assert torch.equal(ht, tok_d.cpu()) and torch.equal(hn, n_d.cpu())
    assert eng.status() == sv.SV_OK


def test_double_buffered_host_rounds_match_device_runs(setup):
    """spec_verify_submit_host / spec_verify_wait_host: rounds alternate
    between the two slots with different inputs each; every round's host
    outputs equal the device run on the same inputs, and a busy slot (or an
    idle one) is refused."""
    dev, wl, W, W_np, inp, eng = setup
    keys = ("hidden", "draft", "q_logits", "uniforms")
    rounds = [si.make_round(wl, W, seed=300 + i) for i in range(6)]
    host = [{k: r[k].cpu().pin_memory() for k in keys} for r in rounds]
    ht = [torch.empty((wl.B, wl.K + 1), dtype=torch.int32).pin_memory() for _ in range(2)]
    hn = [torch.empty((wl.B,), dtype=torch.int32).pin_memory() for _ in range(2)]
    got = []
    for i, hbuf in enumerate(host):
        s = i % 2
        if i >= 2:
            assert sv.spec_verify_wait_host(eng.h, s) == sv.SV_OK
            got.append((ht[s].clone(), hn[s].clone()))
        sv.spec_verify_submit_host(eng.h, s, hbuf["hidden"], W, hbuf["draft"], hbuf["q_logits"],
                                   hbuf["uniforms"], 1.0, ht[s], hn[s])
        if i == 0:
            with pytest.raises(sv.SpecVerifyError) as e:
                sv.spec_verify_submit_host(eng.h, 0, hbuf["hidden"], W, hbuf["draft"],
                                           hbuf["q_logits"], hbuf["uniforms"], 1.0, ht[0], hn[0])
            assert e.value.code == sv.SV_ERR_ARG
    for s in (0, 1):
        assert sv.spec_verify_wait_host(eng.h, s) == sv.SV_OK
        got.append((ht[s].clone(), hn[s].clone()))
    assert sv.spec_verify_wait_host(eng.h, 0) == sv.SV_ERR_ARG
    for r, (t, n) in zip(rounds, got):
        ref_t, ref_n = eng.run(r["hidden"], W, r["draft"], r["q_logits"], r["uniforms"], 1.0)
        assert torch.equal(t, ref_t.cpu()) and torch.equal(n, ref_n.cpu())
    assert eng.status() == sv.SV_OK
