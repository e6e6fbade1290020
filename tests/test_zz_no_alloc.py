"""The allocation-free entry point, spec_verify_run_noalloc.

Some callers cannot allocate device memory at the moment they call in: a
serving runtime that plans every device buffer up front and forbids
cudaMalloc on its request path (cudaMalloc may synchronise the device and
fragments a caching allocator), or a plugin host that passes the library
nothing but input and output pointers.  For them the library offers an
entry point without a handle whose scratch lives in a fixed device array
inside the library.  These tests call it through the C ABI and require its
outputs to equal those of the handle-based spec_verify_run on the same
inputs, for two calls in a row (the second call finds the first call's data
still in the array), and to equal the CPU oracle's outside flagged rounds.
They also check its error contract: a bad draft token spoils only its own
sequence (outputs -1, no status word), and the next call is right again.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import spec_inputs as si
import speculative_decoding_verification_22_gb300 as sv
from gpu_common import compare_tokens, oracle_verify

pytestmark = pytest.mark.gpu


def _noalloc_call(wl, inp, W, T, out_t, out_n):
    cfg = sv.sv_config_t(wl.V, wl.d, wl.B, wl.K, sv.SV_BF16 if wl.dtype == "bf16" else sv.SV_FP32,
                         torch.cuda.current_stream().cuda_stream)
    p = lambda t: None if t is None else t.data_ptr()
    return sv.load_library().spec_verify_run_noalloc(
        ctypes.byref(cfg), p(inp["hidden"]), p(W), p(inp["draft"]), p(inp["q_logits"]),
        p(inp["uniforms"]), float(T), p(out_t), p(out_n))


@pytest.mark.parametrize("name,over,T", [
    ("llama8b", {}, 1.0),
    ("llama8b", {}, 0.0),
    ("tiny", {}, 1.0),
    ("tiny", dict(dtype="bf16", B=8, K=3, V=5000, d=1024, w_std=1 / 32), 0.7),
    # an odd number of 64-wide k blocks (single-block TMA stages) and a
    # vocabulary that is not a multiple of 4 (logits stored lane by lane)
    ("tiny", dict(dtype="bf16", B=2, K=3, V=4999, d=960, w_std=1 / 31), 1.0),
])
def test_noalloc_matches_the_handle_path_twice_in_a_row(name, over, T):
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl = si.workload(name, **over)
    W = si.make_weights(wl, seed=77, device=dev)
    W_np = si.to_oracle(W)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    for call in range(2):
        inp = si.make_round(wl, W, seed=500 + call, T=T)
        ref_t, ref_n = eng.run(inp["hidden"], W, inp["draft"], inp["q_logits"],
                               inp["uniforms"], T)
        assert eng.status() == sv.SV_OK
        out_t = torch.full((wl.B, wl.K + 1), -7, dtype=torch.int32, device=dev)
        out_n = torch.full((wl.B,), -7, dtype=torch.int32, device=dev)
        assert _noalloc_call(wl, inp, W, T, out_t, out_n) == sv.SV_OK
        torch.cuda.synchronize()
        # token ids and accept counts are compared exactly, as everywhere
        assert torch.equal(out_t, ref_t), (call, out_t, ref_t)
        assert torch.equal(out_n, ref_n), (call, out_n, ref_n)
        assert bool((out_n >= 0).all())
        # and the oracle, on the same inputs (flagged rounds excepted)
        ref = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"],
                            inp["uniforms"], T)
        got = {"tokens": out_t.cpu().numpy(), "n_accepted": out_n.cpu().numpy()}
        assert compare_tokens(got, ref, T)[0] == 0, call
    eng.close()


def test_noalloc_rejects_shapes_beyond_its_array():
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl = si.workload("sweep", B=64, K=5)   # 384 rows of 128256 fp32 logits
    small = si.workload("tiny", dtype="bf16", B=1, K=1, V=1000, d=64)
    W = si.make_weights(small, seed=1, device=dev)
    inp = si.make_round(small, W, seed=2)
    out_t = torch.empty((wl.B, wl.K + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((wl.B,), dtype=torch.int32, device=dev)
    # the shape check comes before any pointer is touched
    assert _noalloc_call(wl, inp, W, 1.0, out_t, out_n) == sv.SV_ERR_SHAPE


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_noalloc_bad_token_spoils_only_its_sequence(T):
    # No status word on this path: a draft token outside [0, V) marks its
    # own sequence -1, the others are verified as usual, and the next call
    # (which finds the failed call's counters in the array) is right again.
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl = si.workload("tiny", dtype="bf16", B=4, K=4, V=3000, d=256, w_std=1 / 16)
    W = si.make_weights(wl, seed=81, device=dev)
    W_np = si.to_oracle(W)
    inp = si.make_round(wl, W, seed=82, T=T)
    bad = dict(inp)
    bad["draft"] = inp["draft"].clone()
    bad["draft"][2, 1] = wl.V
    out_t = torch.full((wl.B, wl.K + 1), -7, dtype=torch.int32, device=dev)
    out_n = torch.full((wl.B,), -7, dtype=torch.int32, device=dev)
    assert _noalloc_call(wl, bad, W, T, out_t, out_n) == sv.SV_OK
    torch.cuda.synchronize()
    assert int(out_n[2]) == -1 and bool((out_t[2] == -1).all())
    keep = [0, 1, 3]
    ref_keep = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"],
                             inp["uniforms"], T, rows=keep)
    got = {"tokens": out_t.cpu().numpy(), "n_accepted": out_n.cpu().numpy()}
    assert compare_tokens(got, ref_keep, T, seqs=keep)[0] == 0
    ref = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"], inp["uniforms"], T)
    # the next call, valid, against the handle path and the oracle
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    ref_t, ref_n = eng.run(inp["hidden"], W, inp["draft"], inp["q_logits"], inp["uniforms"], T)
    assert eng.status() == sv.SV_OK
    assert _noalloc_call(wl, inp, W, T, out_t, out_n) == sv.SV_OK
    torch.cuda.synchronize()
    assert torch.equal(out_t, ref_t) and torch.equal(out_n, ref_n)
    got = {"tokens": out_t.cpu().numpy(), "n_accepted": out_n.cpu().numpy()}
    assert compare_tokens(got, ref, T)[0] == 0
    eng.close()
