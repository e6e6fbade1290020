"""GPU parity of the FP8 E4M3 LM head (reading R13) against the CPU oracle
on the same quantised values: logits within 2e-2 and probabilities within
1e-5 of the oracle's exact ones, token ids and accept counts bit-exact
except flagged rounds, at a small ragged shape and at the Llama-8B shape
(sampled and greedy); and the argument checks of the FP8 entry point."""
import numpy as np
import pytest
import torch

import oracle
import spec_inputs as si
import speculative_decoding_verification_22_gb300 as sv
from gpu_common import check_numerics, compare_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _fp8_case(dev, wl, T, seed, point_mass=False):
    W8, ws = si.make_fp8_weights(wl, seed=seed, device=dev)
    inp = si.make_fp8_round(wl, W8, ws, seed=seed + 1, T=T)
    q = None if point_mass else inp["q_logits"]
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, "fp8", device=dev)
    tok, n = eng.run_fp8(inp["hidden8"], inp["h_scale"], W8, ws, inp["draft"], q,
                         inp["uniforms"], T)
    assert eng.status() == sv.SV_OK
    ref = oracle.verify_fp8(si.to_oracle(inp["hidden8"]), si.to_oracle(inp["h_scale"]),
                            si.to_oracle(W8), si.to_oracle(ws), si.to_oracle(inp["draft"]),
                            None if q is None else si.to_oracle(q),
                            si.to_oracle(inp["uniforms"]), T, want_logits=True)
    got = {"tokens": tok.cpu().numpy(), "n_accepted": n.cpu().numpy()}
    return eng, got, ref


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_fp8_parity_small(dev, T):
    wl = si.workload("tiny", dtype="bf16", V=1000, d=256, B=3, K=4, w_std=1 / 16.0)
    eng, got, ref = _fp8_case(dev, wl, T, seed=121)
    check_numerics(eng, ref, wl, T)
    bad, flagged = compare_tokens(got, ref, T)
    assert bad == 0 and flagged <= 1
    eng.close()


@pytest.mark.parametrize("B,K,T", [(1, 4, 1.0), (8, 7, 0.7), (8, 7, 0.0)])
def test_fp8_parity_llama8b(dev, B, K, T):
    wl = si.workload("llama8b", B=B, K=K, T=T)
    eng, got, ref = _fp8_case(dev, wl, T, seed=131 + B)
    dl = check_numerics(eng, ref, wl, T)
    bad, flagged = compare_tokens(got, ref, T)
    assert bad == 0 and flagged <= 1, (bad, flagged, dl)
    eng.close()


def test_fp8_point_mass_drafts(dev):
    wl = si.workload("llama8b", B=2, K=4, T=1.0)
    eng, got, ref = _fp8_case(dev, wl, 1.0, seed=141, point_mass=True)
    bad, flagged = compare_tokens(got, ref, 1.0)
    assert bad == 0 and flagged <= 1
    eng.close()


def test_fp8_argument_checks(dev):
    wl = si.workload("tiny", dtype="bf16", V=1000, d=256, B=1, K=2)
    W8, ws = si.make_fp8_weights(wl, seed=151, device=dev)
    inp = si.make_fp8_round(wl, W8, ws, seed=152, T=1.0)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, "fp8", device=dev)
    out_t = torch.empty((1, 3), dtype=torch.int32, device=dev)
    out_n = torch.empty((1,), dtype=torch.int32, device=dev)
    with pytest.raises(sv.SpecVerifyError) as e:   # the plain entry carries no scales
        sv.spec_verify_run(eng.h, inp["hidden8"], W8, inp["draft"], inp["q_logits"],
                           inp["uniforms"], 1.0, out_t, out_n)
    assert e.value.code == sv.SV_ERR_ARG
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_run_fp8(eng.h, inp["hidden8"], None, W8, ws, inp["draft"],
                               inp["q_logits"], inp["uniforms"], 1.0, out_t, out_n)
    assert e.value.code == sv.SV_ERR_ARG
    with pytest.raises(sv.SpecVerifyError) as e:   # a tree call carries no scales either
        sv.spec_verify_tree_greedy(eng.h, inp["hidden8"], W8, inp["draft"],
                                   torch.tensor([[-1, 0]], dtype=torch.int32, device=dev),
                                   out_t, None, out_n)
    assert e.value.code == sv.SV_ERR_ARG
    assert eng.status() == sv.SV_OK
    eng.close()
    # a bf16 handle refuses the FP8 entry point
    eng2 = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, "bf16", device=dev)
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_run_fp8(eng2.h, inp["hidden8"], inp["h_scale"], W8, ws, inp["draft"],
                               inp["q_logits"], inp["uniforms"], 1.0, out_t, out_n)
    assert e.value.code == sv.SV_ERR_ARG
    eng2.close()
