"""Pins of the oracle's FP8 LM head (reading R13): the E4M3 decoding
against values fixed by the format (largest finite 448, the smallest normal
2^-6, the subnormals m * 2^-9, one NaN code per sign) and against torch's
float8_e4m3fn conversion for all 256 codes, and the scaled logits against a
plain matmul of the decoded values (the special case that reduces to a
library routine)."""
import numpy as np
import torch

import oracle
import spec_inputs as si


def test_e4m3_values_fixed_by_the_format():
    codes = np.array([0x00, 0x80, 0x38, 0xB8, 0x7E, 0xFE, 0x08, 0x01, 0x07, 0x40, 0x7F, 0xFF],
                     dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    assert v[0] == 0.0 and v[1] == 0.0 and np.signbit(v[1])
    assert v[2] == 1.0 and v[3] == -1.0
    assert v[4] == 448.0 and v[5] == -448.0
    assert v[6] == 2.0 ** -6            # smallest normal
    assert v[7] == 2.0 ** -9            # smallest subnormal
    assert v[8] == 7 * 2.0 ** -9        # largest subnormal
    assert v[9] == 2.0                  # exponent 8, mantissa 0
    assert np.isnan(v[10]) and np.isnan(v[11])


def test_e4m3_all_codes_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    nan = np.isnan(t)
    assert np.array_equal(np.isnan(v), nan)
    assert np.array_equal(v[~nan], t[~nan])


def test_fp8_logits_are_scaled_products_of_the_decoded_values():
    rng = np.random.default_rng(8)
    B, K, V, d = 2, 3, 70, 48
    H = torch.from_numpy(rng.standard_normal((B, K + 1, d)).astype(np.float32))
    W = torch.from_numpy((rng.standard_normal((V, d)) * 0.02).astype(np.float32))
    h8, hs = si.quantize_rows_e4m3(H)
    w8, ws = si.quantize_rows_e4m3(W)
    x = rng.integers(0, V, size=(B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    ql = rng.standard_normal((B, K, V)).astype(np.float32)
    out = oracle.verify_fp8(h8.numpy(), hs.numpy(), w8.numpy(), ws.numpy(), x, ql, u, 1.0,
                            want_logits=True)
    Hd = oracle.e4m3_decode(h8.numpy()).reshape(B * (K + 1), d)
    Wd = oracle.e4m3_decode(w8.numpy())
    want = (hs.numpy().reshape(-1).astype(np.float64)[:, None]
            * ws.numpy().astype(np.float64)[None, :]) * (Hd @ Wd.T)
    assert np.allclose(out["logits"], want, rtol=1e-13, atol=1e-15)
    # and the rule on them is the rule: the same tokens as the fp32 path fed
    # the same logits through an identity embedding
    L = out["logits"].reshape(B, K + 1, V).astype(np.float32)
    for b in range(B):
        ref = oracle.verify(L[b:b + 1].copy(), np.eye(V, dtype=np.float32), x[b:b + 1],
                            ql[b:b + 1], u[b:b + 1], 1.0)
        exact = out["dist"][b] > 1e-6 and ref["dist"][0] > 1e-6
        if exact:
            assert np.array_equal(ref["tokens"][0], out["tokens"][b])
