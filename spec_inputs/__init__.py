"""Seeded synthetic inputs for the verify-and-sample step.

Both sides of every parity check (the CUDA library and the CPU oracle) read
the tensors made here.  This module holds none of the step's arithmetic: no
softmax, no acceptance test, no residual, no draw.  It only draws random
numbers and shapes them like the workloads on the pages (Llama-3.1-8B- and
70B-sized LM heads, K = 3..7 drafts, small batches):

* LM-head weights W [V, d] ~ N(0, std^2), rounded once to bf16 (or kept in
  fp32 for the tiny configuration, std = 1/sqrt(d)).
* hidden states [B, K+1, d] ~ N(0, 1), rounded once to bf16 (or fp32).
* draft logits q_logits [B, K, V] = L + sigma * z, z ~ N(0, 1), where L is a
  plain fp32 torch matmul of the hidden states against W.  This only places
  the synthetic draft near the target so that the acceptance rate lands near
  the requested alpha; any values are valid inputs, and both sides read the
  same stored bits.  sigma comes from ``draft_noise_table.json``, a table
  written by ``oracle/calibrate_draft_noise.py``.
* draft tokens x_i drawn from softmax(q_logits_i / T) by the Gumbel-max
  trick (argmax of q_logits / T + Gumbel noise); at T == 0 the draft's own
  argmax.  Drawing the proposals is the draft model's job, not the verify
  step's.
* uniforms [B, K+1] on the grid {0, 2^-24, ..., 1 - 2^-24} (exact fp32).

All randomness comes from a ``torch.Generator`` seeded per call; the same
seed on the same device type gives the same bits.
"""
from __future__ import annotations

import bisect
import json
import math
import os
from dataclasses import dataclass, field

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))


@dataclass(frozen=True)
class Workload:
    name: str
    V: int
    d: int
    B: int
    K: int
    T: float
    dtype: str             # "bf16" or "fp32"
    w_std: float
    alpha: float | None = None                 # one target acceptance rate
    alpha_range: tuple | None = None           # per-sequence U(lo, hi)
    note: str = field(default="", compare=False)


def workload(name: str, **over) -> Workload:
    """The configurations of the verify step: shapes, temperatures and draft
    acceptance targets of the synthetic workloads."""
    base = {
        "tiny": dict(V=1000, d=256, B=1, K=4, T=1.0, dtype="fp32",
                     w_std=1.0 / 16.0, alpha=None, sigma_fixed=0.5,
                     note="V=1000, d=256, B=1, K=4, fp32, T=1, draft noise 0.5"),
        "llama8b": dict(V=128256, d=4096, B=1, K=4, T=1.0, dtype="bf16",
                        w_std=0.02, alpha=0.8,
                        note="Llama-3.1-8B-shaped LM head, B=1, K=4, T=1"),
        "llama8b_b8k7": dict(V=128256, d=4096, B=8, K=7, T=0.7, dtype="bf16",
                             w_std=0.02, alpha_range=(0.5, 0.9),
                             note="8B shape, B=8, K=7, T=0.7, alpha~U(0.5,0.9)"),
        "llama70b": dict(V=128256, d=8192, B=4, K=4, T=1.0, dtype="bf16",
                         w_std=0.02, alpha=0.75,
                         note="Llama-70B-shaped LM head, B=4, K=4, T=1"),
        "sweep": dict(V=128256, d=4096, B=1, K=4, T=1.0, dtype="bf16",
                      w_std=0.02, alpha=0.7,
                      note="8B shape batch sweep, T=1, alpha~0.7"),
    }[name]
    base = dict(base)
    base.update(over)
    sigma_fixed = base.pop("sigma_fixed", None)
    wl = Workload(name=name, **base)
    object.__setattr__(wl, "_sigma_fixed", sigma_fixed)
    return wl


def _noise_table():
    with open(os.path.join(_HERE, "draft_noise_table.json")) as f:
        return json.load(f)


def draft_noise(alpha: float, logit_spread: float, T: float) -> float:
    """sigma (in logit units) that gives acceptance ~alpha, by linear
    interpolation in the calibration table (keyed by s/T, storing sigma/T)."""
    tab = _noise_table()
    alphas = tab["alphas"]
    scaled = logit_spread / (T if T > 0 else 1.0)
    keys = sorted(float(k) for k in tab["spreads"])
    k = min(keys, key=lambda s: abs(s - scaled))
    row = tab["spreads"][f"{k:.2f}"]
    a = min(max(alpha, alphas[0]), alphas[-1])
    i = min(max(bisect.bisect_left(alphas, a), 1), len(alphas) - 1)
    w = (a - alphas[i - 1]) / (alphas[i] - alphas[i - 1])
    s_over_T = row[i - 1] + w * (row[i] - row[i - 1])
    return s_over_T * (T if T > 0 else 1.0)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def torch_dtype(wl: Workload):
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def make_weights(wl: Workload, seed: int, device="cpu") -> torch.Tensor:
    """W [V, d] ~ N(0, w_std^2) in the workload's dtype."""
    g = _gen(seed, device)
    W = torch.empty((wl.V, wl.d), dtype=torch.float32, device=device)
    rows = 8192
    for v0 in range(0, wl.V, rows):
        v1 = min(wl.V, v0 + rows)
        W[v0:v1].normal_(0.0, wl.w_std, generator=g)
    return W.to(torch_dtype(wl))


def make_round(wl: Workload, W: torch.Tensor, seed: int, device=None,
               T: float | None = None) -> dict:
    """One round's inputs: hidden [B, K+1, d], draft [B, K] int32,
    q_logits [B, K, V] fp32, uniforms [B, K+1] fp32, and the per-sequence
    draft noise actually used."""
    device = W.device if device is None else torch.device(device)
    T = wl.T if T is None else float(T)
    g = _gen(seed, device)
    B, K, V, d = wl.B, wl.K, wl.V, wl.d
    hidden = torch.randn((B, K + 1, d), generator=g, device=device,
                         dtype=torch.float32).to(torch_dtype(wl))
    sig_fixed = getattr(wl, "_sigma_fixed", None)
    spread = math.sqrt(d) * wl.w_std
    if sig_fixed is not None:
        sigmas = torch.full((B,), float(sig_fixed))
    elif wl.alpha_range is not None:
        lo, hi = wl.alpha_range
        alphas = lo + (hi - lo) * torch.rand((B,), generator=g, device=device).cpu()
        sigmas = torch.tensor([draft_noise(float(a), spread, T) for a in alphas])
    else:
        sigmas = torch.full((B,), draft_noise(wl.alpha, spread, T))
    if K > 0:
        est = torch.matmul(hidden[:, :K, :].float().reshape(B * K, d),
                           W.float().t()).reshape(B, K, V)
        z = torch.randn((B, K, V), generator=g, device=device)
        q_logits = (est + sigmas.to(device).view(B, 1, 1) * z).float().contiguous()
        if T > 0:
            gum = torch.rand((B, K, V), generator=g, device=device)
            gum = gum.clamp_min(1e-30)
            gumbel = -torch.log(-torch.log(gum))
            draft = torch.argmax(q_logits / T + gumbel, dim=-1)
        else:
            draft = torch.argmax(q_logits, dim=-1)
        draft = draft.to(torch.int32).contiguous()
    else:
        q_logits = torch.zeros((B, 0, V), dtype=torch.float32, device=device)
        draft = torch.zeros((B, 0), dtype=torch.int32, device=device)
    uniforms = (torch.randint(0, 1 << 24, (B, K + 1), generator=g,
                              device=device).to(torch.float32)
                * (2.0 ** -24)).contiguous()
    return {"hidden": hidden.contiguous(), "draft": draft, "q_logits": q_logits,
            "uniforms": uniforms, "sigma": sigmas}


def draw_drafts(q_logits: torch.Tensor, T: float, n: int, seed: int) -> torch.Tensor:
    """n more draft proposals for the same draft logits q_logits [B, K, V]:
    each x_i drawn from softmax(q_logits_i / T) by the Gumbel-max trick (the
    draft model's own sampling, as in make_round; argmax at T == 0).
    Returns int32 [n, B, K]."""
    g = _gen(seed, q_logits.device)
    B, K, V = q_logits.shape
    out = torch.empty((n, B, K), dtype=torch.int32, device=q_logits.device)
    if K == 0:
        return out
    scaled = q_logits / T if T > 0 else q_logits
    chunk = max(1, (1 << 27) // max(1, B * K * V))   # ~0.5 GB of noise at a time
    for i0 in range(0, n, chunk):
        m = min(chunk, n - i0)
        if T > 0:
            gum = torch.rand((m, B, K, V), generator=g, device=q_logits.device).clamp_min(1e-30)
            out[i0:i0 + m] = torch.argmax(scaled.unsqueeze(0) - torch.log(-torch.log(gum)),
                                          dim=-1).to(torch.int32)
        else:
            out[i0:i0 + m] = torch.argmax(scaled, dim=-1).to(torch.int32).unsqueeze(0)
    return out


def draw_uniforms(n: int, B: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """n more sets of uniforms [n, B, K+1] on the 2^-24 grid (exact fp32)."""
    g = _gen(seed, device)
    return (torch.randint(0, 1 << 24, (n, B, K + 1), generator=g, device=device)
            .to(torch.float32) * (2.0 ** -24)).contiguous()


def to_oracle(t: torch.Tensor):
    """Host numpy view for the oracle: bf16 as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


# ---------------------------------------------------------------------------
# FP8 E4M3 inputs (input shaping for the FP8 LM head)
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0


def quantize_rows_e4m3(x: torch.Tensor):
    """Per-row FP8 E4M3 quantisation: scale = max|x| / 448 per row (fp32),
    codes = x / scale converted by torch's float8_e4m3fn (round to nearest
    even).  Returns (codes as uint8 [..., d], scales fp32 [...])."""
    xf = x.float()
    scale = (xf.abs().amax(dim=-1).clamp_min(1e-30) / E4M3_MAX).float()
    q = (xf / scale.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).contiguous(), scale.contiguous()


def dequantize_e4m3(codes: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    return codes.view(torch.float8_e4m3fn).float() * scale.unsqueeze(-1)


def make_fp8_weights(wl: Workload, seed: int, device="cpu"):
    """The bf16-shaped weights of the workload, quantised per vocabulary row:
    (W8 uint8 [V, d], w_scale fp32 [V])."""
    W = make_weights(wl, seed=seed, device=device)
    return quantize_rows_e4m3(W)


def make_fp8_round(wl: Workload, W8: torch.Tensor, w_scale: torch.Tensor, seed: int,
                   T: float | None = None) -> dict:
    """make_round on the dequantised weights, with the hidden states
    quantised per row: adds hidden8 [B, K+1, d] uint8 and h_scale [B, K+1]."""
    Wd = dequantize_e4m3(W8, w_scale)
    r = make_round(wl, Wd, seed, T=T)
    h8, hs = quantize_rows_e4m3(r["hidden"])
    r["hidden8"], r["h_scale"] = h8, hs
    return r
