"""Helpers shared by the GPU tests: move seeded inputs to the device, run the
library through its C ABI, and compare with the oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import synth

# Tolerance stated for the GEMM output: max|y - y_ref| / max|y_ref| <= 2e-3.
REL_TOL = 2e-3
# Engineering bound for this kernel's arithmetic: (q - z) enters the tensor
# cores exactly and x is bf16, so every product is exact; only fp32
# accumulation rounds (within a group in the MMA, then one fp32 FMA per group),
# which stays far below 2e-5 of max|y| at these K.
ARITH_TOL = 2e-5


def dev() -> torch.device:
    return torch.device("cuda:0")


def proj(name: str, **kw) -> synth.Projection:
    return dataclasses.replace(synth.CONFIGS[name], **kw)


def to_dev_host_inputs(p: synth.Projection):
    """Host-generated inputs (numpy) and their device copies (q packed on the GPU)."""
    import weight_only_bit_wq_gb300 as wq

    w = synth.gen_weights(p)
    x = synth.gen_x(p)
    d = dev()
    q_d = torch.from_numpy(w["q"]).to(d)
    dv = {
        "q": q_d,
        "wq": wq.wq_pack(q_d, p.bits),
        "s": torch.from_numpy(w["s"].view(np.int16)).to(d),
        "z": torch.from_numpy(w["z"]).to(d),
        "x": torch.from_numpy(x.view(np.int16)).to(d),
    }
    return w, x, dv


def rel_err(y: np.ndarray, y_ref: np.ndarray) -> float:
    den = np.abs(y_ref).max()
    return float(np.abs(y.astype(np.float64) - y_ref).max() / (den if den > 0 else 1.0))


def oracle_gemm(p, w, x, rows=None):
    wq_ref = oracle.pack(w["q"], p.bits)
    return oracle.gemm_f64(x, wq_ref, w["s"], w["z"], p.K, p.group, p.bits)


def u32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def check_activation(got: np.ndarray, y64: np.ndarray, exact_frac: float = 0.98) -> None:
    """The device activation against the oracle's.  The device starts from the
    fp32 sums, which the GEMM bar lets differ from the exact ones by up to
    ARITH_TOL x max|y|; that error passes through silu(g) * u (|silu'| < 1.1)
    and, where g or u is near zero, can span more than one bf16 step.  So each
    element must lie within one bf16 step plus that propagated error of the
    oracle's value, and most elements must be bit-equal."""
    ref = oracle.swiglu_bf16(y64)
    assert got.shape == ref.shape
    g, u = y64[:, 0::2], y64[:, 1::2]
    delta = ARITH_TOL * np.abs(y64).max()
    sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    dsilu = sig * (1.0 + g * (1.0 - sig))
    reff = synth.bf16_bits_to_f32(ref)
    gotf = synth.bf16_bits_to_f32(got)
    step = np.spacing(np.abs(reff).astype(np.float32)).astype(np.float64) * 65536.0
    bound = step + (np.abs(dsilu * u) + np.abs(silu)) * delta
    assert (np.abs(gotf.astype(np.float64) - reff) <= bound).all()
    assert (got == ref).mean() > exact_frac
