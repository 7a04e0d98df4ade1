"""Helpers for the GPU parity tests: run the CUDA library and the oracle on the same seeded
inputs and measure their disagreement.

Error measure (the tolerance is a "max relative error"): per (batch, head) slice,
max |O - O_ref| / max |O_ref|, then the maximum over slices.  Element-wise ratios are not used:
signed values cancel inside V~ and make single elements near zero meaningless to divide by.
"""
import numpy as np

import oracle
from linear_latent_routing_gb300.inputs import make_inputs, to_numpy

TOL = {"f32": 1e-5, "bf16": 2e-2}


def normwise_error(O, ref):
    O = np.asarray(O, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ax = tuple(range(2, O.ndim))
    num = np.abs(O - ref).max(axis=ax)
    den = np.abs(ref).max(axis=ax)
    return float((num / np.maximum(den, 1e-300)).max())


def rowwise_error(O, ref):
    O = np.asarray(O, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.abs(O - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return float((num / np.maximum(den, 1e-300)).max())


def to_device(inputs, device="cuda"):
    return {k: v.to(device).contiguous() for k, v in inputs.items()}


def gpu_forward(w, dev, flags=0, stream=None):
    from linear_latent_routing_gb300 import gma
    return gma.forward(dev["QX"], dev["KX"], dev["V"], dev["mu"], dev["raw"], dev["logits"],
                       w.causal, eps=w.eps, var_floor=w.var_floor, flags=flags, stream=stream,
                       check=True)


def oracle_forward(w, host, b=None, h=None, n=None):
    """Oracle output for all slices, or for slice (b, h) truncated to its first n tokens
    (exact for the causal variant, whose first n rows see only the first n tokens)."""
    a = to_numpy(host)
    if b is None:
        return oracle.forward(w.causal, a["QX"], a["KX"], a["V"], a["mu"], a["raw"], a["logits"],
                              w.var_floor, w.eps)
    sl = slice(0, n)
    return oracle.forward(w.causal, a["QX"][b:b + 1, h:h + 1, sl], a["KX"][b:b + 1, h:h + 1, sl],
                          a["V"][b:b + 1, h:h + 1, sl], a["mu"][h:h + 1], a["raw"][h:h + 1],
                          a["logits"][h:h + 1], w.var_floor, w.eps)


def case(w):
    host = make_inputs(w)
    return host


def compare_every_token(w, O, host, heads_per_call=4):
    """Every token of every slice of O against the oracle, a few heads per oracle call (the
    oracle runs one slice per host thread)."""
    worst = 0.0
    a = to_numpy(host)
    for h0 in range(0, w.H, heads_per_call):
        h1 = min(w.H, h0 + heads_per_call)
        ref = oracle_heads(w, a, h0, h1)
        got = O[:, h0:h1].float().cpu().numpy()
        assert np.isfinite(got).all()
        worst = max(worst, normwise_error(got, ref))
    return worst


def oracle_heads(w, a, h0, h1, b0=0, b1=None):
    """Oracle output of heads [h0, h1) and batch rows [b0, b1); `a` holds the inputs as numpy."""
    b1 = w.B if b1 is None else b1
    return oracle.forward(w.causal, a["QX"][b0:b1, h0:h1], a["KX"][b0:b1, h0:h1], a["V"][b0:b1, h0:h1],
                          a["mu"][h0:h1], a["raw"][h0:h1], a["logits"][h0:h1], w.var_floor, w.eps)
