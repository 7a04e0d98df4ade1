"""GPU parity of the backward pass (gma_backward) against the fp64 oracle's backward, both
variants, on the same seeded inputs and output gradients.

Tolerance (normwise: max |g - g_ref| / max |g_ref|, per (b, h) slice for dQX, dKX, dV and per
head for dmu, draw, dlogits): 1e-4 when the gradients come out in fp32, 2e-2 when dQX, dKX, dV
are rounded to bf16.  Derivation of the fp32 figure: every step runs in fp32 from inputs exact
in fp32; the responsibilities carry the forward's ~1e-5 relative logit error (d_r = 64 terms of
magnitude ~3 summed in fp32), the segment sums add ~sqrt(N) u, and the softmax backward
dL = Gamma (dGamma - <Gamma, dGamma>) subtracts a common part of dGamma, which can amplify
relative error by a small factor; 1e-4 leaves room for that, and is still 100 times below the
size of any dropped term (the oracle pins check each term separately)."""
import numpy as np
import pytest
import torch

import oracle
from linear_latent_routing_gb300 import inputs as W
from parity import normwise_error

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_latent_routing_gb300 import build
    build.build()


def _gma():
    from linear_latent_routing_gb300 import gma
    return gma


def _dO(w):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed) + 2024)
    d = torch.randn(w.B, w.H, w.N, w.d_v, generator=g, dtype=torch.float32)
    return d.to(torch.bfloat16) if w.dtype == "bf16" else d


def _head_err(g, ref):
    g = np.asarray(g, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ax = tuple(range(1, g.ndim))
    return float((np.abs(g - ref).max(axis=ax) / np.maximum(np.abs(ref).max(axis=ax), 1e-300)).max())


def _run(w, causal):
    gma = _gma()
    host = W.make_inputs(w)
    dO = _dO(w)
    dev = {k: v.cuda() for k, v in host.items()}
    got = gma.backward(dev["QX"], dev["KX"], dev["V"], dev["mu"], dev["raw"], dev["logits"], dO.cuda(),
                       causal, eps=w.eps, var_floor=w.var_floor, check=True)
    got = [t.float().cpu().numpy() for t in got]
    a = W.to_numpy(host)
    ref = oracle.backward(causal, a["QX"], a["KX"], a["V"], a["mu"], a["raw"], a["logits"], w.var_floor,
                          w.eps, dO.float().numpy())
    return got, ref


CASES = [
    W.scaled(W.TINY_BIDIR_F32, B=2, H=2, N=130),
    W.scaled(W.LM_CAUSAL, B=1, H=2, N=200, dtype="f32"),
    W.scaled(W.LM_CAUSAL, B=1, H=2, N=200),
    W.scaled(W.LRA_BIDIR, B=2, H=1, N=97),
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=150, d_r=128, K=40, d_v=16, dtype="f32"),
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=70, K=1, dtype="f32"),
    # one token: O = v a / (a + eps) and the routing gradients are eps-sized differences of
    # O(1) terms, which fp32 cannot resolve at eps = 1e-6 (the oracle's fp64 can); a larger eps
    # keeps the case well conditioned while it still checks the one-token code path
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=1, K=16, dtype="f32", eps=0.1),
    W.scaled(W.LONG_CAUSAL, B=1, H=1, N=129, K=300, dtype="f32"),
    # bf16 with two component tiles (K = 128): the softmax step on its own (row dot products, dL
    # formed by the dx kernel) rather than folded into dGamma, and d_v = 128
    W.scaled(W.LONG_CAUSAL, B=2, H=1, N=150),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.dtype}_B{w.B}H{w.H}N{w.N}r{w.d_r}K{w.K}v{w.d_v}")
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_matches_oracle(w, causal):
    got, ref = _run(w, causal)
    names = ["dQX", "dKX", "dV", "dmu", "draw", "dlogits"]
    tol_act = TOL[w.dtype]
    for name, g, r in zip(names, got, ref):
        assert np.isfinite(g).all(), name
        if name in ("dQX", "dKX", "dV"):
            err = normwise_error(g, r)
            assert err <= tol_act, (name, err)
        else:
            err = _head_err(g, r)
            assert err <= TOL["f32"], (name, err)


def test_backward_is_deterministic():
    gma = _gma()
    w = W.scaled(W.LM_CAUSAL, B=2, H=2, N=300)
    host = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    dO = _dO(w).cuda()
    a = gma.backward(host["QX"], host["KX"], host["V"], host["mu"], host["raw"], host["logits"], dO, True,
                     check=True)
    b = gma.backward(host["QX"], host["KX"], host["V"], host["mu"], host["raw"], host["logits"], dO, True,
                     check=True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_full_size_heads():
    """The benchmarked backward workload (causal, B=4, H=8, N=2048, K=64) in one call, as the
    benchmark runs it; every gradient of two heads against the oracle: all four batch rows of
    each head, so that the parameter gradients (summed over the batch) are complete."""
    gma = _gma()
    w = W.BACKWARD
    host = W.make_inputs(w)
    dO = _dO(w)
    dev = {k: v.cuda() for k, v in host.items()}
    got = gma.backward(dev["QX"], dev["KX"], dev["V"], dev["mu"], dev["raw"], dev["logits"], dO.cuda(),
                       True, eps=w.eps, var_floor=w.var_floor, check=True)
    got = [t.float().cpu().numpy() for t in got]
    a = W.to_numpy(host)
    d = dO.float().numpy()
    names = ["dQX", "dKX", "dV", "dmu", "draw", "dlogits"]
    for h in (0, w.H - 1):
        hs = slice(h, h + 1)
        ref = oracle.backward(True, a["QX"][:, hs], a["KX"][:, hs], a["V"][:, hs], a["mu"][hs], a["raw"][hs],
                              a["logits"][hs], w.var_floor, w.eps, d[:, hs])
        for i, (name, r) in enumerate(zip(names, ref)):
            g = got[i][:, hs] if i < 3 else got[i][hs]
            assert np.isfinite(g).all(), name
            err = normwise_error(g, r) if i < 3 else _head_err(g, r)
            assert err <= (TOL[w.dtype] if i < 3 else TOL["f32"]), (h, name, err)
