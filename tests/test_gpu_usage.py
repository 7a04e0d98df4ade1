"""GPU parity of the component-usage diagnostics (gma_usage) against the fp64 oracle.

Hard assignments are decided by floating point, so they are compared where they are unique: a
token whose assignment differs from the oracle's must be a near tie, i.e. the oracle's
responsibility of the component the GPU chose is within a relative DELTA of the largest one
(DELTA = 1e-5 for the fp32 family, 3e-2 for the tensor-core family, whose logits carry ~1e-2
nats of fp16 rounding).  Counts, used components and the entropy are integers or functions of
integers: they must equal the oracle's histogram of the GPU's own assignments exactly (entropy to
fp32 rounding).  Masses (sums of responsibilities) compare normwise per head: 1e-5 (fp32 family)
or 2e-2 (tensor-core family)."""
import numpy as np
import pytest
import torch

import oracle
from linear_latent_routing_gb300 import inputs as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_latent_routing_gb300 import build
    build.build()


def _gma():
    from linear_latent_routing_gb300 import gma
    return gma


def _check(w, X, host, flags=0, heads=None):
    gma = _gma()
    dev = {k: v.cuda() for k, v in host.items()}
    Xd = X.cuda()
    u = gma.usage(Xd, dev["mu"], dev["raw"], dev["logits"], var_floor=w.var_floor, flags=flags,
                  check=True)
    u = {k: v.cpu().numpy() for k, v in u.items()}
    shape = gma.make_shape(w.B, w.H, X.shape[2], w.d_r, w.K, 16,
                           gma.GMA_BF16 if X.dtype == torch.bfloat16 else gma.GMA_F32,
                           1e-6, w.var_floor, flags)
    tc = gma.gma_kernel_family(shape, gma.GMA_VARIANT_USAGE) == 1
    delta, mtol = (3e-2, 2e-2) if tc else (1e-5, 1e-5)
    a = W.to_numpy({"X": X, "mu": host["mu"], "raw": host["raw"], "logits": host["logits"]})
    heads = list(range(w.H)) if heads is None else heads
    for h in heads:
        ref = oracle.usage(a["X"][:, h:h + 1], a["mu"][h:h + 1], a["raw"][h:h + 1],
                           a["logits"][h:h + 1], w.var_floor)
        ga = u["assign"][:, h:h + 1].astype(np.int64)
        # assignments: equal, or a near tie of the oracle's posterior
        diff = ga != ref["assign"]
        if diff.any():
            X1 = a["X"][:, h]
            for b, i in zip(*np.nonzero(diff[:, 0])):
                g = oracle.responsibilities(X1[b, i:i + 1], a["mu"][h], a["raw"][h], a["logits"][h],
                                            w.var_floor)[0]
                assert g[ga[b, 0, i]] >= g.max() * (1 - delta), (h, b, i, g.max(), g[ga[b, 0, i]])
        assert diff.mean() < 0.01
        # histogram of the GPU's own assignments: exact
        counts, used, ent = oracle.usage_from_assign(ga, w.K)
        assert (u["counts"][h] == counts[0]).all()
        assert u["used"][h] == used[0]
        assert abs(u["entropy"][h] - ent[0]) <= 1e-5
        # masses
        err = np.abs(u["mass"][h] - ref["mass"][0]).max() / np.abs(ref["mass"][0]).max()
        assert err <= mtol, err
        assert np.isclose(u["mass"][h].sum(), w.B * X.shape[2], rtol=1e-4)


CASES = [
    W.scaled(W.LM_CAUSAL, B=2, H=3, N=700),
    W.scaled(W.LM_CAUSAL, B=1, H=2, N=333, dtype="f32"),
    W.scaled(W.LRA_BIDIR, B=3, H=2, N=130),
    W.scaled(W.LONG_CAUSAL, B=1, H=2, N=1000),
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=64, K=1),
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=1, K=16),
    W.scaled(W.K_SWEEP[3], B=1, H=1, N=300),
    W.scaled(W.LM_CAUSAL, B=1, H=2, N=257, d_r=128, K=48),
    W.scaled(W.LM_CAUSAL, B=2, H=2, N=500, d_r=32, K=300),   # tensor cores, components in tiles
    # two tiles: the pre-pass keeps both tables resident and pipelines its steps (argmax and counts
    # merged from the two halves of each row); a partial second tile, then exactly two full ones
    W.scaled(W.LM_CAUSAL, B=2, H=2, N=777, K=200),
    W.scaled(W.LM_CAUSAL, B=1, H=2, N=300, K=256),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.dtype}_B{w.B}H{w.H}N{w.N}r{w.d_r}K{w.K}")
@pytest.mark.parametrize("flags", [0, 1], ids=["default", "simt"])
def test_usage_matches_oracle(w, flags):
    host = W.make_inputs(w)
    _check(w, host["KX"], host, flags=flags)


def test_usage_benchmark_workload_two_heads():
    """The benchmark's keys (B=1, H=16, N=65536, K=128): heads 0 and 9 against the oracle, every
    token, in the benchmark's launch configuration."""
    w = W.LONG_CAUSAL
    host = W.make_inputs(w)
    _check(w, host["KX"], host, heads=[0, 9])


def test_usage_is_deterministic():
    gma = _gma()
    w = W.scaled(W.LM_CAUSAL, B=2, H=2, N=2000)
    host = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    a = gma.usage(host["KX"], host["mu"], host["raw"], host["logits"], check=True)
    b = gma.usage(host["KX"], host["mu"], host["raw"], host["logits"], check=True)
    for k in a:
        assert torch.equal(a[k], b[k]), k
