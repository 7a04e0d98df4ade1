"""GPU parity of cross-attention (gma_forward_cross: N_q queries, N_k keys) against the fp64
oracle's forward_cross on the same seeded inputs.  Tolerances as for the forward pass: 1e-5
(fp32 inputs) / 2e-2 (bf16 inputs), normwise per slice."""
import numpy as np
import pytest
import torch

import oracle
from linear_latent_routing_gb300 import inputs as W
from parity import TOL, normwise_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_latent_routing_gb300 import build
    build.build()


def _gma():
    from linear_latent_routing_gb300 import gma
    return gma


def _inputs(w, n_q, n_k):
    """Queries are the first n_q rows of the workload's Q_X, keys and values the first n_k rows
    of its K_X and V (the workload is drawn with N = max(n_q, n_k))."""
    host = W.make_inputs(W.scaled(w, N=max(n_q, n_k)))
    host["QX"] = host["QX"][:, :, :n_q].contiguous()
    host["KX"] = host["KX"][:, :, :n_k].contiguous()
    host["V"] = host["V"][:, :, :n_k].contiguous()
    return host


def _run(w, n_q, n_k, flags=0, slices=None):
    gma = _gma()
    host = _inputs(w, n_q, n_k)
    dev = {k: v.cuda() for k, v in host.items()}
    O = gma.forward_cross(dev["QX"], dev["KX"], dev["V"], dev["mu"], dev["raw"], dev["logits"],
                          eps=w.eps, var_floor=w.var_floor, flags=flags, check=True)
    O = O.float().cpu().numpy()
    a = W.to_numpy(host)
    if slices is None:
        ref = oracle.forward_cross(a["QX"], a["KX"], a["V"], a["mu"], a["raw"], a["logits"],
                                   w.var_floor, w.eps)
        return O, ref
    outs, refs = [], []
    for b, h in slices:
        refs.append(oracle.forward_cross(a["QX"][b:b + 1, h:h + 1], a["KX"][b:b + 1, h:h + 1],
                                         a["V"][b:b + 1, h:h + 1], a["mu"][h:h + 1],
                                         a["raw"][h:h + 1], a["logits"][h:h + 1], w.var_floor,
                                         w.eps))
        outs.append(O[b:b + 1, h:h + 1])
    return np.concatenate(outs, axis=1), np.concatenate(refs, axis=1)


CASES = [
    (W.scaled(W.LRA_BIDIR, B=2, H=2), 777, 300),
    (W.scaled(W.LRA_BIDIR, B=1, H=2), 129, 2049),
    (W.scaled(W.LRA_BIDIR, B=1, H=1), 1, 5),
    (W.scaled(W.LRA_BIDIR, B=1, H=1), 500, 1),
    (W.scaled(W.LM_CAUSAL, B=1, H=2, causal=False), 1000, 257),
    (W.scaled(W.LONG_CAUSAL, B=1, H=1, causal=False), 300, 1500),
    (W.scaled(W.TINY_BIDIR_F32, H=2), 300, 1000),
    (W.scaled(W.TINY_BIDIR_F32), 1, 1),
    (W.scaled(W.LM_CAUSAL, B=1, H=1, d_r=128, K=40, d_v=32, causal=False), 200, 333),
    (W.scaled(W.K_SWEEP[3], B=1, H=1, causal=False), 130, 260),
    (W.scaled(W.LRA_BIDIR, B=2, H=1, K=200), 777, 300),              # components in tiles
    (W.scaled(W.LM_CAUSAL, B=1, H=2, K=300, causal=False), 129, 1000),
]


def _id(c):
    w, n_q, n_k = c
    return f"{w.dtype}_B{w.B}H{w.H}q{n_q}k{n_k}r{w.d_r}K{w.K}v{w.d_v}"


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("flags", [0, 1], ids=["default", "simt"])
def test_cross_matches_oracle(case, flags):
    w, n_q, n_k = case
    O, ref = _run(w, n_q, n_k, flags=flags)
    assert np.isfinite(O).all()
    assert normwise_error(O, ref) <= TOL[w.dtype]


def test_cross_with_equal_lengths_is_the_bidirectional_forward():
    """n_k == N runs exactly the bidirectional path: identical bits."""
    gma = _gma()
    w = W.scaled(W.LRA_BIDIR, B=2, H=2, N=600)
    host = W.make_inputs(w)
    dev = {k: v.cuda() for k, v in host.items()}
    a = gma.forward_cross(dev["QX"], dev["KX"], dev["V"], dev["mu"], dev["raw"], dev["logits"],
                          eps=w.eps, var_floor=w.var_floor, check=True)
    b = gma.forward(dev["QX"], dev["KX"], dev["V"], dev["mu"], dev["raw"], dev["logits"], False,
                    eps=w.eps, var_floor=w.var_floor, check=True)
    assert torch.equal(a, b)


def test_cross_full_size_sampled_slices():
    """The classification-shaped workload at full batch (B=32, H=8): 4096 queries against 2048
    keys, eight sampled slices against the oracle."""
    w = W.LRA_BIDIR
    slices = [(0, 0), (3, 7), (11, 2), (17, 5), (22, 1), (27, 6), (30, 3), (31, 7)]
    O, ref = _run(w, 4096, 2048, slices=slices)
    assert normwise_error(O, ref) <= TOL[w.dtype]


def test_cross_benchmark_workload_sampled_slices():
    """The cross-attention benchmark workload (B=8, H=16, 2048 queries, 16384 keys, its own
    draws), six sampled slices against the oracle, in the benchmark's launch configuration."""
    gma = _gma()
    w = W.CROSS
    host = W.make_inputs(w)
    dev = {k: v.cuda() for k, v in host.items()}
    O = gma.forward_cross(dev["QX"], dev["KX"], dev["V"], dev["mu"], dev["raw"], dev["logits"],
                          eps=w.eps, var_floor=w.var_floor, check=True).float().cpu().numpy()
    a = W.to_numpy(host)
    for b, h in [(0, 0), (1, 9), (3, 15), (4, 4), (6, 11), (7, 2)]:
        ref = oracle.forward_cross(a["QX"][b:b + 1, h:h + 1], a["KX"][b:b + 1, h:h + 1],
                                   a["V"][b:b + 1, h:h + 1], a["mu"][h:h + 1], a["raw"][h:h + 1],
                                   a["logits"][h:h + 1], w.var_floor, w.eps)
        assert normwise_error(O[b:b + 1, h:h + 1], ref) <= TOL[w.dtype]
