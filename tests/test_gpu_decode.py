"""GPU parity of the autoregressive decode step (gma_decode_step) against the fp64 oracle.

Each case runs T steps on the device, feeding the state back, and compares every step's output
and the final state with the oracle's decode step on the same seeded inputs.  Tolerances: the
output as in the forward parity tests (normwise per slice, 1e-5 for fp32 inputs, 2e-2 for bf16
outputs); the fp32 state, and fp32 outputs from bf16 inputs (exact in fp32, so only the fp32
arithmetic differs), 1e-5 normwise, widened to 1e-4 where d_r = 128 sums 128 squared distances
into each logit in fp32."""
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


def _run_steps(w, S0, flags=0):
    """T = w.N decode steps on the GPU and in the oracle from state S0 [B,H,K,d_v+1] (CPU fp32)."""
    gma = _gma()
    host = W.make_inputs(w)
    dev = {k: v.cuda().contiguous() for k, v in host.items()}
    S = S0.cuda().contiguous()
    a = W.to_numpy(host)
    S_ref = S0.double().numpy()
    outs, refs = [], []
    for t in range(w.N):
        o = gma.decode_step(dev["QX"][:, :, t].contiguous(), dev["KX"][:, :, t].contiguous(),
                            dev["V"][:, :, t].contiguous(), dev["mu"], dev["raw"], dev["logits"], S,
                            eps=w.eps, var_floor=w.var_floor, flags=flags, check=True)
        outs.append(o.float().cpu().numpy())
        o_ref, S_ref = oracle.decode_step(a["QX"][:, :, t], a["KX"][:, :, t], a["V"][:, :, t],
                                          a["mu"], a["raw"], a["logits"], w.var_floor, w.eps, S_ref)
        refs.append(o_ref)
    torch.cuda.synchronize()
    # [B, H, T, d_v]: one slice per (b, h), as the forward tests measure
    return (np.stack(outs, axis=2), np.stack(refs, axis=2), S.cpu().double().numpy(), S_ref)


def _fp32_tol(w):
    return 1e-4 if w.d_r >= 128 else 1e-5


CASES = [
    W.scaled(W.LM_CAUSAL, B=2, H=3, N=12),
    W.scaled(W.LM_CAUSAL, B=2, H=3, N=12, dtype="f32"),
    W.scaled(W.DECODE, B=3, H=2, N=6),
    W.scaled(W.DECODE, B=1, H=2, N=4, d_r=128, K=1024, d_v=128),
    W.scaled(W.DECODE, B=2, H=1, N=5, d_r=16, K=1, d_v=16),
    W.scaled(W.DECODE, B=1, H=3, N=5, d_r=32, K=100, d_v=32, dtype="f32"),
    # K not a multiple of 4: rows off 16-byte boundaries, the plain kernel (5 chunks, ragged tail)
    W.scaled(W.DECODE, B=2, H=2, N=3, K=130),
    W.scaled(W.DECODE, B=1, H=2, N=3, d_r=16, K=301, d_v=16),
    # more slices than SMs: each persistent CTA streams several slices' chunks through its ring
    W.scaled(W.DECODE, B=25, H=16, N=3, K=256),
]


def _id(w):
    return f"{w.dtype}_B{w.B}H{w.H}T{w.N}r{w.d_r}K{w.K}v{w.d_v}"


@pytest.mark.parametrize("w", CASES, ids=_id)
@pytest.mark.parametrize("start", ["zero", "state"])
def test_decode_steps_match_oracle(w, start):
    S0 = (torch.zeros(w.B, w.H, w.K, w.d_v + 1) if start == "zero"
          else W.make_decode_state(w, scale=3.0))
    O, ref, S, S_ref = _run_steps(w, S0)
    assert np.isfinite(O).all() and np.isfinite(S).all()
    tol_o = TOL[w.dtype] if w.dtype == "bf16" else _fp32_tol(w)
    assert normwise_error(O, ref) <= tol_o
    assert normwise_error(S, S_ref) <= _fp32_tol(w)


@pytest.mark.parametrize("w", [W.scaled(W.DECODE, B=2, H=2, N=4),
                               W.scaled(W.DECODE, B=1, H=2, N=3, d_r=128, K=1024, d_v=128)], ids=_id)
def test_decode_fp32_output_from_bf16_inputs(w):
    """With GMA_FLAG_OUT_F32 the output is not rounded to bf16: fp32 agreement."""
    gma = _gma()
    O, ref, S, S_ref = _run_steps(w, W.make_decode_state(w), flags=gma.GMA_FLAG_OUT_F32)
    assert normwise_error(O, ref) <= _fp32_tol(w)
    assert normwise_error(S, S_ref) <= _fp32_tol(w)


def test_decode_continues_the_causal_forward():
    """Decoding token by token from an empty state gives the causal forward's rows: step t's
    output is row t of the forward pass over the first t + 1 tokens (oracle forward)."""
    w = W.scaled(W.LM_CAUSAL, B=1, H=2, N=10, dtype="f32")
    O, _, _, _ = _run_steps(w, torch.zeros(w.B, w.H, w.K, w.d_v + 1))
    a = W.to_numpy(W.make_inputs(w))
    F = oracle.forward(True, a["QX"], a["KX"], a["V"], a["mu"], a["raw"], a["logits"],
                       w.var_floor, w.eps)
    assert normwise_error(O, F) <= 1e-5


def test_decode_full_batch_matches_oracle():
    """The benchmark's decode batch (B=128 sequences x 16 heads, K=128, d_v=128), one step from a
    non-zero state, every slice against the oracle."""
    w = W.scaled(W.DECODE, N=1)
    O, ref, S, S_ref = _run_steps(w, W.make_decode_state(w, scale=10.0))
    assert normwise_error(O, ref) <= TOL["bf16"]
    assert normwise_error(S, S_ref) <= 1e-5


def test_decode_rejects_bad_arguments():
    gma = _gma()
    w = W.scaled(W.DECODE, B=1, H=2, N=1)
    host = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    S = torch.zeros(w.B, w.H, w.K, w.d_v + 1, device="cuda")
    with pytest.raises(ValueError):
        gma.decode_step(host["QX"][:, :, 0], host["KX"][:, :, 0], host["V"][:, :, 0], host["mu"],
                        host["raw"], host["logits"], S[:, :, :-1].contiguous())
    # N != 1 through the C ABI: refused before anything is enqueued
    shape = gma.make_shape(w.B, w.H, 2, w.d_r, w.K, w.d_v, gma.GMA_BF16)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    q = host["QX"]
    r = gma.gma_decode_step(shape, q.data_ptr(), q.data_ptr(), host["V"].data_ptr(),
                            host["mu"].data_ptr(), host["raw"].data_ptr(), host["logits"].data_ptr(),
                            S.data_ptr(), ws.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert r == gma.GMA_ERR_INVALID_ARG
