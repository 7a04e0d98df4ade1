"""GPU parity of the single-launch causal kernel (GMA_FLAG_SINGLE_PASS): the page's causal read
(Méthodologie §3, prefix sums over j <= i) computed in one launch after the parameter kernel, with
the key responsibilities never written to memory and the segments' memories exchanged by a
decoupled look-back.  Compared with the fp64 oracle on the same seeded inputs (bf16 bound 2e-2,
normwise per slice, see tests/parity.py)."""
import numpy as np
import pytest
import torch

from linear_latent_routing_gb300 import inputs as W
from parity import TOL, compare_every_token, gpu_forward, normwise_error, oracle_forward, rowwise_error, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gma():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_latent_routing_gb300 import build
    build.build()
    from linear_latent_routing_gb300 import gma as g
    return g


def _shape(gma, w, flags):
    return gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v, gma.GMA_BF16, w.eps, w.var_floor, flags=flags)


# Causal bf16 shapes the tensor-core family takes with K <= 128: every d_r and d_v, ragged
# sequences, one token, one component, and slices cut into many one-chunk segments (the planner
# gives small problems one chunk per segment, so the look-back walks over several predecessors).
SMALL = [
    W.scaled(W.LM_CAUSAL, B=1, H=2, N=1000),
    W.scaled(W.LONG_CAUSAL, B=1, H=2, N=1500),
    W.scaled(W.LONG_CAUSAL, B=2, H=3, N=4000),
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=1, K=16),
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=129, K=1),
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=300, d_r=16, K=8, d_v=16),
    W.scaled(W.LM_CAUSAL, B=1, H=2, N=700, d_r=32, K=32, d_v=64),
    W.scaled(W.LM_CAUSAL, B=1, H=1, N=520, d_r=32, K=100, d_v=32),
    W.scaled(W.LM_CAUSAL, B=2, H=1, N=2200, d_r=16, K=128, d_v=128),
    W.scaled(W.K_SWEEP[0], B=1, H=2, N=3000),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"B{w.B}H{w.H}N{w.N}r{w.d_r}K{w.K}v{w.d_v}")
def test_small_cases_match_oracle(gma, w):
    assert gma.gma_kernel_family(_shape(gma, w, gma.GMA_FLAG_SINGLE_PASS), gma.GMA_VARIANT_CAUSAL) == 1
    host = W.make_inputs(w)
    dev = to_device(host)
    O = gpu_forward(w, dev, flags=gma.GMA_FLAG_SINGLE_PASS).float().cpu().numpy()
    ref = oracle_forward(w, host)
    err = normwise_error(O, ref)
    print(f"{w.name} single pass: normwise {err:.3e}, rowwise {rowwise_error(O, ref):.3e}")
    assert np.isfinite(O).all()
    assert err <= TOL["bf16"], (err, rowwise_error(O, ref))


@pytest.mark.parametrize("w", [W.LM_CAUSAL, W.LONG_CAUSAL], ids=lambda w: w.name)
def test_full_size_every_token(gma, w):
    """The causal benchmark workloads at full size, in the launch configuration the benchmark
    times for this variant: every token of every slice (at the long-context size, 64 segments per
    slice exchange their memories by look-back)."""
    host = W.make_inputs(w)
    dev = to_device(host)
    O = gpu_forward(w, dev, flags=gma.GMA_FLAG_SINGLE_PASS)
    torch.cuda.synchronize()
    del dev
    err = compare_every_token(w, O, host)
    print(f"{w.name} single pass: normwise {err:.3e} over every token of every slice")
    assert err <= TOL["bf16"], err


def test_one_launch_after_the_parameter_kernel(gma):
    """The call launches the parameter kernel and the single-launch kernel, nothing else (the
    default path adds the segment pass, which stores Gamma_K, and the scan)."""
    w = W.scaled(W.LONG_CAUSAL, B=1, H=4, N=8192)
    host = W.make_inputs(w)
    dev = to_device(host)
    gpu_forward(w, dev, flags=gma.GMA_FLAG_SINGLE_PASS)   # (first call: module load, set-up)
    torch.cuda.synchronize()
    gma.gma_timing_enable(64)
    O = gpu_forward(w, dev, flags=gma.GMA_FLAG_SINGLE_PASS)
    torch.cuda.synchronize()
    names = [n for n, _ in gma.gma_timing_read(64)]
    gma.gma_timing_enable(0)
    assert names == ["tc_params", "tc_causal_single_launch"], names
    assert normwise_error(O.float().cpu().numpy(), oracle_forward(w, host)) <= TOL["bf16"]


def test_repeat_calls_agree(gma):
    """Segments add their predecessors' memories in whichever order the look-back finds them
    published, so two calls may differ in rounding; both stay within the bound, and close."""
    w = W.scaled(W.LONG_CAUSAL, B=1, H=4, N=20000)
    host = W.make_inputs(w)
    dev = to_device(host)
    a = gpu_forward(w, dev, flags=gma.GMA_FLAG_SINGLE_PASS).float()
    b = gpu_forward(w, dev, flags=gma.GMA_FLAG_SINGLE_PASS).float()
    ref = oracle_forward(w, host)
    assert normwise_error(a.cpu().numpy(), ref) <= TOL["bf16"]
    assert normwise_error(b.cpu().numpy(), ref) <= TOL["bf16"]
    assert (a - b).abs().max().item() <= 1e-3 * float(np.abs(ref).max())


@pytest.mark.parametrize("change", [dict(K=200), dict(dtype="f32"), dict(d_r=128)],
                         ids=["K200", "fp32", "dr128"])
def test_shapes_outside_the_family_are_rejected(gma, change):
    w = W.scaled(W.LM_CAUSAL, B=1, H=1, N=256, **change)
    dt = gma.GMA_F32 if w.dtype == "f32" else gma.GMA_BF16
    s = gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v, dt, w.eps, w.var_floor, flags=gma.GMA_FLAG_SINGLE_PASS)
    assert gma.gma_workspace_size(s, gma.GMA_VARIANT_CAUSAL) == 0
    assert gma.gma_kernel_family(s, gma.GMA_VARIANT_CAUSAL) == -1
    host = W.make_inputs(w)
    dev = to_device(host)
    with pytest.raises(gma.GmaError) as e:
        gpu_forward(w, dev, flags=gma.GMA_FLAG_SINGLE_PASS)
    assert e.value.status == gma.GMA_ERR_UNSUPPORTED_SHAPE
