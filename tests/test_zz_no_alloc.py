"""gma_forward_causal_noalloc: the causal entry point for callers that cannot allocate device
memory (allocator callbacks, plugins whose host owns every allocation, loops that must not call
cudaMalloc).  It takes its workspace from a fixed array inside the library instead of from the
caller, so it is checked here against the regular entry point, gma_forward_causal, on the same
inputs, twice in a row (the second call reuses the array the first one left behind).

This file is named to be collected last, so that a run that stops at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from linear_latent_routing_gb300 import inputs as W
from parity import TOL, normwise_error, oracle_forward, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gma():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_latent_routing_gb300 import build
    build.build()
    from linear_latent_routing_gb300 import gma as g
    return g


def _shape(g, w):
    return g.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v,
                        g.GMA_BF16 if w.dtype == "bf16" else g.GMA_F32, w.eps, w.var_floor)


def test_noalloc_matches_regular_entry_point_twice(gma):
    w = W.scaled(W.LM_CAUSAL, B=1, H=2, N=1000)
    host = W.make_inputs(w)
    dev = to_device(host)
    shape = _shape(gma, w)
    ptrs = [dev[k].data_ptr() for k in ("QX", "KX", "V", "mu", "raw", "logits")]
    stream = torch.cuda.current_stream().cuda_stream

    # the existing entry point, with a caller-owned workspace
    ws_n = gma.gma_workspace_size(shape, gma.GMA_VARIANT_CAUSAL)
    assert 0 < ws_n <= gma.GMA_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    O_ref = torch.empty(w.B, w.H, w.N, w.d_v, dtype=torch.bfloat16, device="cuda")
    assert gma.gma_forward_causal(shape, *ptrs, O_ref.data_ptr(), ws.data_ptr(), ws_n,
                                  stream) == 0
    assert gma.gma_check_workspace(ws.data_ptr(), stream) == 0
    ref = O_ref.float().cpu().numpy()

    for _ in range(2):
        O = torch.full((w.B, w.H, w.N, w.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        r = gma.gma_forward_causal_noalloc(shape, *ptrs, O.data_ptr(), stream)
        assert r == 0, gma.gma_status_string(r)
        assert gma.gma_noalloc_check(stream) == 0
        torch.cuda.synchronize()
        got = O.float().cpu().numpy()
        assert np.isfinite(got).all()
        assert normwise_error(got, ref) <= TOL["bf16"]
    # and both against the oracle
    assert normwise_error(got, oracle_forward(w, host)) <= TOL["bf16"]


def _sizes(gma, w):
    full = _shape(gma, w)
    small = gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v, gma.GMA_BF16, w.eps, w.var_floor,
                           flags=gma.GMA_FLAG_RECOMPUTE_KEYS)
    return (full, gma.gma_workspace_size(full, gma.GMA_VARIANT_CAUSAL),
            gma.gma_workspace_size(small, gma.GMA_VARIANT_CAUSAL))


def test_noalloc_falls_back_to_the_smaller_workspace(gma):
    """A shape whose default workspace exceeds the array but whose recompute-keys workspace fits
    runs as if GMA_FLAG_RECOMPUTE_KEYS were set."""
    w = W.scaled(W.LM_CAUSAL, B=1, H=16, N=32768)
    shape, n_full, n_small = _sizes(gma, w)
    assert n_full > gma.GMA_NOALLOC_SCRATCH_BYTES >= n_small
    host = W.make_inputs(w)
    dev = to_device(host)
    ptrs = [dev[k].data_ptr() for k in ("QX", "KX", "V", "mu", "raw", "logits")]
    stream = torch.cuda.current_stream().cuda_stream
    O = torch.full((w.B, w.H, w.N, w.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    r = gma.gma_forward_causal_noalloc(shape, *ptrs, O.data_ptr(), stream)
    assert r == 0, gma.gma_status_string(r)
    from parity import gpu_forward
    ref = gpu_forward(w, dev, flags=gma.GMA_FLAG_RECOMPUTE_KEYS)
    torch.cuda.synchronize()
    assert torch.equal(O, ref)
    n = 2048
    exact = oracle_forward(w, host, b=0, h=w.H - 1, n=n)
    assert normwise_error(O[0:1, w.H - 1:w.H, :n].float().cpu().numpy(), exact) <= TOL["bf16"]


def test_noalloc_rejects_shapes_beyond_its_scratch(gma):
    # 512 heads: the per-head tables and segment memories alone exceed the array, whatever the
    # segment split, so the call must return before enqueuing anything.  Every pointer is null:
    # if a change ever let such a call past the size check, the regular entry point would reject
    # the null pointers (GMA_ERR_INVALID_ARG) before anything is enqueued.
    w = W.scaled(W.LONG_CAUSAL, H=512, N=4096)
    shape, n_full, n_small = _sizes(gma, w)
    assert n_small > gma.GMA_NOALLOC_SCRATCH_BYTES
    r = gma.gma_forward_causal_noalloc(shape, *([None] * 7), None)
    assert r == 4   # GMA_ERR_WORKSPACE
    bad = gma.make_shape(1, 1, 10, 48, 8, 16, gma.GMA_BF16)
    assert gma.gma_forward_causal_noalloc(bad, *([None] * 7), None) == 2   # unsupported d_r
    ok_shape = _shape(gma, W.scaled(W.LM_CAUSAL, B=1, H=1, N=100))
    assert gma.gma_forward_causal_noalloc(ok_shape, *([None] * 7), None) == 1   # null pointers


def test_noalloc_check_reports_a_device_side_condition(gma):
    """A condition only the device can find reaches the caller through gma_noalloc_check: raw
    variances of -20 with no floor give 1/sigma^2 near 5e8, beyond the fp16 table the tensor
    cores read, which the table kernel records as GMA_ERR_RANGE.  A normal call afterwards
    reports GMA_OK again (each call clears the condition)."""
    w = W.scaled(W.LM_CAUSAL, B=1, H=1, N=300)
    host = W.make_inputs(w)
    host["raw"] = torch.full_like(host["raw"], -20.0)
    dev = to_device(host)
    shape = gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v, gma.GMA_BF16, w.eps, 0.0)
    assert gma.gma_kernel_family(shape, gma.GMA_VARIANT_CAUSAL) == 1
    ptrs = [dev[k].data_ptr() for k in ("QX", "KX", "V", "mu", "raw", "logits")]
    stream = torch.cuda.current_stream().cuda_stream
    O = torch.empty(w.B, w.H, w.N, w.d_v, dtype=torch.bfloat16, device="cuda")
    assert gma.gma_forward_causal_noalloc(shape, *ptrs, O.data_ptr(), stream) == 0
    assert gma.gma_noalloc_check(stream) == 3   # GMA_ERR_RANGE
    good = to_device(W.make_inputs(w))
    shape = _shape(gma, w)
    ptrs = [good[k].data_ptr() for k in ("QX", "KX", "V", "mu", "raw", "logits")]
    assert gma.gma_forward_causal_noalloc(shape, *ptrs, O.data_ptr(), stream) == 0
    assert gma.gma_noalloc_check(stream) == 0
