"""The device-side timeout path, exercised without faulting or hanging the GPU.

Every wait of the tensor-core kernels is bounded.  GMA_FLAG_TEST_WITHHOLD (test only) shortens
the bound to about a millisecond and makes the key pass withhold one row-phase hand-off (the
signal that the first chunk's [x^2, x] tile is built, a barrier only CUDA-core threads arrive
on).  The waits on it run out, the kernel records GMA_ERR_TIMEOUT in the workspace header, every
role leaves its loop and the tensor memory is released.  The test checks that the call returns,
that gma_check_workspace reports the timeout, and that the next call on the same stream and
workspace runs normally and matches the oracle (which it could not do if an aborted CTA had kept
its tensor memory: the next CTAs would wait for it)."""
import time

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


@pytest.mark.parametrize("w,single", [(W.scaled(W.LONG_CAUSAL, B=1, H=2, N=1500), False),
                                      (W.scaled(W.LRA_BIDIR, B=2, H=1, N=900), False),
                                      (W.scaled(W.LONG_CAUSAL, B=2, H=2, N=1500), True)],
                         ids=["causal", "bidirectional", "causal_single_pass"])
def test_withheld_handoff_times_out_and_next_call_is_clean(gma, w, single):
    """With the single-launch causal kernel only the first segment of each slice withholds the
    hand-off; every other segment (twelve per slice here) must learn of it through the look-back
    and stop instead of waiting for a prefix that never comes."""
    host = W.make_inputs(w)
    dev = to_device(host)
    variant = gma.GMA_VARIANT_CAUSAL if w.causal else gma.GMA_VARIANT_BIDIRECTIONAL
    fn = gma.gma_forward_causal if w.causal else gma.gma_forward_bidirectional
    base = gma.GMA_FLAG_SINGLE_PASS if single else 0
    test = gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v, gma.GMA_BF16, w.eps, w.var_floor,
                          flags=base | gma.GMA_FLAG_TEST_WITHHOLD)
    normal = gma.make_shape(w.B, w.H, w.N, w.d_r, w.K, w.d_v, gma.GMA_BF16, w.eps, w.var_floor, flags=base)
    assert gma.gma_kernel_family(test, variant) == 1
    ws_n = gma.gma_workspace_size(normal, variant)
    assert gma.gma_workspace_size(test, variant) == ws_n
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    O = torch.empty(w.B, w.H, w.N, w.d_v, dtype=torch.bfloat16, device="cuda")
    ptrs = [dev[k].data_ptr() for k in ("QX", "KX", "V", "mu", "raw", "logits")]
    st = torch.cuda.Stream()
    sh = st.cuda_stream

    t0 = time.time()
    assert fn(test, *ptrs, O.data_ptr(), ws.data_ptr(), ws_n, sh) == 0
    status = gma.gma_check_workspace(ws.data_ptr(), sh)
    took = time.time() - t0
    assert status == gma.GMA_ERR_TIMEOUT, gma.gma_status_string(status)
    assert took < 10.0   # millisecond waits, not the one-second production bound per wait

    for _ in range(2):
        O.fill_(float("nan"))
        assert fn(normal, *ptrs, O.data_ptr(), ws.data_ptr(), ws_n, sh) == 0
        assert gma.gma_check_workspace(ws.data_ptr(), sh) == 0
        got = O.float().cpu().numpy()
        assert np.isfinite(got).all()
        assert normwise_error(got, oracle_forward(w, host)) <= TOL["bf16"]
