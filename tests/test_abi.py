"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and exports every
function include/gma.h declares; validation and workspace sizing behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    from linear_latent_routing_gb300 import build
    build.build()
    from linear_latent_routing_gb300 import gma
    return gma


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(gma_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("gma_responsibilities", "gma_forward_bidirectional", "gma_forward_causal",
              "gma_workspace_size", "gma_check_workspace", "gma_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(g):
    lib = ctypes.CDLL(g.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(g):
    for code in range(8):
        s = g.gma_status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert g.gma_status_string(99) == "unknown status"
    assert g.gma_version() >= 100


def _shape(g, **kw):
    d = dict(B=2, H=3, N=100, d_r=64, K=64, d_v=64, dtype=g.GMA_BF16)
    d.update(kw)
    return g.make_shape(**d)


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_workspace_size_valid_shapes(g, variant):
    s = _shape(g)
    n = g.gma_workspace_size(s, variant)
    assert n > 256 and n % 256 == 0
    assert g.gma_kernel_family(s, variant) in (0, 1)


@pytest.mark.parametrize("bad", [dict(B=0), dict(N=-1), dict(K=0), dict(K=1025), dict(d_r=48),
                                 dict(d_v=8), dict(dtype=7), dict(eps=-1.0),
                                 dict(var_floor=float("nan")), dict(flags=0x80)])
def test_invalid_shapes_have_no_workspace(g, bad):
    s = _shape(g, **bad)
    assert g.gma_workspace_size(s, g.GMA_VARIANT_CAUSAL) == 0
    assert g.gma_kernel_family(s, g.GMA_VARIANT_CAUSAL) == -1


def test_single_pass_flag_validation(g):
    """GMA_FLAG_SINGLE_PASS exists in the tensor-core family only: a causal shape that family
    cannot take (fp32 inputs here, on any machine) has no workspace and no family with it, while
    the same shape without the flag is valid; the bidirectional entry points ignore the flag; an
    undefined flag bit is still refused."""
    sp = g.GMA_FLAG_SINGLE_PASS
    f32 = _shape(g, dtype=g.GMA_F32, flags=sp)
    assert g.gma_workspace_size(f32, g.GMA_VARIANT_CAUSAL) == 0
    assert g.gma_kernel_family(f32, g.GMA_VARIANT_CAUSAL) == -1
    assert g.gma_workspace_size(_shape(g, dtype=g.GMA_F32), g.GMA_VARIANT_CAUSAL) > 0
    assert g.gma_workspace_size(f32, g.GMA_VARIANT_BIDIRECTIONAL) == \
        g.gma_workspace_size(_shape(g, dtype=g.GMA_F32), g.GMA_VARIANT_BIDIRECTIONAL) > 0
    assert g.gma_workspace_size(_shape(g, flags=0x10), g.GMA_VARIANT_CAUSAL) == 0


def test_single_pass_header_value_matches_binding(g):
    text = open(os.path.join(ROOT, "include", "gma.h")).read()
    m = re.search(r"#define GMA_FLAG_SINGLE_PASS (0x[0-9a-fA-F]+)u", text)
    assert m and int(m.group(1), 16) == g.GMA_FLAG_SINGLE_PASS


def test_responsibilities_ignore_value_dimension(g):
    s = _shape(g, d_v=7)
    assert g.gma_workspace_size(s, g.GMA_VARIANT_RESPONSIBILITIES) > 0
    assert g.gma_workspace_size(s, g.GMA_VARIANT_CAUSAL) == 0


def test_workspace_grows_linearly_in_sequence_length(g):
    # the page's profiling claim: activation memory O(N K) at fixed K
    sizes = [g.gma_workspace_size(_shape(g, N=n), g.GMA_VARIANT_CAUSAL) for n in (4096, 8192, 16384)]
    d1, d2 = sizes[1] - sizes[0], sizes[2] - sizes[1]
    assert abs(d2 - 2 * d1) <= 4096


def test_bad_arguments_rejected_before_any_device_work(g):
    s = _shape(g)
    ws_n = g.gma_workspace_size(s, g.GMA_VARIANT_CAUSAL)
    fake = 1 << 20   # never dereferenced: validation fails first
    args = [fake] * 7
    # null pointer
    r = g.gma_forward_causal(s, None, *args[1:], fake, ws_n, None)
    assert r == 1
    # misaligned pointer
    r = g.gma_forward_causal(s, fake + 8, *args[1:], fake, ws_n, None)
    assert r == 1
    # workspace too small / misaligned
    r = g.gma_forward_causal(s, *args, fake, ws_n - 1, None)
    assert r == 4
    r = g.gma_forward_causal(s, *args, fake + 16, ws_n, None)
    assert r == 4
    # unsupported shape
    r = g.gma_forward_bidirectional(_shape(g, d_v=24), *args, fake, ws_n, None)
    assert r == 2
    r = g.gma_responsibilities(_shape(g, K=2000), *args[:5], fake, ws_n, None)
    assert r == 2


def test_no_device_is_reported_without_a_gpu(g):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    s = _shape(g)
    ws_n = g.gma_workspace_size(s, g.GMA_VARIANT_CAUSAL)
    fake = 1 << 20
    r = g.gma_forward_causal(s, *([fake] * 7), fake, ws_n, None)
    assert r == 7


def test_decode_step_validation(g):
    """gma_decode_step takes N == 1 only and refuses null pointers before touching the device;
    its workspace and kernel family follow the decode variant."""
    s1 = _shape(g, N=1)
    s2 = _shape(g, N=2)
    assert g.gma_workspace_size(s1, g.GMA_VARIANT_DECODE) > 0
    assert g.gma_workspace_size(s2, g.GMA_VARIANT_DECODE) == 0
    assert g.gma_kernel_family(s1, g.GMA_VARIANT_DECODE) == 0
    assert g.gma_kernel_family(s2, g.GMA_VARIANT_DECODE) == -1
    assert g.gma_decode_step(s2, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == g.GMA_ERR_INVALID_ARG
    assert g.gma_decode_step(s1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == g.GMA_ERR_INVALID_ARG
    assert g.gma_decode_step(_shape(g, N=1, K=0), 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) != g.GMA_OK


def test_cross_workspace_and_validation(g):
    """Cross-attention: n_k >= 1; with n_k == N the workspace is the bidirectional one; invalid
    arguments are refused before anything is enqueued."""
    s = _shape(g, N=100)
    assert g.gma_workspace_size_cross(s, 0) == 0
    assert g.gma_workspace_size_cross(s, -3) == 0
    assert g.gma_workspace_size_cross(s, 100) == g.gma_workspace_size(s, g.GMA_VARIANT_BIDIRECTIONAL)
    assert g.gma_workspace_size_cross(s, 5000) > g.gma_workspace_size_cross(s, 100)
    f32 = _shape(g, N=100, dtype=g.GMA_F32)
    assert g.gma_workspace_size_cross(f32, 7) > 0
    assert g.gma_forward_cross(s, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == g.GMA_ERR_INVALID_ARG
    assert g.gma_forward_cross(s, 50, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == g.GMA_ERR_INVALID_ARG


def test_usage_workspace_and_validation(g):
    s = _shape(g, N=100, K=100)
    f32 = _shape(g, N=100, K=100, dtype=g.GMA_F32)
    # the fp32 CUDA-core family keeps the responsibilities of every token; the tensor-core family
    # computes the diagnostics in the responsibilities pass and keeps per-CTA sums only
    assert g.gma_workspace_size(f32, g.GMA_VARIANT_USAGE) >= 2 * 3 * 100 * 100 * 4
    n = g.gma_workspace_size(s, g.GMA_VARIANT_USAGE)
    if g.gma_kernel_family(s, g.GMA_VARIANT_USAGE) == 1:   # (the family needs the CUDA driver)
        assert 0 < n < 2 * 3 * 100 * 100 * 4
    else:
        assert n >= 2 * 3 * 100 * 100 * 4
    assert g.gma_kernel_family(s, g.GMA_VARIANT_USAGE) == g.gma_kernel_family(s, g.GMA_VARIANT_RESPONSIBILITIES)
    assert g.gma_workspace_size(_shape(g, N=100, K=0), g.GMA_VARIANT_USAGE) == 0
    assert g.gma_usage(s, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == g.GMA_ERR_INVALID_ARG


def test_backward_workspace_and_validation(g):
    s = _shape(g, N=100)
    assert g.gma_workspace_size(s, g.GMA_VARIANT_BACKWARD) >= 4 * 2 * 3 * 100 * 64 * 4
    assert g.gma_kernel_family(s, g.GMA_VARIANT_BACKWARD) == 0
    assert g.gma_backward(s, 0, *([0] * 15), None) == g.GMA_ERR_INVALID_ARG
    assert g.gma_backward(s, 2, *([0] * 15), None) == g.GMA_ERR_INVALID_ARG
