"""ctypes binding over ``libgma.so`` (declared in ``include/gma.h``).

The ``gma_*`` functions have the C names and arguments (plain integers for pointers and the
stream).  ``forward`` / ``responsibilities`` marshal torch CUDA tensors into those calls: they
check dtypes and contiguity, allocate the output and workspace with torch, and pass the current
stream.  Every step of the computation runs in the library's CUDA kernels; there is no other
implementation behind this module, and importing it fails if the library is missing.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgma.so")

GMA_OK = 0
STATUS_NAMES = {0: "GMA_OK", 1: "GMA_ERR_INVALID_ARG", 2: "GMA_ERR_UNSUPPORTED_SHAPE",
                3: "GMA_ERR_RANGE", 4: "GMA_ERR_WORKSPACE", 5: "GMA_ERR_CUDA",
                6: "GMA_ERR_TIMEOUT", 7: "GMA_ERR_NO_DEVICE"}
globals().update({name: code for code, name in STATUS_NAMES.items()})
GMA_F32, GMA_BF16 = 0, 1
GMA_FLAG_SIMT = 0x1
GMA_FLAG_OUT_F32 = 0x2
GMA_FLAG_RECOMPUTE_KEYS = 0x4
GMA_FLAG_SINGLE_PASS = 0x8
GMA_FLAG_TEST_WITHHOLD = 0x80000000   # tests of the timeout path only (see include/gma.h)
(GMA_VARIANT_RESPONSIBILITIES, GMA_VARIANT_BIDIRECTIONAL, GMA_VARIANT_CAUSAL, GMA_VARIANT_DECODE,
 GMA_VARIANT_USAGE, GMA_VARIANT_BACKWARD) = 0, 1, 2, 3, 4, 5


class gma_shape_t(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("d_r", ctypes.c_int), ("K", ctypes.c_int), ("d_v", ctypes.c_int),
                ("dtype", ctypes.c_int), ("eps", ctypes.c_float), ("var_floor", ctypes.c_float),
                ("flags", ctypes.c_uint)]


class GmaError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} "
                         f"({gma_status_string(status)})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libgma.so is not built ({LIB_PATH}); run "
                          "linear_latent_routing_gb300.build.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, sp = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(gma_shape_t)
    lib.gma_workspace_size.argtypes = [sp, ctypes.c_int]
    lib.gma_workspace_size.restype = sz
    lib.gma_responsibilities.argtypes = [sp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gma_responsibilities.restype = ctypes.c_int
    for name in ("gma_forward_bidirectional", "gma_forward_causal"):
        fn = getattr(lib, name)
        fn.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        fn.restype = ctypes.c_int
    lib.gma_backward.argtypes = [sp, ctypes.c_int] + [vp] * 14 + [sz, vp]
    lib.gma_backward.restype = ctypes.c_int
    lib.gma_usage.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gma_usage.restype = ctypes.c_int
    lib.gma_workspace_size_cross.argtypes = [sp, ctypes.c_int]
    lib.gma_workspace_size_cross.restype = sz
    lib.gma_forward_cross.argtypes = [sp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gma_forward_cross.restype = ctypes.c_int
    lib.gma_decode_step.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gma_decode_step.restype = ctypes.c_int
    lib.gma_forward_causal_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.gma_forward_causal_noalloc.restype = ctypes.c_int
    lib.gma_noalloc_check.argtypes = [vp]
    lib.gma_noalloc_check.restype = ctypes.c_int
    lib.gma_check_workspace.argtypes = [vp, vp]
    lib.gma_check_workspace.restype = ctypes.c_int
    lib.gma_kernel_family.argtypes = [sp, ctypes.c_int]
    lib.gma_kernel_family.restype = ctypes.c_int
    lib.gma_status_string.argtypes = [ctypes.c_int]
    lib.gma_status_string.restype = ctypes.c_char_p
    lib.gma_timing_enable.argtypes = [ctypes.c_int]
    lib.gma_timing_enable.restype = ctypes.c_int
    lib.gma_timing_read.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float),
                                    ctypes.c_int]
    lib.gma_timing_read.restype = ctypes.c_int
    lib.gma_kernel_name.argtypes = [ctypes.c_int]
    lib.gma_kernel_name.restype = ctypes.c_char_p
    lib.gma_version.argtypes = []
    lib.gma_version.restype = ctypes.c_int
    return lib


_lib = _load()
lib = _lib


# ------------------------------------------------------------------ the C entry points

def make_shape(B, H, N, d_r, K, d_v, dtype, eps=1e-6, var_floor=1e-3, flags=0):
    return gma_shape_t(int(B), int(H), int(N), int(d_r), int(K), int(d_v), int(dtype),
                       float(eps), float(var_floor), int(flags))


def gma_workspace_size(shape, variant):
    return int(_lib.gma_workspace_size(ctypes.byref(shape), int(variant)))


def gma_kernel_family(shape, variant):
    return int(_lib.gma_kernel_family(ctypes.byref(shape), int(variant)))


def gma_responsibilities(shape, X, mu, raw_var, prior_logits, gamma, workspace, workspace_bytes,
                         stream):
    return int(_lib.gma_responsibilities(ctypes.byref(shape), X, mu, raw_var, prior_logits,
                                         gamma, workspace, int(workspace_bytes), stream))


def gma_forward_bidirectional(shape, QX, KX, V, mu, raw_var, prior_logits, O, workspace,
                              workspace_bytes, stream):
    return int(_lib.gma_forward_bidirectional(ctypes.byref(shape), QX, KX, V, mu, raw_var,
                                              prior_logits, O, workspace, int(workspace_bytes),
                                              stream))


def gma_forward_causal(shape, QX, KX, V, mu, raw_var, prior_logits, O, workspace,
                       workspace_bytes, stream):
    return int(_lib.gma_forward_causal(ctypes.byref(shape), QX, KX, V, mu, raw_var,
                                       prior_logits, O, workspace, int(workspace_bytes), stream))


def gma_backward(shape, causal, QX, KX, V, mu, raw_var, prior_logits, dO, dQX, dKX, dV, dmu, draw_var,
                 dprior_logits, workspace, workspace_bytes, stream):
    return int(_lib.gma_backward(ctypes.byref(shape), int(causal), QX, KX, V, mu, raw_var, prior_logits,
                                 dO, dQX, dKX, dV, dmu, draw_var, dprior_logits, workspace,
                                 int(workspace_bytes), stream))


def gma_usage(shape, X, mu, raw_var, prior_logits, assign, counts, mass, used, entropy, workspace,
              workspace_bytes, stream):
    return int(_lib.gma_usage(ctypes.byref(shape), X, mu, raw_var, prior_logits, assign, counts,
                              mass, used, entropy, workspace, int(workspace_bytes), stream))


def gma_workspace_size_cross(shape, n_k):
    return int(_lib.gma_workspace_size_cross(ctypes.byref(shape), int(n_k)))


def gma_forward_cross(shape, n_k, QX, KX, V, mu, raw_var, prior_logits, O, workspace,
                      workspace_bytes, stream):
    return int(_lib.gma_forward_cross(ctypes.byref(shape), int(n_k), QX, KX, V, mu, raw_var,
                                      prior_logits, O, workspace, int(workspace_bytes), stream))


def gma_decode_step(shape, qx, kx, v, mu, raw_var, prior_logits, state, o, workspace,
                    workspace_bytes, stream):
    return int(_lib.gma_decode_step(ctypes.byref(shape), qx, kx, v, mu, raw_var, prior_logits,
                                    state, o, workspace, int(workspace_bytes), stream))


GMA_NOALLOC_SCRATCH_BYTES = 32 << 20


def gma_forward_causal_noalloc(shape, QX, KX, V, mu, raw_var, prior_logits, O, stream):
    return int(_lib.gma_forward_causal_noalloc(ctypes.byref(shape), QX, KX, V, mu, raw_var,
                                               prior_logits, O, stream))


def gma_noalloc_check(stream):
    return int(_lib.gma_noalloc_check(stream))


def gma_check_workspace(workspace, stream):
    return int(_lib.gma_check_workspace(workspace, stream))


def gma_status_string(status):
    return _lib.gma_status_string(int(status)).decode()


def gma_version():
    return int(_lib.gma_version())


def gma_timing_enable(capacity):
    return int(_lib.gma_timing_enable(int(capacity)))


def gma_timing_read(cap=65536):
    """[(kernel name, ms), ...] for the launches recorded since the last read."""
    ids = (ctypes.c_int * cap)()
    ms = (ctypes.c_float * cap)()
    n = int(_lib.gma_timing_read(ids, ms, cap))
    if n < 0:
        raise GmaError(5, "gma_timing_read")
    return [(_lib.gma_kernel_name(ids[i]).decode(), float(ms[i])) for i in range(n)]


def gma_kernel_name(kernel_id):
    return _lib.gma_kernel_name(int(kernel_id)).decode()


# ------------------------------------------------------------------ torch marshalling

def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return GMA_BF16
    if t.dtype == torch.float32:
        return GMA_F32
    raise TypeError(f"activations must be bf16 or fp32, got {t.dtype}")


def _check(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream_handle(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace_for(shape, variant, device):
    torch = _torch()
    n = gma_workspace_size(shape, variant)
    if n == 0:
        raise GmaError(2, "gma_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward(QX, KX, V, mu, raw_var, prior_logits, causal, eps=1e-6, var_floor=1e-3, flags=0,
            out=None, workspace=None, stream=None, check=False):
    """GMA forward on torch CUDA tensors; returns O [B, H, N, d_v].

    QX, KX [B,H,N,d_r] and V [B,H,N,d_v] share one dtype (bf16 or fp32); mu, raw_var [H,K,d_r]
    and prior_logits [H,K] are fp32.  ``check=True`` synchronises and raises on a device-side
    condition recorded in the workspace.
    """
    torch = _torch()
    for t, n in ((QX, "QX"), (KX, "KX"), (V, "V")):
        _check(t, n, QX.dtype)
    for t, n in ((mu, "mu"), (raw_var, "raw_var"), (prior_logits, "prior_logits")):
        _check(t, n, torch.float32)
    B, H, N, d_r = QX.shape
    d_v = V.shape[-1]
    K = mu.shape[1]
    if KX.shape != QX.shape or V.shape[:3] != QX.shape[:3]:
        raise ValueError("QX, KX and V must agree on [B, H, N]")
    if mu.shape != (H, K, d_r) or raw_var.shape != (H, K, d_r) or prior_logits.shape != (H, K):
        raise ValueError("mu, raw_var must be [H, K, d_r] and prior_logits [H, K]")
    shape = make_shape(B, H, N, d_r, K, d_v, _dtype_code(QX), eps, var_floor, flags)
    variant = GMA_VARIANT_CAUSAL if causal else GMA_VARIANT_BIDIRECTIONAL
    if out is None:
        odt = torch.float32 if (flags & GMA_FLAG_OUT_F32) else QX.dtype
        out = torch.empty(B, H, N, d_v, dtype=odt, device=QX.device)
    if workspace is None:
        workspace = workspace_for(shape, variant, QX.device)
    fn = gma_forward_causal if causal else gma_forward_bidirectional
    st = _stream_handle(stream)
    r = fn(shape, QX.data_ptr(), KX.data_ptr(), V.data_ptr(), mu.data_ptr(), raw_var.data_ptr(),
           prior_logits.data_ptr(), out.data_ptr(), workspace.data_ptr(), workspace.numel(), st)
    if r != GMA_OK:
        raise GmaError(r, fn.__name__)
    if check:
        r = gma_check_workspace(workspace.data_ptr(), st)
        if r != GMA_OK:
            raise GmaError(r, "gma_check_workspace")
    return out


def forward_cross(QX, KX, V, mu, raw_var, prior_logits, eps=1e-6, var_floor=1e-3, flags=0,
                  out=None, workspace=None, stream=None, check=False):
    """Cross-attention on torch CUDA tensors; returns O [B, H, N_q, d_v].

    QX [B,H,N_q,d_r], KX [B,H,N_k,d_r] and V [B,H,N_k,d_v] share one dtype (bf16 or fp32); mu,
    raw_var [H,K,d_r] and prior_logits [H,K] are fp32.
    """
    torch = _torch()
    for t, n in ((QX, "QX"), (KX, "KX"), (V, "V")):
        _check(t, n, QX.dtype)
    for t, n in ((mu, "mu"), (raw_var, "raw_var"), (prior_logits, "prior_logits")):
        _check(t, n, torch.float32)
    B, H, N_q, d_r = QX.shape
    N_k = KX.shape[2]
    d_v = V.shape[-1]
    K = mu.shape[1]
    if KX.shape != (B, H, N_k, d_r) or V.shape[:3] != (B, H, N_k):
        raise ValueError("KX must be [B, H, N_k, d_r] and V [B, H, N_k, d_v]")
    if mu.shape != (H, K, d_r) or raw_var.shape != (H, K, d_r) or prior_logits.shape != (H, K):
        raise ValueError("mu, raw_var must be [H, K, d_r] and prior_logits [H, K]")
    shape = make_shape(B, H, N_q, d_r, K, d_v, _dtype_code(QX), eps, var_floor, flags)
    if out is None:
        odt = torch.float32 if (flags & GMA_FLAG_OUT_F32) else QX.dtype
        out = torch.empty(B, H, N_q, d_v, dtype=odt, device=QX.device)
    if workspace is None:
        n = gma_workspace_size_cross(shape, N_k)
        if n == 0:
            raise GmaError(2, "gma_workspace_size_cross")
        workspace = torch.empty(n, dtype=torch.uint8, device=QX.device)
    st = _stream_handle(stream)
    r = gma_forward_cross(shape, N_k, QX.data_ptr(), KX.data_ptr(), V.data_ptr(), mu.data_ptr(),
                          raw_var.data_ptr(), prior_logits.data_ptr(), out.data_ptr(),
                          workspace.data_ptr(), workspace.numel(), st)
    if r != GMA_OK:
        raise GmaError(r, "gma_forward_cross")
    if check:
        r = gma_check_workspace(workspace.data_ptr(), st)
        if r != GMA_OK:
            raise GmaError(r, "gma_check_workspace")
    return out


def responsibilities(X, mu, raw_var, prior_logits, var_floor=1e-3, flags=0, out=None,
                     workspace=None, stream=None, check=False):
    """Posterior responsibilities gamma [B, H, N, K] of X [B, H, N, d_r] on torch CUDA tensors."""
    torch = _torch()
    _check(X, "X")
    for t, n in ((mu, "mu"), (raw_var, "raw_var"), (prior_logits, "prior_logits")):
        _check(t, n, torch.float32)
    B, H, N, d_r = X.shape
    K = mu.shape[1]
    shape = make_shape(B, H, N, d_r, K, 16, _dtype_code(X), 0.0, var_floor, flags)
    if out is None:
        odt = torch.float32 if (flags & GMA_FLAG_OUT_F32) or X.dtype == torch.float32 else X.dtype
        out = torch.empty(B, H, N, K, dtype=odt, device=X.device)
    if workspace is None:
        workspace = workspace_for(shape, GMA_VARIANT_RESPONSIBILITIES, X.device)
    st = _stream_handle(stream)
    r = gma_responsibilities(shape, X.data_ptr(), mu.data_ptr(), raw_var.data_ptr(),
                             prior_logits.data_ptr(), out.data_ptr(), workspace.data_ptr(),
                             workspace.numel(), st)
    if r != GMA_OK:
        raise GmaError(r, "gma_responsibilities")
    if check:
        r = gma_check_workspace(workspace.data_ptr(), st)
        if r != GMA_OK:
            raise GmaError(r, "gma_check_workspace")
    return out


def decode_step(qx, kx, v, mu, raw_var, prior_logits, state, eps=1e-6, var_floor=1e-3, flags=0,
                out=None, workspace=None, stream=None, check=False):
    """One autoregressive decode step on torch CUDA tensors; returns o [B, H, d_v].

    qx, kx [B, H, d_r] and v [B, H, d_v] share one dtype (bf16 or fp32); state [B, H, K, d_v + 1]
    fp32 is updated in place; mu, raw_var [H, K, d_r] and prior_logits [H, K] are fp32.
    """
    torch = _torch()
    for t, n in ((qx, "qx"), (kx, "kx"), (v, "v")):
        _check(t, n, qx.dtype)
    for t, n in ((mu, "mu"), (raw_var, "raw_var"), (prior_logits, "prior_logits"), (state, "state")):
        _check(t, n, torch.float32)
    B, H, d_r = qx.shape
    d_v = v.shape[-1]
    K = mu.shape[1]
    if kx.shape != qx.shape or v.shape[:2] != qx.shape[:2] or state.shape != (B, H, K, d_v + 1):
        raise ValueError("qx, kx [B, H, d_r], v [B, H, d_v] and state [B, H, K, d_v + 1] must agree")
    shape = make_shape(B, H, 1, d_r, K, d_v, _dtype_code(qx), eps, var_floor, flags)
    if out is None:
        odt = torch.float32 if (flags & GMA_FLAG_OUT_F32) else qx.dtype
        out = torch.empty(B, H, d_v, dtype=odt, device=qx.device)
    if workspace is None:
        workspace = workspace_for(shape, GMA_VARIANT_DECODE, qx.device)
    st = _stream_handle(stream)
    r = gma_decode_step(shape, qx.data_ptr(), kx.data_ptr(), v.data_ptr(), mu.data_ptr(),
                        raw_var.data_ptr(), prior_logits.data_ptr(), state.data_ptr(), out.data_ptr(),
                        workspace.data_ptr(), workspace.numel(), st)
    if r != GMA_OK:
        raise GmaError(r, "gma_decode_step")
    if check:
        r = gma_check_workspace(workspace.data_ptr(), st)
        if r != GMA_OK:
            raise GmaError(r, "gma_check_workspace")
    return out


def usage(X, mu, raw_var, prior_logits, var_floor=1e-3, flags=0, workspace=None, stream=None,
          check=False):
    """Component-usage diagnostics of X [B, H, N, d_r] (torch CUDA tensor) under each head's GMM.

    Returns a dict of CUDA tensors: assign [B, H, N] int32, counts [H, K] int32, mass [H, K]
    fp32, used [H] int32, entropy [H] fp32 (see gma_usage in include/gma.h).
    """
    torch = _torch()
    _check(X, "X")
    for t, n in ((mu, "mu"), (raw_var, "raw_var"), (prior_logits, "prior_logits")):
        _check(t, n, torch.float32)
    B, H, N, d_r = X.shape
    K = mu.shape[1]
    if mu.shape != (H, K, d_r) or raw_var.shape != (H, K, d_r) or prior_logits.shape != (H, K):
        raise ValueError("mu, raw_var must be [H, K, d_r] and prior_logits [H, K]")
    shape = make_shape(B, H, N, d_r, K, 16, _dtype_code(X), 1e-6, var_floor, flags)
    dev = X.device
    out = {"assign": torch.empty(B, H, N, dtype=torch.int32, device=dev),
           "counts": torch.empty(H, K, dtype=torch.int32, device=dev),
           "mass": torch.empty(H, K, dtype=torch.float32, device=dev),
           "used": torch.empty(H, dtype=torch.int32, device=dev),
           "entropy": torch.empty(H, dtype=torch.float32, device=dev)}
    if workspace is None:
        workspace = workspace_for(shape, GMA_VARIANT_USAGE, dev)
    st = _stream_handle(stream)
    r = gma_usage(shape, X.data_ptr(), mu.data_ptr(), raw_var.data_ptr(), prior_logits.data_ptr(),
                  out["assign"].data_ptr(), out["counts"].data_ptr(), out["mass"].data_ptr(),
                  out["used"].data_ptr(), out["entropy"].data_ptr(), workspace.data_ptr(),
                  workspace.numel(), st)
    if r != GMA_OK:
        raise GmaError(r, "gma_usage")
    if check:
        r = gma_check_workspace(workspace.data_ptr(), st)
        if r != GMA_OK:
            raise GmaError(r, "gma_check_workspace")
    return out


def backward(QX, KX, V, mu, raw_var, prior_logits, dO, causal, eps=1e-6, var_floor=1e-3, workspace=None,
             stream=None, check=False):
    """Gradients of sum(dO * O) for the forward pass with the same arguments (torch CUDA tensors).

    Returns (dQX, dKX, dV, dmu, draw_var, dprior_logits): the first three in the inputs' dtype,
    the parameter gradients fp32 and summed over the batch.
    """
    torch = _torch()
    for t, n in ((QX, "QX"), (KX, "KX"), (V, "V"), (dO, "dO")):
        _check(t, n, QX.dtype)
    for t, n in ((mu, "mu"), (raw_var, "raw_var"), (prior_logits, "prior_logits")):
        _check(t, n, torch.float32)
    B, H, N, d_r = QX.shape
    d_v = V.shape[-1]
    K = mu.shape[1]
    if KX.shape != QX.shape or V.shape[:3] != QX.shape[:3] or dO.shape != V.shape:
        raise ValueError("QX, KX [B,H,N,d_r] and V, dO [B,H,N,d_v] must agree")
    shape = make_shape(B, H, N, d_r, K, d_v, _dtype_code(QX), eps, var_floor, 0)
    outs = [torch.empty_like(QX), torch.empty_like(KX), torch.empty_like(V), torch.empty_like(mu),
            torch.empty_like(raw_var), torch.empty_like(prior_logits)]
    if workspace is None:
        workspace = workspace_for(shape, GMA_VARIANT_BACKWARD, QX.device)
    st = _stream_handle(stream)
    r = gma_backward(shape, 1 if causal else 0, QX.data_ptr(), KX.data_ptr(), V.data_ptr(), mu.data_ptr(),
                     raw_var.data_ptr(), prior_logits.data_ptr(), dO.data_ptr(),
                     *[t.data_ptr() for t in outs], workspace.data_ptr(), workspace.numel(), st)
    if r != GMA_OK:
        raise GmaError(r, "gma_backward")
    if check:
        r = gma_check_workspace(workspace.data_ptr(), st)
        if r != GMA_OK:
            raise GmaError(r, "gma_check_workspace")
    return tuple(outs)

