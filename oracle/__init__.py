"""fp64 CPU oracle for the Gaussian Mixture Attention (GMA) forward pass.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()`` and by the CPU
baseline leg of ``bench.py``.  The CUDA library never imports, links or calls anything here, and
this package imports nothing from the CUDA library.

Two independent formulations of the same definition
(page "Attention par Mélange Gaussien (GMA)", gist.science/fr/paper/2606.18283, Méthodologie):

* ``forward`` / ``responsibilities`` / ``params`` -- the linear (latent-memory) form in plain C,
  fp64, one token at a time (``gma_oracle.c``);
* ``oracle.bruteforce`` -- the explicit N x N affinity form in numpy fp64, for tiny inputs.

Inputs are numpy arrays (any float dtype; they are widened to float64 exactly).
"""
import ctypes
import numpy as np

from .build import build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gmao_params.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, ctypes.c_double, dp, dp]
        lib.gmao_params.restype = None
        lib.gmao_responsibilities.argtypes = [ctypes.c_int] * 3 + [dp] * 4 + [ctypes.c_double, dp]
        lib.gmao_responsibilities.restype = None
        lib.gmao_forward.argtypes = ([ctypes.c_int] * 7 + [dp] * 6
                                     + [ctypes.c_double, ctypes.c_double, dp, ctypes.c_int])
        lib.gmao_forward.restype = ctypes.c_int
        lib.gmao_decode_step.argtypes = [ctypes.c_int] * 5 + [dp] * 6 + [ctypes.c_double] * 2 + [dp] * 2
        lib.gmao_decode_step.restype = None
        lib.gmao_forward_cross.argtypes = ([ctypes.c_int] * 7 + [dp] * 6
                                           + [ctypes.c_double, ctypes.c_double, dp])
        lib.gmao_forward_cross.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def params(raw, logits, var_floor):
    """sigma^2 = softplus(raw) + var_floor and log pi = log softmax(logits), for one head.

    raw: [K, d_r]; logits: [K].  Returns (var [K, d_r], logpi [K]) as float64.
    """
    raw = _f64(raw)
    logits = _f64(logits)
    K, d_r = raw.shape
    var = np.empty((K, d_r))
    logpi = np.empty(K)
    _load().gmao_params(K, d_r, _p(raw), _p(logits), float(var_floor), _p(var), _p(logpi))
    return var, logpi


def responsibilities(X, mu, raw, logits, var_floor):
    """GMM posterior responsibilities p(z = k | x) of the rows of X for one head.

    X: [N, d_r]; mu, raw: [K, d_r]; logits: [K].  Returns gamma [N, K] float64.
    """
    X = _f64(X)
    mu = _f64(mu)
    raw = _f64(raw)
    logits = _f64(logits)
    N, d_r = X.shape
    K = mu.shape[0]
    g = np.empty((N, K))
    _load().gmao_responsibilities(N, d_r, K, _p(X), _p(mu), _p(raw), _p(logits),
                                  float(var_floor), _p(g))
    return g


def forward(causal, QX, KX, V, mu, raw, logits, var_floor, eps, nthreads=0, return_threads=False):
    """GMA forward output O [B, H, N, d_v] (float64) for all slices.

    QX, KX: [B, H, N, d_r]; V: [B, H, N, d_v]; mu, raw: [H, K, d_r]; logits: [H, K].
    ``causal`` selects the prefix-sum variant.  ``nthreads`` caps the OpenMP threads (0 = all).
    """
    QX = _f64(QX)
    KX = _f64(KX)
    V = _f64(V)
    mu = _f64(mu)
    raw = _f64(raw)
    logits = _f64(logits)
    B, H, N, d_r = QX.shape
    d_v = V.shape[-1]
    K = mu.shape[1]
    assert KX.shape == QX.shape and V.shape[:3] == QX.shape[:3]
    assert mu.shape == (H, K, d_r) and raw.shape == (H, K, d_r) and logits.shape == (H, K)
    O = np.empty((B, H, N, d_v))
    used = _load().gmao_forward(int(bool(causal)), B, H, N, d_r, K, d_v, _p(QX), _p(KX), _p(V),
                                _p(mu), _p(raw), _p(logits), float(var_floor), float(eps), _p(O),
                                int(nthreads))
    return (O, used) if return_threads else O


def decode_step(qx, kx, v, mu, raw, logits, var_floor, eps, state):
    """One autoregressive step of the causal variant for every (batch, head) slice.

    qx, kx: [B, H, d_r]; v: [B, H, d_v]; state: [B, H, K, d_v + 1] (the prefix memory V~ and, in
    the last column, the normaliser Z).  Returns (o [B, H, d_v], the updated state), float64;
    the state passed in is not modified.
    """
    qx = _f64(qx)
    kx = _f64(kx)
    v = _f64(v)
    mu = _f64(mu)
    raw = _f64(raw)
    logits = _f64(logits)
    S = np.array(state, dtype=np.float64, copy=True, order="C")
    B, H, d_r = qx.shape
    d_v = v.shape[-1]
    K = mu.shape[1]
    assert S.shape == (B, H, K, d_v + 1)
    o = np.empty((B, H, d_v))
    _load().gmao_decode_step(B, H, d_r, K, d_v, _p(qx), _p(kx), _p(v), _p(mu), _p(raw), _p(logits),
                             float(var_floor), float(eps), _p(S), _p(o))
    return o, S


def forward_cross(QX, KX, V, mu, raw, logits, var_floor, eps):
    """Cross-attention on the bidirectional path: O [B, H, Nq, d_v] (float64).

    QX: [B, H, Nq, d_r]; KX: [B, H, Nk, d_r]; V: [B, H, Nk, d_v].
    """
    QX = _f64(QX)
    KX = _f64(KX)
    V = _f64(V)
    mu = _f64(mu)
    raw = _f64(raw)
    logits = _f64(logits)
    B, H, Nq, d_r = QX.shape
    Nk = KX.shape[2]
    d_v = V.shape[-1]
    K = mu.shape[1]
    assert KX.shape == (B, H, Nk, d_r) and V.shape[:3] == (B, H, Nk)
    O = np.empty((B, H, Nq, d_v))
    _load().gmao_forward_cross(B, H, Nq, Nk, d_r, K, d_v, _p(QX), _p(KX), _p(V), _p(mu), _p(raw),
                               _p(logits), float(var_floor), float(eps), _p(O))
    return O



def usage_from_assign(assign, K):
    """Usage statistics of hard assignments, per head.

    assign: [B, H, N] integer component indices.  Returns (counts [H, K] int64, used [H] int64,
    entropy [H] float64): counts[h, k] = number of tokens of head h assigned to k; used = number
    of components with a non-zero count; entropy = -sum_k p_k ln p_k / ln K with p = counts /
    tokens (0 log 0 = 0), the usage entropy normalised to [0, 1] (0 for K = 1).
    """
    assign = np.asarray(assign)
    B, H, N = assign.shape
    counts = np.zeros((H, K), dtype=np.int64)
    for h in range(H):
        counts[h] = np.bincount(assign[:, h, :].reshape(-1), minlength=K)[:K]
    used = (counts > 0).sum(axis=1)
    entropy = np.zeros(H)
    if K > 1:
        for h in range(H):
            p = counts[h] / max(counts[h].sum(), 1)
            nz = p[p > 0]
            entropy[h] = float(-(nz * np.log(nz)).sum() / np.log(K))
    return counts, used, entropy


def usage(X, mu, raw, logits, var_floor):
    """Component-usage diagnostics of the rows of X under each head's GMM (the page's
    interpretability measurements, Résultats et Performance: components used, usage entropy,
    hard assignments).

    X: [B, H, N, d_r]; mu, raw: [H, K, d_r]; logits: [H, K].  Returns a dict of
    assign [B, H, N] int64 (argmax_k of the posterior, the lowest k on ties), mass [H, K] float64
    (sum over tokens of the responsibilities), gamma_max [B, H, N] float64 (the largest
    responsibility of each token) and counts, used, entropy as in usage_from_assign.
    """
    X = _f64(X)
    B, H, N, _ = X.shape
    K = np.asarray(mu).shape[1]
    assign = np.empty((B, H, N), dtype=np.int64)
    gmax = np.empty((B, H, N))
    mass = np.zeros((H, K))
    for h in range(H):
        for b in range(B):
            g = responsibilities(X[b, h], mu[h], raw[h], logits[h], var_floor)
            assign[b, h] = np.argmax(g, axis=1)
            gmax[b, h] = g.max(axis=1)
            mass[h] += g.sum(axis=0)
    counts, used, entropy = usage_from_assign(assign, K)
    return {"assign": assign, "mass": mass, "gamma_max": gmax, "counts": counts, "used": used,
            "entropy": entropy}


def backward(causal, QX, KX, V, mu, raw, logits, var_floor, eps, dO):
    """Gradients of sum(dO * O) with respect to every input of the forward pass (the page's
    training path: Méthodologie §3, end-to-end training by backpropagation through the softmax
    posteriors and the ratio), written out from the explicit affinity form, one slice at a time.

    QX, KX: [B, H, N, d_r]; V, dO: [B, H, N, d_v]; mu, raw: [H, K, d_r]; logits: [H, K].
    Returns (dQX, dKX, dV, dmu, draw, dlogits) in float64, the parameter gradients summed over
    the batch.

    Per slice, with A = Gamma_Q Gamma_K^T (lower triangle kept for the causal variant),
    num = A V, den = A 1 + eps, O = num / den:
      dnum = dO / den,  dden = -rowsum(dO * num) / den^2,  dA = dnum V^T + dden 1^T (masked),
      dV = A^T dnum,  dGamma_Q = dA Gamma_K,  dGamma_K = dA^T Gamma_Q,
      dL = Gamma * (dGamma - rowsum(Gamma * dGamma))             (softmax over components),
    and through L_k = log pi_k - 1/2 sum_d [(x_d - mu_kd)^2 / s_kd + log s_kd], s = softplus(raw)
    + floor, log pi = logits - logsumexp(logits):
      dx_d   = -sum_k dL_k (x_d - mu_kd) / s_kd
      dmu_kd = sum_rows dL_k (x_d - mu_kd) / s_kd
      ds_kd  = sum_rows dL_k [ (x_d - mu_kd)^2 / (2 s_kd^2) - 1 / (2 s_kd) ],  draw = ds * sigmoid(raw)
      dlogits_j = sum_rows dL_j - pi_j sum_rows sum_k dL_k.
    """
    QX, KX, V, dO = _f64(QX), _f64(KX), _f64(V), _f64(dO)
    mu, raw, logits = _f64(mu), _f64(raw), _f64(logits)
    B, H, N, d_r = QX.shape
    K = mu.shape[1]
    dQX = np.zeros_like(QX)
    dKX = np.zeros_like(KX)
    dV = np.zeros_like(V)
    dmu = np.zeros_like(mu)
    ds = np.zeros_like(raw)
    dlogpi = np.zeros((H, K))
    mask = np.tril(np.ones((N, N))) if causal else np.ones((N, N))
    for h in range(H):
        var, logpi = params(raw[h], logits[h], var_floor)
        w = 1.0 / var
        for b in range(B):
            GQ = responsibilities(QX[b, h], mu[h], raw[h], logits[h], var_floor)
            GK = responsibilities(KX[b, h], mu[h], raw[h], logits[h], var_floor)
            A = (GQ @ GK.T) * mask
            num = A @ V[b, h]
            den = A.sum(axis=1) + eps
            dnum = dO[b, h] / den[:, None]
            dden = -(dO[b, h] * num).sum(axis=1) / den ** 2
            dA = (dnum @ V[b, h].T + dden[:, None]) * mask
            dV[b, h] = A.T @ dnum
            for X, G, dG, dX in ((QX[b, h], GQ, dA @ GK, dQX[b, h]), (KX[b, h], GK, dA.T @ GQ, dKX[b, h])):
                dL = G * (dG - (G * dG).sum(axis=1, keepdims=True))
                diff = X[:, None, :] - mu[h][None, :, :]                  # [N, K, d_r]
                t = dL[:, :, None] * w[None, :, :] * diff
                dX[...] = -t.sum(axis=1)
                dmu[h] += t.sum(axis=0)
                ds[h] += (dL[:, :, None] * (0.5 * w[None] ** 2 * diff ** 2 - 0.5 * w[None])).sum(axis=0)
                dlogpi[h] += dL.sum(axis=0)
    pi = np.exp(logits - logits.max(axis=1, keepdims=True))
    pi /= pi.sum(axis=1, keepdims=True)
    dlogits = dlogpi - pi * dlogpi.sum(axis=1, keepdims=True)
    draw = ds / (1.0 + np.exp(-raw))
    return dQX, dKX, dV, dmu, draw, dlogits
