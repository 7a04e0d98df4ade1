"""Explicit-affinity (N x N) form of GMA in numpy fp64 -- the second, independent oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  For tiny inputs only: it materialises the
N x N affinity that the linear form avoids.

Page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283), Méthodologie §2:
the implicit affinity is A~ = Gamma_Q Gamma_K^T, and O = Gamma_Q V~ / (Gamma_Q Z + eps) with
V~ = Gamma_K^T V and Z = Gamma_K^T 1.  By associativity this is O = A~ V / (A~ 1 + eps); the
causal variant (§3) keeps only keys j <= i, i.e. A~ masked to its lower triangle.

The posterior here is assembled from library routines (scipy's normal log-density and softmax),
not from the C oracle's expression, so agreement between the two pins both.
"""
import numpy as np
from scipy.special import softmax, log_softmax
from scipy.stats import norm


def softplus(r):
    r = np.asarray(r, dtype=np.float64)
    return np.logaddexp(0.0, r)


def posterior(X, mu, var, logits):
    """p(z = k | x) for each row of X via scipy: [N, K]."""
    X = np.asarray(X, dtype=np.float64)
    logp = norm.logpdf(X[:, None, :], loc=mu[None, :, :], scale=np.sqrt(var)[None, :, :]).sum(-1)
    logp = logp + log_softmax(np.asarray(logits, dtype=np.float64))[None, :]
    return softmax(logp, axis=1)


def affinity(QX, KX, mu, raw, logits, var_floor):
    """A~ = Gamma_Q Gamma_K^T for one (batch, head) slice."""
    var = softplus(raw) + var_floor
    gq = posterior(QX, np.asarray(mu, np.float64), var, logits)
    gk = posterior(KX, np.asarray(mu, np.float64), var, logits)
    return gq @ gk.T


def forward_slice(causal, QX, KX, V, mu, raw, logits, var_floor, eps):
    A = affinity(QX, KX, mu, raw, logits, var_floor)
    if causal:
        A = np.tril(A)
    V = np.asarray(V, dtype=np.float64)
    return (A @ V) / (A.sum(axis=1, keepdims=True) + eps)


def forward(causal, QX, KX, V, mu, raw, logits, var_floor, eps):
    """O [B, H, N, d_v] by the explicit affinity, slice by slice."""
    B, H = QX.shape[:2]
    out = np.empty(V.shape[:3] + (V.shape[-1],), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            out[b, h] = forward_slice(causal, QX[b, h], KX[b, h], V[b, h], mu[h], raw[h],
                                      logits[h], var_floor, eps)
    return out
