"""Seeded synthetic inputs for the GMA forward pass, shared by the tests, the benchmark and the
smoke check.  This module only draws random numbers and names workloads; it holds none of the
method's arithmetic, and it serves the CUDA library and the oracle alike.

Recipe (the page's own workloads are WikiText-103 language modelling and Long-Range Arena
classification; their datasets are not used -- tensors of the same shapes stand in for them):

* one ``torch.Generator('cpu')`` seeded per workload;
* draw order, all fp32: Q_X, K_X, V, mu, raw variance, prior logits;
* Q_X, K_X ~ N(0, 1); V ~ N(0, 1) or U(-1, 1); mu ~ N(0, mu_std); raw ~ N(0, raw_std);
  prior logits ~ N(0, 1)  (N(0, s) names the standard deviation s);
* activations are then rounded to bf16 (round-to-nearest-even) for bf16 workloads; the GMM
  parameters stay fp32.
"""
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    causal: bool
    B: int
    H: int
    N: int
    d_r: int
    K: int
    d_v: int
    dtype: str = "bf16"          # "bf16" or "f32": the activation / output type
    seed: int = 0
    v_dist: str = "normal"       # "normal": N(0,1); "uniform": U(-1,1)
    mu_std: float = 1.0
    raw_std: float = 0.5
    logit_std: float = 1.0
    eps: float = 1e-6
    var_floor: float = 1e-3
    N_k: int = 0                 # cross-attention: keys per slice (0: the same N as the queries)

    @property
    def keys(self) -> int:
        return self.N_k or self.N

    @property
    def tokens(self) -> int:
        return self.B * self.N

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.N

    @property
    def key_heads(self) -> int:
        return self.B * self.H * self.keys


def _ws(name, causal, B, H, N, d_r, K, d_v, **kw):
    return Workload(name, causal, B, H, N, d_r, K, d_v, **kw)


# The five benchmark workloads.  Names say what they are; sizes are in the names and fields.
TINY_BIDIR_F32 = _ws("bidir_f32_b1h1_n256_dr16_k8_dv32", False, 1, 1, 256, 16, 8, 32,
                     dtype="f32", seed=0)
LM_CAUSAL = _ws("causal_bf16_b4h8_n2048_dr64_k64_dv64", True, 4, 8, 2048, 64, 64, 64, seed=1)
LRA_BIDIR = _ws("bidir_bf16_b32h8_n4096_dr32_k32_dv64", False, 32, 8, 4096, 32, 32, 64, seed=2,
                v_dist="uniform", mu_std=1.5)
LONG_CAUSAL = _ws("causal_bf16_b1h16_n65536_dr64_k128_dv128", True, 1, 16, 65536, 64, 128, 128,
                  seed=3)
K_SWEEP = tuple(_ws(f"causal_bf16_b2h16_n16384_dr64_k{k}_dv128", True, 2, 16, 16384, 64, k, 128,
                    seed=4) for k in (16, 64, 256, 1024))
N_SWEEP = tuple(_ws(f"causal_bf16_b2h16_n{n}_dr64_k64_dv128", True, 2, 16, n, 64, 64, 128,
                    seed=4) for n in (4096, 8192, 16384, 32768, 65536, 131072))

# Autoregressive decoding with the long-context head shape: B sequences x H heads each take one
# new token per step.  N is the number of steps drawn (one row of Q_X, K_X and V per step); the
# per-slice state is K x (d_v + 1) fp32, 135 MB for the whole batch (above the 129 MB L2).
DECODE = _ws("decode_bf16_b128h16_dr64_k128_dv128", True, 128, 16, 8, 64, 128, 128, seed=5)

# Cross-attention (bidirectional, separate key set): a short query sequence reading a long one,
# as a decoder reads an encoder's output; N = 2048 queries, N_k = 16384 keys per slice.
CROSS = _ws("cross_bf16_b8h16_nq2048_nk16384_dr64_k64_dv64", False, 8, 16, 2048, 64, 64, 64, seed=6,
            N_k=16384)

# Component-usage diagnostics of one long sequence's routing rows (Q_X of this workload), with
# the long-context head shape: B=1, H=16, N=65536, d_r=64, K=128 (d_v unused).
USAGE = _ws("usage_bf16_b1h16_n65536_dr64_k128", False, 1, 16, 65536, 64, 128, 16, seed=7)

# Backward pass of the LM-shaped causal layer (the page's training path): B=4, H=8, N=2048,
# d_r=64, K=64, d_v=64, bf16 activations; the output gradient dO is drawn after the inputs from
# its own generator (seed + 2024), N(0, 1).
BACKWARD = _ws("backward_causal_bf16_b4h8_n2048_dr64_k64_dv64", True, 4, 8, 2048, 64, 64, 64, seed=8)

ALL_WORKLOADS = (TINY_BIDIR_F32, LM_CAUSAL, LRA_BIDIR, LONG_CAUSAL) + K_SWEEP + N_SWEEP + (CROSS, USAGE,
                                                                                         BACKWARD)


def by_name(name: str) -> Workload:
    for w in ALL_WORKLOADS + (DECODE,):
        if w.name == name:
            return w
    raise KeyError(name)


def scaled(w: Workload, **changes) -> Workload:
    """The same recipe with some sizes changed (smaller parity cases)."""
    return replace(w, name=w.name + "_scaled", **changes)


def make_inputs(w: Workload):
    """Draw one workload's inputs on the CPU.

    Returns a dict of CPU tensors: QX [B,H,N,d_r], KX [B,H,N_k,d_r], V [B,H,N_k,d_v] (bf16 or
    fp32; N_k = N but for cross-attention workloads), mu, raw [H,K,d_r] fp32, logits [H,K] fp32.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    B, H, N, d_r, K, d_v = w.B, w.H, w.N, w.d_r, w.K, w.d_v
    Nk = w.keys
    QX = torch.randn(B, H, N, d_r, generator=g, dtype=torch.float32)
    KX = torch.randn(B, H, Nk, d_r, generator=g, dtype=torch.float32)
    if w.v_dist == "uniform":
        V = torch.rand(B, H, Nk, d_v, generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        V = torch.randn(B, H, Nk, d_v, generator=g, dtype=torch.float32)
    mu = torch.randn(H, K, d_r, generator=g, dtype=torch.float32) * w.mu_std
    raw = torch.randn(H, K, d_r, generator=g, dtype=torch.float32) * w.raw_std
    logits = torch.randn(H, K, generator=g, dtype=torch.float32) * w.logit_std
    if w.dtype == "bf16":
        QX, KX, V = QX.to(torch.bfloat16), KX.to(torch.bfloat16), V.to(torch.bfloat16)
    return {"QX": QX, "KX": KX, "V": V, "mu": mu, "raw": raw, "logits": logits}


def to_numpy(inputs):
    """fp32 numpy views of an input dict (bf16 widens to fp32 exactly)."""
    return {k: v.float().numpy() for k, v in inputs.items()}


def make_decode_state(w: Workload, scale: float = 1.0, seed: int = 1000):
    """A non-zero starting decode state [B, H, K, d_v + 1] fp32 on the CPU, drawn from its own
    generator: memory columns ~ N(0, scale), the last (normaliser) column ~ U(0.5, 1.5) * scale,
    positive like any sum of responsibilities."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed) + int(seed))
    S = torch.randn(w.B, w.H, w.K, w.d_v + 1, generator=g, dtype=torch.float32) * scale
    S[..., w.d_v] = (torch.rand(w.B, w.H, w.K, generator=g, dtype=torch.float32) + 0.5) * scale
    return S

