"""Seeded synthetic calibration activations and weights for GPTQ layer workloads.

This module only *draws inputs*; it holds none of the quantization method's arithmetic,
and it is the one piece shared by the CUDA path's tests/bench and the CPU oracle (both
receive the very same bits from it).

The pages quantize real LLM layers on a few hundred calibration forward passes ("tm_gptq_
math", "Post-training quantization and the per-layer objective"); no dataset or trained
model is available here, so seeded synthetic inputs of the same shapes stand in:

* activations: ``X_chan = A Z`` with ``Z ~ N(0, 1)`` and a seeded mixing matrix
  ``A = I + G / sqrt(d)`` (``G ~ N(0, 1)``) that correlates the channels; stored
  token-major ``[n_tok, d_in]``.  Optional dead channels (identically zero) and outlier
  channels (scaled by 20) are picked by a seeded channel permutation;
* ReLU-sparse heavy-tailed activations for down-projections: the mixed channels are
  standardised, divided by ``sqrt(V / 4)`` with ``V ~ chi^2_4`` drawn elementwise
  (Student-t with 4 degrees of freedom marginals, correlation kept) and passed through
  ``max(s - tau, 0)`` with ``tau`` the t4 60th percentile (about 60 % zeros);
* weights ``W ~ N(0, std^2)`` drawn in float32 and stored as bf16 or float32.

Tokens are drawn in chunks of 2048 with one seed per chunk, so the first ``n`` tokens of
a long draw equal a short draw of ``n`` tokens (a token prefix is a valid sample).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

CHUNK_TOKENS = 2048
OUTLIER_FACTOR = 20.0
T4_Q60 = 0.2707222947075976  # 60th percentile of Student's t with 4 degrees of freedom

_STREAMS = {"A": 1, "Z": 2, "W": 3, "perm": 4, "V": 5}


def _seed(base: int, stream: str, index: int = 0) -> int:
    """Mix (base seed, stream name, index) into one 63-bit seed (splitmix64 finalizer)."""
    z = (int(base) * 0x9E3779B97F4A7C15 + _STREAMS[stream] * 0xBF58476D1CE4E5B9
         + int(index) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    z ^= z >> 31
    return z & 0x7FFFFFFFFFFFFFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@dataclass(frozen=True)
class ActivationSpec:
    """How one layer's calibration inputs are drawn."""
    d_in: int
    n_tok: int
    dtype: str = "f16"            # "f16" | "bf16" | "f32"
    n_dead: int = 0
    n_outlier: int = 0
    relu_t4: bool = False         # ReLU-sparse Student-t(4) down-projection inputs
    seed: int = 1000


@dataclass(frozen=True)
class LayerSpec:
    """One linear layer: weight shape/dtype and the activations it sees."""
    name: str
    d_out: int
    act: ActivationSpec
    w_std: float = 0.02
    w_dtype: str = "bf16"
    w_seed: int = 0


@dataclass(frozen=True)
class Workload:
    """A named workload: the layers it quantizes and at which bit widths."""
    name: str
    layers: tuple
    bits: tuple = (4,)
    block: int = 128
    damp: float = 0.01
    note: str = ""
    extra: dict = field(default_factory=dict)


def mixing_matrix(d: int, seed: int, device="cpu") -> torch.Tensor:
    """``A = I + G / sqrt(d)`` with seeded ``G ~ N(0, 1)``, float32 ``[d, d]``."""
    g = _gen(device, _seed(seed, "A"))
    G = torch.randn(d, d, generator=g, device=device, dtype=torch.float32)
    A = G / math.sqrt(d)
    A.diagonal().add_(1.0)
    return A


def channel_roles(spec: ActivationSpec, device="cpu"):
    """Seeded ``(dead_idx, outlier_idx)`` channel index tensors."""
    g = _gen("cpu", _seed(spec.seed, "perm"))
    perm = torch.randperm(spec.d_in, generator=g)
    dead = perm[: spec.n_dead]
    outl = perm[spec.n_dead: spec.n_dead + spec.n_outlier]
    return dead.to(device), outl.to(device)


def activations(spec: ActivationSpec, device="cpu", n_tok: int | None = None,
                tok_start: int = 0, A: torch.Tensor | None = None, out=None) -> torch.Tensor:
    """Token-major ``[n, d_in]`` activations in ``spec.dtype`` for tokens
    ``[tok_start, tok_start + n)`` (``n`` defaults to ``spec.n_tok - tok_start``).

    ``tok_start`` must be a multiple of the 2048-token chunk.  ``out`` may be a
    preallocated tensor of the right shape/dtype/device to fill in place.
    """
    n = spec.n_tok - tok_start if n_tok is None else int(n_tok)
    if tok_start % CHUNK_TOKENS:
        raise ValueError("tok_start must be a multiple of the chunk size")
    d = spec.d_in
    dt = _DTYPES[spec.dtype]
    if A is None:
        A = mixing_matrix(d, spec.seed, device)
    dead, outl = channel_roles(spec, device)
    if spec.relu_t4:
        rownorm = torch.linalg.vector_norm(A, dim=1)
    if out is None:
        out = torch.empty(n, d, dtype=dt, device=device)
    done = 0
    c = tok_start // CHUNK_TOKENS
    while done < n:
        take = min(CHUNK_TOKENS, n - done)
        g = _gen(device, _seed(spec.seed, "Z", c))
        Z = torch.randn(d, CHUNK_TOKENS, generator=g, device=device, dtype=torch.float32)
        Xc = (A @ Z).T.contiguous()          # [chunk, d] token-major
        if spec.relu_t4:
            Xc /= rownorm                    # per-channel standardisation
            gv = _gen(device, _seed(spec.seed, "V", c))
            V = torch.randn(4, CHUNK_TOKENS, d, generator=gv, device=device,
                            dtype=torch.float32).square_().sum(0)
            Xc /= torch.sqrt(V / 4.0)
            Xc = torch.clamp_min(Xc - T4_Q60, 0.0)
        if spec.n_outlier:
            Xc[:, outl] *= OUTLIER_FACTOR
        if spec.n_dead:
            Xc[:, dead] = 0.0
        out[done:done + take] = Xc[:take].to(dt)
        done += take
        c += 1
    return out


def weights(d_out: int, d_in: int, std: float, dtype: str, seed: int,
            device="cpu") -> torch.Tensor:
    """``W ~ N(0, std^2)`` drawn in float32, stored in ``dtype``; ``[d_out, d_in]``."""
    g = _gen(device, _seed(seed, "W"))
    W = torch.randn(d_out, d_in, generator=g, device=device, dtype=torch.float32) * std
    return W.to(_DTYPES[dtype])


def upper_factor(d: int, seed: int, coupling: float = 0.5, device="cpu") -> torch.Tensor:
    """A seeded upper-triangular ``[d, d]`` float32 matrix with positive diagonal: a valid
    inverse-Hessian factor input for the sweep at sizes where no Hessian is factored for it
    (any such U is the upper Cholesky factor of the inverse of the SPD matrix (U^T U)^-1).

    Diagonal ``exp(N(0, 0.25))``, strictly upper entries ``coupling * N(0, 1) / sqrt(d)``
    scaled by their row's diagonal.
    """
    g = _gen(device, _seed(seed, "A", 7))
    diag = torch.exp(0.5 * torch.randn(d, generator=g, device=device, dtype=torch.float32))
    U = torch.randn(d, d, generator=g, device=device, dtype=torch.float32)
    U.mul_(coupling / math.sqrt(d))
    U = torch.triu(U, diagonal=1)
    U.mul_(diag[:, None])
    U.diagonal().copy_(diag)
    return U


def layer_weights(layer: LayerSpec, device="cpu") -> torch.Tensor:
    return weights(layer.d_out, layer.act.d_in, layer.w_std, layer.w_dtype,
                   layer.act.seed * 131 + layer.w_seed, device)


# ---------------------------------------------------------------------------------------
# The five workloads (shapes and distributions of the benchmarked layers)
# ---------------------------------------------------------------------------------------

def _workloads():
    w = {}
    a = ActivationSpec(d_in=256, n_tok=512, dtype="f32", seed=1000)
    w["layer256_n512"] = Workload(
        "layer256_n512", (LayerSpec("linear", 256, a, 0.02, "f32"),), bits=(4,),
        note="d_out=256 d_in=256, 512 fp32 tokens, correlated channels, fp32 W")
    a = ActivationSpec(d_in=4096, n_tok=262144, dtype="f16", n_dead=41, n_outlier=8,
                       seed=1001)
    w["layer4096_n262144"] = Workload(
        "layer4096_n262144", (LayerSpec("linear", 4096, a, 0.02, "bf16"),), bits=(4,),
        note="d_out=4096 d_in=4096, 262144 fp16 tokens (128 x 2048), 8 outlier "
             "channels x20, 41 dead channels, bf16 W")
    up = ActivationSpec(d_in=4096, n_tok=131072, dtype="f16", seed=1002)
    dn = ActivationSpec(d_in=11008, n_tok=131072, dtype="f16", relu_t4=True, seed=1012)
    w["mlp11008_n131072"] = Workload(
        "mlp11008_n131072",
        (LayerSpec("up_proj", 11008, up, 0.02, "bf16"),
         LayerSpec("down_proj", 4096, dn, 0.02, "bf16")), bits=(4,),
        note="up 11008x4096 and down 4096x11008 (ReLU-sparse Student-t4 inputs), "
             "131072 fp16 tokens")
    qkv = ActivationSpec(d_in=4096, n_tok=131072, dtype="f16", seed=1003)
    o = ActivationSpec(d_in=4096, n_tok=131072, dtype="f16", seed=1013)
    gu = ActivationSpec(d_in=4096, n_tok=131072, dtype="f16", seed=1023)
    dn4 = ActivationSpec(d_in=11008, n_tok=131072, dtype="f16", relu_t4=True, seed=1033)
    w["block7b_n131072"] = Workload(
        "block7b_n131072",
        (LayerSpec("q_proj", 4096, qkv, 0.02, "bf16", 1),
         LayerSpec("k_proj", 4096, qkv, 0.02, "bf16", 2),
         LayerSpec("v_proj", 4096, qkv, 0.02, "bf16", 3),
         LayerSpec("o_proj", 4096, o, 0.02, "bf16", 4),
         LayerSpec("gate_proj", 11008, gu, 0.02, "bf16", 5),
         LayerSpec("up_proj", 11008, gu, 0.02, "bf16", 6),
         LayerSpec("down_proj", 4096, dn4, 0.02, "bf16", 7)), bits=(3, 4),
        note="7B-shaped block, hidden 4096 / MLP 11008, q/k/v share one Hessian, "
             "gate/up share one, 131072 fp16 tokens, 3- and 4-bit")
    a = ActivationSpec(d_in=28672, n_tok=65536, dtype="f16", n_dead=143, n_outlier=16,
                       seed=1004)
    w["downproj28672_n65536"] = Workload(
        "downproj28672_n65536", (LayerSpec("down_proj", 8192, a, 0.01, "bf16"),),
        bits=(4,),
        note="d_out=8192 d_in=28672, 65536 fp16 tokens, 16 outlier channels x20, "
             "143 dead channels, W ~ N(0, 0.01^2) bf16")
    return w


WORKLOADS = _workloads()
