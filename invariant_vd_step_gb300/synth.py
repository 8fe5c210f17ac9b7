"""Seeded synthetic inputs shared by the CUDA path, its tests and the oracle.

This module only *draws* inputs: model shapes, random-init bf16 weights,
token streams, context lengths and page permutations.  It holds none of the
decoder's arithmetic, so that the CUDA path and the CPU oracle, which both
consume these arrays, stay independent of each other.

Model shapes follow the workloads of the Vosti evaluation ("Vosti:
Specifying, Implementing, and Verifying Deterministic LLM Inference",
evaluation section: Llama3.1-8B and Gemma3-4B) plus a tiny Llama-style
decoder used for exhaustive invariance runs.  Pretrained weights are not
available, so every matrix is drawn i.i.d. N(0, 0.02) and rounded to bf16;
norm gains are 1.0 unless a test asks for random gains.
"""

from __future__ import annotations

import dataclasses
import hashlib
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class ModelSpec:
    """Shape and numerics configuration of a Llama/Gemma-style decoder.

    Layer ``i`` is a *global* attention layer iff ``local_global_period == 0``
    or ``(i + 1) % local_global_period == 0``; other layers are *local*
    sliding-window layers with ``sliding_window`` keys (the key at the row's
    own position included).
    """

    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rms_eps: float = 1e-5
    act: str = "swiglu"  # "swiglu" (silu(g)*u) or "geglu" (gelu_tanh(g)*u)
    qk_norm: bool = False
    rope_theta: float = 1e4  # global layers
    rope_theta_local: float = 1e4  # local (sliding-window) layers
    sliding_window: int = 0  # 0: no local layers
    local_global_period: int = 0  # 0: every layer global
    page_size: int = 16
    # Gemma-3 block: embeddings times bf16(sqrt(d)); RMSNorm gains (1 + w);
    # sandwich norms (a norm on the attention and FFN outputs before each
    # residual add, weights post_attn_norm / post_ffn_norm).
    embed_scale: bool = False
    norm_offset: bool = False
    sandwich_norm: bool = False

    @property
    def qkv_dim(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def attn_dim(self) -> int:
        return self.n_heads * self.head_dim

    def layer_is_local(self, i: int) -> bool:
        if self.sliding_window <= 0 or self.local_global_period <= 0:
            return False
        return (i + 1) % self.local_global_period != 0

    def layer_window(self, i: int) -> int:
        return self.sliding_window if self.layer_is_local(i) else 0

    def layer_theta(self, i: int) -> float:
        return self.rope_theta_local if self.layer_is_local(i) else self.rope_theta

    def with_(self, **kw) -> "ModelSpec":
        return dataclasses.replace(self, **kw)


# Tiny Llama-style decoder: 2 layers, d 256, 4 q / 2 kv heads, hd 64,
# SwiGLU 768, vocab 2048, eps 1e-5, RoPE theta 1e4.
TINY = ModelSpec("tiny-llama", 2, 256, 4, 2, 64, 768, 2048, rope_theta=1e4)

# Llama-3.1-8B shape.  theta 5e5, no llama3 frequency scaling.
LLAMA8B = ModelSpec("llama3.1-8b-shape", 32, 4096, 32, 8, 128, 14336, 128256,
                    rope_theta=5e5, rope_theta_local=5e5)
# One decoder layer of the 8B shape plus the LM head (decode sweep workload).
LLAMA8B_1L = LLAMA8B.with_(name="llama3.1-8b-shape-1layer", n_layers=1)

# Gemma-3-4B shape: QK-RMSNorm, GeGLU, 5 local (window 1024) : 1 global,
# and the Gemma-3 block (embedding scale, (1 + w) norm gains, sandwich norms).
GEMMA3_4B = ModelSpec("gemma3-4b-shape", 34, 2560, 8, 4, 256, 10240, 262144,
                      act="geglu", qk_norm=True, rope_theta=1e6,
                      rope_theta_local=1e4, sliding_window=1024,
                      local_global_period=6, rms_eps=1e-6, embed_scale=True,
                      norm_offset=True, sandwich_norm=True)

SPECS = {s.name: s for s in (TINY, LLAMA8B, LLAMA8B_1L, GEMMA3_4B)}


def _subseed(seed: int, name: str) -> int:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def weight_shapes(spec: ModelSpec) -> dict:
    """Name -> shape of every weight tensor (row-major, [out][in] for matrices)."""
    d, hd, F, V = spec.d_model, spec.head_dim, spec.ffn_dim, spec.vocab
    shapes = {"embed": (V, d), "final_norm": (d,), "lm_head": (V, d)}
    for i in range(spec.n_layers):
        p = f"layers.{i}."
        shapes[p + "attn_norm"] = (d,)
        shapes[p + "wqkv"] = (spec.qkv_dim, d)  # rows: q heads, k heads, v heads
        if spec.qk_norm:
            shapes[p + "q_norm"] = (hd,)
            shapes[p + "k_norm"] = (hd,)
        shapes[p + "wo"] = (d, spec.attn_dim)
        if spec.sandwich_norm:
            shapes[p + "post_attn_norm"] = (d,)
            shapes[p + "post_ffn_norm"] = (d,)
        shapes[p + "ffn_norm"] = (d,)
        shapes[p + "w_gate_up"] = (2 * F, d)  # rows 0..F-1 gate, F..2F-1 up
        shapes[p + "w_down"] = (d, F)
    return shapes


def _is_gain(name: str) -> bool:
    return name.endswith("norm")


def make_weights(spec: ModelSpec, seed: int = 0, device="cpu", std: float = 0.02,
                 gain_std: float = 0.0, zero: bool = False, exclude=()) -> dict:
    """Random-init bf16 weights, one independent generator stream per tensor.

    Matrices ~ N(0, std) rounded to bf16; norm gains are 1 + N(0, gain_std)
    (exactly 1.0 for gain_std == 0).  With ``spec.norm_offset`` the stored
    weight w is the gain minus one, N(0, gain_std).  ``zero=True`` gives the
    all-zero model.  Tensors named in ``exclude`` are left out (the others
    are unchanged: each tensor has its own stream).
    """
    out = {}
    for name, shape in weight_shapes(spec).items():
        if name in exclude:
            continue
        if zero:
            out[name] = torch.zeros(shape, dtype=torch.bfloat16, device=device)
            continue
        g = torch.Generator(device=device)
        g.manual_seed(_subseed(seed, name))
        if _is_gain(name):
            t = torch.full(shape, 0.0 if spec.norm_offset else 1.0, dtype=torch.float32, device=device)
            if gain_std > 0:
                t += gain_std * torch.randn(shape, generator=g, device=device)
        else:
            t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            t.mul_(std)
        out[name] = t.to(torch.bfloat16)
        del t
    return out


def bf16_to_u16(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a numpy uint16 array (CPU copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def weights_to_numpy(weights: dict) -> dict:
    """bf16 weights as raw uint16 bit arrays (the oracle's input format)."""
    return {k: bf16_to_u16(v) for k, v in weights.items()}


def make_tokens(n: int, vocab: int, seed: int = 1) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def make_prompts(n_req: int, len_lo: int, len_hi: int, vocab: int, seed: int = 1,
                 shared_prefix: int = 0, n_sharing: int = 0) -> list:
    """``n_req`` uniform-random prompts with lengths U[len_lo, len_hi].

    The first ``n_sharing`` prompts start with the same ``shared_prefix``
    tokens (lengths are then at least shared_prefix + 1).
    """
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, vocab, size=shared_prefix).astype(np.int32)
    prompts = []
    for r in range(n_req):
        L = int(rng.integers(len_lo, len_hi + 1))
        toks = rng.integers(0, vocab, size=L).astype(np.int32)
        if r < n_sharing and shared_prefix > 0:
            L = max(L, shared_prefix + 1)
            toks = np.concatenate([prefix, rng.integers(0, vocab, size=L - shared_prefix).astype(np.int32)])
        prompts.append(toks)
    return prompts


def make_context_lengths(n: int, lo: int, hi: int, seed: int = 3) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=n).astype(np.int32)


def page_permutation(num_pages: int, seed: int = 2) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.permutation(num_pages).astype(np.int32)


def make_normal_bf16(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def make_small_int_bf16(shape, seed: int, lo: int = -8, hi: int = 8, device="cpu") -> torch.Tensor:
    """Small integers stored as bf16 (exactly representable)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randint(lo, hi + 1, shape, generator=g, device=device)
    return t.to(torch.bfloat16)


def make_logits(rows: int, vocab: int, seed: int, std: float = 1.0, ties: bool = False) -> np.ndarray:
    """fp32 logits; with ``ties`` some rows repeat their maximum."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, vocab)) * std).astype(np.float32)
    if ties and vocab > 4:
        for r in range(0, rows, 2):
            j = int(np.argmax(x[r]))
            k = int(rng.integers(0, vocab))
            x[r, k] = x[r, j]
    return x
