"""Seeded synthetic inputs for sliding-window attention with sinks.

This module holds the workload recipes and the seeded generators that both the GPU path and the
oracle are fed from. It holds none of the attention arithmetic: it only draws iid N(0, 1) tensors,
rounds them to the storage dtype and, where a workload asks for it, multiplies the keys at the first
few positions by 4 (exact in bf16 and fp32, a power of two) so that they behave as attention sinks.

Draws use torch's seeded generators. A tensor is drawn once, on one device, and the same bytes go
to both sides (the oracle receives a host copy), so the two devices' generators never need to agree.

Workload shapes follow the head shapes of the models the pages discuss: Llama-2-7B (H=32, d=128),
Llama-2-13B (H=40, d=128; 4 sink + 1020 recent slots, 20K tokens, page "滑窗与固定稀疏",
table tbl-attn-fixed-sink-ppl) and Mistral-7B (window 4096, eq attn-fixed-rf; 4 sinks from the
hyper.ai summary of arXiv 2608.28444).
"""
from __future__ import annotations

import dataclasses
import math

import torch

# Tensor ids mixed into the seed so that q, k and v (and decode streams) are independent draws.
TID_Q, TID_K, TID_V = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "prefill" | "decode" | "chunked"
    B: int
    H: int
    L: int               # sequence length (prefill/chunked) or number of decode steps
    d: int
    w: int
    s: int
    dtype: str           # "bf16" | "f32"
    sink_boost: bool     # keys at positions 0..3 multiplied by 4
    chunk: int = 0       # chunk length for chunked prefill
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


# The five workloads; the first three tiny ones are the fp32 correctness shapes.
WORKLOADS = {
    "prefill_tiny_f32_w16_s4": Workload("prefill_tiny_f32_w16_s4", "prefill", 1, 1, 64, 16, 16, 4, "f32", False, seed=1001),
    "prefill_tiny_f32_w16_s0": Workload("prefill_tiny_f32_w16_s0", "prefill", 1, 1, 64, 16, 16, 0, "f32", False, seed=1001),
    "prefill_tiny_f32_w64_s0": Workload("prefill_tiny_f32_w64_s0", "prefill", 1, 1, 64, 16, 64, 0, "f32", False, seed=1001),
    "prefill_llama7b_L8192_w1024_s4": Workload("prefill_llama7b_L8192_w1024_s4", "prefill", 1, 32, 8192, 128, 1024, 4, "bf16", False, seed=1002),
    "prefill_mistral_B2_L32768_w4096_s0": Workload("prefill_mistral_B2_L32768_w4096_s0", "prefill", 2, 32, 32768, 128, 4096, 0, "bf16", False, seed=1003),
    "prefill_mistral_B2_L32768_w4096_s4": Workload("prefill_mistral_B2_L32768_w4096_s4", "prefill", 2, 32, 32768, 128, 4096, 4, "bf16", False, seed=1003),
    "decode_llama13b_B64_w1024_s4_20480": Workload("decode_llama13b_B64_w1024_s4_20480", "decode", 64, 40, 20480, 128, 1024, 4, "bf16", True, seed=1004),
    "chunked_mistral_L131072_w4096_s4_C4096": Workload("chunked_mistral_L131072_w4096_s4_C4096", "chunked", 1, 32, 131072, 128, 4096, 4, "bf16", True, chunk=4096, seed=1005),
}


def _gen(device, seed: int, tid: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + tid * 7919 + 17)
    return g


def normal(shape, seed: int, tid: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """iid N(0, 1) drawn in fp32 from a seeded generator on ``device``, rounded to ``dtype`` (RNE)."""
    x = torch.randn(tuple(shape), generator=_gen(device, seed, tid), device=device, dtype=torch.float32)
    return x.to(dtype)


def boost_sinks(k: torch.Tensor, n: int = 4, factor: float = 4.0, seq_dim: int = -2, pos0: int = 0) -> torch.Tensor:
    """Multiply the keys at absolute positions < n by ``factor`` in place (exact for a power of two).
    ``pos0`` is the absolute position of index 0 along ``seq_dim``."""
    L = k.shape[seq_dim]
    hi = min(n - pos0, L)
    if hi > 0:
        k.narrow(seq_dim, 0, hi).mul_(factor)
    return k


def prefill_inputs(B, H, L, d, seed, dtype=torch.bfloat16, device="cpu", sink_boost=False):
    """q, k, v of shape [B, H, L, d]."""
    q = normal((B, H, L, d), seed, TID_Q, dtype, device)
    k = normal((B, H, L, d), seed, TID_K, dtype, device)
    v = normal((B, H, L, d), seed, TID_V, dtype, device)
    if sink_boost:
        boost_sinks(k)
    return q, k, v


def workload_inputs(wl: Workload, device="cpu"):
    """The full input set of a prefill/chunked workload ([B, H, L, d] each), or of a decode workload
    (per-step q/k/v streams [B, H, steps, d])."""
    return prefill_inputs(wl.B, wl.H, wl.L, wl.d, wl.seed, wl.torch_dtype, device, wl.sink_boost)


def bigbird_pattern(L: int, block: int, n_global_blocks: int, r: int, seed: int):
    """A BigBird-style pattern for the block-sparse prefill (fixed-sparsity page, BigBird section: global tokens
    inside the sequence (ITC) plus r random key blocks per query block).  The global tokens are the first
    n_global_blocks blocks; each query block qb draws r distinct key blocks uniformly from its causal blocks
    0..qb (all of them when there are fewer than r), -1 filling unused entries.  The draw is seeded (numpy), and
    the same arrays go to the library and to the oracle.  Returns (globals list, rand int32 [ceil(L/block), r])."""
    import numpy as np
    rng = np.random.default_rng(seed)
    nqb = (L + block - 1) // block
    globals_ = list(range(min(L, n_global_blocks * block)))
    rand = np.full((nqb, r), -1, dtype=np.int32)
    for qb in range(nqb):
        k = min(r, qb + 1)
        if k > 0:
            rand[qb, :k] = np.sort(rng.choice(qb + 1, size=k, replace=False))
    return globals_, rand


def rand_blocks_dict(rand):
    """The random key blocks as {query block: [key blocks]} (the oracle's form), -1 entries dropped."""
    return {qb: [int(x) for x in row if x >= 0] for qb, row in enumerate(rand)}


def hedgehog_weights(d: int, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """A stand-in for the learned Hedgehog projection wf [d, d/2] (no trained weights are available): iid
    N(0, 1/d) entries, so that f(x) = x wf has unit variance for x ~ N(0, I)."""
    g = _gen(device, seed, 7)
    x = torch.randn((d, d // 2), generator=g, device=device, dtype=torch.float32) / float(d) ** 0.5
    return x.to(dtype)
