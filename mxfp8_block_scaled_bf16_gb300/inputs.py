"""Seeded synthetic inputs for the five workloads.

This module holds random-number recipes only -- none of the quantization or
GEMM arithmetic -- so both the CUDA path and the CPU oracle can be fed from it.
All tensors are drawn on the CPU with ``torch.Generator`` in fp32 and cast to
bf16 (round to nearest even); the GPU copy is made by the caller.

Workload recipes (shapes from the pages' settings; distributions and seeds
are stated readings where the pages give none):

* single linear forward: x, W bf16[256,512] ~ N(0,1), x then W from one
  generator seeded 0;
* Llama-3-8B MLP up-projection: x[16384,4096] ~ N(0,1) (seed 0),
  W[14336,4096] ~ N(0,0.02^2) (seed 1), dy[16384,14336] ~ N(0,1e-4) i.e.
  sigma 0.01 (seed 2); SR seed 1234; RHT signs from seed 7;
* quantize sweep: [M,4096], M in {2048, 8192, 32768, 131072}, values
  0.1 * Student-t(3) (seed 0) with 4 of 4096 channels (0.1%) scaled by 10,
  the channels drawn from seed 1;
* Qwen3-8B-shaped linear stack: per layer l, generator seeded 1000+l;
* MoE grouped linear: 64 experts, 65536 tokens; group sizes = bincount of
  65536 draws from p(k) ~ k^-1.1 on k = 1..64 with numpy default_rng(3).
"""
from __future__ import annotations

import numpy as np
import torch

LLAMA3_8B_UP = dict(M=16384, N=14336, K=4096)
QUANT_SWEEP_M = (2048, 8192, 32768, 131072)
QUANT_SWEEP_K = 4096
SR_SEED = 1234
RHT_SIGN_SEED = 7


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, gen: torch.Generator) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 then rounded to bf16."""
    t = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def rht_sign_vector(seed: int = RHT_SIGN_SEED) -> np.ndarray:
    """16 random signs: b ~ randint(0, 2), s = 1 - 2b."""
    b = torch.randint(0, 2, (16,), generator=_gen(seed))
    return (1 - 2 * b).to(torch.int8).numpy()


def single_linear(seed: int = 0):
    g = _gen(seed)
    x = normal_bf16((256, 512), 1.0, g)
    w = normal_bf16((256, 512), 1.0, g)
    return x, w


def llama_up(M: int = LLAMA3_8B_UP["M"], N: int = LLAMA3_8B_UP["N"], K: int = LLAMA3_8B_UP["K"]):
    x = normal_bf16((M, K), 1.0, _gen(0))
    w = normal_bf16((N, K), 0.02, _gen(1))
    dy = normal_bf16((M, N), 0.01, _gen(2))
    return x, w, dy


def student_t3_outliers(M: int, K: int = QUANT_SWEEP_K, seed: int = 0, outlier_seed: int = 1):
    """0.1 * t(3) with round(0.001*K) channels (at least 1) gained by 10."""
    g = _gen(seed)
    z = torch.randn(M, K, generator=g, dtype=torch.float32)
    chi2 = torch.zeros(M, K, dtype=torch.float32)
    for _ in range(3):
        n = torch.randn(M, K, generator=g, dtype=torch.float32)
        chi2.addcmul_(n, n)
    t = z / torch.sqrt(chi2 / 3.0)
    t.mul_(0.1)
    n_out = max(1, round(0.001 * K))
    ch = torch.randperm(K, generator=_gen(outlier_seed))[:n_out]
    t[:, ch] *= 10.0
    return t.to(torch.bfloat16)


def zipf_group_sizes(n_groups: int = 64, n_tokens: int = 65536, s: float = 1.1, seed: int = 3):
    """bincount of n_tokens draws from the truncated Zipf p(k) ~ k^-s, k=1..G."""
    rng = np.random.default_rng(seed)
    k = np.arange(1, n_groups + 1, dtype=np.float64)
    p = k ** (-s)
    p /= p.sum()
    draws = rng.choice(n_groups, size=n_tokens, p=p)
    return np.bincount(draws, minlength=n_groups).astype(np.int64)


def moe_grouped(n_groups: int = 64, n_tokens: int = 65536, K: int = 4096, N: int = 1536):
    sizes = zipf_group_sizes(n_groups, n_tokens)
    x = normal_bf16((n_tokens, K), 1.0, _gen(0))
    w = normal_bf16((n_groups, N, K), 0.02, _gen(1))
    dy = normal_bf16((n_tokens, N), 0.01, _gen(2))
    return sizes, x, w, dy


QWEN3_8B_STACK = dict(n_layers=36, hidden=4096, kv_dim=1024, mlp=12288, tokens=2048 * 8,
                      vocab=151936, bf16_tail=6)


QWEN3_LINEARS = (("q", "hidden", "hidden"), ("k", "kv_dim", "hidden"), ("v", "kv_dim", "hidden"),
                 ("o", "hidden", "hidden"), ("gate", "mlp", "hidden"), ("up", "mlp", "hidden"),
                 ("down", "hidden", "mlp"))


def qwen3_layer_weights(layer: int, hidden: int = 4096, kv_dim: int = 1024, mlp: int = 12288,
                        device: str = "cpu"):
    """The seven linears of one layer as (name, W[out,in]) ~ N(0, 0.02^2), drawn
    from a generator seeded 1000 + layer on `device` (the full stack is 7.9e9
    parameters, so the benchmark draws it on the GPU; the CPU and GPU streams
    differ, both are seeded)."""
    g = torch.Generator(device=device)
    g.manual_seed(1000 + layer)
    dims = {"hidden": hidden, "kv_dim": kv_dim, "mlp": mlp}
    out = []
    for n, o, i in QWEN3_LINEARS:
        t = torch.randn(dims[o], dims[i], generator=g, dtype=torch.float32, device=device)
        out.append((n, t.mul_(0.02).to(torch.bfloat16)))
    return out


def normal_bf16_on(shape, std: float, seed: int, device: str) -> torch.Tensor:
    """N(0, std^2) bf16 drawn on `device` from a generator seeded `seed`."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)
