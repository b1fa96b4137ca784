"""Seeded synthetic inputs for the deterministic multi-writer reduction.

This module only makes inputs.  It holds no reduction arithmetic: both the
GPU library and the CPU oracle consume the exact bytes made here.  All values
come from seeded torch generators (CPU generator for the routing tables, the
target device's generator for the large value tensors), so the same seed on
the same device and torch build gives the same bytes.

Workloads (shapes follow the cases the pages name):
  * MoE token combine / unpermute ("Megatron-LM determinism developer
    reference", section 3.1): T tokens each routed to top-k of E experts by a
    softmax over N(0,1) logits, weights renormalised over the chosen k.  The
    permuted rows are expert-major, tokens ascending inside an expert (the
    stable (expert id, original token id) order of "DeepSeek-V4 book, Ch 09",
    section 3.2); idx = token id, w = routing weight.
  * Sparse-attention backward key-gradient scatter (Ch 09, section 3.1):
    Q queries each select K distinct keys of S, key ranks drawn with
    probability proportional to r^-s (Zipf), without replacement, via
    Gumbel-top-k; rank -> key id through a seeded permutation so hot keys are
    scattered; source order i = q*K + j with keys ascending in a query;
    contributions N(0, sigma^2) in bf16; no weight.
  * Router scores for the sorted router top-k and the route plan: softmax
    probabilities of N(0,1) logits [T, E] (the score function is the caller's,
    so the inputs are the probabilities themselves).
  * Split-K partials (Ch 09, section 3.3): [S, R*C] float32, values
    z * 2^U with z ~ N(0,1), U ~ Uniform[-8, 8) (mixed magnitudes).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class ScatterCase:
    name: str
    idx: torch.Tensor            # int32 [N], destination of each physical row
    x: torch.Tensor              # [N, H] float32 or bfloat16 (rows may be padded: x.stride(0) = ldx)
    w: Optional[torch.Tensor]    # float32 [N] or None
    M: int
    out_dtype: torch.dtype       # torch.float32 or torch.bfloat16
    src_id: Optional[torch.Tensor] = None   # int64 [N] or None
    meta: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return int(self.idx.numel())

    @property
    def H(self) -> int:
        return int(self.x.shape[1])

    def compulsory_bytes(self) -> int:
        """Sources read once, outputs written once, indices and weights read once."""
        xb = self.N * self.H * self.x.element_size()
        wb = 0 if self.w is None else self.N * 4
        ib = self.N * 4
        ob = self.M * self.H * (4 if self.out_dtype == torch.float32 else 2)
        return xb + wb + ib + ob


def _cpu_gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(seed)


def _dev_gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(seed)


def _fill_normal(shape, dtype, std: float, seed: int, device, rows_per_chunk: int = 1 << 16) -> torch.Tensor:
    """N(0, std^2) values drawn as float32 then rounded to `dtype`, chunked to bound peak memory."""
    out = torch.empty(shape, dtype=dtype, device=device)
    g = _dev_gen(seed, device)
    n = shape[0]
    for r0 in range(0, n, rows_per_chunk):
        r1 = min(n, r0 + rows_per_chunk)
        blk = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            blk.mul_(std)
        out[r0:r1].copy_(blk)
    return out


def moe_routing(T: int, E: int, k: int, seed: int):
    """(expert [T, k] int64, weight [T, k] float32): top-k of softmax(N(0,1) logits), renormalised.

    Ties between equal logits go to the lower expert id (stable sort).
    """
    g = _cpu_gen(seed)
    logits = torch.randn(T, E, generator=g, dtype=torch.float32)
    probs = torch.softmax(logits.double(), dim=1)
    order = torch.sort(-logits, dim=1, stable=True).indices[:, :k]
    top = probs.gather(1, order)
    top = top / top.sum(dim=1, keepdim=True)
    return order, top.float()


def router_scores(T: int, E: int, seed: int, device="cpu") -> torch.Tensor:
    """float32 [T, E] router probabilities: softmax of N(0,1) logits, taken in fp64 and rounded once."""
    g = _cpu_gen(seed)
    logits = torch.randn(T, E, generator=g, dtype=torch.float32)
    return torch.softmax(logits.double(), dim=1).float().to(device)


def moe_combine(T: int, E: int, k: int, H: int, x_dtype=torch.bfloat16, out_dtype=torch.bfloat16,
                seed: int = 2, device="cpu", ldx: Optional[int] = None, name: Optional[str] = None) -> ScatterCase:
    """Permuted expert outputs [T*k, H] (expert-major rows) combined back into [T, H]."""
    experts, weights = moe_routing(T, E, k, seed)
    e_flat = experts.reshape(-1)
    t_flat = torch.arange(T, dtype=torch.int64).repeat_interleave(k)
    w_flat = weights.reshape(-1)
    rows = torch.argsort(e_flat * T + t_flat)          # keys are unique: (expert, token)
    idx = t_flat[rows].to(torch.int32)
    w = w_flat[rows].contiguous()
    N = T * k
    ld = H if ldx is None else ldx
    xfull = _fill_normal((N, ld), x_dtype, 1.0, seed * 7919 + 1, device)
    x = xfull[:, :H]
    return ScatterCase(name=name or f"moe_combine T={T} E={E} k={k} H={H}",
                       idx=idx.to(device), x=x, w=w.to(device), M=T, out_dtype=out_dtype,
                       meta={"T": T, "E": E, "k": k, "experts_of_row": e_flat[rows]})


def zipf_key_lists(Q: int, K: int, S: int, s: float, seed: int, device="cpu", chunk: int = 512) -> torch.Tensor:
    """int64 [Q, K]: for each query K distinct key ids, ascending.

    Ranks r = 1..S are drawn with probability proportional to r^-s without
    replacement (Gumbel-top-k on log r^-s), then mapped to key ids by a seeded
    random permutation so that hot keys are spread over the id space.
    """
    if K > S:
        raise ValueError("K must not exceed S")
    gperm = _cpu_gen(seed)
    pi = torch.randperm(S, generator=gperm).to(device)
    logp = (-s * torch.log(torch.arange(1, S + 1, dtype=torch.float64, device=device))).unsqueeze(0)
    g = _dev_gen(seed * 104729 + 3, device)
    out = torch.empty((Q, K), dtype=torch.int64, device=device)
    tiny = torch.finfo(torch.float64).tiny
    for q0 in range(0, Q, chunk):
        q1 = min(Q, q0 + chunk)
        u = torch.rand((q1 - q0, S), generator=g, dtype=torch.float64, device=device).clamp_(min=tiny)
        scores = logp - torch.log(-torch.log(u))
        ranks = torch.topk(scores, K, dim=1, sorted=False).indices
        keys = pi[ranks]
        out[q0:q1] = torch.sort(keys, dim=1).values
    return out


def sparse_key_scatter(Q: int, K: int, S: int, H: int, zipf_s: float = 1.1, sigma: float = 0.02,
                       seed: int = 4, device="cpu", x_dtype=torch.bfloat16, out_dtype=torch.float32,
                       name: Optional[str] = None) -> ScatterCase:
    """dK contributions of Q queries x K selected keys, scattered into S key rows."""
    keys = zipf_key_lists(Q, K, S, zipf_s, seed, device=device)
    idx = keys.reshape(-1).to(torch.int32)
    x = _fill_normal((Q * K, H), x_dtype, sigma, seed * 7919 + 5, device)
    return ScatterCase(name=name or f"sparse_key_scatter Q={Q} K={K} S={S} H={H} zipf={zipf_s}",
                       idx=idx, x=x, w=None, M=S, out_dtype=out_dtype,
                       meta={"Q": Q, "K": K, "S": S, "zipf_s": zipf_s})


def embedding_backward(T: int, V: int, H: int, zipf_s: float = 1.0, sigma: float = 0.02, seed: int = 6,
                       device="cpu", x_dtype=torch.bfloat16, name: Optional[str] = None) -> ScatterCase:
    """Token-embedding backward: the output gradients dY [T, H] of T tokens are
    added into the fp32 weight gradient [V, H] at each token's id (index_add_).

    Token ids are drawn with replacement from Zipf(zipf_s) over the vocabulary
    (rank r with probability proportional to r^-s, the usual shape of token
    frequencies), ranks mapped to ids by a seeded random permutation.
    """
    g = _cpu_gen(seed)
    p = torch.arange(1, V + 1, dtype=torch.float64) ** (-zipf_s)
    ranks = torch.multinomial(p / p.sum(), T, replacement=True, generator=g)
    ids = torch.randperm(V, generator=g)[ranks].to(torch.int32)
    x = _fill_normal((T, H), x_dtype, sigma, seed * 7919 + 7, device)
    return ScatterCase(name=name or f"embedding_backward T={T} V={V} H={H} zipf={zipf_s}",
                       idx=ids.to(device), x=x, w=None, M=V, out_dtype=torch.float32,
                       meta={"T": T, "V": V, "zipf_s": zipf_s, "accumulate": True})


def splitk_partials(S: int, R: int, C: int, seed: int = 5, device="cpu") -> torch.Tensor:
    """float32 [S, R*C] with values z * 2^U, z ~ N(0,1), U ~ Uniform[-8, 8)."""
    g = _dev_gen(seed * 7919 + 11, device)
    z = torch.randn((S, R * C), generator=g, dtype=torch.float64, device=device)
    u = torch.rand((S, R * C), generator=g, dtype=torch.float64, device=device) * 16.0 - 8.0
    return (z * torch.exp2(u)).to(torch.float32)


def splitk_gemm_inputs(R: int, K: int, C: int, seed: int = 5, device="cpu"):
    """Inputs of a split-K GEMM out = A @ W.T: A bf16 [R, K] ~ N(0, 1) and W bf16
    [C, K] ~ N(0, 1) * 2^-5 (the transposed right operand, K contiguous)."""
    A = _fill_normal((R, K), torch.bfloat16, 1.0, seed * 7919 + 11, device)
    W = _fill_normal((C, K), torch.bfloat16, 2.0 ** -5, seed * 7919 + 13, device)
    return A, W


# --- the five workloads at full size, and small versions for fast parity runs ---

FULL = {
    "tiny_moe": dict(kind="moe", T=64, E=8, k=2, H=128, x_dtype=torch.float32, out_dtype=torch.float32, seed=1),
    "moe_combine": dict(kind="moe", T=4096, E=128, k=8, H=4096, x_dtype=torch.bfloat16,
                        out_dtype=torch.bfloat16, seed=2),
    "ep_invariance": dict(kind="moe", T=16384, E=256, k=8, H=7168, x_dtype=torch.bfloat16,
                          out_dtype=torch.bfloat16, seed=3),
    "sparse_key_scatter": dict(kind="sparse", Q=16384, K=512, S=65536, H=128, zipf_s=1.1, sigma=0.02, seed=4),
    "splitk": dict(kind="splitk", S=56, R=16384, C=24, seed=5),
    # beyond the five: the embedding backward (index_add_ into a 128K-row gradient)
    "embedding_backward": dict(kind="embedding", T=32768, V=131072, H=4096, zipf_s=1.0, sigma=0.02, seed=6),
}

SMALL = {
    "tiny_moe": FULL["tiny_moe"],
    "moe_combine": dict(kind="moe", T=384, E=32, k=8, H=1096, x_dtype=torch.bfloat16,
                        out_dtype=torch.bfloat16, seed=12),
    "ep_invariance": dict(kind="moe", T=512, E=64, k=8, H=712, x_dtype=torch.bfloat16,
                          out_dtype=torch.bfloat16, seed=13),
    "sparse_key_scatter": dict(kind="sparse", Q=640, K=128, S=4096, H=128, zipf_s=1.1, sigma=0.02, seed=14),
    "splitk": dict(kind="splitk", S=56, R=1000, C=24, seed=15),
    "embedding_backward": dict(kind="embedding", T=3000, V=2048, H=200, zipf_s=1.0, sigma=0.02, seed=16),
}


MEDIUM = {
    # same shapes with a quarter of the queries / tokens: sources still far larger than L2,
    # small enough for multi-pass profiler captures
    "sparse_key_scatter": dict(kind="sparse", Q=4096, K=512, S=65536, H=128, zipf_s=1.1, sigma=0.02, seed=24),
    "moe_combine": FULL["moe_combine"],
    "ep_invariance": dict(kind="moe", T=4096, E=256, k=8, H=7168, x_dtype=torch.bfloat16,
                          out_dtype=torch.bfloat16, seed=23),
    "tiny_moe": FULL["tiny_moe"],
    "splitk": FULL["splitk"],
    "embedding_backward": dict(kind="embedding", T=8192, V=131072, H=4096, zipf_s=1.0, sigma=0.02, seed=26),
}


def make(name: str, size: str = "full", device="cpu"):
    """Build a named workload ('full', 'medium' or 'small').  Returns a ScatterCase or a split-K tensor."""
    spec = dict({"full": FULL, "medium": MEDIUM, "small": SMALL}[size][name])
    kind = spec.pop("kind")
    if kind == "moe":
        return moe_combine(device=device, name=f"{name}[{size}]", **spec)
    if kind == "sparse":
        return sparse_key_scatter(device=device, name=f"{name}[{size}]", **spec)
    if kind == "embedding":
        return embedding_backward(device=device, name=f"{name}[{size}]", **spec)
    return splitk_partials(spec["S"], spec["R"], spec["C"], seed=spec["seed"], device=device)


def ep_shard_rows(case: ScatterCase, P: int):
    """Row counts of P expert shards: shard q holds experts [q*E/P, (q+1)*E/P) (contiguous row ranges)."""
    E = case.meta["E"]
    if E % P:
        raise ValueError("P must divide E")
    ex = case.meta["experts_of_row"]
    per = E // P
    return [int(((ex >= q * per) & (ex < (q + 1) * per)).sum()) for q in range(P)]


def split_rows(x: torch.Tensor, rows) -> list:
    """Copy consecutive row ranges of x into separate allocations (one per shard)."""
    out, r = [], 0
    for n in rows:
        out.append(x[r:r + n].clone())
        r += n
    return out


def round_up(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["ScatterCase", "moe_routing", "moe_combine", "zipf_key_lists", "sparse_key_scatter",
           "embedding_backward", "splitk_partials", "splitk_gemm_inputs", "FULL", "MEDIUM", "SMALL", "make", "ep_shard_rows", "split_rows", "round_up", "cdiv"]
