"""Seeded synthetic workloads for the NVFP4 MoE expert forward.

This module only draws random inputs; it holds none of the NVFP4 arithmetic, so
the CUDA path and the CPU oracle can both consume its tensors.

Shapes and distributions follow the five workloads the kernels are measured on:

* ``tiny``     T=64,    K=256,  I=128,  E=8,   top-2, uniform routing
* ``linear``   M=4096,  K=7168, N=4096, one expert (shared-expert linear); the
               activation has 1% of its 16-element blocks all zero, 1% scaled
               far below the tensor maximum (2^-20 of it, so that the block
               underflows once the global scale is applied) and 1% scaled to a
               raw maximum in [2^-10, 6*2^-9) (blocks that are small in raw
               value but normal after the global scale)
* ``decode``   T=128,   K=7168, I=2048, E=256, top-8, uniform routing
* ``prefill``  T=8192,  same layer shape
* ``skewed``   T=16384, same layer shape, Zipf(1.2) expert popularity over a
               seeded permutation of the experts, 16 seeded experts never chosen
* ``dsv4_decode`` / ``dsv4_prefill``  T=128 / 8192, K=7168, I=3072, E=384,
               top-6, uniform routing: the DeepSeek-V4 routed-expert shape the
               pages name ("NVFP4 MegaMoE Kernel" README, model notes: 384
               experts, top-6, intermediate 3072)

x ~ N(0, 1) BF16, router logits ~ N(0, 1) f32 (the top-k of iid logits is a
uniformly random k-subset), weights ~ N(0, 0.02) BF16. W1 is drawn as (E, 2I, K)
with rows [gate | up] (the transpose of the (E, K, 2I) statement, K
contiguous), W2 as (E, K, I). For the skewed workload the logits are
log(p_e) + Gumbel(0, 1) noise (top-k of that is sampling without replacement
proportionally to p) with -inf for the never-chosen experts.

``gs_h`` is the pre-computed global scale of the SwiGLU output that the L1
epilogue requantizes with; it is part of the workload, a constant chosen so
that no block of h saturates on these distributions.
"""
from dataclasses import dataclass
import math

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    K: int
    I: int
    E: int
    k: int
    routing: str = "uniform"
    zipf_s: float = 1.2
    n_dead: int = 0
    gs_h: float = 28.0

    @property
    def M(self) -> int:
        return self.T * self.k

    def flops(self) -> float:
        """Useful FLOPs of one forward: L1 (2*M*K*2I) + L2 (2*M*I*K)."""
        return 6.0 * self.M * self.K * self.I


@dataclass(frozen=True)
class LinearConfig:
    name: str
    M: int
    K: int
    N: int
    zero_frac: float = 0.01
    underflow_frac: float = 0.01
    small_raw_frac: float = 0.01

    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


CONFIGS = {
    "tiny": MoEConfig("tiny", T=64, K=256, I=128, E=8, k=2, gs_h=1344.0),
    "linear": LinearConfig("linear", M=4096, K=7168, N=4096),
    "decode": MoEConfig("decode", T=128, K=7168, I=2048, E=256, k=8, gs_h=28.0),
    "prefill": MoEConfig("prefill", T=8192, K=7168, I=2048, E=256, k=8, gs_h=28.0),
    "skewed": MoEConfig("skewed", T=16384, K=7168, I=2048, E=256, k=8, routing="zipf",
                        zipf_s=1.2, n_dead=16, gs_h=28.0),
    # the h distribution depends on K and the weight scale, not on I, so the
    # same pre-computed gs_h leaves h unsaturated
    "dsv4_decode": MoEConfig("dsv4_decode", T=128, K=7168, I=3072, E=384, k=6, gs_h=28.0),
    "dsv4_prefill": MoEConfig("dsv4_prefill", T=8192, K=7168, I=3072, E=384, k=6, gs_h=28.0),
    # profiler-sized cases: the same layer and the same rows per expert as
    # prefill / decode, with 32 experts (0.8 GB of weights, still above L2)
    "prefill_small": MoEConfig("prefill_small", T=1024, K=7168, I=2048, E=32, k=8, gs_h=28.0),
    "decode_small": MoEConfig("decode_small", T=16, K=7168, I=2048, E=32, k=8, gs_h=28.0),
    # profiler-sized skewed case: 32 experts (2 never chosen) with the same
    # Zipf(1.2) popularity, so the heaviest expert still spans many activation
    # tiles that share each weight tile (0.8 GB of weights)
    "skewed_small": MoEConfig("skewed_small", T=2048, K=7168, I=2048, E=32, k=8, routing="zipf",
                              zipf_s=1.2, n_dead=2, gs_h=28.0),
    # profiler-sized case for the HBM-bound kernels (quantize, combine): 32768
    # routed rows, so the L2 output the combine reads (470 MB) exceeds L2
    "prefill_med": MoEConfig("prefill_med", T=4096, K=7168, I=2048, E=32, k=8, gs_h=28.0),
    # profiler-sized case of the front at the prefill token count: 65536 routed
    # rows (the front's quantize + scatter then runs as its own kernel) with
    # 32 experts, ~2 GB on the device
    "prefill_e32": MoEConfig("prefill_e32", T=8192, K=7168, I=2048, E=32, k=8, gs_h=28.0),
}

# independent sub-streams of one seed
_X, _LOGITS, _W1, _W2, _EDITS, _ZIPF = range(6)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + stream * 7919 + 17)
    return g


def _randn(shape, std, seed, stream, device, dtype):
    g = _gen(seed, stream, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def moe_inputs(cfg: MoEConfig, seed: int = 0, device="cpu", weights=True):
    """x (T,K) bf16, logits (T,E) f32, w1 (E,2I,K) bf16, w2 (E,K,I) bf16."""
    T, K, I, E = cfg.T, cfg.K, cfg.I, cfg.E
    out = {"cfg": cfg}
    out["x"] = _randn((T, K), 1.0, seed, _X, device, torch.bfloat16)
    if cfg.routing == "uniform":
        out["logits"] = _randn((T, E), 1.0, seed, _LOGITS, device, torch.float32)
    elif cfg.routing == "zipf":
        out["logits"] = _zipf_logits(cfg, seed, device)
    else:
        raise ValueError(cfg.routing)
    if weights:
        out["w1"] = torch.empty((E, 2 * I, K), dtype=torch.bfloat16, device=device)
        out["w2"] = torch.empty((E, K, I), dtype=torch.bfloat16, device=device)
        for e in range(E):
            out["w1"][e] = expert_weight(cfg, seed, 1, e, device)
            out["w2"][e] = expert_weight(cfg, seed, 2, e, device)
    out["gs_h"] = float(cfg.gs_h)
    return out


def expert_weight(cfg: MoEConfig, seed: int, which: int, e: int, device="cpu"):
    """W1[e] (which=1, shape (2I, K)) or W2[e] (which=2, shape (K, I)), drawn
    from a generator of its own so one expert can be drawn alone; the values
    equal moe_inputs()'s on the same device type."""
    shape = (2 * cfg.I, cfg.K) if which == 1 else (cfg.K, cfg.I)
    stream = (_W1 if which == 1 else _W2) * 100003 + e + 1
    return _randn(shape, 0.02, seed, stream, device, torch.bfloat16)


def _zipf_logits(cfg: MoEConfig, seed: int, device):
    g = _gen(seed, _ZIPF, "cpu")
    E = cfg.E
    order = torch.randperm(E, generator=g)
    rank = torch.empty(E, dtype=torch.float64)
    rank[order] = torch.arange(1, E + 1, dtype=torch.float64)
    p = rank.pow(-cfg.zipf_s)
    dead = torch.randperm(E, generator=g)[: cfg.n_dead]
    logp = p.log()
    logp[dead] = -math.inf
    u = torch.rand((cfg.T, E), generator=_gen(seed, _LOGITS, "cpu"), dtype=torch.float64)
    u = u.clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u).clamp_max(-1e-300))
    logits = (logp[None, :] + gumbel).to(torch.float32)
    return logits.to(device)


def linear_inputs(cfg: LinearConfig, seed: int = 0, device="cpu"):
    """x (M,K) bf16 with block edits, w (1,N,K) bf16."""
    M, K, N = cfg.M, cfg.K, cfg.N
    x = _randn((M, K), 1.0, seed, _X, "cpu", torch.float32)
    blocks = x.view(M, K // 16, 16)
    nb = blocks.shape[0] * blocks.shape[1]
    amax_x = x.abs().max()
    top = int(x.abs().argmax()) // 16          # the block holding the maximum stays
    g = _gen(seed, _EDITS, "cpu")
    perm = torch.randperm(nb, generator=g)
    perm = perm[perm != top]
    n0 = int(nb * cfg.zero_frac)
    n1 = int(nb * cfg.underflow_frac)
    n2 = int(nb * cfg.small_raw_frac)
    flat = blocks.view(nb, 16)
    zero_idx = perm[:n0]
    under_idx = perm[n0:n0 + n1]
    small_idx = perm[n0 + n1:n0 + n1 + n2]
    flat[zero_idx] = 0.0
    # scale each chosen block so that its own maximum is amax_x * 2^-20
    sub = flat[under_idx]
    sub = sub / sub.abs().amax(dim=1, keepdim=True) * (amax_x * 2.0 ** -20)
    flat[under_idx] = sub
    # raw maximum uniform in [2^-10, 6 * 2^-9)
    sub = flat[small_idx]
    target = 2.0 ** -10 + torch.rand((n2, 1), generator=g) * (6 * 2.0 ** -9 - 2.0 ** -10)
    flat[small_idx] = sub / sub.abs().amax(dim=1, keepdim=True) * target
    w = _randn((1, N, K), 0.02, seed, _W1, device, torch.bfloat16)
    return {"cfg": cfg, "x": x.to(torch.bfloat16).to(device), "w": w,
            "zero_blocks": zero_idx, "underflow_blocks": under_idx, "small_raw_blocks": small_idx}


def bf16_bits(t: torch.Tensor):
    """A BF16 tensor as a numpy uint16 array of its bit patterns (on the host)."""
    import numpy as np
    if t.dtype != torch.bfloat16:
        raise TypeError("bf16_bits expects a bfloat16 tensor, got %s" % t.dtype)
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
