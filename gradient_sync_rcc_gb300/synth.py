"""Seeded synthetic inputs shaped like the workloads the pages describe.

This module only draws random numbers; it holds none of the collectives' or
the optimizer's arithmetic.  The same arrays feed both the CUDA library and
the CPU oracle in the tests, so the two sides never generate data of their own.

Streams are keyed by a tuple (workload, rank, tensor, step, ...) on top of a
fixed base seed, so any one rank buffer can be regenerated on its own.

Host (numpy, PCG64 through SeedSequence):
  uniform_pm1   U[-1, 1) on the 2^-23 grid (24-bit mantissa values)
  int_pm1000    integers uniform in [-1000, 1000], stored as fp32
  normal        N(0, sigma^2) drawn in fp64, rounded to fp32
  gradient_like N(0, sigma^2) with a Bernoulli(p) fraction scaled by `scale`
  bf16_normal   N(0, 1) rounded to bf16 (torch's CPU conversion), as uint16 bits
  param_sizes   log-uniform integer sizes in [lo, hi]
Device (torch generators, for workloads too large to move through the host):
  gpu_rank_buffers(kind, R, n, dtype, key, device)
"""
import math

import numpy as np

BASE_SEED = 0x5EEDC0DE


def _seq(*key):
    return np.random.SeedSequence([BASE_SEED, *[int(k) & 0xFFFFFFFF for k in key]])


def rng(*key) -> np.random.Generator:
    return np.random.default_rng(_seq(*key))


def seed32(*key) -> int:
    return int(_seq(*key).generate_state(1, np.uint32)[0])


# ----------------------------------------------------------------- host draws

def uniform_pm1(n, *key):
    k = rng(*key).integers(-(1 << 23), 1 << 23, size=n, dtype=np.int64)
    return (k.astype(np.float64) / float(1 << 23)).astype(np.float32)


def int_pm1000(n, *key):
    return rng(*key).integers(-1000, 1001, size=n).astype(np.float32)


def normal(n, sigma, *key):
    return (rng(*key).standard_normal(n) * sigma).astype(np.float32)


def gradient_like(n, *key, sigma=1e-2, p=1e-3, scale=100.0):
    g = rng(*key)
    x = g.standard_normal(n) * sigma
    mask = g.random(n) < p
    x[mask] *= scale
    return x.astype(np.float32)


def bf16_normal(n, *key):
    import torch
    x = torch.from_numpy(rng(*key).standard_normal(n).astype(np.float32))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_uniform_pm1(n, *key):
    import torch
    x = torch.from_numpy(uniform_pm1(n, *key))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def param_sizes(P, lo, hi, *key):
    u = rng(*key).random(P)
    return [int(round(math.exp(math.log(lo) + v * (math.log(hi) - math.log(lo))))) for v in u]


KINDS = {
    "uniform": lambda n, key: uniform_pm1(n, *key),
    "int": lambda n, key: int_pm1000(n, *key),
    "grad": lambda n, key: gradient_like(n, *key),
    "normal1": lambda n, key: normal(n, 1.0, *key),
}


def rank_buffers(kind, R, n, *key):
    """R host arrays, rank r drawn from stream (*key, r)."""
    if kind == "bf16_normal":
        return [bf16_normal(n, *key, r) for r in range(R)]
    if kind == "bf16_uniform":
        return [bf16_uniform_pm1(n, *key, r) for r in range(R)]
    return [KINDS[kind](n, (*key, r)) for r in range(R)]


# --------------------------------------------------------------- device draws

def gpu_draw(kind, n, dtype, key, device):
    """One device tensor of n elements drawn from a torch generator seeded by key."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed32(*key))
    if kind == "uniform":
        k = torch.randint(-(1 << 23), 1 << 23, (n,), generator=g, device=device, dtype=torch.int32)
        x = k.to(torch.float32) * (1.0 / (1 << 23))
    elif kind == "int":
        x = torch.randint(-1000, 1001, (n,), generator=g, device=device,
                          dtype=torch.int32).to(torch.float32)
    elif kind == "grad":
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32) * 1e-2
        mask = torch.rand(n, generator=g, device=device) < 1e-3
        x = torch.where(mask, x * 100.0, x)
    elif kind == "normal1":
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    elif kind.startswith("normal:"):
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32) * float(kind[7:])
    else:
        raise ValueError(kind)
    return x.to(dtype)


def gpu_rank_buffers(kind, R, n, dtype, key, device="cuda"):
    return [gpu_draw(kind, n, dtype, (*key, r), device) for r in range(R)]
