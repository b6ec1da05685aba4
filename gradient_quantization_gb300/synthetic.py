"""Seeded synthetic inputs of the AGoQ quantization workloads.

This module draws random numbers and casts them to BF16; it holds none of the
quantization arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  Inputs that the method itself derives (FP8 shards, the INT4 operand
of the weight-gradient product) are quantized by the caller: the tests use
the oracle, the bench uses the library.

Two families of generators share each recipe:

* ``*_np`` functions use numpy's PCG64 and return BF16 bit patterns as
  ``numpy.uint16``.  A tensor is drawn in chunks of ``CHUNK`` consecutive
  elements; chunk c of tensor t comes from its own stream,
  ``PCG64(SeedSequence(seed, spawn_key=(t, c)))``, and within a chunk the
  values are drawn first, then the outlier mask.  The chunks are independent,
  so full-size tensors are drawn by several threads at once (numpy releases
  the GIL while it draws) with the same result as one thread.
* ``*_torch`` functions draw the same distributions on a torch device with a
  seeded ``torch.Generator``; they serve full-size runs, where the host would
  spend minutes drawing numbers.  Their values differ from the numpy ones.

Shapes follow the LLaMA-7B MLP (hidden 4096, FFN 11008), the layer types the
LAAQ section of "AGoQ: Activation and Gradient Quantization for
Memory-Efficient Distributed Training of LLMs" quantizes (RMSNorm and SiLU
inputs); no real activations or weights are used.
"""
import concurrent.futures as _cf
import os

import numpy as np
import torch

# Sizes of the named workloads.
LAAQ_INT4_SHAPE = (2048, 4096)            # one activation, 4-bit round trip
DBCA_RMSNORM_SHAPE = (8192, 4096)         # RMSNorm input
DBCA_SILU_SHAPE = (8192, 11008)           # SiLU/gate input
QUANGRAD_N = 1 << 30                      # flat gradient
QUANGRAD_STEPS = 8                        # micro-batches
REDUCE_N = 1 << 25                        # elements per shard
REDUCE_WS = (8, 64)                       # shard counts
WGRAD_M, WGRAD_N, WGRAD_K = 11008, 4096, 8192


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (library cast) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_tensor_from_bits(bits: np.ndarray) -> torch.Tensor:
    """View uint16 BF16 bit patterns as a torch.bfloat16 CPU tensor (no copy of values)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


# ---------------------------------------------------------------- numpy recipes
CHUNK = 1 << 22   # elements per independently seeded chunk


def chunk_rng(seed, tensor, chunk):
    """The PCG64 generator of chunk ``chunk`` of tensor ``tensor`` under ``seed``."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(tensor, chunk))))


def draw_bf16_np(seed, tensor, n, draw):
    """BF16 bit patterns [n] of one tensor: ``draw(rng, size)`` returns the float32
    values of one chunk; chunks are drawn (and rounded to BF16) in parallel."""
    out = np.empty(n, np.uint16)
    nchunks = (n + CHUNK - 1) // CHUNK

    def one(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        out[lo:hi] = bf16_bits_from_f32(draw(chunk_rng(seed, tensor, c), hi - lo))

    if nchunks <= 1:
        for c in range(nchunks):
            one(c)
    else:
        with _cf.ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(one, range(nchunks)))
    return out


def outlier_normal_np(rng, n, p=1e-3, factor=20.0, sd=1.0):
    """sd * N(0,1) float32 draws, then a Bernoulli(p) mask (drawn after the
    values) whose entries are multiplied by ``factor``."""
    x = rng.standard_normal(n, dtype=np.float32)
    if sd != 1.0:
        x *= np.float32(sd)
    mask = rng.random(n, dtype=np.float32) < p
    x[mask] *= np.float32(factor)
    return x


def laaq_activation_np(seed=0, tokens=LAAQ_INT4_SHAPE[0], hidden=LAAQ_INT4_SHAPE[1]):
    """BF16 activation [tokens x hidden]: N(0,1) with 0.1% of entries x20 (tensor 0)."""
    return draw_bf16_np(seed, 0, tokens * hidden, outlier_normal_np).reshape(tokens, hidden)


def dbca_activations_np(seed=1, tokens=DBCA_RMSNORM_SHAPE[0], hidden=DBCA_RMSNORM_SHAPE[1],
                        ffn=DBCA_SILU_SHAPE[1]):
    """(RMSNorm input [tokens x hidden] (tensor 0), SiLU input [tokens x ffn] (tensor 1)),
    Student-t nu=4, BF16."""
    t4 = lambda rng, m: rng.standard_t(4, m).astype(np.float32)   # noqa: E731
    return (draw_bf16_np(seed, 0, tokens * hidden, t4).reshape(tokens, hidden),
            draw_bf16_np(seed, 1, tokens * ffn, t4).reshape(tokens, ffn))


def quangrad_grad_np(seed=2, step=0, n=QUANGRAD_N):
    """Micro-batch ``step`` (tensor ``step``): N(0, sd 1e-3), 0.01% of entries x1000, BF16."""
    draw = lambda rng, m: outlier_normal_np(rng, m, p=1e-4, factor=1000.0, sd=1e-3)   # noqa: E731
    return draw_bf16_np(seed, step, n, draw)


def quangrad_grads_np(seed=2, n=QUANGRAD_N, steps=QUANGRAD_STEPS):
    """Yield the ``steps`` BF16 micro-batch gradients in order."""
    for k in range(steps):
        yield quangrad_grad_np(seed, k, n)


def reduce_shard_values_np(seed=3, W=8, n=REDUCE_N):
    """BF16 values of W shards [W][n]: shard r (tensor r + 1) is N(0, sd 1e-2 * j_r),
    with the factors j_r ~ U[0.5, 2) drawn first, from tensor 0's stream.  The
    caller block-quantizes each shard to FP8."""
    j = chunk_rng(seed, 0, 0).uniform(0.5, 2.0, W).astype(np.float32)
    out = np.empty((W, n), np.uint16)
    for r in range(W):
        sd = np.float32(np.float32(1e-2) * j[r])
        out[r] = draw_bf16_np(seed, r + 1, n,
                              lambda rng, m, sd=sd: rng.standard_normal(m, dtype=np.float32) * sd)
    return out


def wgrad_inputs_np(seed=4, M=WGRAD_M, N=WGRAD_N, K=WGRAD_K):
    """(dY BF16 [K x M] ~ N(0, sd 1e-2) (tensor 0), X BF16 [K x N] ~ N(0,1) with
    0.1% x20 (tensor 1)).  The caller quantizes X with the 4-bit LAAQ rule."""
    dy = draw_bf16_np(seed, 0, K * M,
                      lambda rng, m: rng.standard_normal(m, dtype=np.float32) * np.float32(1e-2))
    x = draw_bf16_np(seed, 1, K * N, outlier_normal_np)
    return dy.reshape(K, M), x.reshape(K, N)


def wgrad_exact_sum_inputs_np(seed=5, M=WGRAD_M, N=WGRAD_N, K=WGRAD_K):
    """(dY BF16 [K x M], X BF16 [K x N]) on a power-of-two grid, for checks whose
    FP32 accumulation must be exact in any summation order.  dY = i * 2^-6 with
    i uniform in -3..3; each 128-element block of an X row is c * 2^e with c
    uniform in -7..7, e uniform in -4..0 per block, and element 0 of the block
    set to +-7 * 2^e (random sign) so that the block absmax is 7 * 2^e.  Draw
    order: dY integers, X integers, block exponents, block signs."""
    rng = np.random.default_rng(seed)
    dy = rng.integers(-3, 4, K * M).astype(np.float32) * np.float32(2.0 ** -6)
    c = rng.integers(-7, 8, (K, N // 128, 128)).astype(np.float32)
    e = rng.integers(-4, 1, (K, N // 128, 1))
    sign = np.where(rng.random((K, N // 128)) < 0.5, -1.0, 1.0).astype(np.float32)
    c[:, :, 0] = 7.0 * sign
    x = (c * np.ldexp(np.float32(1.0), e).astype(np.float32)).astype(np.float32)
    return bf16_bits_from_f32(dy).reshape(K, M), bf16_bits_from_f32(x.reshape(-1)).reshape(K, N)


# ---------------------------------------------------------------- torch recipes
def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def outlier_normal_torch(gen, n, device, p=1e-3, factor=20.0, sd=1.0):
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    if sd != 1.0:
        x.mul_(sd)
    mask = torch.rand(n, generator=gen, device=device, dtype=torch.float32) < p
    x[mask] *= factor
    return x.to(torch.bfloat16)


def student_t4_torch(gen, n, device):
    """Student-t with 4 degrees of freedom from its definition z / sqrt(chi2_4 / 4)."""
    z = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    chi2 = torch.zeros(n, device=device, dtype=torch.float32)
    for _ in range(4):
        u = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        chi2.addcmul_(u, u)
    return (z / torch.sqrt(chi2 / 4.0)).to(torch.bfloat16)


def laaq_activation_torch(seed=0, device="cuda", tokens=LAAQ_INT4_SHAPE[0],
                          hidden=LAAQ_INT4_SHAPE[1]):
    g = _gen(device, seed)
    return outlier_normal_torch(g, tokens * hidden, device).view(tokens, hidden)


def dbca_activations_torch(seed=1, device="cuda", tokens=DBCA_RMSNORM_SHAPE[0],
                           hidden=DBCA_RMSNORM_SHAPE[1], ffn=DBCA_SILU_SHAPE[1]):
    g = _gen(device, seed)
    a = student_t4_torch(g, tokens * hidden, device).view(tokens, hidden)
    b = student_t4_torch(g, tokens * ffn, device).view(tokens, ffn)
    return a, b


def quangrad_grad_torch(seed=2, step=0, device="cuda", n=QUANGRAD_N):
    """Micro-batch ``step`` of the accumulation workload (each step has its own stream)."""
    g = _gen(device, seed * 1000003 + step)
    return outlier_normal_torch(g, n, device, p=1e-4, factor=1000.0, sd=1e-3)


def reduce_shard_values_torch(seed=3, W=8, device="cuda", n=REDUCE_N):
    g = _gen(device, seed)
    j = torch.rand(W, generator=g, device=device) * 1.5 + 0.5
    out = torch.empty((W, n), device=device, dtype=torch.bfloat16)
    for r in range(W):
        v = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        out[r] = (v * (1e-2 * j[r])).to(torch.bfloat16)
    return out


def wgrad_inputs_torch(seed=4, device="cuda", M=WGRAD_M, N=WGRAD_N, K=WGRAD_K):
    g = _gen(device, seed)
    dy = (torch.randn(K * M, generator=g, device=device) * 1e-2).to(torch.bfloat16).view(K, M)
    x = outlier_normal_torch(g, K * N, device).view(K, N)
    return dy, x
