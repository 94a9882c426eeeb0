"""Seeded bf16 tensors shaped like hidden-4096 transformer linear layers.

Recipe (the same for every test and for the benchmark):
  * generator: numpy PCG64 seeded by SeedSequence([stream, seed]), so every tensor of a
    workload has its own independent stream;
  * N(0, sigma) means mean 0 and standard deviation sigma; samples are drawn in float64,
    multiplied by sigma, narrowed to float32 and rounded to bf16 (round-to-nearest-even,
    done by torch's dtype conversion);
  * outliers: an independent Bernoulli(p) mask (its own stream) multiplies the chosen
    entries by a constant factor before the bf16 rounding;
  * the delayed-scaling sequence draws sigma_t log-uniformly and independently per step.

Tensors come back as numpy uint16 arrays holding bf16 bit patterns, row-major.
"""
import numpy as np
import torch

STREAM_X = 0
STREAM_W = 1
STREAM_DY = 2
STREAM_W2 = 3
STREAM_OUTLIER = 4
STREAM_SIGMA = 99
STREAM_STEP0 = 100


def _rng(seed, stream):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(stream), int(seed)])))


def bf16_bits_from_f32(a):
    """float32 array -> bf16 bit patterns (uint16), round-to-nearest-even via torch."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits):
    """bf16 bit patterns (uint16) -> float32 (exact: bf16 is the top half of float32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_normal(rows, cols, sigma=1.0, seed=0, stream=STREAM_X,
                     outlier_p=0.0, outlier_factor=50.0):
    """A [rows, cols] bf16 tensor of iid N(0, sigma) samples, optionally with outliers."""
    g = _rng(seed, stream)
    a = g.standard_normal((rows, cols)) * float(sigma)
    if outlier_p > 0.0:
        mask = _rng(seed, STREAM_OUTLIER).random((rows, cols)) < outlier_p
        a[mask] *= outlier_factor
    return bf16_bits_from_f32(a.astype(np.float32))


def sigma_schedule(steps, lo=0.5, hi=4.0, seed=0):
    """sigma_t for the delayed-scaling sequence: iid log-uniform in [lo, hi]."""
    g = _rng(seed, STREAM_SIGMA)
    return np.exp(g.uniform(np.log(lo), np.log(hi), size=steps))


def workload_shapes():
    """The five seeded workloads and their tensor shapes (rows, cols) and sigmas."""
    return {
        "tensorwise_256": dict(M=256, N=256, K=256, x_sigma=1.0, w_sigma=1.0),
        "mxfp8_fprop_8192x4096x4096": dict(M=8192, N=4096, K=4096, x_sigma=1.0, w_sigma=0.02,
                                           outlier_p=1e-3, outlier_factor=50.0),
        "blockwise_fwd_bwd_4096": dict(M=4096, N=4096, K=4096, x_sigma=1.0, w_sigma=0.02,
                                       dy_sigma=1e-3),
        "delayed_64_steps_8192x4096x4096": dict(M=8192, N=4096, K=4096, w_sigma=0.02, steps=64,
                                                history_len=1024, sigma_lo=0.5, sigma_hi=4.0),
        "mxfp8_mlp_8192x4096x16384": dict(M=8192, H=4096, F=16384, x_sigma=1.0, w_sigma=0.02,
                                          dy_sigma=1e-3),
    }
