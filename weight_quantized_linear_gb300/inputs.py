"""Seeded synthetic inputs shared by the tests, the benchmark and the CPU oracle's callers.

This module only draws random numbers; it contains none of the quantisation arithmetic, and it
imports nothing from the library or from the oracle.

Recipe (numpy PCG64; one child stream per tensor from ``SeedSequence(seed).spawn(5)`` in the order
weight, activation, weight-outlier mask, activation-outlier mask, gamma):
  * weights W [K, N] fp32 ~ N(0, 0.02); when weight outliers are on, exactly round(0.001 K N)
    positions drawn uniformly without replacement are multiplied by 10;
  * activations X [M, K] ~ N(0, 1); when activation outliers are on, round(0.01 K) input channels
    drawn without replacement are multiplied by 20; then rounded to fp16;
  * RMSNorm weight gamma [K] ~ U(0.5, 1.5), rounded to fp16; eps = 1e-6.
These stand in for the Llama-2-7B / InternLM layers of the source pages, whose weights and
calibration data are not available.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def _streams(seed: int):
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(5)]


def weight(K: int, N: int, seed: int = 0, outliers: bool = False) -> np.ndarray:
    rw, _, rmw, _, _ = _streams(seed)
    W = rw.standard_normal((K, N), dtype=np.float32)
    W *= np.float32(0.02)
    if outliers:
        n_out = int(round(0.001 * K * N))
        if n_out:
            idx = rmw.choice(K * N, size=n_out, replace=False)
            W.reshape(-1)[idx] *= np.float32(10.0)
    return W


def activations(M: int, K: int, seed: int = 0, outlier_channels: bool = False) -> np.ndarray:
    _, rx, _, rmx, _ = _streams(seed)
    X = rx.standard_normal((M, K), dtype=np.float32)
    if outlier_channels:
        n_ch = int(round(0.01 * K))
        if n_ch:
            ch = rmx.choice(K, size=n_ch, replace=False)
            X[:, ch] *= np.float32(20.0)
    return X.astype(np.float16)


def gamma(K: int, seed: int = 0) -> np.ndarray:
    rg = _streams(seed)[4]
    return rg.uniform(0.5, 1.5, size=K).astype(np.float16)


# ----------------------------------------------------------------------------------------------
# The five workload families (Llama-7B-shaped layers).
# ----------------------------------------------------------------------------------------------

def tiny_cases():
    """Tiny W4A16 AWQ linear: M=1, K=N=512, G=128, no outliers, seed 0."""
    return [dict(M=1, K=512, N=512, G=128, w_outliers=False, x_outliers=False)]


def decode_cases():
    """Decode W4A16 GEMV, q_proj shape K=N=4096, G=128, M in {1, 4, 16}, 0.1% weight outliers."""
    return [dict(M=m, K=4096, N=4096, G=128, w_outliers=True, x_outliers=False) for m in (1, 4, 16)]


def sweep_cases():
    """Layer sweep: fused QKV, gate_up, down x G in {32, 64, 128} x M in {1, 8, 32, 128, 256}."""
    shapes = [(4096, 12288), (4096, 22016), (11008, 4096)]
    return [dict(M=m, K=k, N=n, G=g, w_outliers=True, x_outliers=False)
            for (k, n) in shapes for g in (32, 64, 128) for m in (1, 8, 32, 128, 256)]


def prefill_cases():
    """Prefill W4A16: M in {512, 2048, 8192}, K=4096, N in {11008, 4096}, G=128, 1% x20 activation channels."""
    return [dict(M=m, K=4096, N=n, G=128, w_outliers=False, x_outliers=True)
            for m in (512, 2048, 8192) for n in (11008, 4096)]


def w8a8_cases():
    """SmoothQuant block: K=4096, N in {4096, 11008}, M in {1, 16, 512, 4096}, 1% x20 activation channels."""
    return [dict(M=m, K=4096, N=n, w_outliers=False, x_outliers=True)
            for n in (4096, 11008) for m in (1, 16, 512, 4096)]
