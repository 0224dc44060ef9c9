"""Seeded synthetic inputs for the quantized linear layer workloads.

Holds none of the method's arithmetic: only random draws with the shapes and
value distributions of the five workloads, shared by the tests, the
benchmark and (through the tests) the CPU oracle.  Everything is numpy on
the host; callers move arrays to the GPU themselves.

Workloads (default seeds 0..4):
  tiny_w4a16      T=1, N=256, K=512: X ~ N(0,1) fp16; codes ~ U{0..15};
                  fp16 scales ~ U[0.005, 0.02]; symmetric zero-point 8.
  w4a16_decode    T in {1,4,16}; (N,K) in {(4096,4096),(11008,4096),
                  (4096,11008)} (Llama-2-7B-shaped layers): X ~ N(0,1) fp16,
                  W ~ N(0, 0.02) fp32 (quantized g128 asymmetric by the path).
  w4a16_packed_random  already-packed uint4 g128 weights for shapes too large
                  to draw and quantize in fp32: every byte ~ U{0..255} (two
                  codes), fp16 scales ~ U[0.005, 0.02], packed zero-points
                  ~ U{0..255}; X ~ N(0,1) fp16.
  w8a8_sym_bias   T=2048, K=4096, N=4096: X ~ N(0,1) with 1% of channels
                  (41, seeded choice) scaled x20, fp16; W ~ N(0, 0.02) fp32;
                  bias ~ N(0, 0.1) fp16.
  w8a8_azp_token  T=4096, K=4096, N=14336: X ~ U[-1, 3] fp16; W ~ N(0, 0.02)
                  fp32; bias ~ N(0, 0.1) fp16.
  nvfp4_arc       T=2048, K=4096, N=4096, S=128: X ~ N(0,1) with 2% of
                  channels (82, seeded choice) scaled x50, fp16; W ~ N(0, 0.02).
"""

import numpy as np

LLAMA2_7B_LAYERS = ((4096, 4096), (11008, 4096), (4096, 11008))


def _outlier_count(k, frac):
    return int(round(frac * k))


def tiny_w4a16(seed=0, T=1, N=256, K=512):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K), dtype=np.float32).astype(np.float16)
    codes = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    scales = rng.uniform(0.005, 0.02, size=(N, K // 128)).astype(np.float16)
    return {"x": x, "codes": codes, "scales": scales, "zeros": None}


def w4a16_packed_random(seed, T, N, K):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K), dtype=np.float32).astype(np.float16)
    wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.uniform(0.005, 0.02, size=(N, K // 128)).astype(np.float16)
    zeros = rng.integers(0, 256, size=(N, (K // 128 + 1) // 2), dtype=np.uint8)
    return {"x": x, "wq": wq, "scales": scales, "zeros": zeros}


def w4a16_decode(seed=1, T=1, N=4096, K=4096):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K), dtype=np.float32).astype(np.float16)
    w = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    return {"x": x, "w": w}


def w8a8_sym_bias(seed=2, T=2048, K=4096, N=4096, outlier_frac=0.01, outlier_scale=20.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K), dtype=np.float32)
    cols = rng.choice(K, _outlier_count(K, outlier_frac), replace=False)
    x[:, cols] *= np.float32(outlier_scale)
    w = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    bias = (rng.standard_normal(N, dtype=np.float32) * np.float32(0.1)).astype(np.float16)
    return {"x": x.astype(np.float16), "w": w, "bias": bias, "outlier_cols": np.sort(cols)}


def w8a8_azp_token(seed=3, T=4096, K=4096, N=14336):
    rng = np.random.default_rng(seed)
    x = rng.uniform(-1.0, 3.0, size=(T, K)).astype(np.float16)
    w = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    bias = (rng.standard_normal(N, dtype=np.float32) * np.float32(0.1)).astype(np.float16)
    return {"x": x, "w": w, "bias": bias}


def nvfp4_arc(seed=4, T=2048, K=4096, N=4096, S=128, outlier_frac=0.02, outlier_scale=50.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K), dtype=np.float32)
    cols = rng.choice(K, _outlier_count(K, outlier_frac), replace=False)
    x[:, cols] *= np.float32(outlier_scale)
    w = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    return {"x": x.astype(np.float16), "w": w, "S": S, "outlier_cols": np.sort(cols)}
