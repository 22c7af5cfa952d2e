"""Seeded synthetic inputs for the sharded-GEMM workloads.

This module only draws random numbers and stores them in the element types the
path consumes; it holds none of the method's arithmetic (no products, no
slicing, no sums, no quantization), so both the CUDA path and the CPU oracle
may take their inputs from it.

Conventions:
* numpy PCG64 generators; one sub-stream per tensor, spawned from
  ``SeedSequence(seed)`` in the fixed order in which a workload lists them;
* ``normal(std)`` means standard deviation ``std``;
* bfloat16 tensors are returned as their uint16 bit patterns, rounded from the
  float32 draw to nearest-even.

Workload shapes are the ones the pages use as stand-ins: an MLX-style
``Linear(2, 2)`` worked example, a Llama-7B-shaped MLP (4096 -> 11008) and
gated FFN (gate / up 4096 -> 11008, down 11008 -> 4096), SUMMA
on an 8192-square product, Llama-shaped fused-QKV / output projections with an
OPT-sized vocabulary (50272) LM head, and a Llama-70B-shaped MLP (8192 <->
28672) for the 4-bit quantized pair.
"""
from __future__ import annotations

import math

import numpy as np

SEED = 0


def streams(seed: int, n: int) -> list[np.random.Generator]:
    """``n`` independent PCG64 generators spawned from ``seed``."""
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rnd = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + rnd) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """float32 values of bfloat16 bit patterns (exact)."""
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_f32(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def normal_bf16(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return f32_to_bf16_bits(normal_f32(g, shape, std))


def uniform_f32(g: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return g.uniform(lo, hi, size=shape).astype(np.float32)


# ------------------------------------------------------------------ workloads
def worked(seed: int = SEED) -> dict:
    """MLX worked example: x (4, 2) float32 U[-1, 1]; column-parallel
    Linear(2 -> 2, bias) then row-parallel Linear(2 -> 2, bias), N = 2.
    Weights and biases U[-1/sqrt(2), 1/sqrt(2)] (MLX's scale sqrt(1/in))."""
    gx, gw1, gb1, gw2, gb2 = streams(seed, 5)
    sc = math.sqrt(1.0 / 2.0)
    return dict(
        name="worked", N=2, dtype="f32",
        x=uniform_f32(gx, (4, 2), -1.0, 1.0),
        w1=uniform_f32(gw1, (2, 2), -sc, sc), b1=uniform_f32(gb1, (2,), -sc, sc),
        w2=uniform_f32(gw2, (2, 2), -sc, sc), b2=uniform_f32(gb2, (2,), -sc, sc),
    )


def mlp(seed: int = SEED, T: int = 512, D: int = 4096, F: int = 11008, N: int = 4,
        bias_std: float = 0.0) -> dict:
    """Column -> row MLP pair: x (T, D) bf16 N(0,1); W1 (F, D), W2 (D, F) bf16
    N(0, 0.02); biases zero (or N(0, bias_std) when bias_std > 0, float32)."""
    gx, gw1, gb1, gw2, gb2 = streams(seed, 5)
    b1 = normal_f32(gb1, (F,), bias_std) if bias_std else np.zeros((F,), np.float32)
    b2 = normal_f32(gb2, (D,), bias_std) if bias_std else np.zeros((D,), np.float32)
    return dict(
        name="mlp", N=N, T=T, D=D, F=F, dtype="bf16",
        x=normal_bf16(gx, (T, D), 1.0),
        w1=normal_bf16(gw1, (F, D), 0.02), b1=b1,
        w2=normal_bf16(gw2, (D, F), 0.02), b2=b2,
    )


def ffn(seed: int = SEED, T: int = 512, D: int = 4096, F: int = 11008, N: int = 4,
        bias_std: float = 0.0) -> dict:
    """Gated (Llama) FFN: x (T, D) bf16 N(0,1); gate W1 (F, D), up W3 (F, D),
    down W2 (D, F) bf16 N(0, 0.02); biases zero (or N(0, bias_std) float32)."""
    gx, gw1, gw3, gw2, gb1, gb3, gb2 = streams(seed, 7)

    def bias(g, n):
        return normal_f32(g, (n,), bias_std) if bias_std else np.zeros((n,), np.float32)
    return dict(
        name="ffn", N=N, T=T, D=D, F=F, dtype="bf16",
        x=normal_bf16(gx, (T, D), 1.0),
        w1=normal_bf16(gw1, (F, D), 0.02), w3=normal_bf16(gw3, (F, D), 0.02),
        w2=normal_bf16(gw2, (D, F), 0.02),
        b1=bias(gb1, F), b3=bias(gb3, F), b2=bias(gb2, D),
    )


def grad_output(seed: int = SEED, T: int = 512, D: int = 4096) -> dict:
    """An incoming output gradient dy (T, D) bf16 N(0, 1) for a backward step
    (its own seed stream, so it is independent of the forward's inputs)."""
    (g,) = streams(seed + 1000003, 1)
    return dict(name="grad", T=T, D=D, dy=normal_bf16(g, (T, D), 1.0))


def summa(seed: int = SEED, M: int = 8192, K: int = 8192, Ncols: int = 8192) -> dict:
    """SUMMA Y = X A: X (M, K), A (K, Ncols) bf16 N(0, 1/sqrt(K))."""
    gx, ga = streams(seed, 2)
    std = 1.0 / math.sqrt(K)
    return dict(name="summa", M=M, K=K, Ncols=Ncols, dtype="bf16",
                X=normal_bf16(gx, (M, K), std), A=normal_bf16(ga, (K, Ncols), std))


def qkv(seed: int = SEED, T: int = 16, D: int = 4096, V: int = 50272, N: int = 8,
        bias_std: float = 0.0) -> dict:
    """Fused-QKV attention projections and a vocab-parallel LM head, N = 8.

    x (T, D) bf16 N(0,1); W_qkv (3D, D) [Q; K; V stacked], W_o (D, D) and the
    LM head W (V, D), all bf16 N(0, 0.02); biases zero unless bias_std > 0.
    The W_o input is x itself, split by columns across the N shards."""
    gx, gq, go, gl, gbq, gbo = streams(seed, 6)
    bq = normal_f32(gbq, (3 * D,), bias_std) if bias_std else np.zeros((3 * D,), np.float32)
    bo = normal_f32(gbo, (D,), bias_std) if bias_std else np.zeros((D,), np.float32)
    return dict(
        name="qkv", N=N, T=T, D=D, V=V, dtype="bf16",
        x=normal_bf16(gx, (T, D), 1.0),
        w_qkv=normal_bf16(gq, (3 * D, D), 0.02), b_qkv=bq,
        w_o=normal_bf16(go, (D, D), 0.02), b_o=bo,
        w_lm=normal_bf16(gl, (V, D), 0.02),
    )


def q4(seed: int = SEED, T: int = 16, D: int = 8192, F: int = 28672, N: int = 8) -> dict:
    """4-bit quantized pair: float32 source weights W_up (F, D) and W_down (D, F)
    N(0, 0.02) (quantized later), x (T, D) bf16 N(0, 1)."""
    gx, gu, gd = streams(seed, 3)
    return dict(
        name="q4", N=N, T=T, D=D, F=F, dtype="bf16",
        x=normal_bf16(gx, (T, D), 1.0),
        w_up=normal_f32(gu, (F, D), 0.02),
        w_down=normal_f32(gd, (D, F), 0.02),
    )
