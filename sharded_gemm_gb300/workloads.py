"""The sharded-GEMM workloads as device-resident objects with one ``step()``.

Each class takes host arrays from ``synth`` (or arrays the caller prepared),
moves them to the GPU once, slices the weights into their N shard buffers
with ``tp_shard_weight`` (a1), allocates the outputs, and exposes ``step()``:
one pass of that workload's hot path through the C ABI.  Nothing here does
arithmetic of its own.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (tp_all_to_sharded, tp_all_to_sharded_dx, tp_bias_grad, tp_gated_all_to_sharded,
               tp_mx_all_to_sharded, tp_mx_quantize, tp_mx_sharded_to_all,
               tp_sharded_dw, tp_sharded_to_all_dx, tp_gathered_to_sharded, tp_q4_all_to_sharded,
               tp_q4_quantize,
               tp_q4_sharded_to_all, tp_shard_weight, tp_sharded_to_all, tp_sharded_to_sharded, tp_summa)


def to_device(a: np.ndarray, kind: str, device="cuda") -> torch.Tensor:
    """Host array -> device tensor. kind: 'bf16' (uint16 bits), 'f16', 'f32', 'u32'."""
    a = np.ascontiguousarray(a)
    if kind == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif kind == "f16":
        t = torch.from_numpy(a.view(np.float16) if a.dtype == np.uint16 else a.astype(np.float16))
    elif kind == "f32":
        t = torch.from_numpy(a.astype(np.float32))
    elif kind == "u32":
        t = torch.from_numpy(a.view(np.int32))
    else:
        raise ValueError(kind)
    return t.to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> host float64 (bf16 / f16 / f32 values are exact)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


class MLPPair:
    """Column-parallel W1 (out dims split on axis 0) feeding row-parallel W2
    (split on its last axis); the intermediate stays sharded (bf16)."""

    def __init__(self, cfg: dict, device="cuda", mid_dtype=torch.bfloat16, out_dtype=torch.float32):
        self.N = N = cfg["N"]
        kind = cfg["dtype"]
        self.x = to_device(cfg["x"], kind, device)
        w1 = to_device(cfg["w1"], kind, device)
        w2 = to_device(cfg["w2"], kind, device)
        self.w1 = tp_shard_weight(w1, 0, 1, N)
        self.b1 = tp_shard_weight(to_device(cfg["b1"], "f32", device), 0, 1, N)
        self.w2 = tp_shard_weight(w2, -1, 1, N)
        self.b2 = to_device(cfg["b2"], "f32", device)
        del w1, w2
        T = self.x.shape[0]
        if kind == "f32":
            mid_dtype = torch.float32
        self.mid = [torch.empty((T, self.w1[0].shape[0]), dtype=mid_dtype, device=device) for _ in range(N)]
        self.y = torch.empty((T, self.w2[0].shape[0]), dtype=out_dtype, device=device)
        self.flops = 2.0 * T * (cfg["w1"].shape[0] * cfg["w1"].shape[1] + cfg["w2"].shape[0] * cfg["w2"].shape[1])

    def step(self, x=None, stream=None):
        tp_all_to_sharded(self.x if x is None else x, self.w1, self.b1, out=self.mid, stream=stream)
        tp_sharded_to_all(self.mid, self.w2, self.b2, out=self.y, stream=stream)
        return self.y


class GatedFFN:
    """Llama FFN: gate W1 and up W3 column-parallel on the same x (one gated
    launch writing silu(x W1_r^T) * (x W3_r^T) per shard, bf16), then the
    row-parallel down projection W2 (float32 output)."""

    def __init__(self, cfg: dict, device="cuda", mid_dtype=torch.bfloat16, out_dtype=torch.float32):
        self.N = N = cfg["N"]
        kind = cfg["dtype"]
        self.x = to_device(cfg["x"], kind, device)
        for name, axis in (("w1", 0), ("w3", 0), ("w2", -1)):
            full = to_device(cfg[name], kind, device)
            setattr(self, name, tp_shard_weight(full, axis, 1, N))
            del full
        self.b1 = tp_shard_weight(to_device(cfg["b1"], "f32", device), 0, 1, N)
        self.b3 = tp_shard_weight(to_device(cfg["b3"], "f32", device), 0, 1, N)
        self.b2 = to_device(cfg["b2"], "f32", device)
        T = self.x.shape[0]
        if kind == "f32":
            mid_dtype = torch.float32
        self.h = [torch.empty((T, self.w1[0].shape[0]), dtype=mid_dtype, device=device) for _ in range(N)]
        self.y = torch.empty((T, self.w2[0].shape[0]), dtype=out_dtype, device=device)
        D, F = cfg["D"], cfg["F"]
        self.flops = 2.0 * T * 3 * D * F

    def step(self, x=None, stream=None):
        tp_gated_all_to_sharded(self.x if x is None else x, self.w1, self.w3, self.b1, self.b3, out=self.h,
                                stream=stream)
        tp_sharded_to_all(self.h, self.w2, self.b2, out=self.y, stream=stream)
        return self.y


class MLPGatherScatter:
    """The same two weights as ``MLPPair`` with the input and the output both
    sharded along the model width: an all-gather of the input's column
    shards feeds the column-parallel W1, and the row-parallel W2's partial
    sums are reduce-scattered, so rank c ends with column block c of the
    output (one all-gather and one reduce-scatter per FFN)."""

    def __init__(self, cfg: dict, device="cuda", mid_dtype=torch.bfloat16, out_dtype=torch.float32):
        self.N = N = cfg["N"]
        kind = cfg["dtype"]
        x = to_device(cfg["x"], kind, device)
        self.xs = tp_shard_weight(x, -1, 1, N)
        del x
        w1 = to_device(cfg["w1"], kind, device)
        w2 = to_device(cfg["w2"], kind, device)
        self.w1 = tp_shard_weight(w1, 0, 1, N)
        self.b1 = tp_shard_weight(to_device(cfg["b1"], "f32", device), 0, 1, N)
        self.w2 = tp_shard_weight(w2, -1, 1, N)
        self.b2 = to_device(cfg["b2"], "f32", device)
        del w1, w2
        T = self.xs[0].shape[0]
        if kind == "f32":
            mid_dtype = torch.float32
        D = cfg["w2"].shape[0]
        self.mid = [torch.empty((T, self.w1[0].shape[0]), dtype=mid_dtype, device=device) for _ in range(N)]
        self.ys = [torch.empty((T, D // N), dtype=out_dtype, device=device) for _ in range(N)]
        self.flops = 2.0 * T * (cfg["w1"].shape[0] * cfg["w1"].shape[1] + cfg["w2"].shape[0] * cfg["w2"].shape[1])

    def step(self, xs=None, stream=None):
        tp_gathered_to_sharded(self.xs if xs is None else xs, self.w1, self.b1, out=self.mid, stream=stream)
        tp_sharded_to_sharded(self.mid, self.w2, self.b2, out=self.ys, stream=stream)
        return self.ys


class MLPBackward:
    """Backward step of ``MLPPair`` (no activation between the layers) for an
    incoming gradient dy of its (T, D) output:
      dh_r  = dy @ W2_r                  (row-parallel input gradient, bf16)
      dW2_r = dy^T @ h_r,  db2 = sum_t dy
      dx    = sum_r dh_r @ W1_r          (column-parallel: all-summed, f32)
      dW1_r = dh_r^T @ x,  db1_r = sum_t dh_r
    Weight and bias gradients are float32.  ``h`` is the forward's sharded
    intermediate, computed once at construction."""

    def __init__(self, cfg: dict, dy: np.ndarray, device="cuda"):
        self.fwd = MLPPair(cfg, device=device)
        self.fwd.step()
        f = self.fwd
        self.N = N = f.N
        self.dy = to_device(dy, "bf16", device)
        T, D = self.dy.shape
        Fn = f.w1[0].shape[0]
        self.dh = [torch.empty((T, Fn), dtype=torch.bfloat16, device=device) for _ in range(N)]
        self.dw2 = [torch.empty((D, Fn), dtype=torch.float32, device=device) for _ in range(N)]
        self.db2 = [torch.empty((D,), dtype=torch.float32, device=device)]
        self.dx = torch.empty((T, D), dtype=torch.float32, device=device)
        self.dw1 = [torch.empty((Fn, D), dtype=torch.float32, device=device) for _ in range(N)]
        self.db1 = [torch.empty((Fn,), dtype=torch.float32, device=device) for _ in range(N)]
        self.flops = 4 * 2.0 * T * D * Fn * N

    def launches(self):
        f = self
        p = self.fwd
        return [
            lambda s: tp_sharded_to_all_dx(f.dy, p.w2, out=f.dh, stream=s),
            lambda s: tp_sharded_dw([f.dy] * f.N, p.mid, out=f.dw2, stream=s),
            lambda s: tp_bias_grad([f.dy], out=f.db2, stream=s),
            lambda s: tp_all_to_sharded_dx(f.dh, p.w1, out=f.dx, stream=s),
            lambda s: tp_sharded_dw(f.dh, [p.x] * f.N, out=f.dw1, stream=s),
            lambda s: tp_bias_grad(f.dh, out=f.db1, stream=s),
        ]

    def step(self, stream=None):
        for fn in self.launches():
            fn(stream)
        return self.dx


class Summa:
    def __init__(self, cfg: dict, q: int, device="cuda"):
        self.q = q
        M, K, Nc = cfg["M"], cfg["K"], cfg["Ncols"]
        X = to_device(cfg["X"], cfg["dtype"], device)
        A = to_device(cfg["A"], cfg["dtype"], device)
        bm, bk, bn = M // q, K // q, Nc // q
        self.X = [X[i * bm:(i + 1) * bm, j * bk:(j + 1) * bk].contiguous() for i in range(q) for j in range(q)]
        self.A = [A[i * bk:(i + 1) * bk, j * bn:(j + 1) * bn].contiguous() for i in range(q) for j in range(q)]
        del X, A
        self.Y = [torch.empty((bm, bn), dtype=torch.float32, device=device) for _ in range(q * q)]
        self.flops = 2.0 * M * K * Nc

    def step(self, stream=None):
        return tp_summa(self.q, self.X, self.A, self.Y, stream=stream)


class QKV:
    """Fused QKV (segments=3), row-parallel W_o on x split by columns, and a
    vocab-parallel LM head whose logits land in one gathered (T, V) buffer."""

    def __init__(self, cfg: dict, device="cuda"):
        self.N = N = cfg["N"]
        self.x = to_device(cfg["x"], "bf16", device)
        T, D, V = self.x.shape[0], cfg["D"], cfg["V"]
        wq = to_device(cfg["w_qkv"], "bf16", device)
        self.w_qkv = tp_shard_weight(wq, 0, 3, N)
        self.b_qkv = tp_shard_weight(to_device(cfg["b_qkv"], "f32", device), 0, 3, N)
        del wq
        wo = to_device(cfg["w_o"], "bf16", device)
        self.w_o = tp_shard_weight(wo, -1, 1, N)
        self.b_o = to_device(cfg["b_o"], "f32", device)
        del wo
        wl = to_device(cfg["w_lm"], "bf16", device)
        self.w_lm = tp_shard_weight(wl, 0, 1, N)
        del wl
        self.qkv = [torch.empty((T, 3 * D // N), dtype=torch.bfloat16, device=device) for _ in range(N)]
        self.attn_out = torch.empty((T, D), dtype=torch.float32, device=device)
        self.logits = torch.empty((T, V), dtype=torch.float32, device=device)
        Vn = V // N
        self.logit_views = [self.logits[:, r * Vn:(r + 1) * Vn] for r in range(N)]
        self.x_cols = [self.x[:, r * (D // N):(r + 1) * (D // N)] for r in range(N)]
        self.flops = 2.0 * T * D * (3 * D + D + V)
        self.weight_bytes = 2.0 * D * (3 * D + D + V)

    def step(self, stream=None):
        tp_all_to_sharded(self.x, self.w_qkv, self.b_qkv, out=self.qkv, stream=stream)
        tp_sharded_to_all(self.x_cols, self.w_o, self.b_o, out=self.attn_out, stream=stream)
        tp_all_to_sharded(self.x, self.w_lm, None, out=self.logit_views, stream=stream)
        return self.qkv, self.attn_out, self.logits


class Q4Pair:
    """4-bit affine quantized up (column-parallel) / down (row-parallel) pair.

    ``quantized`` may hold host (codes, scales, biases) for both weights; if
    absent the float32 source weights are quantized on the device (a6)."""

    def __init__(self, cfg: dict, device="cuda", quantized=None):
        self.N = N = cfg["N"]
        self.x = to_device(cfg["x"], "bf16", device)
        T, D, F = self.x.shape[0], cfg["D"], cfg["F"]
        if quantized is None:
            wu = to_device(cfg["w_up"], "f32", device)
            up = tp_q4_quantize(wu)
            del wu
            wd = to_device(cfg["w_down"], "f32", device)
            down = tp_q4_quantize(wd)
            del wd
        else:
            (uq, us, ub), (dq, ds, db) = quantized
            up = (to_device(uq, "u32", device), to_device(us, "f16", device), to_device(ub, "f16", device))
            down = (to_device(dq, "u32", device), to_device(ds, "f16", device), to_device(db, "f16", device))
        self.up = [tp_shard_weight(a, 0, 1, N) for a in up]
        self.down = [tp_shard_weight(a, -1, 1, N) for a in down]
        del up, down
        self.mid = [torch.empty((T, F // N), dtype=torch.bfloat16, device=device) for _ in range(N)]
        self.y = torch.empty((T, D), dtype=torch.float32, device=device)
        self.flops = 2.0 * T * 2 * D * F
        self.weight_bytes = 2 * D * F * (0.5 + 4.0 / 64)

    def step(self, x=None, stream=None):
        tp_q4_all_to_sharded(self.x if x is None else x, *self.up, out=self.mid, stream=stream)
        tp_q4_sharded_to_all(self.mid, *self.down, out=self.y, stream=stream)
        return self.y


class MXPair:
    """MXFP8 up (column-parallel) / down (row-parallel) pair on the 4-bit pair's
    shapes: the float32 source weights are quantized on the device (or
    ``quantized`` holds host (codes, scales) for both), then sliced into the N
    shards (codes and scales on the same axis)."""

    def __init__(self, cfg: dict, device="cuda", quantized=None):
        self.N = N = cfg["N"]
        self.x = to_device(cfg["x"], "bf16", device)
        T, D, F = self.x.shape[0], cfg["D"], cfg["F"]
        if quantized is None:
            wu = to_device(cfg["w_up"], "f32", device)
            up = tp_mx_quantize(wu)
            del wu
            wd = to_device(cfg["w_down"], "f32", device)
            down = tp_mx_quantize(wd)
            del wd
        else:
            (uc, us), (dc, ds) = quantized
            up = tuple(torch.from_numpy(a).to(device) for a in (uc, us))
            down = tuple(torch.from_numpy(a).to(device) for a in (dc, ds))
        self.up = [tp_shard_weight(a, 0, 1, N) for a in up]
        self.down = [tp_shard_weight(a, -1, 1, N) for a in down]
        del up, down
        self.mid = [torch.empty((T, F // N), dtype=torch.bfloat16, device=device) for _ in range(N)]
        self.y = torch.empty((T, D), dtype=torch.float32, device=device)
        self.flops = 2.0 * T * 2 * D * F
        self.weight_bytes = 2 * D * F * (1.0 + 1.0 / 32)

    def step(self, x=None, stream=None):
        tp_mx_all_to_sharded(self.x if x is None else x, *self.up, out=self.mid, stream=stream)
        tp_mx_sharded_to_all(self.mid, *self.down, out=self.y, stream=stream)
        return self.y
