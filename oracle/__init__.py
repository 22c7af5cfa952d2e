"""CPU oracle for the sharded matrix multiply behind tensor-parallel linears.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library (``sharded_gemm_gb300``) never imports, links or
calls it, and it shares no code with the CUDA path: the two meet only through
the seeded input generators in ``sharded_gemm_gb300.synth``, which hold none
of the method's arithmetic.

Everything here is the plain definition, computed in float64:

* linear layers follow "MLX tensor parallelism guide" section 2.1/2.2: weight
  ``(output_dims, input_dims)``, ``y = x @ W.T + b``;
* parameter slicing follows the same page, section 3.2 (``_shard``): split the
  array into ``segments`` equal parts along the axis, split each part into
  ``N`` equal parts, keep part ``r`` of each and concatenate them in order;
* the column-parallel layer (section 2.1) is the local linear of each shard
  with no communication; the row-parallel layer (section 2.2) sums the local
  partial products over all shards and adds the bias once, after the sum;
* the gated FFN follows the same page, sections 5.2-5.3: gate (w1) and up
  (w3) projections are both column-parallel, and the elementwise
  ``silu(gate) * up`` runs on each rank's shard;
* backward: the column-parallel layer's input gradient is the all_sum of the
  ranks' local gradients (MLX guide, sum_gradients), the row-parallel one's
  needs none; weight gradients are dy^T x per shard; bias gradients are row
  sums; the 2-D layer's backward products are Matmul_ABT_2D / Matmul_ATB_2D
  of the SUMMA page and its bias is added per column block (add_bias_2d);
* the reduce-scatter and all-gather variants follow "sharded matrices"
  notes, cases 2 and 3 and the collective-primitive table: the reduce-scatter
  adds the ranks' partial products in rank order and gives rank c column
  block c of the sum; the all-gather joins the input's column shards in rank
  order before the column-parallel product;
* SUMMA follows "ColossalAI 2D tensor parallel via SUMMA", equations (1) and
  (2): block ``Y_ij`` is the sum over steps ``t = 0..q-1`` of ``X_it A_tj``,
  accumulated in step order;
* the 4-bit affine quantized weight (same MLX page, section 2.3: group_size 64,
  bits 4, mode "affine") dequantizes to ``s[o, g] * q[o, k] + b[o, g]`` with
  ``g = k // group_size``;
* the "mxfp8" mode of the same section (no per-group biases) is the OCP
  microscaling FP8 format: E4M3 codes, one power-of-two E8M0 scale per 32
  consecutive elements; ``W_hat[o, k] = e4m3(q[o, k]) * 2^(s[o, k // 32] - 127)``.

The matrix products run in the naive C loops of ``oracle.c`` (pinned against
``numpy.matmul`` by the tests); slicing and sums use numpy directly.

Pins (see ``tests/test_oracle.py``): closed-form shard index rule, brute-force
slicing, the sharded == unsharded invariant, the SUMMA q=2 block identity and
the blockwise-identity special case, the ABT / ATB block identities and
numpy transposes, the adjoint identity <dy, f(x)> = <f^T(dy), x> of every
gradient, integer bias-gradient sums, SiLU closed forms, the gated
sharded == unsharded invariant, the all-gather / reduce-scatter transpose
identity, the sharded == unsharded invariant of both collective
variants, the dequant identity on brute-force and constant-code inputs, the
quantizer round-trip bound, the E4M3 value table's closed forms, its rounding at every
midpoint and the MXFP8 scale choice, error bound and exact grid, and the worked-example shapes
from the MLX page.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-shared", "-fPIC", _SRC, "-o", tmp]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        i64 = ctypes.c_int64
        dp = ctypes.POINTER(ctypes.c_double)
        for name in ("orc_gemm_nt", "orc_gemm_nn"):
            fn = getattr(lib, name)
            fn.argtypes = [i64, i64, i64, dp, i64, dp, i64, dp, i64]
            fn.restype = None
        lib.orc_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the C loops use (OpenMP's default: all host cores)."""
    return int(_load().orc_num_threads())


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


# ---------------------------------------------------------------- widening
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (uint16) as float64."""
    u = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f16_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact value of float16 numbers (or their uint16 bit patterns) as float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.float16)
    return a.astype(np.float64)


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """float64 copy of ``a`` holding ``dtype`` values ('bf16' bits, 'f16', 'f32')."""
    if dtype == "bf16":
        return bf16_to_f64(a)
    if dtype == "f16":
        return f16_to_f64(a)
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "f64":
        return np.asarray(a, dtype=np.float64)
    raise ValueError(dtype)


# ---------------------------------------------------------------- products
def linear(x: np.ndarray, w: np.ndarray, b: np.ndarray | None = None) -> np.ndarray:
    """y = x @ w.T (+ b) in float64; x (T, K), w (O, K), b (O,)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    T, K = x.shape
    O, K2 = w.shape
    if K != K2:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    y = np.empty((T, O), dtype=np.float64)
    if T and O:
        _load().orc_gemm_nt(T, O, K, _dp(x), K, _dp(w), K, _dp(y), O)
    if b is not None:
        y = y + np.asarray(b, dtype=np.float64)[None, :]
    return y


def matmul(X: np.ndarray, A: np.ndarray) -> np.ndarray:
    """Y = X @ A in float64; X (M, K), A (K, N)."""
    X = np.ascontiguousarray(X, dtype=np.float64)
    A = np.ascontiguousarray(A, dtype=np.float64)
    M, K = X.shape
    K2, N = A.shape
    if K != K2:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    Y = np.empty((M, N), dtype=np.float64)
    if M and N:
        _load().orc_gemm_nn(M, N, K, _dp(X), K, _dp(A), N, _dp(Y), N)
    return Y


# ---------------------------------------------------------------- slicing
def shard(w: np.ndarray, axis: int, segments: int, n: int) -> list[np.ndarray]:
    """``_shard`` of one parameter: the N rank slices, byte-exact.

    Split ``w`` along ``axis`` into ``segments`` equal parts, split every part
    into ``n`` equal parts, and give rank ``r`` the concatenation (in segment
    order) of part ``r`` of each segment.  Equal splits need the axis length
    to be a multiple of ``segments * n``; otherwise this raises ValueError.
    """
    w = np.asarray(w)
    ax = axis % w.ndim
    if segments < 1 or n < 1:
        raise ValueError("segments and n must be >= 1")
    if w.shape[ax] % (segments * n):
        raise ValueError("Cannot shard the output of size %d across %d devices."
                         % (w.shape[ax], segments * n))
    segs = np.split(w, segments, axis=ax)
    out = []
    for r in range(n):
        pieces = [np.split(seg, n, axis=ax)[r] for seg in segs]
        out.append(np.ascontiguousarray(np.concatenate(pieces, axis=ax)))
    return out


def check_all_to_sharded_dims(output_dims: int, n: int) -> None:
    """Constructor check of the column-parallel layer (MLX page, section 2.1)."""
    if output_dims % n != 0:
        raise ValueError("Cannot shard the output of size %d across %d devices."
                         % (output_dims, n))


# ---------------------------------------------------------------- layers
def all_to_sharded(x, w_shards, b_shards=None):
    """Column-parallel linear: rank r computes x @ W_r.T + b_r, nothing summed."""
    out = []
    for r, w in enumerate(w_shards):
        b = None if b_shards is None else b_shards[r]
        out.append(linear(x, w, b))
    return out


def sharded_to_all(x_shards, w_shards, b=None):
    """Row-parallel linear: partials x_r @ W_r.T summed over r = 0..N-1 in
    ascending order, then the bias added once."""
    total = None
    for x, w in zip(x_shards, w_shards):
        p = linear(x, w)
        total = p if total is None else total + p
    if b is not None:
        total = total + np.asarray(b, dtype=np.float64)[None, :]
    return total


# ---------------------------------------------------------------- backward
def all_to_sharded_dx(dy_shards, w_shards):
    """Input gradient of the column-parallel layer.  Its forward passes x
    through sum_gradients (MLX guide, gradient aggregation in backward:
    identity forward, all_sum of the gradient backward), so the ranks' local
    gradients dy_r @ W_r are summed, r ascending."""
    total = None
    for dy, w in zip(dy_shards, w_shards):
        p = matmul(dy, w)
        total = p if total is None else total + p
    return total


def sharded_to_all_dx(dy, w_shards):
    """Input gradient of the row-parallel layer: dy is replicated (the forward
    ended in all_sum), so rank r's slice is dy @ W_r, no communication."""
    return [matmul(dy, w) for w in w_shards]


def sharded_dw(dy_list, x_list):
    """Weight gradients: dW_r = dy_r^T @ x_r (column-parallel: x_r = x;
    row-parallel: dy_r = dy)."""
    return [matmul(np.ascontiguousarray(np.asarray(dy, dtype=np.float64).T), x)
            for dy, x in zip(dy_list, x_list)]


def bias_grad(dy_groups):
    """Bias gradient: the bias is added to every row, so its gradient is the
    sum over rows of the output gradient, over each group's matrices in order."""
    out = []
    for group in dy_groups:
        acc = None
        for d in group:
            cs = np.asarray(d, dtype=np.float64).sum(axis=0)
            acc = cs if acc is None else acc + cs
        out.append(acc)
    return out


# ---------------------------------------------------------------- gated FFN
def silu(a):
    """SiLU, a * sigmoid(a) = a / (1 + exp(-a)), in float64 (the gate of the
    Llama FFN the MLX guide shards, sections 5.2-5.4).  For a below about -709
    exp(-a) overflows to infinity and the quotient is -0, the limit."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def gated_all_to_sharded(x, w1_shards, w3_shards, b1_shards=None, b3_shards=None):
    """Gate (w1) and up (w3) projections, both column-parallel on the same
    input (MLX guide, section 5.2), combined elementwise on each rank's shard
    (section 5.3): h_r = silu(x @ W1_r.T + b1_r) * (x @ W3_r.T + b3_r)."""
    out = []
    for r, (w1, w3) in enumerate(zip(w1_shards, w3_shards)):
        g = linear(x, w1, None if b1_shards is None else b1_shards[r])
        u = linear(x, w3, None if b3_shards is None else b3_shards[r])
        out.append(silu(g) * u)
    return out


# ---------------------------------------------------------------- collectives
def all_gather(shards, axis: int):
    """AllGather over the group ("sharded matrices" notes, primitive table):
    every rank receives all N shards joined in rank order along ``axis``."""
    return np.concatenate([np.asarray(s, dtype=np.float64) for s in shards], axis=axis)


def reduce_scatter(partials, axis: int):
    """ReduceScatter over the group (same table): the N partial results are
    added in rank order 0..N-1, the sum is cut along ``axis`` into N equal
    contiguous blocks, and rank c receives block c."""
    n = len(partials)
    total = None
    for p in partials:
        p = np.asarray(p, dtype=np.float64)
        total = p if total is None else total + p
    length = total.shape[axis]
    if length % n:
        raise ValueError("cannot scatter an axis of %d over %d ranks" % (length, n))
    w = length // n
    return [np.take(total, np.arange(c * w, (c + 1) * w), axis=axis) for c in range(n)]


def sharded_to_sharded(x_shards, w_shards, b=None):
    """Row-parallel linear whose partial products are reduce-scattered over
    the output columns instead of all-reduced ("sharded matrices" notes, case
    3, second option): rank c receives column block c of sum_r x_r @ W_r.T
    and adds block c of the layer's bias once, after the sum."""
    n = len(x_shards)
    partials = [linear(x, w) for x, w in zip(x_shards, w_shards)]
    ys = reduce_scatter(partials, axis=1)
    if b is not None:
        b = np.asarray(b, dtype=np.float64)
        w = b.shape[0] // n
        ys = [y + b[None, c * w:(c + 1) * w] for c, y in enumerate(ys)]
    return ys


def gathered_to_sharded(x_shards, w_shards, b_shards=None):
    """Case 2 of the same notes, standard route: all-gather the input, which
    is sharded along its contraction axis (columns), then every rank's local
    column-parallel linear x @ W_r.T + b_r."""
    return all_to_sharded(all_gather(x_shards, axis=1), w_shards, b_shards)


def summa(X_blocks, A_blocks, q: int):
    """SUMMA on a q x q grid: Y_ij = sum_{t=0}^{q-1} X_it A_tj, t ascending.

    Blocks are indexed i*q + j.  Returns the q*q output blocks.
    """
    if len(X_blocks) != q * q or len(A_blocks) != q * q:
        raise ValueError("need q*q blocks of each operand")
    Y = []
    for i in range(q):
        for j in range(q):
            acc = None
            for t in range(q):
                p = matmul(X_blocks[i * q + t], A_blocks[t * q + j])
                acc = p if acc is None else acc + p
            Y.append(acc)
    return Y


def summa_linear(X_blocks, A_blocks, b_blocks, q: int):
    """Linear2D forward: SUMMA's Y_ij plus column block j's bias (the piece
    add_bias_2d gathers along the column group), added after the q steps."""
    Y = summa(X_blocks, A_blocks, q)
    if b_blocks is None:
        return Y
    return [Y[i * q + j] + np.asarray(b_blocks[j], dtype=np.float64)[None, :]
            for i in range(q) for j in range(q)]


def summa_abt(A_blocks, B_blocks, q: int):
    """Matmul_ABT_2D (the SUMMA page, backward): C = A B^T on the grid,
    C_ij = sum_{t=0}^{q-1} A_it B_jt^T, t ascending."""
    C = []
    for i in range(q):
        for j in range(q):
            acc = None
            for t in range(q):
                p = matmul(A_blocks[i * q + t], np.ascontiguousarray(np.asarray(B_blocks[j * q + t]).T))
                acc = p if acc is None else acc + p
            C.append(acc)
    return C


def summa_atb(A_blocks, B_blocks, q: int):
    """Matmul_ATB_2D (same page): C = A^T B on the grid,
    C_ij = sum_{t=0}^{q-1} A_ti^T B_tj, t ascending."""
    C = []
    for i in range(q):
        for j in range(q):
            acc = None
            for t in range(q):
                p = matmul(np.ascontiguousarray(np.asarray(A_blocks[t * q + i]).T), B_blocks[t * q + j])
                acc = p if acc is None else acc + p
            C.append(acc)
    return C


def blocks(M: np.ndarray, q: int) -> list[np.ndarray]:
    """Split a matrix into its q x q grid of equal blocks, index i*q + j."""
    R, C = M.shape
    if R % q or C % q:
        raise ValueError("matrix %dx%d not divisible by q=%d" % (R, C, q))
    r, c = R // q, C // q
    return [np.ascontiguousarray(M[i * r:(i + 1) * r, j * c:(j + 1) * c])
            for i in range(q) for j in range(q)]


def unblock(B: list[np.ndarray], q: int) -> np.ndarray:
    """Inverse of ``blocks``."""
    return np.concatenate([np.concatenate(B[i * q:(i + 1) * q], axis=1) for i in range(q)], axis=0)


# ---------------------------------------------------------------- 4-bit affine
def unpack_codes(packed: np.ndarray, k: int) -> np.ndarray:
    """uint32 words (8 codes each, element k at bits 4*(k mod 8)) -> codes."""
    packed = np.asarray(packed, dtype=np.uint32)
    rows = packed.shape[0]
    out = np.empty((rows, packed.shape[1] * 8), dtype=np.uint8)
    for e in range(8):
        out[:, e::8] = (packed >> np.uint32(4 * e)) & np.uint32(0xF)
    return out[:, :k]


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """codes (rows, K) in 0..15 with K % 8 == 0 -> uint32 (rows, K/8)."""
    codes = np.asarray(codes, dtype=np.uint32)
    rows, k = codes.shape
    if k % 8:
        raise ValueError("K must be a multiple of 8")
    words = np.zeros((rows, k // 8), dtype=np.uint32)
    for e in range(8):
        words |= codes[:, e::8] << np.uint32(4 * e)
    return words


def quantize_affine4(w: np.ndarray, group_size: int = 64):
    """Affine 4-bit quantization of a float32 weight (rows, K), per row in
    groups of ``group_size`` consecutive input elements.

    Per group: s = (max - min) / 15 in float32 (1 if that is 0), b = min;
    both stored as float16 (round to nearest even; s = 1 if it rounds to 0).
    Codes: q = clamp(round_half_even((w - b) / s), 0, 15) with w, s, b as
    float32 and each operation rounded to float32.
    Returns (packed uint32 (rows, K/8), scales f16 (rows, K/g), biases f16).
    """
    w = np.asarray(w, dtype=np.float32)
    rows, k = w.shape
    if k % group_size:
        raise ValueError("K must be a multiple of group_size")
    g = w.reshape(rows, k // group_size, group_size)
    mn = g.min(axis=2)
    mx = g.max(axis=2)
    s = ((mx - mn) / np.float32(15.0)).astype(np.float32)
    s = np.where(s == 0, np.float32(1.0), s)
    s16 = s.astype(np.float16)
    s16 = np.where(s16 == 0, np.float16(1.0), s16)
    b16 = mn.astype(np.float16)
    d = (g - b16.astype(np.float32)[:, :, None]).astype(np.float32)
    v = (d / s16.astype(np.float32)[:, :, None]).astype(np.float32)
    q = np.clip(np.rint(v), 0, 15).astype(np.uint32).reshape(rows, k)
    return pack_codes(q), s16, b16


def dequant_affine4(packed: np.ndarray, scales: np.ndarray, biases: np.ndarray,
                    group_size: int = 64) -> np.ndarray:
    """W_hat[o, k] = s[o, k // g] * q[o, k] + b[o, k // g] in float64."""
    s = f16_to_f64(scales)
    b = f16_to_f64(biases)
    k = s.shape[1] * group_size
    q = unpack_codes(packed, k).astype(np.float64)
    gi = np.arange(k) // group_size
    return s[:, gi] * q + b[:, gi]


def q4_all_to_sharded(x, packed_shards, scale_shards, bias_q_shards, group_size=64, b_shards=None):
    """Quantized column-parallel linear: rank r computes x @ W_hat_r.T (+ b_r)."""
    w = [dequant_affine4(p, s, b, group_size)
         for p, s, b in zip(packed_shards, scale_shards, bias_q_shards)]
    return all_to_sharded(x, w, b_shards)


def q4_sharded_to_all(x_shards, packed_shards, scale_shards, bias_q_shards, group_size=64, b=None):
    """Quantized row-parallel linear: sum_r x_r @ W_hat_r.T in rank order (+ b)."""
    w = [dequant_affine4(p, s, bq, group_size)
         for p, s, bq in zip(packed_shards, scale_shards, bias_q_shards)]
    return sharded_to_all(x_shards, w, b)


# ---------------------------------------------------------------- mxfp8
# The MLX guide (section 2.3, and the distributed tests of section 4) names a
# second quantization mode, "mxfp8", passed through sharding like the affine
# one and with no per-group biases.  Its format is the microscaling FP8 of the
# OCP MX specification: blocks of 32 consecutive input elements share one
# power-of-two scale stored as an 8-bit exponent (E8M0, value 2^(s - 127)),
# and each element is an FP8 E4M3 number (1 sign, 4 exponent bits with bias 7,
# 3 mantissa bits; exponent field 0 is subnormal; 0x7F / 0xFF are NaN, so the
# largest finite magnitude is 448).  The quantized matmul keeps x in its own
# type and multiplies by the dequantized weight.
MX_GROUP = 32
MX_EMAX_ELEM = 8  # exponent of the largest E4M3 normal (448 = 1.75 * 2^8)


def e4m3_value(byte: int) -> float:
    """Value of one E4M3 code from the format's definition (NaN for 0x7F, 0xFF)."""
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9          # subnormal: m/8 * 2^(1-7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def e4m3_from_f64(v: np.ndarray) -> np.ndarray:
    """Round to the nearest finite E4M3 code, ties to the even code (even
    mantissa), magnitudes above 448 saturating to 448, the sign kept (a
    negative value that rounds to zero gives -0, 0x80).  Written as a search
    over the 127 non-negative finite codes 0x00..0x7E (their values ascend
    with the code), so it follows the definition directly."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.minimum(np.abs(v), 448.0)
    pos = E4M3_TABLE[:0x7F]                                  # codes 0..126, ascending
    hi = np.searchsorted(pos, mag, side="left")             # first code with value >= mag
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - pos[lo]
    d_hi = pos[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    # the sign is kept, also when the magnitude rounds to zero (-0 is 0x80)
    sign = np.signbit(v).astype(np.uint8) << 7
    return (code | sign).astype(np.uint8)


def quantize_mxfp8(w: np.ndarray):
    """MXFP8 quantization of a float32 weight (rows, K), per row in blocks of
    32 consecutive input elements (OCP MX conversion):
      X = floor(log2(max |w| of the block)) - 8, clamped to [-127, 127]
      (X = -127 for an all-zero block); scale byte = X + 127;
      code = E4M3 round-to-nearest-even, saturating, of w / 2^X.
    Returns (codes uint8 (rows, K), scales uint8 (rows, K/32))."""
    w = np.asarray(w, dtype=np.float32)
    rows, k = w.shape
    if k % MX_GROUP:
        raise ValueError("K must be a multiple of 32")
    g = w.reshape(rows, k // MX_GROUP, MX_GROUP).astype(np.float64)
    amax = np.abs(g).max(axis=2)
    _, ex = np.frexp(amax)                 # amax = f * 2^ex, f in [0.5, 1)
    X = np.where(amax > 0, ex - 1 - MX_EMAX_ELEM, -127)
    X = np.clip(X, -127, 127)
    codes = e4m3_from_f64(g / np.ldexp(1.0, X)[:, :, None])
    return codes.reshape(rows, k), (X + 127).astype(np.uint8)


def dequant_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W_hat[o, k] = e4m3(code[o, k]) * 2^(scale[o, k // 32] - 127) in float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    k = codes.shape[1]
    gi = np.arange(k) // MX_GROUP
    return E4M3_TABLE[codes] * np.ldexp(1.0, scales.astype(np.int64) - 127)[:, gi]


def mx_all_to_sharded(x, code_shards, scale_shards, b_shards=None):
    """MXFP8 column-parallel linear: rank r computes x @ W_hat_r.T (+ b_r)."""
    return all_to_sharded(x, [dequant_mxfp8(c, s) for c, s in zip(code_shards, scale_shards)], b_shards)


def mx_sharded_to_all(x_shards, code_shards, scale_shards, b=None):
    """MXFP8 row-parallel linear: sum_r x_r @ W_hat_r.T in rank order (+ b)."""
    return sharded_to_all(x_shards, [dequant_mxfp8(c, s) for c, s in zip(code_shards, scale_shards)], b)
