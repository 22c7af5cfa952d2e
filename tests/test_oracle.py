"""Pins for the CPU oracle, against facts that do not come from the oracle.

Each ``check_*`` helper takes the oracle routine under test as an argument so
that ``test_oracle_mutations.py`` can hand it a deliberately broken copy and
show that the pin notices.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from sharded_gemm_gb300 import synth

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ products
def check_linear_vs_numpy(linear):
    for (T, K, O) in [(1, 1, 1), (3, 5, 7), (17, 64, 33), (64, 130, 96)]:
        x = RNG.standard_normal((T, K))
        w = RNG.standard_normal((O, K))
        b = RNG.standard_normal(O)
        ref = np.matmul(x, w.T) + b
        got = linear(x, w, b)
        assert got.shape == (T, O)
        err = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
        assert err <= 1e-12, err


def check_matmul_vs_numpy(matmul):
    for (M, K, N) in [(1, 1, 1), (5, 3, 7), (33, 64, 17), (40, 96, 72)]:
        X = RNG.standard_normal((M, K))
        A = RNG.standard_normal((K, N))
        ref = np.matmul(X, A)
        got = matmul(X, A)
        assert got.shape == (M, N)
        assert np.linalg.norm(got - ref) <= 1e-12 * np.linalg.norm(ref)


def test_linear_vs_numpy():
    check_linear_vs_numpy(oracle.linear)


def test_matmul_vs_numpy():
    check_matmul_vs_numpy(oracle.matmul)


def test_linear_small_integers_exact():
    # Integer-valued operands: every product and partial sum is exact in fp64,
    # so the result must equal the integer dot products bit for bit.
    x = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.float64)
    w = np.array([[1, 0, -1], [2, 1, 0]], dtype=np.float64)
    b = np.array([10, -10], dtype=np.float64)
    y = oracle.linear(x, w, b)
    assert np.array_equal(y, np.array([[1 - 3 + 10, 2 + 2 - 10], [4 - 6 + 10, 8 + 5 - 10]]))


# ------------------------------------------------------------------ slicing
def closed_form_rows(O, S, N, r):
    """Global row of local row i of shard r: (i // w)*(O/S) + r*w + (i % w)."""
    w = O // (S * N)
    return [(i // w) * (O // S) + r * w + (i % w) for i in range(O // N)]


def check_shard_closed_form(shard):
    for (O, C, S, N) in [(8, 3, 1, 2), (12, 2, 3, 2), (24, 5, 3, 4), (16, 1, 2, 8), (6, 4, 1, 1)]:
        w = RNG.integers(0, 2**16, size=(O, C), dtype=np.uint16)
        parts = shard(w, 0, S, N)
        assert len(parts) == N
        for r in range(N):
            assert parts[r].dtype == w.dtype
            assert np.array_equal(parts[r], w[closed_form_rows(O, S, N, r)])
        # axis -1: the same rule on columns
        wt = np.ascontiguousarray(w.T)
        parts = shard(wt, -1, S, N)
        for r in range(N):
            assert np.array_equal(parts[r], wt[:, closed_form_rows(O, S, N, r)])


def test_shard_closed_form():
    check_shard_closed_form(oracle.shard)


def test_shard_fused_qkv_by_hand():
    # A fused [Q; K; V] weight with 4 rows each, N = 2: rank 0 holds rows
    # 0-1 of Q, K and V; rank 1 rows 2-3 of each (segments=3 slicing).
    w = np.arange(12, dtype=np.uint32)[:, None] * np.uint32(10) + np.arange(2, dtype=np.uint32)
    p = oracle.shard(w, 0, 3, 2)
    assert p[0][:, 0].tolist() == [0, 10, 40, 50, 80, 90]
    assert p[1][:, 0].tolist() == [20, 30, 60, 70, 100, 110]


def test_shard_concat_identity():
    for dt in (np.uint16, np.uint32, np.float32, np.float16):
        w = RNG.standard_normal((24, 16)).astype(dt) if dt in (np.float32, np.float16) else \
            RNG.integers(0, 1000, size=(24, 16)).astype(dt)
        for N in (1, 2, 4, 8):
            assert np.array_equal(np.concatenate(oracle.shard(w, 0, 1, N), axis=0), w)
            assert np.array_equal(np.concatenate(oracle.shard(w, 1, 1, N), axis=1), w)


def test_shard_bruteforce_tiny():
    # Every element lands in exactly one shard; within a shard, order follows
    # (segment, position) of the original.
    for (L, S, N) in [(4, 1, 2), (6, 3, 2), (12, 2, 3), (8, 2, 2)]:
        w = np.arange(L, dtype=np.int64)
        parts = oracle.shard(w, 0, S, N)
        seen = sorted(v for p in parts for v in p.tolist())
        assert seen == list(range(L))
        seg = L // S
        for r, p in enumerate(parts):
            for v in p.tolist():
                assert (v % seg) // (seg // N) == r
            assert p.tolist() == sorted(p.tolist())


def test_shard_not_divisible_raises():
    with pytest.raises(ValueError):
        oracle.shard(np.zeros((10, 4)), 0, 3, 2)
    with pytest.raises(ValueError):
        oracle.shard(np.zeros((4, 10)), -1, 1, 4)


def test_worked_example_shapes(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example.json")))
    N = g["N"]
    cfg = synth.worked()
    x = oracle.widen(cfg["x"], "f32")
    assert list(x.shape) == g["x_shape"]
    w1 = oracle.shard(cfg["w1"], 0, 1, N)
    b1 = oracle.shard(cfg["b1"], 0, 1, N)
    assert all(list(p.shape) == g["all_to_sharded"]["weight_slice_shape"] for p in w1)
    y1 = oracle.all_to_sharded(x, [oracle.widen(p, "f32") for p in w1], [oracle.widen(p, "f32") for p in b1])
    assert all(list(y.shape) == g["all_to_sharded"]["per_rank_output_shape"] for y in y1)
    w2 = oracle.shard(cfg["w2"], -1, 1, N)
    assert all(list(p.shape) == g["sharded_to_all"]["weight_slice_shape"] for p in w2)
    partials = [oracle.linear(y1[r], oracle.widen(w2[r], "f32")) for r in range(N)]
    assert all(list(p.shape) == g["sharded_to_all"]["per_rank_partial_shape"] for p in partials)
    y2 = oracle.sharded_to_all(y1, [oracle.widen(p, "f32") for p in w2], oracle.widen(cfg["b2"], "f32"))
    assert list(y2.shape) == g["sharded_to_all"]["output_shape"]
    # and the chain equals the unsharded two-layer model
    full = oracle.linear(oracle.linear(x, oracle.widen(cfg["w1"], "f32"), oracle.widen(cfg["b1"], "f32")),
                         oracle.widen(cfg["w2"], "f32"), oracle.widen(cfg["b2"], "f32"))
    assert np.allclose(y2, full, rtol=0, atol=1e-14)


def test_divisibility_message(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example.json")))["divisibility_error"]
    with pytest.raises(ValueError) as e:
        oracle.check_all_to_sharded_dims(g["output_dims"], g["N"])
    assert str(e.value) == g["message"]
    oracle.check_all_to_sharded_dims(4096, 8)


# ------------------------------------------------------------------ invariants
def check_col_invariant(all_to_sharded, shard):
    for (T, K, O, S, N) in [(5, 8, 12, 1, 2), (3, 16, 24, 3, 4), (7, 9, 16, 1, 8)]:
        x = RNG.standard_normal((T, K))
        w = RNG.standard_normal((O, K))
        b = RNG.standard_normal(O)
        full = np.matmul(x, w.T) + b
        ys = all_to_sharded(x, shard(w, 0, S, N), shard(b, 0, S, N))
        for r in range(N):
            ref = full[:, closed_form_rows(O, S, N, r)]
            assert np.abs(ys[r] - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


def check_row_invariant(sharded_to_all, shard):
    for (T, K, O, N) in [(5, 8, 6, 2), (3, 64, 10, 4), (9, 24, 7, 8), (2, 3, 2, 1)]:
        x = RNG.standard_normal((T, K))
        w = RNG.standard_normal((O, K))
        b = RNG.standard_normal(O)
        full = np.matmul(x, w.T) + b
        y = sharded_to_all(shard(x, -1, 1, N), shard(w, -1, 1, N), b)
        assert np.abs(y - full).max() <= 1e-12 * (1 + np.abs(full).max())


def test_col_equals_unsharded():
    check_col_invariant(oracle.all_to_sharded, oracle.shard)


def test_row_equals_unsharded():
    check_row_invariant(oracle.sharded_to_all, oracle.shard)


def test_row_bias_added_once_after_sum():
    # With zero inputs the partials vanish; the output must be exactly b
    # (an implementation adding b per shard would give N*b).
    N = 4
    x = np.zeros((3, 8))
    w = RNG.standard_normal((5, 8))
    b = RNG.standard_normal(5)
    y = oracle.sharded_to_all(oracle.shard(x, -1, 1, N), oracle.shard(w, -1, 1, N), b)
    assert np.array_equal(y, np.broadcast_to(b, (3, 5)))


def test_pair_equals_unsharded_mlp_small():
    # Column -> row pair with the intermediate kept sharded (MLX page section 4).
    T, D, F, N = 6, 16, 24, 4
    x = RNG.standard_normal((T, D))
    w1, b1 = RNG.standard_normal((F, D)), RNG.standard_normal(F)
    w2, b2 = RNG.standard_normal((D, F)), RNG.standard_normal(D)
    mid = oracle.all_to_sharded(x, oracle.shard(w1, 0, 1, N), oracle.shard(b1, 0, 1, N))
    y = oracle.sharded_to_all(mid, oracle.shard(w2, -1, 1, N), b2)
    ref = np.matmul(np.matmul(x, w1.T) + b1, w2.T) + b2
    assert np.abs(y - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


# ------------------------------------------------------------------ backward
def _ints(shape, lo=-4, hi=5):
    return RNG.integers(lo, hi, shape).astype(np.float64)


def _dot(a, b):
    return float(np.sum(np.asarray(a) * np.asarray(b)))


def check_col_adjoint(all_to_sharded_dx, sharded_dw, shard):
    # The column-parallel forward y_r = x W_r^T is linear in x and in W, so
    # its gradients are the adjoints:  sum_r <dy_r, x W_r^T> = <dx, x> =
    # sum_r <dW_r, W_r>.  Small integers keep all three sums exact.
    for (T, K, O, N) in [(3, 5, 8, 2), (4, 6, 12, 4), (2, 3, 8, 8), (5, 4, 3, 1)]:
        x, w = _ints((T, K)), _ints((O, K))
        ws = shard(w, 0, 1, N)
        dys = [_ints((T, O // N)) for _ in range(N)]
        lhs = sum(_dot(dy, x @ wr.T) for dy, wr in zip(dys, ws))
        dx = all_to_sharded_dx(dys, ws)
        assert dx.shape == (T, K)
        assert _dot(dx, x) == lhs
        dws = sharded_dw(dys, [x] * N)
        assert [d.shape for d in dws] == [wr.shape for wr in ws]
        assert sum(_dot(d, wr) for d, wr in zip(dws, ws)) == lhs


def check_row_adjoint(sharded_to_all_dx, sharded_dw, shard):
    # Row-parallel forward y = sum_r x_r W_r^T:
    # <dy, y> = sum_r <dx_r, x_r> = sum_r <dW_r, W_r>.
    for (T, K, O, N) in [(3, 8, 5, 2), (4, 12, 6, 4), (2, 8, 3, 8), (5, 3, 4, 1)]:
        x, w = _ints((T, K)), _ints((O, K))
        xs, ws = shard(x, -1, 1, N), shard(w, -1, 1, N)
        dy = _ints((T, O))
        lhs = _dot(dy, sum(xr @ wr.T for xr, wr in zip(xs, ws)))
        dxs = sharded_to_all_dx(dy, ws)
        assert [d.shape for d in dxs] == [xr.shape for xr in xs]
        assert sum(_dot(d, xr) for d, xr in zip(dxs, xs)) == lhs
        dws = sharded_dw([dy] * N, xs)
        assert sum(_dot(d, wr) for d, wr in zip(dws, ws)) == lhs


def check_bias_grad_closed_form(bias_grad):
    # dy[t, c] = t + 2c: the column sums are T(T-1)/2 + 2cT; two matrices in a
    # group add; and <dy, 1 b^T> = <db, b> for the bias's own adjoint.
    T, C = 7, 5
    t, c = np.meshgrid(np.arange(T), np.arange(C), indexing="ij")
    dy = (t + 2 * c).astype(np.float64)
    got = bias_grad([[dy], [dy, 3 * dy]])
    expect = T * (T - 1) / 2 + 2 * np.arange(C) * T
    assert np.array_equal(got[0], expect)
    assert np.array_equal(got[1], 4 * expect)
    b = _ints((C,))
    d2 = _ints((T, C))
    assert _dot(d2, np.broadcast_to(b, (T, C))) == _dot(bias_grad([[d2]])[0], b)


def check_summa_backward(summa_abt, summa_atb):
    # Block identities of Matmul_ABT_2D / Matmul_ATB_2D at q = 2, written out.
    A = RNG.standard_normal((8, 6))
    B = RNG.standard_normal((10, 6))
    Ab, Bb = oracle.blocks(A, 2), oracle.blocks(B, 2)
    A00, A01, A10, A11 = Ab
    B00, B01, B10, B11 = Bb
    expect = [A00 @ B00.T + A01 @ B01.T, A00 @ B10.T + A01 @ B11.T,
              A10 @ B00.T + A11 @ B01.T, A10 @ B10.T + A11 @ B11.T]
    for e, g in zip(expect, summa_abt(Ab, Bb, 2)):
        assert g.shape == e.shape and np.abs(g - e).max() <= 1e-12 * (1 + np.abs(e).max())
    P = RNG.standard_normal((6, 8))
    Q = RNG.standard_normal((6, 10))
    Pb, Qb = oracle.blocks(P, 2), oracle.blocks(Q, 2)
    P00, P01, P10, P11 = Pb
    Q00, Q01, Q10, Q11 = Qb
    expect = [P00.T @ Q00 + P10.T @ Q10, P00.T @ Q01 + P10.T @ Q11,
              P01.T @ Q00 + P11.T @ Q10, P01.T @ Q01 + P11.T @ Q11]
    for e, g in zip(expect, summa_atb(Pb, Qb, 2)):
        assert g.shape == e.shape and np.abs(g - e).max() <= 1e-12 * (1 + np.abs(e).max())
    # q = 4 against numpy's transposed products
    X = RNG.standard_normal((16, 12))
    Y = RNG.standard_normal((8, 12))
    got = oracle.unblock(summa_abt(oracle.blocks(X, 4), oracle.blocks(Y, 4), 4), 4)
    assert np.abs(got - X @ Y.T).max() <= 1e-12 * (1 + np.abs(X @ Y.T).max())
    Z = RNG.standard_normal((12, 8))
    got = oracle.unblock(summa_atb(oracle.blocks(X.T.copy(), 4), oracle.blocks(Z, 4), 4), 4)
    assert np.abs(got - X @ Z).max() <= 1e-12 * (1 + np.abs(X @ Z).max())


def test_col_gradients_are_adjoints():
    check_col_adjoint(oracle.all_to_sharded_dx, oracle.sharded_dw, oracle.shard)


def test_row_gradients_are_adjoints():
    check_row_adjoint(oracle.sharded_to_all_dx, oracle.sharded_dw, oracle.shard)


def test_col_dx_equals_unsharded():
    # the all-summed input gradient is the unsharded dy @ W
    T, K, O, N = 5, 16, 12, 4
    dy, w = RNG.standard_normal((T, O)), RNG.standard_normal((O, K))
    dx = oracle.all_to_sharded_dx(oracle.shard(dy, -1, 1, N), oracle.shard(w, 0, 1, N))
    assert np.abs(dx - dy @ w).max() <= 1e-12 * (1 + np.abs(dy @ w).max())


def test_bias_grad_closed_form():
    check_bias_grad_closed_form(oracle.bias_grad)


def test_summa_backward_identities():
    check_summa_backward(oracle.summa_abt, oracle.summa_atb)


def test_summa_backward_adjoint():
    # Y = X A on the grid: <dY, X A> = <dY A^T, X> = <X^T dY, A>, i.e.
    # dX = ABT(dY, A) and dA = ATB(X, dY).
    q = 2
    X, A, dY = _ints((6, 4)), _ints((4, 8)), _ints((6, 8))
    Xb, Ab, dYb = oracle.blocks(X, q), oracle.blocks(A, q), oracle.blocks(dY, q)
    lhs = _dot(dY, X @ A)
    dX = oracle.unblock(oracle.summa_abt(dYb, Ab, q), q)
    dA = oracle.unblock(oracle.summa_atb(Xb, dYb, q), q)
    assert _dot(dX, X) == lhs
    assert _dot(dA, A) == lhs
    assert oracle.unblock(oracle.summa(Xb, Ab, q), q).shape == dY.shape


def test_summa_linear_bias_per_column_block():
    # X = 0: every block is exactly its column block's bias
    q = 2
    Xb = oracle.blocks(np.zeros((4, 6)), q)
    Ab = oracle.blocks(RNG.standard_normal((6, 8)), q)
    b = [RNG.standard_normal(4) for _ in range(q)]
    Y = oracle.summa_linear(Xb, Ab, b, q)
    for i in range(q):
        for j in range(q):
            assert np.array_equal(Y[i * q + j], np.broadcast_to(b[j], (2, 4)))


# ------------------------------------------------------------------ gated FFN
def check_silu_closed_forms(silu):
    # sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4 in closed form.
    l3 = math.log(3.0)
    assert silu(np.array([0.0]))[0] == 0.0
    assert abs(silu(np.array([l3]))[0] - 0.75 * l3) <= 1e-15
    assert abs(silu(np.array([-l3]))[0] + 0.25 * l3) <= 1e-15
    # silu(a) - silu(-a) = a (since sigmoid(a) + sigmoid(-a) = 1)
    a = RNG.standard_normal(64) * 6
    assert np.abs(silu(a) - silu(-a) - a).max() <= 1e-13
    # against the tanh form of the logistic function, sigmoid(a) = (1 + tanh(a/2)) / 2
    b = np.linspace(-30, 30, 121)
    assert np.abs(silu(b) - b * 0.5 * (1 + np.tanh(b / 2))).max() <= 1e-13
    # limits
    assert silu(np.array([-1000.0]))[0] == 0.0
    assert silu(np.array([1000.0]))[0] == 1000.0


def check_gated_invariant(gated, shard):
    # Rank r's gated output equals columns r*F/N.. of the unsharded
    # silu(x W1^T + b1) * (x W3^T + b3), the SiLU written with tanh.
    def silu_t(a):
        return a * 0.5 * (1 + np.tanh(a / 2))
    for (T, K, F, N) in [(5, 8, 12, 2), (3, 64, 24, 4), (7, 9, 16, 8), (2, 3, 2, 1)]:
        x = RNG.standard_normal((T, K))
        w1, w3 = RNG.standard_normal((F, K)), RNG.standard_normal((F, K))
        b1, b3 = RNG.standard_normal(F), RNG.standard_normal(F)
        full = silu_t(np.matmul(x, w1.T) + b1) * (np.matmul(x, w3.T) + b3)
        hs = gated(x, shard(w1, 0, 1, N), shard(w3, 0, 1, N), shard(b1, 0, 1, N), shard(b3, 0, 1, N))
        Fn = F // N
        assert len(hs) == N
        for r in range(N):
            ref = full[:, r * Fn:(r + 1) * Fn]
            assert hs[r].shape == ref.shape
            assert np.abs(hs[r] - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


def test_silu_closed_forms():
    check_silu_closed_forms(oracle.silu)


def test_gated_equals_unsharded():
    check_gated_invariant(oracle.gated_all_to_sharded, oracle.shard)


def test_gated_unit_up_gives_activation():
    # W3 = 0 and b3 = 1: the up projection is one everywhere and the output
    # is the activated gate alone.
    x = RNG.standard_normal((4, 16))
    w1 = RNG.standard_normal((8, 16))
    hs = oracle.gated_all_to_sharded(x, oracle.shard(w1, 0, 1, 2), [np.zeros((4, 16))] * 2, None,
                                     [np.ones(4)] * 2)
    assert np.array_equal(np.concatenate(hs, axis=1), oracle.silu(oracle.linear(x, w1)))


def test_gated_ffn_then_row_parallel():
    # The guide's FFN: gate and up all-to-sharded, down (w2) sharded-to-all.
    T, D, F, N = 5, 16, 24, 4
    x = RNG.standard_normal((T, D))
    w1, w3, w2 = RNG.standard_normal((F, D)), RNG.standard_normal((F, D)), RNG.standard_normal((D, F))
    hs = oracle.gated_all_to_sharded(x, oracle.shard(w1, 0, 1, N), oracle.shard(w3, 0, 1, N))
    y = oracle.sharded_to_all(hs, oracle.shard(w2, -1, 1, N))
    a = np.matmul(x, w1.T)
    ref = np.matmul(a * 0.5 * (1 + np.tanh(a / 2)) * np.matmul(x, w3.T), w2.T)
    assert np.abs(y - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


# ------------------------------------------------------------------ collectives
def check_all_gather_closed_form(all_gather):
    # Joining the equal column (or row) blocks of a matrix in rank order must
    # give the matrix back exactly.
    x = RNG.standard_normal((6, 12))
    for N in (1, 2, 3, 4, 6, 12):
        w = 12 // N
        cols = [x[:, r * w:(r + 1) * w] for r in range(N)]
        assert np.array_equal(all_gather(cols, 1), x)
    rows = [x[r * 2:(r + 1) * 2] for r in range(3)]
    assert np.array_equal(all_gather(rows, 0), x)


def check_reduce_scatter_closed_form(reduce_scatter):
    # Partials (r + 1) * M sum to N(N+1)/2 * M; rank c must get block c.
    # Integer entries keep every sum exact.
    for (T, w, N) in [(2, 3, 2), (3, 2, 4), (1, 4, 8), (2, 5, 1)]:
        M = RNG.integers(-50, 50, (T, w * N)).astype(np.float64)
        got = reduce_scatter([(r + 1) * M for r in range(N)], 1)
        assert len(got) == N
        for c in range(N):
            assert np.array_equal(got[c], N * (N + 1) // 2 * M[:, c * w:(c + 1) * w])


def check_gather_scatter_transpose(all_gather, reduce_scatter):
    # The notes' "AllGather and ReduceScatter are transposes of each other":
    # for u = (u_0..u_{N-1}) and per-rank v_r,
    #   sum_r <AG(u), v_r> == sum_c <u_c, RS(v)_c>.
    # Integer entries make both sides exact.
    for (T, w, N) in [(3, 2, 2), (4, 5, 4), (2, 3, 8)]:
        u = [RNG.integers(-9, 10, (T, w)).astype(np.float64) for _ in range(N)]
        v = [RNG.integers(-9, 10, (T, w * N)).astype(np.float64) for _ in range(N)]
        g = all_gather(u, 1)
        lhs = sum(float(np.sum(g * vr)) for vr in v)
        rs = reduce_scatter(v, 1)
        rhs = sum(float(np.sum(uc * rc)) for uc, rc in zip(u, rs))
        assert lhs == rhs


def check_rs_invariant(sharded_to_sharded, shard):
    # Rank c's block of the reduce-scattered output equals columns
    # c*O/N.. of the unsharded x @ W.T + b.
    for (T, K, O, N) in [(5, 8, 6, 2), (3, 64, 12, 4), (9, 24, 16, 8), (2, 3, 2, 1)]:
        x = RNG.standard_normal((T, K))
        w = RNG.standard_normal((O, K))
        b = RNG.standard_normal(O)
        full = np.matmul(x, w.T) + b
        ys = sharded_to_sharded(shard(x, -1, 1, N), shard(w, -1, 1, N), b)
        On = O // N
        assert len(ys) == N
        for c in range(N):
            ref = full[:, c * On:(c + 1) * On]
            assert ys[c].shape == ref.shape
            assert np.abs(ys[c] - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


def check_rs_bias_once(sharded_to_sharded, shard):
    # Zero input: every partial vanishes and block c must be exactly bias
    # block c (adding it per partial would give N times the bias).
    N = 4
    x = np.zeros((3, 8))
    w = RNG.standard_normal((8, 8))
    b = RNG.standard_normal(8)
    ys = sharded_to_sharded(shard(x, -1, 1, N), shard(w, -1, 1, N), b)
    for c in range(N):
        assert np.array_equal(ys[c], np.broadcast_to(b[c * 2:(c + 1) * 2], (3, 2)))


def check_ag_invariant(gathered_to_sharded, shard):
    # Input sharded along its contraction axis, gathered, then rank r's
    # column-parallel product: equals columns r*O/N.. of x @ W.T + b.
    for (T, K, O, N) in [(5, 8, 6, 2), (3, 64, 12, 4), (9, 24, 16, 8), (2, 3, 2, 1)]:
        x = RNG.standard_normal((T, K))
        w = RNG.standard_normal((O, K))
        b = RNG.standard_normal(O)
        full = np.matmul(x, w.T) + b
        ys = gathered_to_sharded(shard(x, -1, 1, N), shard(w, 0, 1, N), shard(b, 0, 1, N))
        On = O // N
        for r in range(N):
            ref = full[:, r * On:(r + 1) * On]
            assert ys[r].shape == ref.shape
            assert np.abs(ys[r] - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


def test_all_gather_closed_form():
    check_all_gather_closed_form(oracle.all_gather)


def test_reduce_scatter_closed_form():
    check_reduce_scatter_closed_form(oracle.reduce_scatter)


def test_gather_scatter_transpose():
    check_gather_scatter_transpose(oracle.all_gather, oracle.reduce_scatter)


def test_reduce_scatter_not_divisible_raises():
    with pytest.raises(ValueError):
        oracle.reduce_scatter([np.zeros((2, 6))] * 4, 1)


def test_rs_equals_unsharded():
    check_rs_invariant(oracle.sharded_to_sharded, oracle.shard)


def test_rs_bias_added_once_after_sum():
    check_rs_bias_once(oracle.sharded_to_sharded, oracle.shard)


def test_rs_blocks_join_to_all_reduce():
    # Case 3's two options give the same numbers: the reduce-scattered blocks
    # side by side are the all-reduced output.
    T, K, O, N = 4, 32, 16, 4
    x = RNG.standard_normal((T, K))
    w = RNG.standard_normal((O, K))
    b = RNG.standard_normal(O)
    xs, ws = oracle.shard(x, -1, 1, N), oracle.shard(w, -1, 1, N)
    ys = oracle.sharded_to_sharded(xs, ws, b)
    y = oracle.sharded_to_all(xs, ws, b)
    assert np.abs(np.concatenate(ys, axis=1) - y).max() <= 1e-12 * (1 + np.abs(y).max())


def test_ag_equals_unsharded():
    check_ag_invariant(oracle.gathered_to_sharded, oracle.shard)


def test_ffn_one_gather_one_scatter():
    # The notes' Transformer FFN with F sharded: one all-gather in, one
    # reduce-scatter out; the output comes back sharded like the input.
    T, D, F, N = 5, 16, 24, 4
    x = RNG.standard_normal((T, D))
    w_in, b_in = RNG.standard_normal((F, D)), RNG.standard_normal(F)
    w_out, b_out = RNG.standard_normal((D, F)), RNG.standard_normal(D)
    xs = oracle.shard(x, -1, 1, N)
    mid = oracle.gathered_to_sharded(xs, oracle.shard(w_in, 0, 1, N), oracle.shard(b_in, 0, 1, N))
    out = oracle.sharded_to_sharded(mid, oracle.shard(w_out, -1, 1, N), b_out)
    ref = np.matmul(np.matmul(x, w_in.T) + b_in, w_out.T) + b_out
    assert [o.shape for o in out] == [s.shape for s in xs]
    assert np.abs(np.concatenate(out, axis=1) - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


# ------------------------------------------------------------------ SUMMA
def check_summa_q2_identity(summa):
    # Equations (1) + (2) of the SUMMA page, written out block by block.
    X = RNG.standard_normal((8, 6))
    A = RNG.standard_normal((6, 10))
    Xb, Ab = oracle.blocks(X, 2), oracle.blocks(A, 2)
    X00, X01, X10, X11 = Xb
    A00, A01, A10, A11 = Ab
    expect = [X00 @ A00 + X01 @ A10, X00 @ A01 + X01 @ A11,
              X10 @ A00 + X11 @ A10, X10 @ A01 + X11 @ A11]
    got = summa(Xb, Ab, 2)
    for e, g in zip(expect, got):
        assert g.shape == e.shape
        assert np.abs(g - e).max() <= 1e-12 * (1 + np.abs(e).max())


def test_summa_q2_identity():
    check_summa_q2_identity(oracle.summa)


def test_summa_q1_is_matmul():
    X = RNG.standard_normal((7, 5))
    A = RNG.standard_normal((5, 3))
    (Y,) = oracle.summa([X], [A], 1)
    assert np.abs(Y - X @ A).max() <= 1e-12 * np.abs(X @ A).max()


def test_summa_identity_x_gives_a_exactly():
    for q in (1, 2, 4):
        n = 8 * q
        X = np.eye(n)
        A = RNG.standard_normal((n, n))
        Y = oracle.unblock(oracle.summa(oracle.blocks(X, q), oracle.blocks(A, q), q), q)
        assert np.array_equal(Y, A)


def test_summa_vs_numpy_q4():
    X = RNG.standard_normal((16, 12))
    A = RNG.standard_normal((12, 20))
    Y = oracle.unblock(oracle.summa(oracle.blocks(X, 4), oracle.blocks(A, 4), 4), 4)
    assert np.abs(Y - X @ A).max() <= 1e-12 * np.abs(X @ A).max()


# ------------------------------------------------------------------ 4-bit affine
def test_pack_order_by_hand():
    codes = np.array([[1, 2, 3, 4, 5, 6, 7, 8, 15, 0, 0, 0, 0, 0, 0, 9]], dtype=np.uint8)
    words = oracle.pack_codes(codes)
    assert words.tolist() == [[0x87654321, 0x9000000F]]
    assert np.array_equal(oracle.unpack_codes(words, 16), codes)


def check_dequant_bruteforce(dequant):
    rows, K, g = 3, 16, 8
    packed = RNG.integers(0, 2**32, size=(rows, K // 8), dtype=np.uint64).astype(np.uint32)
    s = RNG.uniform(0.01, 0.1, size=(rows, K // g)).astype(np.float16)
    b = RNG.uniform(-0.5, 0.5, size=(rows, K // g)).astype(np.float16)
    got = dequant(packed, s, b, g)
    for o in range(rows):
        for k in range(K):
            code = (int(packed[o, k // 8]) >> (4 * (k % 8))) & 15
            want = float(s[o, k // g]) * code + float(b[o, k // g])
            assert got[o, k] == want


def test_dequant_bruteforce():
    check_dequant_bruteforce(oracle.dequant_affine4)


def test_q4_constant_codes_closed_form():
    # All codes c: y[t, o] = sum_g (s[o,g] c + b[o,g]) * sum_{k in g} x[t, k].
    T, O, K, g, c = 3, 4, 128, 64, 11
    packed = np.full((O, K // 8), 0x11111111 * c, dtype=np.uint32)
    s = RNG.uniform(0.01, 0.1, size=(O, K // g)).astype(np.float16)
    b = RNG.uniform(-0.5, 0.5, size=(O, K // g)).astype(np.float16)
    x = RNG.standard_normal((T, K))
    y = oracle.q4_all_to_sharded(x, [packed], [s], [b], g)[0]
    xs = x.reshape(T, K // g, g).sum(axis=2)
    ref = xs @ (s.astype(np.float64) * c + b.astype(np.float64)).T
    assert np.abs(y - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


def test_quantize_recovers_exact_grid():
    # w = b + s*code with s, b exact in fp16 and codes spanning 0..15:
    # the quantizer must return those codes, that s and that b.
    s, b = np.float16(0.015625), np.float16(-0.25)
    codes = RNG.integers(0, 16, size=(2, 64)).astype(np.uint8)
    codes[:, 0], codes[:, 1] = 0, 15
    w = (np.float32(b) + np.float32(s) * codes.astype(np.float32)).astype(np.float32)
    packed, sq, bq = oracle.quantize_affine4(w, 64)
    assert np.all(sq == s) and np.all(bq == b)
    assert np.array_equal(oracle.unpack_codes(packed, 64), codes)


def test_quantize_roundtrip_bound():
    w = (RNG.standard_normal((16, 256)) * 0.02).astype(np.float32)
    packed, s, b = oracle.quantize_affine4(w, 64)
    what = oracle.dequant_affine4(packed, s, b, 64)
    sg = np.repeat(s.astype(np.float64), 64, axis=1)
    mn = np.repeat(w.reshape(16, 4, 64).min(axis=2).astype(np.float64), 64, axis=1)
    bound = 0.5 * sg + np.abs(np.repeat(b.astype(np.float64), 64, axis=1) - mn) + 1e-6 * np.abs(w)
    assert np.all(np.abs(what - w) <= bound)


def test_quantize_constant_group_uses_unit_scale():
    w = np.full((1, 64), 0.5, dtype=np.float32)
    packed, s, b = oracle.quantize_affine4(w, 64)
    assert float(s[0, 0]) == 1.0 and float(b[0, 0]) == 0.5
    assert np.all(oracle.unpack_codes(packed, 64) == 0)


def test_q4_row_equals_dequant_unsharded():
    T, O, K, N, g = 2, 6, 512, 4, 64
    w = (RNG.standard_normal((O, K)) * 0.02).astype(np.float32)
    x = RNG.standard_normal((T, K))
    packed, s, b = oracle.quantize_affine4(w, g)
    what = oracle.dequant_affine4(packed, s, b, g)
    ref = x @ what.T
    y = oracle.q4_sharded_to_all(oracle.shard(x, -1, 1, N), oracle.shard(packed, -1, 1, N),
                                 oracle.shard(s, -1, 1, N), oracle.shard(b, -1, 1, N), g)
    assert np.abs(y - ref).max() <= 1e-12 * (1 + np.abs(ref).max())


# ------------------------------------------------------------------ mxfp8
def check_e4m3_table(table):
    # closed forms of the E4M3 definition (bias 7, 3 mantissa bits)
    assert table[0x38] == 1.0 and table[0x7E] == 448.0
    assert table[0x01] == 2.0 ** -9 and table[0x07] == 7 * 2.0 ** -9   # subnormals
    assert table[0x08] == 2.0 ** -6                                       # smallest normal
    assert table[0x3C] == 1.5 and table[0x44] == 3.0 and table[0x30] == 0.5
    assert np.isnan(table[0x7F]) and np.isnan(table[0xFF])
    assert table[0x00] == 0.0 and table[0x80] == 0.0 and np.signbit(table[0x80])
    pos = table[:0x7F]
    assert np.all(np.diff(pos) > 0)                                       # ascending, distinct
    assert np.array_equal(table[0x80:0xFF], -pos)                         # sign mirror


def check_e4m3_rounding(conv, table):
    pos = table[:0x7F]
    codes = np.arange(0x7F)
    assert np.array_equal(conv(pos), codes)                 # representable values are exact
    assert np.array_equal(conv(-pos[1:]), codes[1:] | 0x80)
    mid = (pos[:-1] + pos[1:]) / 2                           # ties go to the even code
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(conv(mid), even)
    eps = (pos[1:] - pos[:-1]) / 1024
    assert np.array_equal(conv(mid - eps), codes[:-1])
    assert np.array_equal(conv(mid + eps), codes[1:])
    assert list(conv(np.array([449.0, 1e9, -500.0]))) == [0x7E, 0x7E, 0xFE]  # saturation
    assert list(conv(np.array([2.0 ** -11, -2.0 ** -11]))) == [0x00, 0x80]    # to zero, sign kept


def check_mx_quantize(quantize, dequant):
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((6, 128)) * np.array([1e-3, 0.02, 1.0, 30.0, 5e3, 1e-30])[:, None]).astype(np.float32)
    w[0, :32] = 0.0                                          # all-zero block
    codes, scales = quantize(w)
    assert codes.shape == (6, 128) and scales.shape == (6, 4)
    assert scales[0, 0] == 0 and not codes[0, :32].any()
    X = scales.astype(np.int64) - 127
    amax = np.abs(w.astype(np.float64)).reshape(6, 4, 32).max(axis=2)
    nz = (amax > 0) & (X > -127)
    # the block maximum lands in E4M3's top binade: 2^(X+8) <= amax < 2^(X+9)
    assert np.all(np.ldexp(1.0, X + 8)[nz] <= amax[nz]) and np.all(amax[nz] < np.ldexp(1.0, X + 9)[nz])
    wh = dequant(codes, scales)
    err = np.abs(wh - w.astype(np.float64))
    bound = np.maximum(np.abs(w) * 2.0 ** -4, np.ldexp(1.0, X - 10).repeat(32, axis=1))
    assert np.all(err <= bound)
    # exact grid: values that are E4M3 numbers times 2^X come back unchanged
    grid = (rng.integers(0, 0x7F, (2, 64)) | (rng.integers(0, 2, (2, 64)) << 7)).astype(np.uint8)
    grid[:, ::32] = 0x78                                     # 256 = 2^8 sets X = 0 in each block
    g = oracle.E4M3_TABLE[grid].astype(np.float32) * np.float32(2.0 ** -5)
    c2, s2 = quantize(g)
    assert np.all(s2 == 127 - 5)
    assert np.array_equal(dequant(c2, s2), g.astype(np.float64))


def test_e4m3_table():
    check_e4m3_table(oracle.E4M3_TABLE)


def test_e4m3_rounding():
    check_e4m3_rounding(oracle.e4m3_from_f64, oracle.E4M3_TABLE)


def test_mx_quantize():
    check_mx_quantize(oracle.quantize_mxfp8, oracle.dequant_mxfp8)


def test_mx_dequant_bruteforce():
    codes = np.array([[0x38, 0xB8, 0x01, 0x7E] * 8], dtype=np.uint8)
    scales = np.array([[127 + 3]], dtype=np.uint8)
    expect = np.array([[8.0, -8.0, 2.0 ** -6, 448.0 * 8] * 8])
    assert np.array_equal(oracle.dequant_mxfp8(codes, scales), expect)


def test_mx_layers_equal_unsharded():
    rng = np.random.default_rng(11)
    T, K, O, N = 3, 256, 16, 4
    x = rng.standard_normal((T, K))
    w = (rng.standard_normal((O, K)) * 0.02).astype(np.float32)
    codes, scales = oracle.quantize_mxfp8(w)
    wh = oracle.dequant_mxfp8(codes, scales)
    b = rng.standard_normal(O)
    ys = oracle.mx_all_to_sharded(x, oracle.shard(codes, 0, 1, N), oracle.shard(scales, 0, 1, N),
                                  oracle.shard(b, 0, 1, N))
    full = np.matmul(x, wh.T) + b
    assert np.abs(np.concatenate(ys, axis=1) - full).max() <= 1e-12 * (1 + np.abs(full).max())
    y = oracle.mx_sharded_to_all(oracle.shard(x, -1, 1, N), oracle.shard(codes, -1, 1, N),
                                 oracle.shard(scales, -1, 1, N), b)
    assert np.abs(y - full).max() <= 1e-12 * (1 + np.abs(full).max())


def test_bf16_widen_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x7F7F], dtype=np.uint16)
    want = [1.0, -1.0, 3.140625, 0.0, 3.3895313892515355e38]
    assert oracle.bf16_to_f64(bits).tolist() == want


def test_num_threads_positive():
    assert oracle.num_threads() >= 1
