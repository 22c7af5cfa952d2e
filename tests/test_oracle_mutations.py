"""Plant a mistake in a copy of an oracle routine (on the CPU) and show that
the corresponding pin in ``test_oracle.py`` fails.  This is evidence that the
pins can tell a right oracle from a plausible wrong one."""
import numpy as np
import pytest

import oracle
import test_oracle as T


def _expect_fail(check, *fns):
    with pytest.raises(AssertionError):
        check(*fns)


def test_mutation_transposed_operand():
    # x @ W instead of x @ W.T (only square shapes survive; others must fail)
    def bad_linear(x, w, b=None):
        if w.shape[0] != w.shape[1]:
            return np.zeros((x.shape[0], w.shape[0]))
        y = x @ w
        return y if b is None else y + b
    _expect_fail(T.check_linear_vs_numpy, bad_linear)


def test_mutation_dropped_bias():
    _expect_fail(T.check_linear_vs_numpy, lambda x, w, b=None: oracle.linear(x, w))


def test_mutation_shard_wrong_rank():
    def bad_shard(w, axis, s, n):
        p = oracle.shard(w, axis, s, n)
        return p[1:] + p[:1]
    _expect_fail(T.check_shard_closed_form, bad_shard)


def test_mutation_shard_ignores_segments():
    _expect_fail(T.check_shard_closed_form, lambda w, a, s, n: oracle.shard(w, a, 1, n))


def test_mutation_row_bias_per_shard():
    def bad_row(xs, ws, b=None):
        tot = sum(oracle.linear(x, w, b) for x, w in zip(xs, ws))
        return tot
    _expect_fail(T.check_row_invariant, bad_row, oracle.shard)


def test_mutation_col_wrong_index():
    def bad_col(x, ws, bs=None):
        return [oracle.linear(x, ws[0], bs[0]) for _ in ws]
    _expect_fail(T.check_col_invariant, bad_col, oracle.shard)


def test_mutation_summa_wrong_block():
    def bad_summa(Xb, Ab, q):
        out = []
        for i in range(q):
            for j in range(q):
                out.append(sum(oracle.matmul(Xb[i * q + t], Ab[j * q + t]) for t in range(q)))
        return out
    _expect_fail(T.check_summa_q2_identity, bad_summa)


def test_mutation_dequant_nibble_order():
    def bad_dequant(packed, s, b, g):
        k = s.shape[1] * g
        codes = np.empty((packed.shape[0], k))
        for e in range(8):
            codes[:, e::8] = (packed >> np.uint32(4 * (7 - e))) & 15
        gi = np.arange(k) // g
        return s.astype(np.float64)[:, gi] * codes + b.astype(np.float64)[:, gi]
    _expect_fail(T.check_dequant_bruteforce, bad_dequant)


def test_mutation_reduce_scatter_wrong_block():
    def bad_rs(parts, axis):
        got = oracle.reduce_scatter(parts, axis)
        return got[1:] + got[:1]
    _expect_fail(T.check_reduce_scatter_closed_form, bad_rs)


def test_mutation_reduce_scatter_transposed_pairing():
    # pairs rank c with the mirrored block N-1-c: a consistent AllGather
    # in rank order no longer transposes it
    def bad_rs(parts, axis):
        return oracle.reduce_scatter(parts, axis)[::-1]
    _expect_fail(T.check_gather_scatter_transpose, oracle.all_gather, bad_rs)


def test_mutation_all_gather_reversed():
    _expect_fail(T.check_all_gather_closed_form, lambda s, axis: oracle.all_gather(s[::-1], axis))


def test_mutation_rs_bias_per_partial():
    def bad_rs(xs, ws, b=None):
        parts = [oracle.linear(x, w, b) for x, w in zip(xs, ws)]
        return oracle.reduce_scatter(parts, 1)
    _expect_fail(T.check_rs_bias_once, bad_rs, oracle.shard)


def test_mutation_rs_scatter_rows():
    # scattering the token axis instead of the output columns
    def bad_rs(xs, ws, b=None):
        parts = [oracle.linear(x, w, b) for x, w in zip(xs, ws)]
        tot = sum(parts)
        return np.array_split(tot, len(xs), axis=0)
    _expect_fail(T.check_rs_invariant, bad_rs, oracle.shard)


def test_mutation_ag_reversed_blocks():
    def bad_ag(xs, ws, bs=None):
        return oracle.all_to_sharded(np.concatenate(xs[::-1], axis=1), ws, bs)
    _expect_fail(T.check_ag_invariant, bad_ag, oracle.shard)


def test_mutation_silu_sign():
    # a * sigmoid(-a) instead of a * sigmoid(a)
    def bad_silu(a):
        a = np.asarray(a, dtype=np.float64)
        with np.errstate(over="ignore"):
            return a / (1.0 + np.exp(a))
    _expect_fail(T.check_silu_closed_forms, bad_silu)


def test_mutation_gated_roles_swapped():
    def bad(x, w1s, w3s, b1s=None, b3s=None):
        return oracle.gated_all_to_sharded(x, w3s, w1s, b3s, b1s)
    _expect_fail(T.check_gated_invariant, bad, oracle.shard)


def test_mutation_gated_up_bias_dropped():
    def bad(x, w1s, w3s, b1s=None, b3s=None):
        return oracle.gated_all_to_sharded(x, w1s, w3s, b1s, None)
    _expect_fail(T.check_gated_invariant, bad, oracle.shard)


def test_mutation_col_dx_wrong_rank():
    def bad(dys, ws):
        n = len(ws)
        return oracle.all_to_sharded_dx(dys, [ws[(r + 1) % n] for r in range(n)])
    _expect_fail(T.check_col_adjoint, bad, oracle.sharded_dw, oracle.shard)


def test_mutation_row_dx_transposed_weight():
    def bad(dy, ws):
        return [oracle.matmul(dy, np.ascontiguousarray(np.flipud(w))) for w in ws]
    _expect_fail(T.check_row_adjoint, bad, oracle.sharded_dw, oracle.shard)


def test_mutation_dw_reversed_k():
    # dW_r with its K index reversed
    def bad(dys, xs):
        return [np.fliplr(g) for g in oracle.sharded_dw(dys, xs)]
    _expect_fail(T.check_col_adjoint, oracle.all_to_sharded_dx, bad, oracle.shard)


def test_mutation_bias_grad_wrong_axis():
    def bad(groups):
        return [sum(np.asarray(d).sum(axis=0)[::-1] for d in g) for g in groups]
    _expect_fail(T.check_bias_grad_closed_form, bad)


def test_mutation_abt_wrong_block():
    def bad(Ab, Bb, q):
        return oracle.summa_abt(Ab, [Bb[(b % q) * q + b // q] for b in range(q * q)], q)
    _expect_fail(T.check_summa_backward, bad, oracle.summa_atb)


def test_mutation_atb_wrong_block():
    def bad(Ab, Bb, q):
        return oracle.summa_atb([Ab[(b % q) * q + b // q] for b in range(q * q)], Bb, q)
    _expect_fail(T.check_summa_backward, oracle.summa_abt, bad)


def test_mutation_e4m3_wrong_bias():
    bad = np.array([oracle.e4m3_value(b) * 0.5 for b in range(256)])
    _expect_fail(T.check_e4m3_table, bad)


def test_mutation_e4m3_ties_away():
    def bad(v):
        v = np.asarray(v, dtype=np.float64)
        out = oracle.e4m3_from_f64(v)
        pos = oracle.E4M3_TABLE[:0x7F]
        mid = (pos[:-1] + pos[1:]) / 2
        hit = np.isin(np.abs(v), mid)
        return np.where(hit, np.searchsorted(pos, np.abs(v)) | (np.signbit(v) << 7), out).astype(np.uint8)
    _expect_fail(T.check_e4m3_rounding, bad, oracle.E4M3_TABLE)


def test_mutation_mx_scale_off_by_one():
    # X = floor(log2 amax) - 7: the block maximum lands one binade low
    def bad(w):
        w = np.asarray(w, dtype=np.float32)
        _, s = oracle.quantize_mxfp8(w)
        s = np.where(s > 0, s + 1, s).astype(np.uint8)
        X = s.astype(np.int64) - 127
        g = w.astype(np.float64) / np.ldexp(1.0, X).repeat(32, axis=1)
        return oracle.e4m3_from_f64(g), s
    _expect_fail(T.check_mx_quantize, bad, oracle.dequant_mxfp8)


def test_mutation_mx_dequant_group_64():
    def bad(codes, scales):
        k = codes.shape[1]
        gi = np.arange(k) // 64
        return oracle.E4M3_TABLE[codes] * np.ldexp(1.0, scales.astype(np.int64) - 127)[:, gi]
    _expect_fail(T.check_mx_quantize, oracle.quantize_mxfp8, bad)
