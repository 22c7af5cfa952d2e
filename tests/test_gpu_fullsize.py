"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times (the same `workloads` objects and calls), checked against the
fp64 oracle on sampled output rows (every row for T <= 16).
"""
import numpy as np
import pytest
import torch

import oracle
import sharded_gemm_gb300 as tp
from sharded_gemm_gb300 import build as tpbuild
from sharded_gemm_gb300 import synth
from sharded_gemm_gb300.workloads import GatedFFN, MLPBackward, MLPGatherScatter, MLPPair, MXPair, Q4Pair, QKV, Summa, to_host
from gpu_util import bf16, check_close, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    tpbuild.build()
    tp.tp_set_policy(tp.TP_POLICY_AUTO)


def test_full_mlp_pair():
    cfg = synth.mlp()
    pair = MLPPair(cfg)
    pair.step()
    assert tp.tp_query_status() == 0
    # 64 of the 512 token rows (both 256-row token tiles), every output column
    rows = sample_rows(cfg["T"], 64)
    x = bf16(cfg["x"])[rows]
    N = cfg["N"]
    w1 = [bf16(p) for p in oracle.shard(cfg["w1"], 0, 1, N)]
    b1 = [p.astype(np.float64) for p in oracle.shard(cfg["b1"], 0, 1, N)]
    ref_mid = oracle.all_to_sharded(x, w1, b1)
    mids = [to_host(m)[rows] for m in pair.mid]
    for r in range(N):
        check_close(mids[r], ref_mid[r], "mid shard %d" % r)
    w2 = [bf16(p) for p in oracle.shard(cfg["w2"], -1, 1, N)]
    check_close(to_host(pair.y)[rows], oracle.sharded_to_all(mids, w2, cfg["b2"]), "y")


def test_full_gated_ffn():
    # Llama FFN at the bench's ffn_gated size: gated gate/up launch, then W2
    cfg = synth.ffn()
    ffn = GatedFFN(cfg)
    ffn.step()
    assert tp.tp_query_status() == 0
    rows = sample_rows(cfg["T"], 48)
    x = bf16(cfg["x"])[rows]
    N = cfg["N"]
    sh = lambda a: [bf16(p) for p in oracle.shard(cfg[a], 0, 1, N)]
    fb = lambda a: [p.astype(np.float64) for p in oracle.shard(cfg[a], 0, 1, N)]
    ref_h = oracle.gated_all_to_sharded(x, sh("w1"), sh("w3"), fb("b1"), fb("b3"))
    hs = [to_host(h)[rows] for h in ffn.h]
    for r in range(N):
        check_close(hs[r], ref_h[r], "h shard %d" % r)
    w2 = [bf16(p) for p in oracle.shard(cfg["w2"], -1, 1, N)]
    check_close(to_host(ffn.y)[rows], oracle.sharded_to_all(hs, w2, cfg["b2"]), "y")


def test_full_mlp_backward():
    # the bench's mlp_bwd step: sampled token rows of dh and dx, sampled
    # output rows of every weight gradient, all of both bias gradients
    cfg = synth.mlp()
    T, D, N = cfg["T"], cfg["D"], cfg["N"]
    dy = synth.grad_output(T=T, D=D)["dy"]
    bw = MLPBackward(cfg, dy)
    bw.step()
    assert tp.tp_query_status() == 0
    rows = sample_rows(T, 32)
    dyv = bf16(dy)
    w1 = [bf16(p) for p in oracle.shard(cfg["w1"], 0, 1, N)]
    w2 = [bf16(p) for p in oracle.shard(cfg["w2"], -1, 1, N)]
    dh = [to_host(d) for d in bw.dh]
    ref_dh = oracle.sharded_to_all_dx(dyv[rows], w2)
    for r in range(N):
        check_close(dh[r][rows], ref_dh[r], "dh %d" % r)
    check_close(to_host(bw.dx)[rows], oracle.all_to_sharded_dx([d[rows] for d in dh], w1), "dx")
    h = [to_host(m) for m in bw.fwd.mid]
    x = bf16(cfg["x"])
    for r in range(N):
        o2 = sample_rows(D, 64, seed=r)
        check_close(to_host(bw.dw2[r])[o2], oracle.sharded_dw([dyv[:, o2]], [h[r]])[0], "dW2 %d" % r)
        o1 = sample_rows(dh[r].shape[1], 64, seed=10 + r)
        check_close(to_host(bw.dw1[r])[o1], oracle.sharded_dw([dh[r][:, o1]], [x])[0], "dW1 %d" % r)
    check_close(to_host(bw.db2[0]), oracle.bias_grad([[dyv]])[0], "db2")
    for r, g in enumerate(oracle.bias_grad([[d] for d in dh])):
        check_close(to_host(bw.db1[r]), g, "db1 %d" % r)


def test_full_mlp_gather_scatter():
    # the MLP pair with width-sharded input and output (all-gather in,
    # reduce-scatter out), the bench's mlp_ag_rs launches
    cfg = synth.mlp()
    ffn = MLPGatherScatter(cfg)
    ffn.step()
    assert tp.tp_query_status() == 0
    rows = sample_rows(cfg["T"], 64)
    N = cfg["N"]
    xs = [bf16(p)[rows] for p in oracle.shard(cfg["x"], -1, 1, N)]
    w1 = [bf16(p) for p in oracle.shard(cfg["w1"], 0, 1, N)]
    b1 = [p.astype(np.float64) for p in oracle.shard(cfg["b1"], 0, 1, N)]
    ref_mid = oracle.gathered_to_sharded(xs, w1, b1)
    mids = [to_host(m)[rows] for m in ffn.mid]
    for r in range(N):
        check_close(mids[r], ref_mid[r], "mid shard %d" % r)
    w2 = [bf16(p) for p in oracle.shard(cfg["w2"], -1, 1, N)]
    ref_y = oracle.sharded_to_sharded(mids, w2, cfg["b2"])
    for c in range(N):
        check_close(to_host(ffn.ys[c])[rows], ref_y[c], "y block %d" % c)


@pytest.mark.parametrize("q", [2, 4])
def test_full_summa(q):
    cfg = synth.summa()
    s = Summa(cfg, q)
    s.step()
    assert tp.tp_query_status() == 0
    bm = cfg["M"] // q
    Xb = [bf16(b) for b in oracle.blocks(cfg["X"], q)]
    Ab = [bf16(b) for b in oracle.blocks(cfg["A"], q)]
    # a seeded sample of 256 local rows per block row i: Y_ij for every j on
    # those rows (the first and last row of the block always included)
    for i in range(q):
        rows = sample_rows(bm, 256, seed=17 * q + i)
        for j in range(q):
            ref = None
            for t in range(q):
                p = oracle.matmul(Xb[i * q + t][rows], Ab[t * q + j])
                ref = p if ref is None else ref + p
            check_close(to_host(s.Y[i * q + j])[rows], ref, "block (%d, %d)" % (i, j))


@pytest.mark.parametrize("T", [1, 16, 2048])
def test_full_qkv(T):
    cfg = synth.qkv(T=T)
    w = QKV(cfg)
    w.step()
    assert tp.tp_query_status() == 0
    N, D = cfg["N"], cfg["D"]
    rows = sample_rows(T, 16 if T <= 16 else 48)  # every token row for T <= 16
    x = bf16(cfg["x"])[rows]
    # fused QKV: shard r holds rows {s*D + r*D/N + i} of W_qkv
    wq = oracle.shard(cfg["w_qkv"], 0, 3, N)
    bq = oracle.shard(cfg["b_qkv"], 0, 3, N)
    for r in range(N):
        check_close(to_host(w.qkv[r])[rows], oracle.linear(x, bf16(wq[r]), bq[r]), "qkv shard %d" % r)
    # W_o: row-parallel over x's column slices
    xs = oracle.shard(cfg["x"], -1, 1, N)
    wo = oracle.shard(cfg["w_o"], -1, 1, N)
    ref_o = oracle.sharded_to_all([bf16(p)[rows] for p in xs], [bf16(p) for p in wo], cfg["b_o"])
    check_close(to_host(w.attn_out)[rows], ref_o, "W_o")
    # vocab-parallel LM head: gathered logits, sampled columns of every shard
    V = cfg["V"]
    cols = np.sort(np.concatenate([r * (V // N) + sample_rows(V // N, 64, seed=r) for r in range(N)]))
    ref_l = oracle.linear(x, bf16(cfg["w_lm"][cols]))
    check_close(to_host(w.logits)[rows][:, cols], ref_l, "LM head")


@pytest.mark.parametrize("T", [1, 16, 256])
def test_full_q4_pair(T):
    cfg = synth.q4(T=T)
    N, D, F = cfg["N"], cfg["D"], cfg["F"]
    up = oracle.quantize_affine4(cfg["w_up"], 64)
    down = oracle.quantize_affine4(cfg["w_down"], 64)
    w = Q4Pair(cfg, quantized=(up, down))
    w.step()
    assert tp.tp_query_status() == 0
    rows = sample_rows(T, 16 if T <= 16 else 48)  # every token row for T <= 16
    x = bf16(cfg["x"])[rows]
    # up: column-parallel, sampled output columns of every shard
    for r in range(N):
        cols = sample_rows(F // N, 64, seed=r)
        g = [a[r * (F // N):(r + 1) * (F // N)][cols] for a in up]
        ref = oracle.q4_all_to_sharded(x, [g[0]], [g[1]], [g[2]], 64)[0]
        check_close(to_host(w.mid[r])[rows][:, cols], ref, "q4 up shard %d" % r)
    # down: row-parallel over the GPU's own intermediate, sampled output columns
    cols = sample_rows(D, 128, seed=11)
    mids = [to_host(m)[rows] for m in w.mid]
    dq = [oracle.shard(a[cols], -1, 1, N) for a in down]
    ref = oracle.q4_sharded_to_all(mids, dq[0], dq[1], dq[2], 64)
    check_close(to_host(w.y)[rows][:, cols], ref, "q4 down")


@pytest.mark.parametrize("T", [1, 16, 256])
def test_full_mx_pair(T):
    cfg = synth.q4(T=T)
    N, D, F = cfg["N"], cfg["D"], cfg["F"]
    up = oracle.quantize_mxfp8(cfg["w_up"])
    down = oracle.quantize_mxfp8(cfg["w_down"])
    w = MXPair(cfg, quantized=(up, down))
    w.step()
    assert tp.tp_query_status() == 0
    rows = sample_rows(T, 16 if T <= 16 else 48)  # every token row for T <= 16
    x = bf16(cfg["x"])[rows]
    for r in range(N):
        cols = sample_rows(F // N, 96, seed=r)
        sl = slice(r * (F // N), (r + 1) * (F // N))
        ref = oracle.mx_all_to_sharded(x, [up[0][sl][cols]], [up[1][sl][cols]])[0]
        check_close(to_host(w.mid[r])[rows][:, cols], ref, "mx up shard %d" % r)
    cols = sample_rows(D, 128, seed=11)
    mids = [to_host(m)[rows] for m in w.mid]
    dq = [oracle.shard(a[cols], -1, 1, N) for a in down]
    ref = oracle.mx_sharded_to_all(mids, dq[0], dq[1])
    check_close(to_host(w.y)[rows][:, cols], ref, "mx down")
