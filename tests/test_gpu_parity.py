"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small cases span several tiles with ragged tails in every dimension and run
under both kernel policies (tensor-core AUTO and the CUDA-core SIMT
cross-check).  Full-size cases use the workloads' real shapes, in the launch
configuration the bench times, and compare sampled outputs.
"""
import hashlib

import numpy as np
import pytest
import torch

import oracle
import sharded_gemm_gb300 as tp
from sharded_gemm_gb300 import build as tpbuild
from sharded_gemm_gb300 import synth
from sharded_gemm_gb300.workloads import (GatedFFN, MLPBackward, MLPGatherScatter, MLPPair, MXPair, Q4Pair, QKV, Summa, to_device,
                                          to_host)
from gpu_util import bf16, check_close, sample_rows

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(2024)


@pytest.fixture(scope="module", autouse=True)
def built():
    tpbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    tp.tp_set_policy(tp.TP_POLICY_AUTO)


@pytest.fixture(params=[tp.TP_POLICY_AUTO, tp.TP_POLICY_SINGLE_SM, tp.TP_POLICY_SIMT],
                ids=["auto", "single_sm", "simt"])
def policy(request):
    tp.tp_set_policy(request.param)
    yield request.param
    tp.tp_set_policy(tp.TP_POLICY_AUTO)


def _status_ok():
    assert tp.tp_query_status() == 0


def rand_bf16(shape, std=1.0):
    return synth.f32_to_bf16_bits((RNG.standard_normal(shape) * std).astype(np.float32))


# ------------------------------------------------------------------ a1 slicing
@pytest.mark.parametrize("dtype", [np.uint16, np.uint32, np.float16, np.uint8, np.uint64])
@pytest.mark.parametrize("axis,S,N,rows,cols", [
    (0, 1, 4, 8, 12), (0, 3, 2, 12, 6), (1, 1, 8, 5, 16), (-1, 3, 4, 3, 24), (0, 1, 1, 7, 3),
    (1, 2, 2, 4, 12)])
def test_shard_weight_bitexact(dtype, axis, S, N, rows, cols):
    w = RNG.integers(0, 255, size=(rows, cols)).astype(dtype)
    dev = torch.from_numpy(w.view({1: np.uint8, 2: np.int16, 4: np.int32, 8: np.int64}[w.itemsize])).cuda()
    got = tp.tp_shard_weight(dev, axis, S, N)
    ref = oracle.shard(w, axis, S, N)
    for r in range(N):
        g = got[r].cpu().numpy().view(dtype)
        assert g.shape == ref[r].shape
        assert g.tobytes() == ref[r].tobytes(), r


def test_shard_weight_bias_1d():
    b = RNG.standard_normal(24).astype(np.float32)
    got = tp.tp_shard_weight(torch.from_numpy(b).cuda(), 0, 3, 4)
    for g, r in zip(got, oracle.shard(b, 0, 3, 4)):
        assert g.cpu().numpy().tobytes() == r.tobytes()


def test_shard_weight_not_divisible_raises():
    with pytest.raises(tp.TPError) as e:
        tp.tp_shard_weight(torch.zeros((10, 4), device="cuda"), 0, 1, 4)
    assert e.value.code == tp.TP_ERR_NOT_DIVISIBLE
    assert "Cannot shard the output of size 10 across 4 devices." in e.value.msg


# ------------------------------------------------------------------ worked example
def test_worked_example(policy):
    cfg = synth.worked()
    pair = MLPPair(cfg)
    pair.step()
    torch.cuda.synchronize()
    _status_ok()
    x = oracle.widen(cfg["x"], "f32")
    w1 = [oracle.widen(p, "f32") for p in oracle.shard(cfg["w1"], 0, 1, 2)]
    b1 = [oracle.widen(p, "f32") for p in oracle.shard(cfg["b1"], 0, 1, 2)]
    w2 = [oracle.widen(p, "f32") for p in oracle.shard(cfg["w2"], -1, 1, 2)]
    ref_mid = oracle.all_to_sharded(x, w1, b1)
    assert [tuple(m.shape) for m in pair.mid] == [(4, 1), (4, 1)]
    assert [tuple(w.shape) for w in pair.w1] == [(1, 2), (1, 2)]
    assert [tuple(w.shape) for w in pair.w2] == [(2, 1), (2, 1)]
    for r in range(2):
        check_close(to_host(pair.mid[r]), ref_mid[r], "mid %d" % r)
    ref = oracle.sharded_to_all([to_host(m) for m in pair.mid], w2, oracle.widen(cfg["b2"], "f32"))
    check_close(to_host(pair.y), ref, "y")
    assert np.abs(to_host(pair.y) - ref).max() < 1e-5


# ------------------------------------------------------------------ a2 column-parallel
@pytest.mark.parametrize("T,K,On,N", [(1, 64, 128, 2), (5, 192, 40, 4), (130, 320, 600, 2),
                                      (300, 200, 264, 3), (17, 512, 256, 8), (256, 128, 512, 1)])
@pytest.mark.parametrize("out_dt", [torch.bfloat16, torch.float32])
def test_all_to_sharded(policy, T, K, On, N, out_dt):
    x = rand_bf16((T, K))
    w = rand_bf16((On * N, K), 0.05)
    b = (RNG.standard_normal(On * N) * 0.1).astype(np.float32)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), 0, 1, N)
    bs = tp.tp_shard_weight(to_device(b, "f32"), 0, 1, N)
    ys = tp.tp_all_to_sharded(to_device(x, "bf16"), ws, bs, out_dtype=out_dt)
    _status_ok()
    ref = oracle.all_to_sharded(bf16(x), [bf16(p) for p in oracle.shard(w, 0, 1, N)],
                                [p.astype(np.float64) for p in oracle.shard(b, 0, 1, N)])
    for r in range(N):
        check_close(to_host(ys[r]), ref[r], "shard %d" % r)


def test_all_to_sharded_gathered_output(policy):
    # vocab-parallel head: every shard writes its columns of one (T, O) buffer
    T, K, N, On = 70, 256, 4, 300
    x = rand_bf16((T, K))
    w = rand_bf16((On * N, K), 0.05)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), 0, 1, N)
    full = torch.full((T, On * N), float("nan"), device="cuda")
    views = [full[:, r * On:(r + 1) * On] for r in range(N)]
    tp.tp_all_to_sharded(to_device(x, "bf16"), ws, None, out=views)
    _status_ok()
    check_close(to_host(full), oracle.linear(bf16(x), bf16(w)), "gathered")


def test_all_to_sharded_fused_qkv_segments(policy):
    T, D, N = 33, 256, 4
    x = rand_bf16((T, D))
    w = rand_bf16((3 * D, D), 0.05)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), 0, 3, N)
    ys = tp.tp_all_to_sharded(to_device(x, "bf16"), ws, None, out_dtype=torch.float32)
    _status_ok()
    full = oracle.linear(bf16(x), bf16(w))
    wl = D // N
    for r in range(N):
        cols = [s * D + r * wl + i for s in range(3) for i in range(wl)]
        check_close(to_host(ys[r]), full[:, cols], "qkv shard %d" % r)


# ------------------------------------------------------------------ a3 row-parallel
@pytest.mark.parametrize("T,Kn,O,N", [(1, 64, 256, 2), (5, 96, 40, 4), (130, 320, 300, 4),
                                      (200, 200, 520, 3), (64, 512, 128, 8), (129, 128, 129, 1)])
def test_sharded_to_all(policy, T, Kn, O, N):
    x = rand_bf16((T, Kn * N))
    w = rand_bf16((O, Kn * N), 0.05)
    b = (RNG.standard_normal(O) * 0.1).astype(np.float32)
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), -1, 1, N)
    y = tp.tp_sharded_to_all(xs, ws, to_device(b, "f32"))
    _status_ok()
    ref = oracle.sharded_to_all([bf16(p) for p in oracle.shard(x, -1, 1, N)],
                                [bf16(p) for p in oracle.shard(w, -1, 1, N)], b.astype(np.float64))
    check_close(to_host(y), ref, "row")


# Small batches (T <= 16) with fewer output tiles than SMs split each tile's
# contraction into k-block ranges summed by an ordered reduction: ranges that
# cross rank boundaries (22 k-blocks per rank), ragged k-blocks and tokens,
# and a column-parallel split inside one rank's contraction.
@pytest.mark.parametrize("T,Kn,O,N", [(1, 1376, 4096, 8), (16, 1376, 1000, 8), (9, 100, 333, 3),
                                      (16, 512, 4096, 8)])
def test_sharded_to_all_small_batch_split(T, Kn, O, N):
    x = rand_bf16((T, Kn * N))
    w = rand_bf16((O, Kn * N), 0.05)
    b = (RNG.standard_normal(O) * 0.1).astype(np.float32)
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), -1, 1, N)
    bd = to_device(b, "f32")
    y = tp.tp_sharded_to_all(xs, ws, bd)
    y2 = tp.tp_sharded_to_all(xs, ws, bd)
    _status_ok()
    assert torch.equal(y, y2)
    ref = oracle.sharded_to_all([bf16(p) for p in oracle.shard(x, -1, 1, N)],
                                [bf16(p) for p in oracle.shard(w, -1, 1, N)], b.astype(np.float64))
    check_close(to_host(y), ref, "row split")


@pytest.mark.parametrize("T,K,On,N", [(1, 4096, 1536, 8), (16, 4096, 1536, 8), (7, 1000, 200, 2)])
def test_all_to_sharded_small_batch_split(T, K, On, N):
    x = rand_bf16((T, K))
    w = rand_bf16((On * N, K), 0.05)
    b = (RNG.standard_normal(On * N) * 0.1).astype(np.float32)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), 0, 1, N)
    bs = tp.tp_shard_weight(to_device(b, "f32"), 0, 1, N)
    ys = tp.tp_all_to_sharded(to_device(x, "bf16"), ws, bs)
    _status_ok()
    ref = oracle.all_to_sharded(bf16(x), [bf16(p) for p in oracle.shard(w, 0, 1, N)],
                                [p.astype(np.float64) for p in oracle.shard(b, 0, 1, N)])
    for r in range(N):
        check_close(to_host(ys[r]), ref[r], "split shard %d" % r)


def test_small_batch_calls_replay_in_a_cuda_graph():
    # The split small-batch path (workspace, arrival counters) and the
    # programmatic launches run unchanged inside a captured CUDA graph once
    # the same calls have run on the capturing stream.
    T, K, O, N = 1, 4096, 4096, 8
    x = to_device(rand_bf16((T, K)), "bf16")
    w = tp.tp_shard_weight(to_device(rand_bf16((O, K), 0.05), "bf16"), -1, 1, N)
    xs = [x[:, r * (K // N):(r + 1) * (K // N)] for r in range(N)]
    wc = tp.tp_shard_weight(to_device(rand_bf16((O, K), 0.05), "bf16"), 0, 1, N)
    y = torch.empty((T, O), dtype=torch.bfloat16, device="cuda")
    yc = [torch.empty((T, O // N), dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            tp.tp_sharded_to_all(xs, w, None, out=y, stream=s)
            tp.tp_all_to_sharded(x, wc, None, out=yc, stream=s)
    s.synchronize()
    ref = [y.clone()] + [t.clone() for t in yc]
    y.zero_()
    for t in yc:
        t.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tp.tp_sharded_to_all(xs, w, None, out=y, stream=s)
        tp.tp_all_to_sharded(x, wc, None, out=yc, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    _status_ok()
    for a, b in zip([y] + yc, ref):
        assert torch.equal(a, b)


def test_graph_replay_survives_a_larger_call_on_the_same_stream():
    # A captured call holds the addresses of its stream's split workspace.  A
    # later call with a larger split (more tiles, more tokens, a 4-bit row-
    # parallel sum) grows that workspace; the buffers the graph addresses must
    # stay allocated and the replay must still give the captured result.
    T, K, O, N = 1, 4096, 4096, 8
    x = to_device(rand_bf16((T, K)), "bf16")
    w = tp.tp_shard_weight(to_device(rand_bf16((O, K), 0.05), "bf16"), -1, 1, N)
    xs = [x[:, r * (K // N):(r + 1) * (K // N)] for r in range(N)]
    y = torch.empty((T, O), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            tp.tp_sharded_to_all(xs, w, None, out=y, stream=s)
    s.synchronize()
    ref = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tp.tp_sharded_to_all(xs, w, None, out=y, stream=s)
    # larger splits on the same stream, outside the capture
    T2, K2, O2 = 16, 8192, 8192
    x2 = to_device(rand_bf16((T2, K2)), "bf16")
    w2 = tp.tp_shard_weight(to_device(rand_bf16((O2, K2), 0.05), "bf16"), -1, 1, N)
    x2s = [x2[:, r * (K2 // N):(r + 1) * (K2 // N)] for r in range(N)]
    y2 = torch.empty((T2, O2), dtype=torch.float32, device="cuda")
    pq, ps, pb = _q4_host(O2, K2, 5)
    q4x = tp.tp_shard_weight(x2[:1].contiguous(), -1, 1, N)
    q4w = [tp.tp_shard_weight(to_device(a, k), -1, 1, N) for a, k in ((pq, "u32"), (ps, "f16"), (pb, "f16"))]
    with torch.cuda.stream(s):
        tp.tp_sharded_to_all(x2s, w2, None, out=y2, stream=s)
        tp.tp_q4_sharded_to_all(q4x, *q4w, stream=s)
    s.synchronize()
    y.zero_()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(y, ref)


def test_sharded_to_all_strided_input_columns(policy):
    # W_o style: x split by columns as strided views of one (T, K) buffer
    T, K, O, N = 48, 512, 192, 8
    x = rand_bf16((T, K))
    w = rand_bf16((O, K), 0.05)
    xd = to_device(x, "bf16")
    views = [xd[:, r * (K // N):(r + 1) * (K // N)] for r in range(N)]
    ws = tp.tp_shard_weight(to_device(w, "bf16"), -1, 1, N)
    y = tp.tp_sharded_to_all(views, ws, None, out_dtype=torch.bfloat16)
    _status_ok()
    check_close(to_host(y), oracle.linear(bf16(x), bf16(w)), "strided row")


def test_mlp_pair_small(policy):
    cfg = synth.mlp(seed=3, T=150, D=256, F=688, N=4, bias_std=0.1)
    pair = MLPPair(cfg)
    pair.step()
    _status_ok()
    x = bf16(cfg["x"])
    ref_mid = oracle.all_to_sharded(x, [bf16(p) for p in oracle.shard(cfg["w1"], 0, 1, 4)],
                                    [p.astype(np.float64) for p in oracle.shard(cfg["b1"], 0, 1, 4)])
    mids = [to_host(m) for m in pair.mid]
    for r in range(4):
        check_close(mids[r], ref_mid[r], "mid %d" % r)
    w2 = [bf16(p) for p in oracle.shard(cfg["w2"], -1, 1, 4)]
    check_close(to_host(pair.y), oracle.sharded_to_all(mids, w2, cfg["b2"].astype(np.float64)), "y (layer)")
    chain = oracle.linear(oracle.linear(x, bf16(cfg["w1"]), cfg["b1"]), bf16(cfg["w2"]), cfg["b2"])
    check_close(to_host(pair.y), chain, "y (end to end)")


# ------------------------------------------------------------------ f4 mxfp8
@pytest.mark.parametrize("rows,K", [(1, 32), (37, 512), (256, 1024)])
def test_mx_quantize_bitexact(rows, K):
    w = (RNG.standard_normal((rows, K)) * 0.02).astype(np.float32)
    w[0, :32] = 0.0                                    # all-zero block
    if K >= 128:
        w[0, 32:64] = -0.0                             # negative zeros
        w[0, 64:96] *= np.float32(1e30)                # large block
        w[0, 96:128] = np.float32(1e-40) * np.arange(32, dtype=np.float32)  # subnormal block
    if rows > 1:
        w[1, :] = np.where(np.arange(K) % 7 == 0, np.float32(3.0), np.float32(-1e-7))  # tiny next to large
    codes, scales = tp.tp_mx_quantize(torch.from_numpy(w).cuda())
    rc, rs = oracle.quantize_mxfp8(w)
    assert scales.cpu().numpy().tobytes() == rs.tobytes()
    assert codes.cpu().numpy().tobytes() == rc.tobytes()


def _mx_host(rows, K, seed):
    w = (np.random.default_rng(seed).standard_normal((rows, K)) * 0.02).astype(np.float32)
    return oracle.quantize_mxfp8(w)


# T <= 4: the CUDA-core GEMV; larger T: the tensor-core kernel (token tiles of
# 16, 32, 64, 128 and 256, split-K with the ordered fixup, a 32-code tail).
@pytest.mark.parametrize("T,K,On,N", [(1, 512, 40, 4), (3, 1024, 130, 2), (4, 96, 7, 1), (2, 2048, 64, 8),
                                      (20, 256, 96, 2), (16, 4096, 130, 2), (5, 96, 128, 1),
                                      (256, 1024, 256, 2), (300, 512, 200, 1), (64, 2048, 384, 4)])
@pytest.mark.parametrize("out_dt", [torch.bfloat16, torch.float32])
def test_mx_all_to_sharded(policy, T, K, On, N, out_dt):
    codes, scales = _mx_host(On * N, K, T + K)
    x = rand_bf16((T, K))
    cs = tp.tp_shard_weight(torch.from_numpy(codes).cuda(), 0, 1, N)
    ss = tp.tp_shard_weight(torch.from_numpy(scales).cuda(), 0, 1, N)
    b = (RNG.standard_normal(On * N) * 0.1).astype(np.float32)
    bs = tp.tp_shard_weight(to_device(b, "f32"), 0, 1, N)
    ys = tp.tp_mx_all_to_sharded(to_device(x, "bf16"), cs, ss, bs, out_dtype=out_dt)
    _status_ok()
    ref = oracle.mx_all_to_sharded(bf16(x), oracle.shard(codes, 0, 1, N), oracle.shard(scales, 0, 1, N),
                                   [p.astype(np.float64) for p in oracle.shard(b, 0, 1, N)])
    for r in range(N):
        check_close(to_host(ys[r]), ref[r], "shard %d" % r)


@pytest.mark.parametrize("T,Kn,O,N", [(1, 512, 40, 4), (2, 64, 130, 3), (4, 256, 64, 8), (1, 3584, 33, 2),
                                      (17, 128, 48, 2), (16, 3584, 260, 8), (256, 1024, 128, 2),
                                      (100, 96, 129, 3)])
def test_mx_sharded_to_all(policy, T, Kn, O, N):
    codes, scales = _mx_host(O, Kn * N, T + Kn)
    x = rand_bf16((T, Kn * N))
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    cs = tp.tp_shard_weight(torch.from_numpy(codes).cuda(), -1, 1, N)
    ss = tp.tp_shard_weight(torch.from_numpy(scales).cuda(), -1, 1, N)
    b = (RNG.standard_normal(O) * 0.1).astype(np.float32)
    y = tp.tp_mx_sharded_to_all(xs, cs, ss, to_device(b, "f32"))
    _status_ok()
    ref = oracle.mx_sharded_to_all([bf16(p) for p in oracle.shard(x, -1, 1, N)], oracle.shard(codes, -1, 1, N),
                                   oracle.shard(scales, -1, 1, N), b.astype(np.float64))
    check_close(to_host(y), ref, "mx row")


def test_mx_pair_small_repeatable():
    cfg = synth.q4(seed=9, T=1, D=1024, F=2048, N=4)
    up = oracle.quantize_mxfp8(cfg["w_up"])
    down = oracle.quantize_mxfp8(cfg["w_down"])
    w = MXPair(cfg, quantized=(up, down))
    y1 = w.step().clone()
    y2 = w.step().clone()
    _status_ok()
    assert torch.equal(y1, y2)
    x = bf16(cfg["x"])
    mid = oracle.mx_all_to_sharded(x, oracle.shard(up[0], 0, 1, 4), oracle.shard(up[1], 0, 1, 4))
    mids = [to_host(m) for m in w.mid]
    for r in range(4):
        check_close(mids[r], mid[r], "up %d" % r)
    ref = oracle.mx_sharded_to_all(mids, oracle.shard(down[0], -1, 1, 4), oracle.shard(down[1], -1, 1, 4))
    check_close(to_host(w.y), ref, "down")


# ------------------------------------------------------------------ f3 backward
@pytest.mark.parametrize("T,On,K,N", [(1, 64, 128, 2), (5, 40, 192, 4), (130, 320, 600, 2),
                                      (300, 264, 200, 3), (64, 256, 512, 8), (129, 128, 129, 1),
                                      (200, 75, 64, 2)])
def test_all_to_sharded_dx(policy, T, On, K, N):
    dy = rand_bf16((T, On * N))
    w = rand_bf16((On * N, K), 0.05)
    dys = tp.tp_shard_weight(to_device(dy, "bf16"), -1, 1, N)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), 0, 1, N)
    dx = tp.tp_all_to_sharded_dx(dys, ws)
    _status_ok()
    ref = oracle.all_to_sharded_dx([bf16(p) for p in oracle.shard(dy, -1, 1, N)],
                                   [bf16(p) for p in oracle.shard(w, 0, 1, N)])
    check_close(to_host(dx), ref, "dx")


@pytest.mark.parametrize("T,O,Kn,N", [(1, 64, 128, 2), (5, 96, 40, 4), (130, 320, 300, 4),
                                      (200, 200, 520, 3), (64, 512, 128, 8)])
def test_sharded_to_all_dx(policy, T, O, Kn, N):
    dy = rand_bf16((T, O))
    w = rand_bf16((O, Kn * N), 0.05)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), -1, 1, N)
    dxs = tp.tp_sharded_to_all_dx(to_device(dy, "bf16"), ws, out_dtype=torch.float32)
    _status_ok()
    ref = oracle.sharded_to_all_dx(bf16(dy), [bf16(p) for p in oracle.shard(w, -1, 1, N)])
    for r in range(N):
        check_close(to_host(dxs[r]), ref[r], "dx %d" % r)


@pytest.mark.parametrize("T,O,K,N,shared", [(1, 128, 64, 2, "x"), (130, 300, 520, 2, "x"),
                                            (512, 256, 384, 4, "dy"), (77, 136, 264, 3, "dy"),
                                            (700, 520, 260, 1, "x"), (64, 40, 72, 8, "x")])
@pytest.mark.parametrize("out_dt", [torch.float32, torch.bfloat16])
def test_sharded_dw(policy, T, O, K, N, shared, out_dt):
    # shared == "x": column-parallel form (per-shard dy, one x);
    # shared == "dy": row-parallel form (one dy, per-shard x)
    if shared == "x":
        dyh = [rand_bf16((T, O)) for _ in range(N)]
        xh = [rand_bf16((T, K))] * N
    else:
        dyh = [rand_bf16((T, O))] * N
        xh = [rand_bf16((T, K)) for _ in range(N)]
    dyd = [to_device(a, "bf16") for a in dyh]
    xd = [to_device(a, "bf16") for a in xh]
    dws = tp.tp_sharded_dw(dyd, xd, out_dtype=out_dt)
    _status_ok()
    ref = oracle.sharded_dw([bf16(a) for a in dyh], [bf16(a) for a in xh])
    for r in range(N):
        check_close(to_host(dws[r]), ref[r], "dW %d" % r)


def test_sharded_dw_empty_batch_is_zero():
    dy = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    out = [torch.full((64, 128), float("nan"), device="cuda") for _ in range(2)]
    tp.tp_sharded_dw([dy, dy], [x, x], out=out)
    _status_ok()
    for o in out:
        assert torch.equal(o, torch.zeros_like(o))


@pytest.mark.parametrize("rows,cols,nout,nin,dt", [(512, 4096, 1, 1, "bf16"), (130, 75, 3, 1, "f32"),
                                                   (1, 33, 2, 2, "bf16"), (0, 64, 1, 1, "f32"),
                                                   (257, 1000, 2, 4, "f16")])
def test_bias_grad(rows, cols, nout, nin, dt):
    hs = [RNG.standard_normal((rows, cols)).astype(np.float32) for _ in range(nout * nin)]
    if dt == "bf16":
        hs = [synth.f32_to_bf16_bits(h) for h in hs]
        vals = [bf16(h) for h in hs]
    elif dt == "f16":
        hs = [h.astype(np.float16) for h in hs]
        vals = [h.astype(np.float64) for h in hs]
    else:
        vals = [h.astype(np.float64) for h in hs]
    db = tp.tp_bias_grad([to_device(h, dt) for h in hs], nin=nin)
    _status_ok()
    ref = oracle.bias_grad([vals[o * nin:(o + 1) * nin] for o in range(nout)])
    for o in range(nout):
        check_close(to_host(db[o]), ref[o], "db %d" % o)


def _blocks_dev(M, q):
    return [to_device(b, "bf16") for b in oracle.blocks(M, q)]


@pytest.mark.parametrize("q,M,K,Nc", [(1, 128, 128, 256), (2, 272, 320, 528), (4, 512, 256, 1024),
                                      (2, 48, 64, 48)])
def test_summa_abt_atb_linear(policy, q, M, K, Nc):
    A = rand_bf16((M, K))
    B = rand_bf16((Nc, K))
    C = tp.tp_summa_abt(q, _blocks_dev(A, q), _blocks_dev(B, q))
    _status_ok()
    ref = oracle.summa_abt([bf16(b) for b in oracle.blocks(A, q)], [bf16(b) for b in oracle.blocks(B, q)], q)
    for b in range(q * q):
        check_close(to_host(C[b]), ref[b], "abt block %d" % b)
    P = rand_bf16((K, M))
    Q = rand_bf16((K, Nc))
    C = tp.tp_summa_atb(q, _blocks_dev(P, q), _blocks_dev(Q, q))
    _status_ok()
    ref = oracle.summa_atb([bf16(b) for b in oracle.blocks(P, q)], [bf16(b) for b in oracle.blocks(Q, q)], q)
    for b in range(q * q):
        check_close(to_host(C[b]), ref[b], "atb block %d" % b)
    X = rand_bf16((M, K))
    Am = rand_bf16((K, Nc))
    bias = [(RNG.standard_normal(Nc // q) * 0.5).astype(np.float32) for _ in range(q)]
    Y = tp.tp_summa_linear(q, _blocks_dev(X, q), _blocks_dev(Am, q), [to_device(b, "f32") for b in bias])
    _status_ok()
    ref = oracle.summa_linear([bf16(b) for b in oracle.blocks(X, q)], [bf16(b) for b in oracle.blocks(Am, q)],
                              [b.astype(np.float64) for b in bias], q)
    for b in range(q * q):
        check_close(to_host(Y[b]), ref[b], "linear block %d" % b)


def test_mlp_backward_small(policy):
    cfg = synth.mlp(seed=8, T=150, D=256, F=688, N=4, bias_std=0.1)
    dy = synth.grad_output(seed=8, T=150, D=256)["dy"]
    bw = MLPBackward(cfg, dy)
    bw.step()
    _status_ok()
    N = 4
    x, dyv = bf16(cfg["x"]), bf16(dy)
    w1 = [bf16(p) for p in oracle.shard(cfg["w1"], 0, 1, N)]
    w2 = [bf16(p) for p in oracle.shard(cfg["w2"], -1, 1, N)]
    h = [to_host(m) for m in bw.fwd.mid]
    ref_dh = oracle.sharded_to_all_dx(dyv, w2)
    dh = [to_host(d) for d in bw.dh]
    for r in range(N):
        check_close(dh[r], ref_dh[r], "dh %d" % r)
    for r, g in enumerate(oracle.sharded_dw([dyv] * N, h)):
        check_close(to_host(bw.dw2[r]), g, "dW2 %d" % r)
    check_close(to_host(bw.db2[0]), oracle.bias_grad([[dyv]])[0], "db2")
    check_close(to_host(bw.dx), oracle.all_to_sharded_dx(dh, w1), "dx")
    for r, g in enumerate(oracle.sharded_dw(dh, [x] * N)):
        check_close(to_host(bw.dw1[r]), g, "dW1 %d" % r)
    for r, g in enumerate(oracle.bias_grad([[d] for d in dh])):
        check_close(to_host(bw.db1[r]), g, "db1 %d" % r)
    # end to end: the unsharded gradient of y = (x W1^T + b1) W2^T + b2
    full_dx = dyv @ bf16(cfg["w2"]) @ bf16(cfg["w1"])
    check_close(to_host(bw.dx), full_dx, "dx (end to end)")


# ------------------------------------------------------------------ f2 gated FFN
@pytest.mark.parametrize("T,K,Fn,N", [(1, 64, 128, 2), (5, 192, 40, 4), (130, 320, 600, 2),
                                      (300, 200, 264, 3), (17, 512, 256, 8), (256, 128, 512, 1),
                                      (600, 1024, 1000, 2), (70, 100, 64, 2)])
@pytest.mark.parametrize("out_dt", [torch.bfloat16, torch.float32])
def test_gated_all_to_sharded(policy, T, K, Fn, N, out_dt):
    x = rand_bf16((T, K))
    w1 = rand_bf16((Fn * N, K), 0.08)
    w3 = rand_bf16((Fn * N, K), 0.08)
    b1 = (RNG.standard_normal(Fn * N) * 0.5).astype(np.float32)
    b3 = (RNG.standard_normal(Fn * N) * 0.5).astype(np.float32)
    w1s = tp.tp_shard_weight(to_device(w1, "bf16"), 0, 1, N)
    w3s = tp.tp_shard_weight(to_device(w3, "bf16"), 0, 1, N)
    b1s = tp.tp_shard_weight(to_device(b1, "f32"), 0, 1, N)
    b3s = tp.tp_shard_weight(to_device(b3, "f32"), 0, 1, N)
    hs = tp.tp_gated_all_to_sharded(to_device(x, "bf16"), w1s, w3s, b1s, b3s, out_dtype=out_dt)
    _status_ok()
    sh = lambda a: [bf16(p) for p in oracle.shard(a, 0, 1, N)]
    fb = lambda a: [p.astype(np.float64) for p in oracle.shard(a, 0, 1, N)]
    ref = oracle.gated_all_to_sharded(bf16(x), sh(w1), sh(w3), fb(b1), fb(b3))
    for r in range(N):
        check_close(to_host(hs[r]), ref[r], "shard %d" % r)


def test_gated_wide_range_and_gathered_output(policy):
    # gate values from about -60 to 60 (SiLU saturating at both ends), no
    # biases, output written as column views of one (T, F) buffer
    T, K, Fn, N = 150, 256, 320, 4
    x = rand_bf16((T, K))
    w1 = rand_bf16((Fn * N, K), 2.0)
    w3 = rand_bf16((Fn * N, K), 0.05)
    w1s = tp.tp_shard_weight(to_device(w1, "bf16"), 0, 1, N)
    w3s = tp.tp_shard_weight(to_device(w3, "bf16"), 0, 1, N)
    full = torch.full((T, Fn * N), float("nan"), device="cuda")
    views = [full[:, r * Fn:(r + 1) * Fn] for r in range(N)]
    tp.tp_gated_all_to_sharded(to_device(x, "bf16"), w1s, w3s, out=views)
    _status_ok()
    ref = oracle.gated_all_to_sharded(bf16(x), [bf16(w1)], [bf16(w3)])[0]
    assert np.abs(oracle.linear(bf16(x), bf16(w1))).max() > 40
    check_close(to_host(full), ref, "gated gathered")


def test_gated_ffn_small(policy):
    cfg = synth.ffn(seed=6, T=150, D=256, F=688, N=4, bias_std=0.1)
    ffn = GatedFFN(cfg)
    ffn.step()
    _status_ok()
    x = bf16(cfg["x"])
    sh = lambda a: [bf16(p) for p in oracle.shard(cfg[a], 0, 1, 4)]
    fb = lambda a: [p.astype(np.float64) for p in oracle.shard(cfg[a], 0, 1, 4)]
    ref_h = oracle.gated_all_to_sharded(x, sh("w1"), sh("w3"), fb("b1"), fb("b3"))
    hs = [to_host(h) for h in ffn.h]
    for r in range(4):
        check_close(hs[r], ref_h[r], "h %d" % r)
    w2 = [bf16(p) for p in oracle.shard(cfg["w2"], -1, 1, 4)]
    check_close(to_host(ffn.y), oracle.sharded_to_all(hs, w2, cfg["b2"].astype(np.float64)), "y (layer)")
    g = oracle.linear(x, bf16(cfg["w1"]), cfg["b1"])
    u = oracle.linear(x, bf16(cfg["w3"]), cfg["b3"])
    chain = oracle.linear(oracle.silu(g) * u, bf16(cfg["w2"]), cfg["b2"])
    check_close(to_host(ffn.y), chain, "y (end to end)")


# ------------------------------------------------------------------ f1 reduce-scatter / all-gather
# (520, 2048, 512, 4): 40 tiles of 128 x 256 per rank need two rounds of
# 4-rank clusters, so the 256-row cluster tiles are taken (ragged last row
# tile); (300, 2752, 256, 4): one round, 128-row cluster tiles; the short-K
# cases take the single-CTA partial kernel or (T <= 16) the swapped tiles.
@pytest.mark.parametrize("T,Kn,On,N", [(1, 64, 128, 2), (5, 96, 40, 4), (130, 320, 75, 4),
                                       (200, 200, 130, 3), (64, 512, 32, 8), (129, 128, 129, 1),
                                       (300, 2752, 256, 4), (520, 2048, 512, 4)])
def test_sharded_to_sharded(policy, T, Kn, On, N):
    x = rand_bf16((T, Kn * N))
    w = rand_bf16((On * N, Kn * N), 0.05)
    b = (RNG.standard_normal(On * N) * 0.1).astype(np.float32)
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), -1, 1, N)
    ys = tp.tp_sharded_to_sharded(xs, ws, to_device(b, "f32"))
    _status_ok()
    ref = oracle.sharded_to_sharded([bf16(p) for p in oracle.shard(x, -1, 1, N)],
                                    [bf16(p) for p in oracle.shard(w, -1, 1, N)], b.astype(np.float64))
    for c in range(N):
        assert tuple(ys[c].shape) == (T, On)
        check_close(to_host(ys[c]), ref[c], "block %d" % c)


def test_sharded_to_sharded_blocks_equal_all_reduce_bits(policy):
    # Both options of case 3 form each partial from zero and add the partials
    # in rank order, so rank c's block is bit for bit columns c*O/N.. of the
    # all-reduced output.
    T, Kn, O, N = 200, 2752, 1024, 4
    x = rand_bf16((T, Kn * N))
    w = rand_bf16((O, Kn * N), 0.05)
    b = (RNG.standard_normal(O) * 0.1).astype(np.float32)
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), -1, 1, N)
    bd = to_device(b, "f32")
    y = tp.tp_sharded_to_all(xs, ws, bd)
    ys = tp.tp_sharded_to_sharded(xs, ws, bd)
    full = torch.full((T, O), float("nan"), device="cuda")
    views = [full[:, c * (O // N):(c + 1) * (O // N)] for c in range(N)]
    tp.tp_sharded_to_sharded(xs, ws, bd, out=views)
    _status_ok()
    for c in range(N):
        assert torch.equal(ys[c], y[:, c * (O // N):(c + 1) * (O // N)]), c
    assert torch.equal(full, y)


@pytest.mark.parametrize("T,Kn,On,N", [(1, 64, 128, 2), (5, 96, 40, 4), (130, 320, 600, 2),
                                       (300, 200, 264, 3), (17, 512, 256, 8), (256, 128, 512, 1),
                                       (70, 100, 64, 2), (260, 1024, 700, 4)])
@pytest.mark.parametrize("out_dt", [torch.bfloat16, torch.float32])
def test_gathered_to_sharded(policy, T, Kn, On, N, out_dt):
    x = rand_bf16((T, Kn * N))
    w = rand_bf16((On * N, Kn * N), 0.05)
    b = (RNG.standard_normal(On * N) * 0.1).astype(np.float32)
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), 0, 1, N)
    bs = tp.tp_shard_weight(to_device(b, "f32"), 0, 1, N)
    ys = tp.tp_gathered_to_sharded(xs, ws, bs, out_dtype=out_dt)
    _status_ok()
    ref = oracle.gathered_to_sharded([bf16(p) for p in oracle.shard(x, -1, 1, N)],
                                     [bf16(p) for p in oracle.shard(w, 0, 1, N)],
                                     [p.astype(np.float64) for p in oracle.shard(b, 0, 1, N)])
    for r in range(N):
        check_close(to_host(ys[r]), ref[r], "shard %d" % r)


@pytest.mark.parametrize("T", [3, 300])
def test_gathered_equals_column_parallel_on_gathered_bits(policy, T):
    # With K/N a multiple of the 64-wide k-block, chaining the gathered blocks
    # runs the same k-blocks in the same order as the column-parallel product
    # of the materialised gathered input: the results agree bit for bit.
    Kn, On, N = 512, 384, 4
    x = rand_bf16((T, Kn * N))
    w = rand_bf16((On * N, Kn * N), 0.05)
    xd = to_device(x, "bf16")
    xs = tp.tp_shard_weight(xd, -1, 1, N)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), 0, 1, N)
    ys = tp.tp_gathered_to_sharded(xs, ws, None, out_dtype=torch.float32)
    ref = tp.tp_all_to_sharded(xd, ws, None, out_dtype=torch.float32)
    _status_ok()
    for r in range(N):
        assert torch.equal(ys[r], ref[r]), r


def test_mlp_gather_scatter_small(policy):
    cfg = synth.mlp(seed=4, T=150, D=256, F=688, N=4, bias_std=0.1)
    ffn = MLPGatherScatter(cfg)
    ffn.step()
    _status_ok()
    x = bf16(cfg["x"])
    ref_mid = oracle.gathered_to_sharded(oracle.shard(x, -1, 1, 4),
                                         [bf16(p) for p in oracle.shard(cfg["w1"], 0, 1, 4)],
                                         [p.astype(np.float64) for p in oracle.shard(cfg["b1"], 0, 1, 4)])
    mids = [to_host(m) for m in ffn.mid]
    for r in range(4):
        check_close(mids[r], ref_mid[r], "mid %d" % r)
    w2 = [bf16(p) for p in oracle.shard(cfg["w2"], -1, 1, 4)]
    ref_y = oracle.sharded_to_sharded(mids, w2, cfg["b2"].astype(np.float64))
    for c in range(4):
        check_close(to_host(ffn.ys[c]), ref_y[c], "y block %d (layer)" % c)
    chain = oracle.linear(oracle.linear(x, bf16(cfg["w1"]), cfg["b1"]), bf16(cfg["w2"]), cfg["b2"])
    check_close(np.concatenate([to_host(y) for y in ffn.ys], axis=1), chain, "y (end to end)")


# ------------------------------------------------------------------ a5 SUMMA
@pytest.mark.parametrize("q,M,K,Nc", [(1, 128, 128, 256), (2, 272, 320, 528), (4, 512, 256, 1024),
                                      (2, 48, 64, 48), (4, 544, 544, 544)])
def test_summa(policy, q, M, K, Nc):
    cfg = synth.summa(seed=5, M=M, K=K, Ncols=Nc)
    s = Summa(cfg, q)
    s.step()
    _status_ok()
    Xb = [bf16(b) for b in oracle.blocks(cfg["X"], q)]
    Ab = [bf16(b) for b in oracle.blocks(cfg["A"], q)]
    ref = oracle.summa(Xb, Ab, q)
    for b in range(q * q):
        check_close(to_host(s.Y[b]), ref[b], "block %d" % b)


def test_summa_identity_x_returns_a(policy):
    q, n = 2, 256
    X = synth.f32_to_bf16_bits(np.eye(n, dtype=np.float32))
    A = rand_bf16((n, n))
    s = Summa(dict(M=n, K=n, Ncols=n, dtype="bf16", X=X, A=A), q)
    s.step()
    _status_ok()
    got = oracle.unblock([to_host(y) for y in s.Y], q)
    assert np.array_equal(got, bf16(A))


# ------------------------------------------------------------------ a6 / a7 4-bit
@pytest.mark.parametrize("rows,K", [(1, 64), (37, 512), (256, 1024)])
def test_quantize_bitexact(rows, K):
    w = (RNG.standard_normal((rows, K)) * 0.02).astype(np.float32)
    w[0, :64] = 0.25                 # constant group -> unit scale
    if K >= 192:
        w[0, 64:128] = np.float32(1e-9) * np.arange(64, dtype=np.float32)   # scale rounds to 0 in f16
        w[0, 128:192] = np.float32(1e-7) * np.arange(64, dtype=np.float32)  # f16-subnormal scale
    wq, sc, qb = tp.tp_q4_quantize(torch.from_numpy(w).cuda())
    rq, rs, rb = oracle.quantize_affine4(w, 64)
    assert wq.cpu().numpy().view(np.uint32).tobytes() == rq.tobytes()
    assert sc.cpu().numpy().tobytes() == rs.tobytes()
    assert qb.cpu().numpy().tobytes() == rb.tobytes()


def _q4_host(rows, K, seed):
    w = (np.random.default_rng(seed).standard_normal((rows, K)) * 0.02).astype(np.float32)
    return oracle.quantize_affine4(w, 64)


# (2, 1088, 37, 3): two tokens, 34 items of 32 per row (a ragged second slab),
# 37 rows (a ragged last block of 4); (1, 64, 1, 1): one group, one row.
# (3, 1024, 200, 2), (9, 1536, 129, 3), (16, 512, 200, 4): the 8-bit tensor-core
# decode (whole 512-element stages; 8- and 16-token operand widths; a ragged
# last 128-row tile); (2, 1024, 300, 2) under single_sm takes it at two tokens.
@pytest.mark.parametrize("T,K,On,N", [(1, 256, 128, 2), (2, 1088, 37, 3), (1, 64, 1, 1), (16, 512, 200, 4),
                                      (40, 1024, 136, 8), (256, 128, 64, 1), (3, 1024, 200, 2),
                                      (9, 1536, 129, 3), (2, 1024, 300, 2), (13, 8192, 128, 1)])
def test_q4_all_to_sharded(policy, T, K, On, N):
    x = rand_bf16((T, K))
    pq, ps, pb = _q4_host(On * N, K, T + K)
    shards = [tp.tp_shard_weight(to_device(a, k), 0, 1, N) for a, k in ((pq, "u32"), (ps, "f16"), (pb, "f16"))]
    ys = tp.tp_q4_all_to_sharded(to_device(x, "bf16"), *shards, out_dtype=torch.float32)
    _status_ok()
    ref = oracle.q4_all_to_sharded(bf16(x), oracle.shard(pq, 0, 1, N), oracle.shard(ps, 0, 1, N),
                                   oracle.shard(pb, 0, 1, N), 64)
    for r in range(N):
        check_close(to_host(ys[r]), ref[r], "q4 col shard %d" % r)


# (2, 192, 75, 5): two tokens, 6 items per rank, 75 rows; (1, 2112, 130, 3):
# 66 items per rank (three slabs, ragged), 130 rows.
# (5, 512, 300, 4), (16, 3584, 200, 2), (8, 1024, 129, 8): the 8-bit decode's
# row-parallel sums (rank partials, and split chunks of a rank's groups, added
# in order by the last arriving warp).
@pytest.mark.parametrize("T,Kn,O,N", [(1, 128, 256, 2), (2, 192, 75, 5), (1, 2112, 130, 3), (16, 64, 130, 8),
                                      (33, 256, 72, 4), (256, 192, 128, 2), (5, 512, 300, 4),
                                      (16, 3584, 200, 2), (8, 1024, 129, 8)])
def test_q4_sharded_to_all(policy, T, Kn, O, N):
    x = rand_bf16((T, Kn * N))
    pq, ps, pb = _q4_host(O, Kn * N, O + Kn)
    b = (RNG.standard_normal(O) * 0.1).astype(np.float32)
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    shards = [tp.tp_shard_weight(to_device(a, k), -1, 1, N) for a, k in ((pq, "u32"), (ps, "f16"), (pb, "f16"))]
    y = tp.tp_q4_sharded_to_all(xs, *shards, bias=to_device(b, "f32"))
    _status_ok()
    ref = oracle.q4_sharded_to_all([bf16(p) for p in oracle.shard(x, -1, 1, N)], oracle.shard(pq, -1, 1, N),
                                   oracle.shard(ps, -1, 1, N), oracle.shard(pb, -1, 1, N), 64, b.astype(np.float64))
    check_close(to_host(y), ref, "q4 row")


# The 8-bit decode's fallback for CTAs whose peers are not resident: each CTA
# prepares every activation item itself instead of waiting for the launch-wide
# count.  The prepared values are the same, so the outputs must be the same
# bytes as the default path's; both sides span several 128-row tiles, ragged
# last tiles and (row-parallel) range splits across rank boundaries.
@pytest.mark.parametrize("layer,T", [("col", 16), ("col", 5), ("row", 16), ("row", 8)])
def test_q4_dec8_prepare_alone_bit_identical(layer, T):
    N = 4
    if layer == "col":
        K, On = 1536, 200
        x = to_device(rand_bf16((T, K)), "bf16")
        pq, ps, pb = _q4_host(On * N, K, 7 + T)
        shards = [tp.tp_shard_weight(to_device(a, k), 0, 1, N) for a, k in ((pq, "u32"), (ps, "f16"), (pb, "f16"))]
        run = lambda: torch.cat(tp.tp_q4_all_to_sharded(x, *shards, out_dtype=torch.float32), dim=1)
    else:
        Kn, O = 3584, 300
        xs = tp.tp_shard_weight(to_device(rand_bf16((T, Kn * N)), "bf16"), -1, 1, N)
        pq, ps, pb = _q4_host(O, Kn * N, 11 + T)
        shards = [tp.tp_shard_weight(to_device(a, k), -1, 1, N) for a, k in ((pq, "u32"), (ps, "f16"), (pb, "f16"))]
        b = to_device((RNG.standard_normal(O) * 0.1).astype(np.float32), "f32")
        run = lambda: tp.tp_q4_sharded_to_all(xs, *shards, bias=b)
    y0 = run().clone()
    _status_ok()
    try:
        tp.tp_debug_prep_alone(True)
        y1 = run().clone()
        _status_ok()
    finally:
        tp.tp_debug_prep_alone(False)
    y2 = run().clone()
    _status_ok()
    assert to_host(y1).tobytes() == to_host(y0).tobytes()
    assert to_host(y2).tobytes() == to_host(y0).tobytes()


def _range_rows(T, K, seed):
    """Activation rows spanning the bfloat16 range, for the 4-bit prefill
    (T > 16): rows far above the float16 maximum (|x| ~ 1e6 > 65504), rows of
    tiny values (~1e-30, below the float16 subnormals), ordinary rows, an
    all-zero row, a row mixing 1e5 and 1 inside it, and rows near 3e4."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K))
    scale = np.ones(T)
    scale[0:8] = 1e6
    scale[8:16] = 1e-30
    scale[24] = 0.0
    scale[26:T] = 3e4
    x = x * scale[:, None]
    x[25, ::2] *= 1e5
    return synth.f32_to_bf16_bits(x.astype(np.float32))


def _check_rows(got, ref, what):
    # Row by row (one token per row), each row divided by its largest |ref|
    # first: the shared bound |d| <= ATOL (|ref| + 1) is written for outputs
    # of order one, and on a 1e6-scale row its absolute floor vanishes, so
    # outputs that cancel to near zero would be held to a bound that the
    # rounding of the row's large terms exceeds.
    for t in range(ref.shape[0]):
        s = float(np.abs(ref[t]).max())
        s = s if s > 0 else 1.0
        check_close(np.asarray(got[t], np.float64) / s, ref[t] / s, "%s token %d" % (what, t))


@pytest.mark.parametrize("T,K,On,N", [(40, 512, 72, 2), (300, 256, 130, 1)])
def test_q4_prefill_keeps_bf16_range_col(policy, T, K, On, N):
    # the prefill takes x in float16 after a per-row power-of-two scaling:
    # rows beyond the float16 range or below its subnormals must come out
    # as the oracle computes them from the bfloat16 values
    x = _range_rows(T, K, T + K)
    pq, ps, pb = _q4_host(On * N, K, 5 + K)
    shards = [tp.tp_shard_weight(to_device(a, k), 0, 1, N) for a, k in ((pq, "u32"), (ps, "f16"), (pb, "f16"))]
    ys = tp.tp_q4_all_to_sharded(to_device(x, "bf16"), *shards, out_dtype=torch.float32)
    _status_ok()
    ref = oracle.q4_all_to_sharded(bf16(x), oracle.shard(pq, 0, 1, N), oracle.shard(ps, 0, 1, N),
                                   oracle.shard(pb, 0, 1, N), 64)
    for r in range(N):
        _check_rows(to_host(ys[r]), ref[r], "q4 prefill range, shard %d" % r)


def test_q4_prefill_keeps_bf16_range_row(policy):
    T, Kn, O, N = 40, 256, 136, 4
    x = _range_rows(T, Kn * N, 77)
    pq, ps, pb = _q4_host(O, Kn * N, 91)
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    shards = [tp.tp_shard_weight(to_device(a, k), -1, 1, N) for a, k in ((pq, "u32"), (ps, "f16"), (pb, "f16"))]
    y = tp.tp_q4_sharded_to_all(xs, *shards, out_dtype=torch.float32)
    _status_ok()
    ref = oracle.q4_sharded_to_all([bf16(p) for p in oracle.shard(x, -1, 1, N)], oracle.shard(pq, -1, 1, N),
                                   oracle.shard(ps, -1, 1, N), oracle.shard(pb, -1, 1, N), 64, None)
    _check_rows(to_host(y), ref, "q4 prefill range, row-parallel")


# ------------------------------------------------------------------ determinism, faults
def _digest(ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()


def test_repeat_runs_bit_identical(policy):
    cfg = synth.mlp(seed=11, T=260, D=512, F=1376, N=4)
    pair = MLPPair(cfg)
    digests = set()
    for _ in range(5):
        pair.y.fill_(0)
        pair.step()
        digests.add(_digest(pair.mid + [pair.y]))
    _status_ok()
    assert len(digests) == 1


def test_bounded_wait_times_out_and_context_survives():
    tp.tp_debug_wait_timeout(50_000_000)
    assert tp.tp_query_status() == tp.TP_ERR_TIMEOUT
    assert tp.tp_query_status() == 0  # the word was cleared
    # the context is still usable
    x = to_device(rand_bf16((8, 64)), "bf16")
    w = [to_device(rand_bf16((16, 64)), "bf16")]
    y = tp.tp_all_to_sharded(x, w, None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_query_status() == 0
    assert torch.isfinite(y[0]).all()


def test_many_pair_tiles_bias_and_determinism():
    # More 256 x 256 pair tiles (80) than pairs of SMs, long K, a bias: sampled
    # rows against the oracle and bit-identical repeats.
    tp.tp_set_policy(tp.TP_POLICY_AUTO)
    T, K, On, N = 300, 2048, 2560, 4
    x = rand_bf16((T, K))
    w = rand_bf16((On * N, K), 0.03)
    b = (RNG.standard_normal(On * N) * 0.5).astype(np.float32)
    ws = tp.tp_shard_weight(to_device(w, "bf16"), 0, 1, N)
    bs = tp.tp_shard_weight(to_device(b, "f32"), 0, 1, N)
    xd = to_device(x, "bf16")
    ys = tp.tp_all_to_sharded(xd, ws, bs, out_dtype=torch.float32)
    _status_ok()
    first = _digest(ys)
    rows = sample_rows(T, 10)
    ref = oracle.all_to_sharded(bf16(x)[rows], [bf16(p) for p in oracle.shard(w, 0, 1, N)],
                                [p.astype(np.float64) for p in oracle.shard(b, 0, 1, N)])
    for r in range(N):
        check_close(to_host(ys[r])[rows], ref[r], "shard %d" % r)
    for _ in range(3):
        ys = tp.tp_all_to_sharded(xd, ws, bs, out_dtype=torch.float32)
        assert _digest(ys) == first
