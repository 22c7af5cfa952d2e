"""GPU test of tp_q4_sharded_to_all_noalloc, the entry point for callers that
cannot allocate device memory (graph-captured serving loops, engines with
their own pool allocator, paths that cannot afford cudaMalloc's implicit
synchronization).  It must give what tp_q4_sharded_to_all gives, call after
call, while taking its split workspace from a fixed array inside the library.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import sharded_gemm_gb300 as tp
from sharded_gemm_gb300 import build as tpbuild
from sharded_gemm_gb300 import synth
from sharded_gemm_gb300.workloads import to_device, to_host
from gpu_util import check_close

pytestmark = pytest.mark.gpu


def _inputs(T, Kn, O, N, seed):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, Kn * N)).astype(np.float32))
    w = (rng.standard_normal((O, Kn * N)) * 0.02).astype(np.float32)
    pq, ps, pb = oracle.quantize_affine4(w, 64)
    b = (rng.standard_normal(O) * 0.1).astype(np.float32)
    xs = tp.tp_shard_weight(to_device(x, "bf16"), -1, 1, N)
    sh = [tp.tp_shard_weight(to_device(a, k), -1, 1, N) for a, k in ((pq, "u32"), (ps, "f16"), (pb, "f16"))]
    return xs, sh, to_device(b, "f32")


@pytest.mark.parametrize("T,Kn,O,N", [(16, 3584, 1000, 8), (1, 512, 260, 4)])
def test_noalloc_matches_allocating_entry_point_on_two_calls(T, Kn, O, N):
    tpbuild.build()
    tp.tp_set_policy(tp.TP_POLICY_AUTO)
    xs, sh, b = _inputs(T, Kn, O, N, seed=T + O)
    ref = tp.tp_q4_sharded_to_all(xs, *sh, bias=b)
    torch.cuda.synchronize()
    ref_h = to_host(ref)
    for _ in range(2):
        out = torch.full((T, O), float("nan"), dtype=torch.float32, device="cuda")
        tp.tp_q4_sharded_to_all_noalloc(xs, *sh, bias=b, out=out)
        torch.cuda.synchronize()
        check_close(to_host(out), ref_h, "noalloc vs allocating entry point")


def test_noalloc_rejects_a_split_larger_than_its_buffer():
    tpbuild.build()
    # prefill-sized call: 32 row tiles x 8 rank partials of 128 x 256 floats = 32 MiB > 8 MiB
    T, Kn, O, N = 300, 64, 4096, 8
    xs, sh, b = _inputs(T, Kn, O, N, seed=1)
    out = torch.zeros((T, O), dtype=torch.float32, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_q4_sharded_to_all_noalloc(xs, *sh, bias=b, out=out)
    assert e.value.code == tp.TP_ERR_UNSUPPORTED
    assert "fixed buffer" in e.value.msg
