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
    ref = oracle.q4_sharded_to_all([oracle.bf16_to_f64(p) for p in oracle.shard(x, -1, 1, N)],
                                   *[oracle.shard(a, -1, 1, N) for a in (pq, ps, pb)], 64, b.astype(np.float64))
    return xs, sh, to_device(b, "f32"), ref


# (16, 3584, 1000, 8): the decode shape of the 8192 x 28672 down projection's
# ranks, split across CTAs through the fixed buffer; (1, 512, 260, 4): one token.
@pytest.mark.parametrize("policy", ["auto", "simt"])
@pytest.mark.parametrize("T,Kn,O,N", [(16, 3584, 1000, 8), (1, 512, 260, 4)])
def test_noalloc_matches_allocating_entry_point_on_two_calls(T, Kn, O, N, policy):
    tpbuild.build()
    tp.tp_set_policy(tp.TP_POLICY_SIMT if policy == "simt" else tp.TP_POLICY_AUTO)
    try:
        xs, sh, b, oref = _inputs(T, Kn, O, N, seed=T + O)
        ref = tp.tp_q4_sharded_to_all(xs, *sh, bias=b)
        torch.cuda.synchronize()
        ref_h = to_host(ref)
        check_close(ref_h, oref, "allocating entry point vs oracle")
        for _ in range(2):
            out = torch.full((T, O), float("nan"), dtype=torch.float32, device="cuda")
            tp.tp_q4_sharded_to_all_noalloc(xs, *sh, bias=b, out=out)
            torch.cuda.synchronize()
            assert tp.tp_query_status() == 0  # the fixed buffer's status word is read too
            got = to_host(out)
            check_close(got, ref_h, "noalloc vs allocating entry point")
            check_close(got, oref, "noalloc vs oracle")
    finally:
        tp.tp_set_policy(tp.TP_POLICY_AUTO)


def test_noalloc_rejects_a_split_larger_than_its_buffer():
    tpbuild.build()
    # prefill-sized call: 32 row tiles x 8 rank partials of 128 x 256 floats = 32 MiB > 8 MiB
    T, Kn, O, N = 300, 64, 4096, 8
    xs, sh, b, _ = _inputs(T, Kn, O, N, seed=1)
    out = torch.zeros((T, O), dtype=torch.float32, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_q4_sharded_to_all_noalloc(xs, *sh, bias=b, out=out)
    assert e.value.code == tp.TP_ERR_UNSUPPORTED
    assert "fixed buffer" in e.value.msg
