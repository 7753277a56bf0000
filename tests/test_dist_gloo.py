"""The multi-rank path of bench.py on CPU: two gloo ranks, one process each.

The block shards by tokens with no data-path collective; the benchmark's only cross-rank steps
are the barrier and the max over ranks of the step time, and the whole-job rate counts every
rank's units against that slowest time.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]
        mx = bench.reduce_max(ms, world, torch.device("cpu"))
        dist.barrier()
        rate = bench.whole_job_rate(100.0, world, mx)
        out[rank] = (mx, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_rate():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (5.0, 2 * 100.0 / 5e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(2.5, 1, None) == 2.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5000.0


# ------------------------------------------------------------------ data-parallel block ----

def _dp_worker(rank, world, port, out):
    import numpy as np
    import torch
    import torch.distributed as dist

    from fp8_transformer_gb300 import dp
    from oracle import block as ob
    from workloads import make_inputs

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m, H, F = 24, 64, 96
        inp = make_inputs("gpt_ln_mlp_bwd", device="cpu", M=world * m, H=H, F=F)
        f = lambda k: inp[k].double().numpy()
        rows = slice(rank * m, (rank + 1) * m)
        scales = dict(x=32.0, w1=2048.0, act=16.0, w2=2048.0, grad=64.0)
        fp8 = {k: np.float32(v) for k, v in scales.items()}
        loc = ob.layernorm_mlp_bwd(f("dy")[rows], f("x")[rows], f("gamma"), f("beta"), f("w1"),
                                   f("w2"), f("b1"), f("b2"), "layernorm", False, inp["eps"],
                                   "gelu", "bf16", fp8=fp8)
        # this rank's gradients as the library stores them, in the flat buckets
        b = dp.GradBuckets(H, F, False, dtype=torch.float32, device="cpu")
        b.dkernel1.copy_(torch.from_numpy(loc["dW1"].value))
        b.dkernel2.copy_(torch.from_numpy(loc["dW2"].value))
        for name, v in (("dbias1", loc["db1"]), ("dbias2", loc["db2"]),
                        ("dgamma", loc["dgamma"]), ("dbeta", loc["dbeta"])):
            getattr(b, name).copy_(torch.from_numpy(np.asarray(v, np.float32)))
        b.allreduce()
        bank = dp.QuantizerBank(dict(x=32.0, kernel1=2048.0, act=16.0, kernel2=2048.0,
                                     grad=64.0), device="cpu")
        fw = loc["fwd"]
        for name, amax in (("x", fw["ln"].amax), ("kernel1", fw["w1"].amax),
                           ("act", fw["a"].amax), ("kernel2", fw["w2"].amax),
                           ("grad", loc["dh"].amax)):
            bank.quantizers[name].amax.fill_(float(amax))
        bank.allreduce_amax()
        out[rank] = dict(weights=b.weights.numpy().copy(), vectors=b.vectors.numpy().copy(),
                         amax=bank.amax.numpy().copy())
    finally:
        dist.destroy_process_group()


def test_data_parallel_exchanges_match_the_whole_batch():
    """Two gloo ranks each run the oracle's FP8 backward on their half of the tokens (standing in
    for the GPU call, which the test cannot run on a CPU) and exchange through
    fp8_transformer_gb300.dp: the summed parameter gradients must match the oracle's backward on
    the whole batch (GEMM rule for the kernels' gradients, each rank's bf16 rounding included;
    1e-4 for the fp32 vectors), and the amax MAX must give the whole batch's amaxes exactly, so
    that every rank derives the same scales."""
    import numpy as np

    from oracle import block as ob
    from parity import assert_gemm_close, assert_reduction_close, rms
    from workloads import make_inputs

    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_dp_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for k in ("weights", "vectors", "amax"):
        assert np.array_equal(res[0][k], res[1][k]), k  # every rank holds the same result
    m, H, F = 24, 64, 96
    inp = make_inputs("gpt_ln_mlp_bwd", device="cpu", M=world * m, H=H, F=F)
    f = lambda k: inp[k].double().numpy()
    fp8 = {k: np.float32(v) for k, v in dict(x=32.0, w1=2048.0, act=16.0, w2=2048.0,
                                             grad=64.0).items()}
    ref = ob.layernorm_mlp_bwd(f("dy"), f("x"), f("gamma"), f("beta"), f("w1"), f("w2"),
                               f("b1"), f("b2"), "layernorm", False, inp["eps"], "gelu", "bf16",
                               fp8=fp8)
    w, v = res[0]["weights"], res[0]["vectors"]
    M = world * m
    ln = ref["fwd"]["ln"].value * ref["fwd"]["ln"].inv()
    dh = ref["dh"].value * ref["dh"].inv()
    assert_gemm_close(w[:H * F].reshape(H, F), ref["dW1"].value, M, rms(ln), rms(dh), what="dW1",
                      stored="bf16")
    assert_gemm_close(w[H * F:].reshape(F, H), ref["dW2"].value, M, rms(ref["a_re"].value),
                      rms(f("dy")), what="dW2", stored="bf16")
    o = 0
    for name, want in (("dbias1", ref["db1"]), ("dbias2", ref["db2"]),
                       ("dgamma", ref["dgamma"]), ("dbeta", ref["dbeta"])):
        n = len(want)
        assert_reduction_close(v[o:o + n], want, what=name)
        o += n
    fw = ref["fwd"]
    want_amax = [fw["ln"].amax, fw["w1"].amax, fw["a"].amax, fw["w2"].amax, ref["dh"].amax]
    assert np.array_equal(res[0]["amax"], np.asarray(want_amax, np.float32))
