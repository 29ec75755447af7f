"""bench.py's work accounting and its profile lookup (CPU only).

The roofline numerator is algorithmic work: 2*M*N*K FLOPs per GEMM (summed over experts)
and the bytes the method must move once: the packed operand with its scales, the BF16
grad_out and the BF16 output.  These are checked against the figures written out by
hand for the five workloads (packed W and X from their shapes, E4M3 scales per 128x128
block, E8M0 per 32, E4M3 per 16 plus a float32 tensor scale).
"""

from types import SimpleNamespace

import numpy as np
import pytest

import bench

MB = 1e6


def _packed(fmt, batch, rows, cols):
    return SimpleNamespace(fmt=fmt, batch=batch, rows=rows, cols=cols)


def _cfg(n):
    if n == 1:
        M, N, K = 64, 128, 256
        return dict(M=M, N=N, K=K, E=1, grouped=False, W=_packed(1, 1, N, K), X=_packed(0, 1, M, K))
    if n == 2:
        M = N = K = 4096
        return dict(M=M, N=N, K=K, E=1, grouped=False, W=_packed(2, 1, N, K), X=_packed(2, 1, M, K))
    if n == 3:
        M, N, K = 8192, 14336, 5120
        return dict(M=M, N=N, K=K, E=1, grouped=False, W=_packed(3, 1, N, K), X=_packed(3, 1, M, K))
    if n == 4:
        E, S, N, K = 64, 16384, 2816, 2048
        return dict(M=S, N=N, K=K, E=E, grouped=True, offsets=np.array([S]), W=_packed(1, E, N, K), X=None)
    E, S, N, K = 128, 32768, 2048, 7168
    return dict(M=S, N=N, K=K, E=E, grouped=True, offsets=np.array([S]), W=_packed(2, E, N, K),
                X=_packed(2, 1, S, K))


# (op, GFLOP, algorithmic MB) per workload, from the shapes:
#   linear dgrad bytes = packed W + scales + 2*M*N (grad_out) + 2*M*K (grad_X)
#   linear wgrad bytes = packed X + scales + 2*M*N + 2*N*K (grad_W)
#   grouped dgrad / wgrad: the same with S rows and E experts of W / E outputs of grad_W
EXPECTED = {
    2: [("dgrad", 137.439, 76.02), ("wgrad", 137.439, 76.02)],
    3: [("dgrad", 1202.591, 360.05), ("wgrad", 1202.591, 405.27)],
    4: [("grouped_dgrad", 188.979, 528.57)],
    5: [("grouped_dgrad", 962.073, 1602.22), ("grouped_wgrad", 962.073, 4017.09)],
}


@pytest.mark.parametrize("n", sorted(EXPECTED))
def test_plan_matches_hand_counts(n):
    got = bench.plan(_cfg(n))
    assert [g[0] for g in got] == [e[0] for e in EXPECTED[n]]
    for (name, flops, nbytes), (_, gflop, mb) in zip(got, EXPECTED[n]):
        assert flops / 1e9 == pytest.approx(gflop, abs=5e-4), name
        assert nbytes / MB == pytest.approx(mb, abs=5e-3), name


def test_packed_bytes_per_format():
    # 256 x 512: BF16 2 B/elem; FP8 1 B + one f32 per 128x128 block; MXFP4 0.5 B + 1/32;
    # NVFP4 0.5 B + 1/16 + one f32 tensor scale
    n = 256 * 512
    assert bench.packed_bytes(_packed(0, 1, 256, 512)) == 2 * n
    assert bench.packed_bytes(_packed(1, 1, 256, 512)) == n + 4 * 2 * 4
    assert bench.packed_bytes(_packed(2, 1, 256, 512)) == n / 2 + n / 32
    assert bench.packed_bytes(_packed(3, 1, 256, 512)) == n / 2 + n / 16 + 4
    # ragged FP8 grid rounds up
    assert bench.packed_bytes(_packed(1, 2, 130, 129)) == 2 * 130 * 129 + 4 * 2 * 2 * 2


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "bsq_gemm_kernel_w.md").write_text(
        "text\n    traffic: op=dgrad bytes=123 source_sha1=aaaa\n    traffic: op=wgrad bytes=456 source_sha1=bbbb\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha1", lambda: "aaaa")
    assert bench.profiled_traffic("w", "dgrad") == 123
    assert bench.profiled_traffic("w", "wgrad") is None       # taken on other sources
    assert bench.profiled_traffic("other", "dgrad") is None   # no capture for the workload


def _rank_main(rank, world, port, values, out):
    import os
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank])
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    # two gloo ranks on the CPU, as the N-GPU bench runs one replica per rank
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    values = [12.5, 40.0]
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(2, port, values, out), nprocs=2, start_method="spawn", join=True)
    assert dict(out) == {0: 40.0, 1: 40.0}


def test_single_process_and_job_throughput():
    assert bench.max_over_ranks(7.0) == 7.0           # no process group: unchanged
    # 2 replicas x 1 TFLOP per step x 10 steps in 20 ms -> 1000 TFLOP/s for the job
    assert bench.job_tflops(2, 1e12, 10, 20.0) == pytest.approx(1000.0)


def test_fused_step_reads_grad_out_once():
    """The fused backward launch of a linear workload moves both packed operands, grad_out
    once and both outputs: MXFP4 4096^3 = 2 x (8.39 MB codes + 0.52 MB scales) + 3 x 33.55 MB."""
    name, flops, nbytes = bench.step_plan(_cfg(2))
    assert name == "backward"
    assert flops / 1e9 == pytest.approx(274.878, abs=5e-3)
    assert nbytes / MB == pytest.approx(118.489, abs=5e-3)
    assert bench.step_plan(_cfg(1)) is None        # W E4M3, X BF16: two launches
    assert bench.step_plan(_cfg(5)) is None        # grouped
