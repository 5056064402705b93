"""Multi-rank host logic on CPU with the gloo backend (world size 2).

1. The sequence-parallel pipeline itself, run with real collectives: each rank holds its own
   un-reduced output for every (padded) token; ReduceScatter along the token dim gives each rank
   the summed rows of its contiguous shard; the rank applies add + RMSNorm + quant to its shard
   (the oracle, tp=1, with its chunk of the replicated residual); AllGather along the token dim
   and unpad. The result must equal the fused single-device call on all partials, bit for bit
   (vllm-ascend SP/FlashComm notes §2.2-2.3, §3.3; PR #18671 notes §2, §5.2).
2. The bench's aggregation over ranks: slowest rank's time, whole-job throughput.
3. The reference arm under torchrun: ranks other than 0 exit without work.
"""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, port):
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD,
                            init_method=f"tcp://127.0.0.1:{port}")


def _gather_rows(t: torch.Tensor) -> torch.Tensor:
    """AllGather along dim 0 (integer payloads travel as int32)."""
    x = t.to(torch.int32).contiguous()
    out = torch.empty((x.shape[0] * WORLD,) + tuple(x.shape[1:]), dtype=torch.int32)
    dist.all_gather_into_tensor(out, x)
    return out


def _sp_pipeline_worker(rank, port, mode):
    _init(rank, port)
    try:
        import oracle
        from sequence_reduce_add_gb300 import synth
        bits = synth.bf16_bits
        T, H = 13, 32
        T_pad = -(-T // WORLD) * WORLD  # pad the token count to a multiple of tp
        S = T_pad // WORLD
        g = torch.Generator().manual_seed(77)  # same draw on every rank
        partials = torch.randint(-8, 9, (WORLD, T_pad, H), generator=g).double()
        partials[:, T:] = 0  # F.pad before the ReduceScatter
        residual = torch.randint(-8, 9, (T_pad, H), generator=g).to(torch.bfloat16)
        weight = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
        bias = torch.randint(-2, 3, (H,), generator=g).to(torch.bfloat16)
        scale = {"fp8_static": 0.05, "nvfp4": 60.0}.get(mode)

        # ReduceScatter(dim 0): sum over ranks, rank r keeps rows [r*S, (r+1)*S)
        shard = torch.empty((S, H), dtype=torch.float64)
        dist.reduce_scatter_tensor(shard, partials[rank].contiguous())
        rows = slice(rank * S, (rank + 1) * S)
        valid = max(0, min(S, T - rank * S))
        local = oracle.fused_reduce_norm(
            bits(shard.to(torch.bfloat16)[None]), bits(residual[rows].contiguous()),
            bits(weight), bits(bias), 1e-6, mode, scale, valid)
        assert local["status"] == 0
        # AllGather(dim 0), then unpad
        gathered = {k: _gather_rows(torch.from_numpy(local[k].astype(np.int64)))
                    for k in ("out", "residual_out") if local[k] is not None}
        if local["out_scales"] is not None:
            sc = local["out_scales"]
            sc = sc.view(np.int32) if sc.dtype == np.float32 else sc.astype(np.int32)
            gathered["out_scales"] = _gather_rows(torch.from_numpy(sc.copy()))

        if rank == 0:
            fused = oracle.fused_reduce_norm(
                bits(partials.to(torch.bfloat16)), bits(residual), bits(weight), bits(bias), 1e-6,
                mode, scale, T)
            assert fused["status"] == 0
            for k, v in gathered.items():
                ref = fused[k]
                ref = ref.view(np.int32) if ref.dtype == np.float32 else ref.astype(np.int32)
                got = v.numpy()
                assert np.array_equal(got[:T], ref[:T]), k       # unpadded rows
                assert not got[T:].any(), k                       # padding rows are zero
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["none", "fp8_static", "fp8_per_token", "nvfp4"])
def test_sp_pipeline_with_collectives_equals_fused_call(mode):
    mp.spawn(_sp_pipeline_worker, args=(_free_port(), mode), nprocs=WORLD, join=True)


def _aggregation_worker(rank, port):
    _init(rank, port)
    try:
        import bench
        my_ms = 10.0 + 5.0 * rank
        worst = bench.max_over_ranks(my_ms, "cpu")
        assert worst == 15.0
        gbs = bench.whole_job_throughput(1_000_000_000, 100, WORLD, worst)
        assert abs(gbs - 1e9 * 100 * WORLD / 0.015 / 1e9) < 1e-6
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_bench_aggregation_over_ranks():
    mp.spawn(_aggregation_worker, args=(_free_port(),), nprocs=WORLD, join=True)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "3", "--warmup", "1"], env=env, capture_output=True,
                          text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr[-500:]
    assert proc.stdout.strip() == ""
