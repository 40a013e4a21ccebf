"""The tensor-parallel linear on a GPU ("The Graph IR", the AllReduce /
AllGather row; "Model and Distributed IR", "Boundary between the layers":
rank-local matmul tasks, a collective, and a reconstructed result equal to
the one-device result).

* Ranks emulated in one process: each rank's local step through the C ABI
  on its shard, the collective stood in for by placing the shards in their
  slots (column split) or adding the FP32 partial sums in rank order (row
  split), then the library's assembly / finishing kernel.  The column split
  is compared with the one-GPU call bit for bit where both sum every output
  in the same order (GEMM shapes with K below the split-K threshold) and
  with the oracle under the contract's rule everywhere; the row split with
  the oracle under the rule (its partial sums are added in another legal
  FP32 order).
* Two processes on the one GPU, each a rank of a gloo group, run the whole
  path (column_parallel_linear, row_parallel_linear); their kernels never
  wait on one another, and the collective runs on the host.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import linear_fp16_gb300 as L
from linear_fp16_gb300 import synth
from tests.parity import check_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _column_emulated(x, w, b, world):
    M, N = x.shape[0], w.shape[0]
    b0, e0 = L.shard_range(N, world, 0)
    slot = max(1, M * (e0 - b0))
    slots = torch.full((world * slot,), float("nan"), dtype=torch.float16, device=DEV)
    for r in range(world):
        nb, ne = L.shard_range(N, world, r)
        if ne > nb:
            L.linear(x, w[nb:ne], b[nb:ne], out=slots[r * slot:r * slot + M * (ne - nb)].view(M, ne - nb))
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    rc = L.poot_linear_gather_columns(slots.data_ptr(), y.data_ptr(), M, N, world, slot,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == L.POOT_OK, L.poot_linear_status_string(rc)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("world", [2, 3, 4, 8])
@pytest.mark.parametrize("M,N,K,dist", [(300, 1000, 520, "normal"), (2047, 1000, 770, "smallint"),
                                        (129, 72, 64, "normal"), (1, 4096, 4096, "normal"),
                                        (8, 1000, 776, "normal"), (512, 2056, 4096, "normal")])
def test_column_split_reconstructs_the_one_gpu_result(world, M, N, K, dist):
    xh, wh, bh = synth.make_inputs(M, N, K, dist, 60 + world + M % 7)
    x, w, b = xh.to(DEV), wh.to(DEV), bh.to(DEV)
    y = _column_emulated(x, w, b, world)
    ok, rep = check_rows(_bits(y), _bits(xh), _bits(wh), _bits(bh), exact=dist == "smallint")
    assert ok, rep
    if M > L.GEMV_MAX_M and K < 1024:
        # the GEMM sums each output in K order whatever the tile: same bits
        assert np.array_equal(_bits(y), _bits(L.linear(x, w, b)))


@pytest.mark.parametrize("world", [2, 3, 4])
@pytest.mark.parametrize("M,N,K,dist", [(300, 520, 1000, "normal"), (2047, 1000, 776, "smallint"),
                                        (8, 2048, 4096, "normal"), (1, 1000, 1032, "normal"),
                                        (256, 4096, 4096, "normal")])
def test_row_split_rounds_once_after_the_reduction(world, M, N, K, dist):
    xh, wh, bh = synth.make_inputs(M, N, K, dist, 70 + world + M % 5)
    x, w, b = xh.to(DEV), wh.to(DEV), bh.to(DEV)
    S = torch.zeros((M, N), dtype=torch.float32, device=DEV)
    for r in range(world):  # the all-reduce, in rank order
        kb, ke = L.shard_range(K, world, r)
        if ke > kb:
            S += L.contract(x[:, kb:ke].contiguous(), w[:, kb:ke].contiguous(), None, out_f32=True)
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    rc = L.poot_linear_f16_finish(S.data_ptr(), b.data_ptr(), y.data_ptr(), M, N,
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == L.POOT_OK, L.poot_linear_status_string(rc)
    torch.cuda.synchronize()
    ok, rep = check_rows(_bits(y), _bits(xh), _bits(wh), _bits(bh), exact=dist == "smallint")
    assert ok, rep


def test_finish_is_the_linear_epilogue_on_a_given_sum():
    # exact sums (small integers): RN16(RN16(S) + b) equals the one-GPU call
    M, N, K = 130, 264, 200
    xh, wh, bh = synth.make_inputs(M, N, K, "smallint", 81)
    x, w, b = xh.to(DEV), wh.to(DEV), bh.to(DEV)
    S = L.contract(x, w, None, out_f32=True)
    for off in (0, 1):  # 16-byte aligned y and an odd element offset (scalar path)
        ybuf = torch.full((M * N + 1,), float("nan"), dtype=torch.float16, device=DEV)
        y = ybuf[off:off + M * N]
        rc = L.poot_linear_f16_finish(S.data_ptr(), b.data_ptr(), y.data_ptr(), M, N,
                                      torch.cuda.current_stream().cuda_stream)
        assert rc == L.POOT_OK
        torch.cuda.synchronize()
        assert np.array_equal(_bits(y.view(M, N)), _bits(L.linear(x, w, b)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, M, N, K, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import linear_fp16_gb300 as L
    from linear_fp16_gb300 import synth
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dev = torch.device("cuda", 0)
    x, w, b = (t.to(dev) for t in synth.make_inputs(M, N, K, "normal", 91))
    nb, ne = L.shard_range(N, world, rank)
    yc = L.column_parallel_linear(x, w[nb:ne].contiguous(), b[nb:ne].contiguous(), N)
    kb, ke = L.shard_range(K, world, rank)
    yr = L.row_parallel_linear(x[:, kb:ke].contiguous(), w[:, kb:ke].contiguous(), b, K)
    torch.cuda.synchronize()
    dist.destroy_process_group()
    out[rank] = (yc.cpu().view(torch.int16).numpy(), yr.cpu().view(torch.int16).numpy())


@pytest.mark.parametrize("world,M,N,K", [(2, 300, 1000, 520), (2, 8, 2048, 1024)])
def test_two_gloo_ranks_on_one_gpu(world, M, N, K):
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, M, N, K, out), nprocs=world, join=True, start_method="spawn")
    xh, wh, bh = synth.make_inputs(M, N, K, "normal", 91)
    ys = [out[r] for r in range(world)]
    for yc, yr in ys:
        for y in (yc, yr):
            ok, rep = check_rows(y.view(np.uint16), _bits(xh), _bits(wh), _bits(bh), exact=False)
            assert ok, rep
    # every rank holds the same result
    for yc, yr in ys[1:]:
        assert np.array_equal(yc, ys[0][0]) and np.array_equal(yr, ys[0][1])
