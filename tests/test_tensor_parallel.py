"""The tensor-parallel linear's host side, on the CPU.

* The shard plan (poot_linear_tp_shard, host logic of the C library):
  contiguous ranges covering the axis in rank order, 8-element multiples
  but the last, balanced, argument errors.
* Two gloo ranks run the collectives of linear_fp16_gb300.tensor_parallel
  on CPU tensors, with each rank's local step computed by the oracle (the
  kernels need a GPU; they are checked in tests/test_gpu_tensor_parallel.py):
  the column split gathers the oracle's column shards into exactly the
  one-device result, and the row split's all-reduced FP32 partial sums,
  rounded once, give a result within the contract's rule of the oracle's
  ("Model and Distributed IR", "Boundary between the layers": the
  reconstructed result equals the source semantics).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import linear_fp16_gb300 as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("extent", [0, 1, 7, 8, 9, 63, 1000, 4096, 14336, 2047])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_shard_plan_covers_the_axis(extent, world):
    ranges = [L.shard_range(extent, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == extent
    for (b0, e0), (b1, e1) in zip(ranges, ranges[1:]):
        assert e0 == b1 and b0 <= e0
    widths = [e - b for b, e in ranges]
    # every shard that ends before the axis does is a multiple of 8 wide
    assert all((e - b) % 8 == 0 for b, e in ranges if e < extent)
    assert max(widths) <= max(8, -(-extent // world) + 7)


@pytest.mark.parametrize("args", [(-1, 2, 0), (8, 0, 0), (8, 2, 2), (8, 2, -1), (1 << 31, 2, 0), (8, 65537, 0)])
def test_shard_plan_argument_errors(args):
    rc, _, _ = L.poot_linear_tp_shard(*args)
    assert rc == L.POOT_ERR_INVALID_ARG


def test_gather_and_finish_argument_errors_before_any_cuda_call():
    S, Y = 0x1000_0000, 0x4000_0000  # never dereferenced
    assert L.poot_linear_gather_columns(S, Y, 4, 16, 2, 4 * 8 - 1, 0) == L.POOT_ERR_INVALID_ARG  # slot too small
    assert L.poot_linear_gather_columns(0, Y, 4, 16, 2, 32, 0) == L.POOT_ERR_INVALID_ARG
    assert L.poot_linear_gather_columns(S + 1, Y, 4, 16, 2, 32, 0) == L.POOT_ERR_MISALIGNED
    assert L.poot_linear_gather_columns(S, S + 64, 4, 16, 2, 32, 0) == L.POOT_ERR_INVALID_ARG  # overlap
    assert L.poot_linear_gather_columns(S, Y, 4, 16, 0, 32, 0) == L.POOT_ERR_INVALID_ARG
    assert L.poot_linear_gather_columns(0, 0, 0, 16, 2, 0, 0) == L.POOT_OK
    B = 0x2000_0000
    assert L.poot_linear_f16_finish(S + 2, B, Y, 4, 16, 0) == L.POOT_ERR_MISALIGNED
    assert L.poot_linear_f16_finish(S, 0, Y, 4, 16, 0) == L.POOT_ERR_INVALID_ARG
    assert L.poot_linear_f16_finish(S, B, S + 64, 4, 16, 0) == L.POOT_ERR_INVALID_ARG  # y overlaps S
    assert L.poot_linear_f16_finish(S, B, B + 16, 4, 16, 0) == L.POOT_ERR_INVALID_ARG  # y overlaps b
    assert L.poot_linear_f16_finish(0, 0, 0, 0, 16, 0) == L.POOT_OK


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bits(t):
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _rank_main(rank, world, port, M, N, K, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle
    from linear_fp16_gb300 import synth, tensor_parallel as tp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x, w, b = synth.make_inputs(M, N, K, "normal", 31)
    # column split: this rank's rows of W and b, the oracle as the local step
    nb, ne = tp.shard_range(N, world, rank)
    w0b, w0e = tp.shard_range(N, world, 0)
    slot = M * (w0e - w0b)
    local = torch.zeros(slot, dtype=torch.float16)
    if ne > nb:
        yr = oracle.linear_f16(_bits(x), _bits(w[nb:ne]), _bits(b[nb:ne]))
        local[:M * (ne - nb)] = torch.from_numpy(yr.view(np.float16).reshape(-1))
    gathered = _bits(tp.all_gather_slots(local))
    y = np.zeros((M, N), np.uint16)
    for r in range(world):  # the layout poot_linear_gather_columns reads
        rb, re = tp.shard_range(N, world, r)
        y[:, rb:re] = gathered[r * slot:r * slot + M * (re - rb)].reshape(M, re - rb)
    # row split: this rank's columns of x and W, FP32 partial sums from the oracle
    kb, ke = tp.shard_range(K, world, rank)
    S = torch.zeros((M, N), dtype=torch.float32)
    if ke > kb:
        S = torch.from_numpy(oracle.contraction(_bits(x[:, kb:ke].contiguous()), _bits(w[:, kb:ke].contiguous()),
                                                None, out_f32=True))
    tp.all_reduce_sum(S)
    dist.destroy_process_group()
    out[rank] = (y, S.numpy())


@pytest.mark.parametrize("world,M,N,K", [(2, 24, 200, 136), (3, 17, 64, 520)])
def test_gloo_collectives_reconstruct_the_one_device_result(world, M, N, K):
    import oracle
    from linear_fp16_gb300 import synth
    from tests.parity import check_rows
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, M, N, K, out), nprocs=world, join=True)
    x, w, b = synth.make_inputs(M, N, K, "normal", 31)
    y_one = oracle.linear_f16(_bits(x), _bits(w), _bits(b))
    for r in range(world):
        y, S = out[r]
        assert np.array_equal(y, y_one)           # column split: bit-identical
        # row split: one rounding of the FP32 sum, then the bias
        p = oracle.f32_to_f16_rn(S.astype(np.float32)).reshape(M, N)
        yk = oracle.f32_to_f16_rn(oracle.f16_to_f32(p).reshape(M, N) + oracle.f16_to_f32(_bits(b))[None, :])
        ok, rep = check_rows(yk.reshape(M, N), _bits(x), _bits(w), _bits(b), exact=False)
        assert ok, rep
