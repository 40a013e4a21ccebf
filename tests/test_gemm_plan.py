"""The GEMM's tile plan (poot_linear_gemm_plan: host logic of the C library,
no GPU): which decomposition each configured shape gets on a 152-SM part,
and the argument errors.  The plans' results are checked on the GPU by the
parity tests; these pin the choices the measurements in the design notes
were taken with."""
import pytest

import linear_fp16_gb300 as L


@pytest.mark.parametrize("M,N,K,want", [
    # toy: one wave of 128 x 64 single-CTA tiles (short K: pairs lose)
    (1024, 1024, 768, {"cluster": 1, "tile_n": 64, "split_k": 1, "tiles": 128}),
    # prefill: CTA pairs, 224-wide tiles, exactly four waves of 76 pairs
    (4096, 4096, 4096, {"cluster": 2, "tile_n": 224, "split_k": 1, "tiles": 304}),
    # MLP up-projection: CTA pairs, full 256-wide tiles
    (8192, 14336, 4096, {"cluster": 2, "tile_n": 256, "split_k": 1}),
    # small M, long K: split-K fills the SMs
    (64, 4096, 4096, {"cluster": 1, "split_k": 4}),
])
def test_plans_of_the_configured_shapes(M, N, K, want):
    rc, plan = L.poot_linear_gemm_plan(M, N, K)
    assert rc == L.POOT_OK
    for k, v in want.items():
        assert plan[k] == v, (k, plan)
    assert plan["k_chunk"] == 1024 and plan["ctas"] == 152


def test_plan_argument_errors():
    assert L.poot_linear_gemm_plan(0, 8, 8)[0] == L.POOT_ERR_INVALID_ARG
    assert L.poot_linear_gemm_plan(8, 8, 1 << 31)[0] == L.POOT_ERR_INVALID_ARG
    assert L.poot_linear_gemm_plan(8, 8, 8, sm_count=1)[0] == L.POOT_ERR_INVALID_ARG
