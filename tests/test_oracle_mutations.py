"""The pins have teeth: each planted oracle mistake fails at least one pin.

The mistakes are compiled into separate copies of the oracle on the CPU
(ORACLE_MUTATION in oracle/oracle_linear.c); the product path is untouched.
"""
import numpy as np
import pytest

import oracle
from tests import exact

MUTATIONS = {
    1: "bias added before the projection rounding",
    2: "W read transposed",
    3: "last term of the sum dropped",
    4: "products rounded to FP16",
    5: "FP16 accumulator",
    6: "bias indexed by row",
    7: "bias subtracted",
}


def _pins_pass(mutation: int) -> bool:
    y = lambda x, w, b: oracle.linear_f16(x, w, b, mutation=mutation).view(np.float16).astype(np.float64)
    for name in ("round_before_bias.txt", "fp32_accumulation.txt", "no_product_rounding.txt",
                 "overflow_boundary.txt", "subnormal_rounding.txt"):
        x, w, b, want = exact.parse_golden(name)
        if not exact.same_values(y(x, w, b), want):
            return False
    rng = np.random.default_rng(3)
    for (M, N, K) in [(2, 3, 5), (3, 2, 7), (4, 4, 16)]:
        x = rng.integers(-4, 5, size=(M, K)).astype(np.float16)
        w = rng.integers(-4, 5, size=(N, K)).astype(np.float16)
        b = rng.integers(-4, 5, size=N).astype(np.float16)
        want = exact.exact_linear(x.view(np.uint16), w.view(np.uint16), b.view(np.uint16))
        if not exact.same_values(y(x, w, b), want):
            return False
    return True


def test_unmutated_oracle_passes_the_pins():
    assert _pins_pass(0)


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation):
    assert not _pins_pass(mutation), MUTATIONS[mutation]
