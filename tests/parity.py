"""The comparison rule, re-exported for the tests (it lives with the oracle,
in ``oracle/parity.py``, so that the benchmark's parity leg uses the same
rule)."""
from oracle.parity import U_RN, U_TRUNC, check_rows, compare, intervals, judge, legal_interval, ulp16  # noqa: F401
