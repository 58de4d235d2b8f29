"""The MUFU throughput self-test returns a plausible rate (the bench reports
the softmax's exponentials against it)."""
import pytest

from ulysses_sequence_attention_seq_gb300 import binding as U

pytestmark = pytest.mark.gpu


def test_ex2_rate_is_plausible():
    rate = U.ulysses_selftest_ex2_rate()
    assert 4.0 < rate < 256.0, rate
