"""Failure detection on the GPU, without a fault: a kernel whose bounded mbarrier
wait expires reports LAGA_ERR_TIMEOUT through laga_mla_check (with the wait
site), the check clears the status word, and the same context then runs a
forward + backward that still matches the oracle."""
import pytest
import torch

from mla_attention_sequence_gb300 import laga
from mla_attention_sequence_gb300.synth import make_inputs

from test_parity_gpu import TC_CASES, TOL, assert_close, built, dev, run_gpu, run_oracle  # noqa: F401

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    d = dev()
    laga.check(d)  # nothing pending from earlier tests
    laga.selftest_timeout(d)
    with pytest.raises(laga.LagaError) as err:
        laga.check(d)
    assert err.value.status == 5, err.value
    assert "site 99" in str(err.value)
    laga.check(d)  # the check cleared the word
    p = TC_CASES["multi_tile"]
    x = make_inputs(p, seed=12)
    assert_close(run_gpu(p, x, "materialize"), run_oracle(p, x), TOL["bf16"], tag="after an expired wait")
    laga.check(d)
