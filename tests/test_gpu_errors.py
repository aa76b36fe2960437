"""Failure detection on the GPU without a fault: the device error word that a
kernel's bounded wait writes when it runs out, read back by
gdr_check_device (GDR_DEVICE_TIMEOUT), both injected from the host and
produced by a real bounded wait on a barrier that nothing completes.  The
context stays usable afterwards."""
import pytest
import torch

import synth
from gpu_util import SCALE, assert_within, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdr():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import gated_delta_rule_varlen_gb300 as m
    m.load()
    m.gdr_check_device()  # start from a clean error word
    return m


def _small_parity():
    lengths = [100, 37]
    x = synth.make_inputs("kda", sum(lengths), 1, 1, 128, seed=21)
    cu = synth.cu_from_lengths(lengths)
    print(assert_within(compare(run_gpu("kda", x, cu), run_oracle(x, cu))))


def test_injected_error_word_is_reported_once(gdr):
    gdr.gdr_inject_device_error(9)
    with pytest.raises(gdr.GdrError) as ei:
        gdr.gdr_check_device()
    assert ei.value.status == gdr.GDR_DEVICE_TIMEOUT
    gdr.gdr_check_device()  # the report cleared the word


def test_bounded_wait_runs_out_and_the_context_survives(gdr):
    gdr.gdr_selftest_wait(5_000_000)  # 5 ms on a barrier that nothing completes
    with pytest.raises(gdr.GdrError) as ei:
        gdr.gdr_check_device()
    assert ei.value.status == gdr.GDR_DEVICE_TIMEOUT
    gdr.gdr_check_device()
    _small_parity()
