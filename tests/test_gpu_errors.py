"""GPU checks of the device error word: the bounded waits give up and report
SMLA_DEV_TIMEOUT without losing the context, and the stream-ordered read
returns what the work queued before it on its stream set, without waiting for
other streams.

The waits here run out because nothing arrives on an mbarrier that only the
self-test kernel itself may arrive on, with a limit the host sets (a few
milliseconds); nothing faults, traps or hangs."""

import numpy as np
import pytest
import torch

from sparse_mla_decode_gb300 import smla, workloads
from tests.gpu_helpers import compare, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_word():
    assert smla.smla_device_error() == 0  # nothing left over from earlier tests
    yield
    smla.smla_device_error()


def test_a_wait_that_nothing_completes_gives_up_and_reports_a_timeout():
    side = torch.cuda.Stream()
    smla.smla_selftest_bounded_wait(False, 2_000_000, stream=side)  # 2 ms
    assert smla.smla_read_device_error(side) == smla.DEV_TIMEOUT
    assert smla.smla_read_device_error(side) == 0  # the read cleared it
    smla.smla_selftest_bounded_wait(True, 2_000_000, stream=side)
    assert smla.smla_read_device_error(side) == 0


def test_the_context_stays_usable_after_a_wait_gave_up():
    smla.smla_selftest_bounded_wait(False, 1_000_000)
    assert smla.smla_read_device_error() == smla.DEV_TIMEOUT
    w = workloads.tiny()
    d = to_device(w)
    out, lse = smla.decode(d["q"], d["pools"], d["indices"], d["lens"], d["sinks"], w["bmm1_scale"],
                           w["bmm2_scale"], w["k_scale"])
    assert smla.smla_read_device_error() == 0
    compare(w, out.float().cpu().numpy(), out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy())


def test_a_stream_ordered_read_sees_its_own_streams_bits():
    w = workloads.small("oob", seed=7, tokens=1, heads=16, width=64, head_dim=576, pool_rows=100)
    w["indices"][0, 10] = 100  # one past the last row
    d = to_device(w)
    torch.cuda.synchronize()
    s1 = torch.cuda.Stream()
    with torch.cuda.stream(s1):
        smla.decode(d["q"], d["pools"], d["indices"], d["lens"], None, w["bmm1_scale"], w["bmm2_scale"],
                    w["k_scale"], stream=s1)
    assert smla.smla_read_device_error(s1) == smla.DEV_INDEX_RANGE
    assert smla.smla_read_device_error(s1) == 0


def test_a_stream_ordered_read_does_not_wait_for_other_streams():
    busy, reader = torch.cuda.Stream(), torch.cuda.Stream()
    done = torch.cuda.Event()
    smla.smla_selftest_bounded_wait(False, 300_000_000, stream=busy)  # gives up after 0.3 s
    done.record(busy)
    # the busy stream's wait has not given up yet, so its bit is not there
    assert smla.smla_read_device_error(reader) == 0
    assert not done.query(), "the read waited for another stream"
    busy.synchronize()
    assert smla.smla_read_device_error(reader) == smla.DEV_TIMEOUT
