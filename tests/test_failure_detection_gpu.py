"""Failure detection on the GPU without a fault: a bounded in-kernel wait that
nothing completes gives up, flags PD_DEVERR_TIMEOUT in the caller's error
word and returns; the context stays usable (a decode right after it matches
the oracle with a clean error word).  Bad inputs that the kernels check
(out-of-range slots, block ids, contexts) are covered by the op tests."""
import pytest
import torch

import pd_inputs
from tests.parity import assert_close, device_err, gpu_store_and_decode, oracle_store_and_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [1_000, 2_000_000])
def test_bounded_wait_times_out_and_context_survives(cuda_lib, limit_ns):
    pd = cuda_lib
    err = device_err()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    pd.pd_selftest_bounded_wait(err, limit_ns)
    b.record()
    torch.cuda.synchronize()
    assert err.item() == pd.PD_DEVERR_TIMEOUT
    assert a.elapsed_time(b) * 1e6 >= 0.9 * limit_ns - 5000      # it did wait (ns)
    # the context is intact: a normal step runs and is exact
    c = pd_inputs.tiny_decode()
    err2 = device_err()
    out, _, _ = gpu_store_and_decode(pd, c, dev_err=err2)
    torch.cuda.synchronize()
    ref, _, _ = oracle_store_and_decode(c)
    assert err2.item() == 0
    assert_close(out, ref, "decode after a timed-out wait")


def test_error_word_accumulates_and_other_bits_stay(cuda_lib):
    pd = cuda_lib
    err = torch.full((1,), pd.PD_DEVERR_SLOT_RANGE, dtype=torch.int32, device="cuda")
    pd.pd_selftest_bounded_wait(err, 10_000)
    torch.cuda.synchronize()
    assert err.item() == pd.PD_DEVERR_SLOT_RANGE | pd.PD_DEVERR_TIMEOUT
