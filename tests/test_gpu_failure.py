"""Failure detection on the GPU without a fault: the bounded wait that every
kernel uses gives up on a barrier that nothing completes, the host reads
PA_ERR_TIMEOUT from the device error word, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

from paged_kv_cache_174_gb300 import ops
from paged_kv_cache_174_gb300 import workloads as W

from gpu_util import assert_attn_close, run_gpu_step, run_oracle_step, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    ops.check_device_errors()  # start clean
    t0 = time.perf_counter()
    ops.selftest_wait_timeout(5_000_000)  # 5 ms
    with pytest.raises(ops.PagedAttnError) as ei:
        ops.check_device_errors()
    assert ei.value.code == 5  # PA_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    ops.check_device_errors()  # the word was cleared by the read


def test_context_is_usable_after_a_timeout():
    ops.selftest_wait_timeout(2_000_000)
    with pytest.raises(ops.PagedAttnError):
        ops.check_device_errors()
    b = W.make_batch("after-timeout", [300, 17], [1, 1], num_q_heads=8, num_kv_heads=2,
                     head_dim=64, block_size=16, num_blocks=40, seed=2)
    _, out = run_gpu_step(b)
    _, _, ref = run_oracle_step(b)
    assert_attn_close(to_f64(out), ref, "decode after a timed-out wait")
