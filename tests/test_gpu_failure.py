"""Failure behaviour on the GPU without a fault: a bounded wait that nothing
completes gives up, reports PA_DEV_ERR_TIMEOUT through the error word, and the
kernel returns; the context stays usable (a decode step afterwards still
matches the oracle). Device-side bad data is covered where it arises (bad
block ids, slots, pairs and lengths in the decode, cache and prefill tests)."""
import time

import numpy as np
import pytest
import torch

from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import workloads as W
from tests.helpers import bits, compare, gpu_step, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("limit_ms", [1, 20])
def test_bounded_wait_gives_up_and_reports(limit_ms):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = B.lib().pa_check_bounded_wait(err.data_ptr(), limit_ms * 1_000_000, None)
    assert st == B.PA_OK
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) & B.PA_DEV_ERR_TIMEOUT
    assert dt >= limit_ms * 1e-3 * 0.9      # it did wait
    assert dt < limit_ms * 1e-3 + 1.0       # and it gave up
    # the context is still usable: a decode step matches the oracle
    wl = W.custom([1, 17, 300], n_q_heads=8, n_kv_heads=2, seed=3, name="after-timeout")
    vals_cpu = W.make_values(wl, poison_tails=True)
    ref, kp, vp = oracle_step(wl, vals_cpu)
    vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
    out, e = gpu_step(wl, vals)
    assert e == 0
    assert np.array_equal(bits(vals["k_pool"]), kp)
    compare(out, ref, wl.name)
