"""Failure handling on the GPU without a fault or a hang: the kernel's
pipeline waits are bounded. With the wait limit cut to 1 ns
(LF_WAIT_LIMIT_NS, a diagnostic), the waits give up before the copies land;
the kernel must report LF_DEVERR_WAIT_TIMEOUT in the device error word,
still retire (every copy in flight is drained with the full limit), and leave
the context usable: the next call with the normal limit is correct."""
import numpy as np
import pytest

import decode_kv_cache_step_gb300 as lf

import _pins
from test_gpu_edges import check_case

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_context_stays_usable(monkeypatch):
    rng = np.random.default_rng(77)
    case = _pins.rand_case(rng, 4, 32, 8, 128, 4096, p_masked=0.1, max_age=9000)
    import torch
    from _gpu import DevState
    lf.device_errors(clear=True)
    monkeypatch.setenv("LF_WAIT_LIMIT_NS", "1")
    dev = DevState(case["k_cache"], case["v_cache"], case["mask"], 32)
    dev.step(case["q"], case["new_k"], case["new_v"], case["write_slot"], 16, 0.088)
    torch.cuda.synchronize()
    flags = lf.device_errors(clear=True)
    assert flags & lf.LF_DEVERR_WAIT_TIMEOUT
    monkeypatch.delenv("LF_WAIT_LIMIT_NS")
    check_case(case, W=16, scale=0.088, where="after a timed-out call")
    assert lf.device_errors(clear=True) == 0
