"""The in-kernel watchdog on the GPU: a wait that nothing completes gives up, the
host reads FA_ERR_DEVICE_TIMEOUT with the wait site, and the context stays usable.

The expired wait is the library's own self-test kernel (one warp waiting on an
mbarrier phase that nothing completes, bounded at about two seconds); no fault,
trap or unbounded loop is involved.
"""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import binding as b, inputs as I

from helpers import check_fwd, to_dev, to_f64

pytestmark = pytest.mark.gpu


def test_watchdog_reports_timeout_and_context_survives():
    import torch
    from tiled_attention_tmem_gb300 import api
    stream = torch.cuda.current_stream().cuda_stream
    assert b.fa_get_device_error(stream)[0] == b.FA_OK
    assert b.fa_watchdog_selftest(stream) == b.FA_OK
    status, site = b.fa_get_device_error(stream)
    assert status == b.FA_ERR_DEVICE_TIMEOUT
    assert site == (6 << 8) | 1
    # Reading the status cleared it, and kernels launched afterwards compute normally.
    assert b.fa_get_device_error(stream)[0] == b.FA_OK
    x = I.make_inputs(1, 2, 256, 128, seed=77)
    q, k, v = (to_dev(t) for t in (x.q, x.k, x.v))
    o, lse = api.attention_forward(q, k, v, 128 ** -0.5, True)
    api.check_device_error()
    qf, kf, vf, _ = x.as_f64()
    o_ref, lse_ref = oracle.forward(qf, kf, vf, 128 ** -0.5, True)
    check_fwd(to_f64(o), to_f64(lse), o_ref, lse_ref, "after watchdog self-test")


def test_kernels_skip_work_while_the_error_word_is_set():
    """Between the expired wait and the host reading it, later launches exit at once
    (they see the error word) instead of computing on a poisoned device state."""
    import torch
    from tiled_attention_tmem_gb300 import api
    stream = torch.cuda.current_stream().cuda_stream
    x = I.make_inputs(1, 1, 128, 64, seed=78)
    q, k, v = (to_dev(t) for t in (x.q, x.k, x.v))
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 1, 128), 7.0, dtype=torch.float32, device=q.device)
    assert b.fa_watchdog_selftest(stream) == b.FA_OK
    api.attention_forward(q, k, v, 0.125, False, out=o, lse=lse)
    # the split-KV forward's part and merge kernels skip as well
    api.attention_forward(q, k, v, 0.125, False, out=o, lse=lse, splits=2)
    status, _ = b.fa_get_device_error(stream)
    assert status == b.FA_ERR_DEVICE_TIMEOUT
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
