"""Failure detection without a GPU fault: the bounded mbarrier wait that every kernel uses gives up
after its limit, records the site in the device error word and returns; the host sees DIT_ETIMEOUT
at the next dit_check and the context keeps working."""

import time

import numpy as np
import pytest
import torch

import diffusion_transformer_gb300 as D
import oracle as O

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_leaves_the_context_usable():
    D.dit_check()                           # start from a clear error word
    D.dit_selftest_bounded_wait(True)       # the barrier completes: no error
    D.dit_check()
    t0 = time.time()
    D.dit_selftest_bounded_wait(False)      # nothing completes the barrier
    with pytest.raises(D.DitError) as e:
        D.dit_check()
    elapsed = time.time() - t0
    assert e.value.status == D.DIT_ETIMEOUT
    assert 0.9 <= elapsed < 30, elapsed     # the 1 s limit, not an endless wait
    D.dit_check()                           # dit_check cleared the word
    g = np.random.default_rng(0)
    x = g.standard_normal((4096, 64), dtype=np.float32)
    v = g.standard_normal((4096, 64), dtype=np.float32)
    xd, vd = torch.from_numpy(x).cuda(), torch.from_numpy(v).cuda()
    D.dit_euler_step(xd, vd, 0.75, 0.5)
    D.dit_check()
    assert np.array_equal(xd.cpu().numpy(), O.euler_step(x, v, 0.75, 0.5))
