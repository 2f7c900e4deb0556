"""Device-side failure detection, made to fire without faulting the GPU.

The tensor-core kernels bound every mbarrier wait: on expiry (or when the
CTA's abort flag is up) they record OS2_ERR_TIMEOUT in the device status word
and return.  os2_wait_selftest runs those same waits on an mbarrier that no
thread arrives at, with a limit of a few milliseconds.  The test reads the
status word from the host, then checks that the context still runs the whole
path bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import rns_emulated_fp64_gb300 as os2
import workloads
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit", [100_000, 4_000_000])
def test_bounded_wait_gives_up_and_status_reaches_host(limit):
    assert os2.get_status() == 0, "status word not clear before the test"
    res = os2.wait_selftest(limit)
    assert res[0] == 1, "a satisfied wait did not complete"
    assert res[1] == 1, "an unsatisfied wait did not give up"
    assert res[2] == 1, "an unsatisfied cluster-scope wait did not give up"
    assert res[3] == 1, "a raised abort flag did not end the wait"
    assert res[4] == 1, "the wait gave up before its limit"
    assert res[5:] == [0, 0, 0]
    assert os2.get_status() == os2.ERR_TIMEOUT
    assert os2.get_status() == 0, "reading the status word clears it"


def test_context_usable_after_timeout():
    os2.wait_selftest(1_000_000)
    assert os2.get_status() == os2.ERR_TIMEOUT
    A, Bt = workloads.make_pair("spread", 300, 260, 700, seed=5, phi=1.0)
    C = os2.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda(), 16, "fast")
    assert os2.get_status() == 0
    ref = orc.gemm_entries(A, Bt, 16, want_X=False, want_c=False, want_G=False)
    assert np.array_equal(C.cpu().numpy().view(np.uint64), ref.C.view(np.uint64))
