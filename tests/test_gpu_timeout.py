"""The bounded waits' timeout path on the GPU, without any fault: one wait on a barrier that
expects bytes no copy delivers gives up after a short limit and reports SV_ST_TIMEOUT; the copy
that was issued lands first; the device then runs verification as usual."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def test_a_wait_that_cannot_complete_reports_timeout(sv):
    st = sv.selftest_wait_timeout(2_000_000)  # about a millisecond of SM cycles
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [sv.ST_TIMEOUT, 1]
    # the context is healthy: a verify call right after matches the oracle
    w = workloads.tiny_greedy()
    got = sv.verify_greedy(w["target"], w["R"], w["k"], 1, w["draft"])
    torch.cuda.synchronize()
    want = oracle.verify_greedy(workloads.host_rows(w["target"]), w["R"], w["k"], 1, w["draft"].cpu().numpy())
    for key in ("accept_len", "tokens", "status"):
        np.testing.assert_array_equal(got[key].cpu().numpy(), want[key], err_msg=key)


def test_timeout_limit_argument_is_checked(sv):
    lib = sv.load()
    buf = torch.zeros(8, dtype=torch.int32, device="cuda")
    import ctypes as C

    assert lib.sv_selftest_wait_timeout(C.c_void_p(buf.data_ptr()), C.c_void_p(buf.data_ptr()), 0, None) == -1
    assert lib.sv_selftest_wait_timeout(C.c_void_p(buf.data_ptr() + 4), C.c_void_p(buf.data_ptr()), 10, None) == -7
