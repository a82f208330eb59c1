"""sv_verify_greedy_noalloc, the greedy entry point for callers that cannot
allocate device memory (a plugin inside a framework that owns the GPU's
memory pool, or a decode loop that may not allocate while serving).

The call goes straight through the C ABI with ctypes and must give exactly
the tokens, accept lengths, branches and status of sv_verify_greedy (which
takes a caller-allocated workspace) on two calls in a row.  This file is
collected last so a run that stops at the first failure has run the rest.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

SV_ERR_LIMIT = -4


def _entry(lib):
    import serving_sampler_gb300 as m

    fn = lib.sv_verify_greedy_noalloc
    P, i32 = C.c_void_p, C.c_int32
    fn.argtypes = [m.SvRows, i32, i32, i32, P, P, P, P, P, P]
    fn.restype = C.c_int
    return fn


def _p(t):
    return C.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_on_two_calls(sv):
    lib = sv.load()
    fn = _entry(lib)
    cases = [(24, 9, 2, 151936, torch.bfloat16, 11), (7, 40, 1, 4100, torch.float32, 12)]
    for R, k, branches, V, dtype, seed in cases:
        w = workloads.greedy_batch(R, k, V, dtype, branches=branches, p_full=0.6, p_first=0.5, seed=seed)
        want = sv.verify_greedy(w["target"], R, k, branches, w["draft"])
        got = {name: torch.full_like(t, -7) for name, t in want.items()}
        stream = torch.cuda.current_stream()
        rc = fn(sv.rows_of(w["target"]), R, k, branches, _p(w["draft"]), _p(got["accept_len"]),
                _p(got["tokens"]), _p(got["branch"]), _p(got["status"]), C.c_void_p(stream.cuda_stream))
        assert rc == 0, lib.sv_status_string(rc)
        torch.cuda.synchronize()
        for name in ("accept_len", "tokens", "branch", "status"):
            np.testing.assert_array_equal(got[name].cpu().numpy(), want[name].cpu().numpy(), err_msg=name)


def test_noalloc_rejects_batches_larger_than_its_scratch(sv):
    lib = sv.load()
    fn = _entry(lib)
    t = torch.zeros(2, 151936, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(4, dtype=torch.int32, device="cuda")
    R, k = 20000, 32  # workspace of about 200 MB, far above the fixed array
    assert lib.sv_verify_greedy_workspace(R, k, 2, 151936) > (8 << 20)
    rc = fn(sv.rows_of(t), R, k, 2, _p(i), _p(i), _p(i), None, None, None)
    assert rc == SV_ERR_LIMIT
