"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side argument checks answer without touching a GPU."""
import ctypes as C
import os
import re
import shutil

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "specverify.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from serving_sampler_gb300 import _build

    _build.build()
    import serving_sampler_gb300 as m

    return m.load()


def test_binding_constants_match_the_header():
    import serving_sampler_gb300 as m

    text = open(HEADER).read()
    st = dict(re.findall(r"SV_(ST_[A-Z_0-9]+)\s*=\s*(\d+)", text))
    for name, v in st.items():
        assert getattr(m, name) == int(v), name
    limits = {}
    for name, v in re.findall(r"#define SV_(MAX_[A-Z]+)\s+(\(?[0-9 <]+\)?)", text):
        a, _, b = v.strip("() ").partition("<<")
        limits[name] = int(a) << int(b) if b else int(a)
    for name in ("MAX_K", "MAX_S", "MAX_NGRAM", "MAX_POOL"):
        assert getattr(m, name) == limits[name], name


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ["sv_verify_greedy", "sv_verify_sample", "sv_cfg_merge_sample", "sv_accept_scan"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in specverify.h but not exported"


def test_every_exported_entry_point_is_declared(lib):
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    import serving_sampler_gb300 as m
    import subprocess

    out = subprocess.run([nm, "-D", "--defined-only", m.LIB_PATH], capture_output=True, text=True, check=True)
    exported = sorted({line.split()[-1] for line in out.stdout.splitlines()
                       if line.split()[-1].startswith("sv_") and " T " in line})
    assert exported == _declared()


def test_status_strings(lib):
    for code in range(0, -9, -1):
        s = lib.sv_status_string(code)
        assert s and s != b"unknown status"
    assert lib.sv_status_string(12345) == b"unknown status"


def test_workspace_sizes(lib):
    assert lib.sv_verify_greedy_workspace(64, 32, 2, 151936) >= 64 * 65 * 16
    assert lib.sv_verify_greedy_workspace(-1, 2, 1, 10) == 0
    assert lib.sv_verify_greedy_workspace(1, 2, 9, 10) == 0  # more branches than SV_MAX_BRANCHES
    assert lib.sv_verify_greedy_workspace(1, 2, 0, 10) == 0
    assert lib.sv_verify_greedy_workspace(1, 2, 8, 10) > 0  # eight branches: 1 + 8 * 2 rows
    assert lib.sv_verify_sample_workspace(128, 7, 151936, 32000) > 0
    assert lib.sv_cfg_merge_sample_workspace(256, 4, 9, 4096) > 0
    assert lib.sv_cfg_merge_sample_workspace(1, 1, 17, 4096) == 0


def _rows(data=0x1000, dtype=0, width=16, stride=16):
    import serving_sampler_gb300 as m

    return m.SvRows(data, dtype, width, stride)


def test_argument_checks_need_no_gpu(lib):
    P = C.c_void_p
    buf = P(0x10000)
    ws = P(0x20000)
    g = lib.sv_verify_greedy
    # R == 0 is a no-op
    assert g(_rows(), 0, 2, 1, buf, buf, buf, None, None, ws, 1 << 20, None) == 0
    assert g(_rows(), -1, 2, 1, buf, buf, buf, None, None, ws, 1 << 20, None) == -1
    assert g(_rows(), 1, 2, 0, buf, buf, buf, None, None, ws, 1 << 20, None) == -1
    assert g(_rows(), 1, 2, 9, buf, buf, buf, None, None, ws, 1 << 20, None) == -4  # SV_ERR_LIMIT
    assert g(_rows(), 1, 0, 2, buf, buf, buf, None, None, ws, 1 << 20, None) == -1
    assert g(_rows(), 1, 257, 1, buf, buf, buf, None, None, ws, 1 << 20, None) == -4
    assert g(_rows(dtype=7), 1, 2, 1, buf, buf, buf, None, None, ws, 1 << 20, None) == -2
    assert g(_rows(stride=8), 1, 2, 1, buf, buf, buf, None, None, ws, 1 << 20, None) == -3
    assert g(_rows(data=0x1001), 1, 2, 1, buf, buf, buf, None, None, ws, 1 << 20, None) == -7
    assert g(_rows(), 1, 2, 1, None, buf, buf, None, None, ws, 1 << 20, None) == -1
    assert g(_rows(), 1, 2, 1, buf, buf, buf, None, None, ws, 16, None) == -6
    assert g(_rows(), 1, 2, 1, buf, buf, buf, None, None, P(0x20010), 1 << 20, None) == -6
    s = lib.sv_accept_scan
    assert s(buf, buf, buf, -2, 3, buf, buf, None) == -1
    assert s(buf, buf, buf, 0, 3, buf, buf, None) == 0
    assert s(buf, buf, None, 2, 3, buf, buf, None) == -1
    pa, pl = lib.sv_pool_append, lib.sv_pool_lookup
    assert pa(buf, buf, 64, buf, 4, 0, None, None) == 0
    assert pa(buf, buf, 64, buf, 4, -1, None, None) == -1
    assert pa(buf, buf, 64, buf, 257, 1, None, None) == -4
    assert pa(buf, buf, (1 << 24) + 1, buf, 4, 1, None, None) == -4
    assert pa(buf, None, 64, buf, 4, 1, None, None) == -1
    assert pa(P(0x10002), buf, 64, buf, 4, 1, None, None) == -7
    assert pl(buf, buf, 64, buf, 4, 0, 8, buf, buf, None) == 0
    assert pl(buf, buf, 64, buf, 65, 1, 8, buf, buf, None) == -4  # N above SV_MAX_NGRAM
    assert pl(buf, buf, 64, buf, 4, 1, 257, buf, buf, None) == -4
    assert pl(buf, buf, 64, None, 4, 1, 8, buf, buf, None) == -1
    assert pl(buf, buf, 64, buf, 4, 1, 8, buf, None, None) == -1
    assert pl(buf, buf, 64, buf, 4, 1, -1, buf, buf, None) == -1
    sa = lib.sv_suffix_append
    assert sa(buf, 8, 0, buf, buf, 4, None) == 0
    assert sa(buf, 0, 3, buf, buf, 4, None) == 0
    assert sa(buf, 65, 1, buf, buf, 4, None) == -4
    assert sa(buf, 8, 1, buf, buf, 257, None) == -4
    assert sa(buf, 8, 1, None, buf, 4, None) == -1
    assert sa(buf, -1, 1, buf, buf, 4, None) == -1
    st = lib.sv_selftest_wait_timeout
    st.argtypes = [P, P, C.c_int64, P]
    assert st(buf, buf, 0, None) == -1          # the wait's limit must be positive
    assert st(P(0x10004), buf, 10, None) == -7  # the copy source must be 16-byte aligned
    c = lib.sv_cfg_merge_sample
    base = (C.c_int32 * 2)(0, 16)
    assert c(_rows(), _rows(width=8), C.cast(base, P), None, 2, 3.0, _rows(data=None), 1, 1, buf, buf, buf, buf,
             buf, None, None, ws, 1 << 20, None) == -3
    assert c(_rows(), _rows(), C.cast(base, P), None, 17, 3.0, _rows(data=None), 1, 1, buf, buf, buf, buf,
             buf, None, None, ws, 1 << 20, None) == -4


def test_sampling_limits_need_no_gpu(lib):
    P = C.c_void_p
    buf = P(0x10000)
    ws = P(0x20000)
    smp = lib.sv_verify_sample

    def call(target, R, k, d2t=None, plan=None, draft_rows=None):
        return smp(target, draft_rows or _rows(width=target.width), d2t, plan, R, k, buf, buf, buf, buf, buf,
                   None, None, None, None, ws, 1 << 30, None)

    # identity map, vocabulary above the race's chunk-table limit (819,200 ids)
    wide = _rows(width=819208, stride=819208)
    assert call(wide, 1, 1) == -4
    # R * (k + 1) must stay below 2^31
    assert call(_rows(), 1 << 24, 255) == -4
    # a d2t plan must be 256-byte aligned
    assert call(_rows(), 1, 1, d2t=buf, plan=P(0x20010), draft_rows=_rows(width=8)) == -6
    # the plan calls reject impossible sizes before anything runs
    assert lib.sv_d2t_plan_bytes(0, 5) == 0
    assert lib.sv_d2t_plan_build(buf, 70000, 151936, ws, 1 << 30, None) == -4


def test_binding_fails_loudly_without_library(tmp_path):
    import serving_sampler_gb300 as m

    saved = m._lib
    m._lib = None
    try:
        with pytest.raises(RuntimeError):
            m.load(str(tmp_path / "missing.so"))
    finally:
        m._lib = saved


def test_valid_call_without_device_reports_no_device(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    P = C.c_void_p
    buf = P(0x10000)
    rc = lib.sv_verify_greedy(_rows(), 1, 2, 1, buf, buf, buf, None, None, P(0x20000), 1 << 20, None)
    assert rc == -8


def test_noalloc_argument_errors_match_the_workspace_entry(lib):
    """sv_verify_greedy_noalloc answers every argument error with sv_verify_greedy's code, in
    sv_verify_greedy's order (no GPU is touched before the arguments pass)."""
    P = C.c_void_p
    buf = P(0x10000)
    ws = P(0x20000)
    g, na = lib.sv_verify_greedy, lib.sv_verify_greedy_noalloc
    cases = [
        (_rows(), 0, 2, 1, buf),            # R == 0: a no-op
        (_rows(), -1, 2, 1, buf),
        (_rows(), 1, 2, 0, buf),
        (_rows(), 1, 2, 9, buf),            # more branches than SV_MAX_BRANCHES: SV_ERR_LIMIT
        (_rows(), 1, 0, 2, buf),
        (_rows(), 1, 257, 1, buf),
        (_rows(), -1, 2, 9, buf),           # two errors: the first check decides
        (_rows(dtype=7), 1, 257, 1, buf),
        (_rows(dtype=7), 1, 2, 1, buf),
        (_rows(stride=8), 1, 2, 1, buf),
        (_rows(data=0x1001), 1, 2, 1, buf),
        (_rows(), 1, 2, 1, None),           # no draft tokens
        (_rows(), 1, 2, 1, P(0x10002)),     # misaligned draft tokens
    ]
    for t, R, k, br, d in cases:
        want = g(t, R, k, br, d, buf, buf, None, None, ws, 1 << 30, None)
        assert want != 0 or R == 0
        assert na(t, R, k, br, d, buf, buf, None, None, None) == want, (R, k, br)
