"""serving_sampler_gb300 -- Python binding of the specverify C library.

The binding only marshals arguments: it turns torch tensors into raw device
pointers and sizes, calls the C entry points of ``libspecverify.so`` through
ctypes on the current CUDA stream, and raises on a non-zero return code.
Every step of verification runs in the library's CUDA kernels; there is no
fallback.  If the library has not been built, ``load()`` raises.

Entry points (same names as the C ABI in include/specverify.h):
  verify_greedy, verify_sample, cfg_merge_sample, accept_scan
"""
from __future__ import annotations

import ctypes as C
import os

from . import _build

LIB_PATH = _build.LIB

SV_BF16, SV_F32 = 0, 1
ST_TOKEN_RANGE, ST_BAD_LOGITS, ST_OFF_SUPPORT, ST_RESIDUAL_ZERO = 1, 2, 4, 8
ST_BAD_TEMP, ST_BAD_D2T, ST_TIMEOUT, ST_POOL_FULL = 16, 32, 64, 128
MAX_K, MAX_S, MAX_NGRAM, MAX_POOL = 256, 16, 64, 1 << 24

# kernels launched by one call of each entry point (reported by the benchmark)
# kernels one call launches: verify_sample with a prebuilt d2t plan (or the identity map)
# launches 2, and 2 more when it builds the plan itself; d2t_plan launches 2
LAUNCHES = {"verify_greedy": 2, "verify_greedy_top2": 2, "infer_modality": 2, "pool_append": 1, "pool_lookup": 1, "suffix_append": 1, "verify_sample": 2, "verify_sample_plan_in_call": 4, "d2t_plan": 2,
            "cfg_merge_sample": 2, "accept_scan": 1}


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, text: str):
        super().__init__(f"specverify error {code}: {text}")
        self.code = code


class SvRows(C.Structure):
    _fields_ = [("data", C.c_void_p), ("dtype", C.c_int32), ("width", C.c_int32), ("row_stride", C.c_int64)]


_lib = None


def load(path: str | None = None):
    """Load libspecverify.so (built in-tree by ``_build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first (python -c 'import __graft_entry__ as g; g.build()')"
        )
    lib = C.CDLL(path)
    P, i32, sz, f32 = C.c_void_p, C.c_int32, C.c_size_t, C.c_float
    lib.sv_status_string.argtypes = [C.c_int]
    lib.sv_status_string.restype = C.c_char_p
    lib.sv_verify_greedy_workspace.argtypes = [i32, i32, i32, i32]
    lib.sv_verify_greedy_workspace.restype = sz
    lib.sv_verify_greedy.argtypes = [SvRows, i32, i32, i32, P, P, P, P, P, P, sz, P]
    lib.sv_verify_greedy.restype = C.c_int
    lib.sv_verify_greedy_top2_workspace.argtypes = [i32, i32, i32, i32]
    lib.sv_verify_greedy_top2_workspace.restype = sz
    lib.sv_verify_greedy_top2.argtypes = [SvRows, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
    lib.sv_verify_greedy_top2.restype = C.c_int
    lib.sv_infer_modality_workspace.argtypes = [i32, i32]
    lib.sv_infer_modality_workspace.restype = sz
    lib.sv_infer_modality.argtypes = [SvRows, i32, P, i32, P, P, P, P, P, P, sz, P]
    lib.sv_infer_modality.restype = C.c_int
    lib.sv_verify_sample_workspace.argtypes = [i32, i32, i32, i32]
    lib.sv_verify_sample_workspace.restype = sz
    lib.sv_verify_sample.argtypes = [SvRows, SvRows, P, P, i32, i32, P, P, P, P, P, P, P, P, P, P, sz, P]
    lib.sv_d2t_plan_bytes.argtypes = [i32, i32]
    lib.sv_d2t_plan_bytes.restype = sz
    lib.sv_d2t_plan_build.argtypes = [P, i32, i32, P, sz, P]
    lib.sv_d2t_plan_build.restype = C.c_int
    lib.sv_verify_sample.restype = C.c_int
    lib.sv_cfg_merge_sample_workspace.argtypes = [i32, i32, i32, i32]
    lib.sv_cfg_merge_sample_workspace.restype = sz
    lib.sv_cfg_merge_sample.argtypes = [SvRows, SvRows, P, P, i32, f32, SvRows, i32, i32, P, P, P, P, P, P,
                                        P, P, sz, P]
    lib.sv_cfg_merge_sample.restype = C.c_int
    lib.sv_pool_append.argtypes = [P, P, i32, P, i32, i32, P, P]
    lib.sv_pool_lookup.argtypes = [P, P, i32, P, i32, i32, i32, P, P, P]
    lib.sv_suffix_append.argtypes = [P, i32, i32, P, P, i32, P]
    lib.sv_accept_scan.argtypes = [P, P, P, i32, i32, P, P, P]
    lib.sv_accept_scan.restype = C.c_int
    lib.sv_selftest_wait_timeout.argtypes = [P, P, C.c_int64, P]
    lib.sv_selftest_wait_timeout.restype = C.c_int
    _lib = lib
    return lib


def _check(rc: int):
    if rc != 0:
        raise SpecVerifyError(rc, load().sv_status_string(rc).decode())


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def rows_of(t, width: int | None = None) -> SvRows:
    """Describe a 2-D CUDA tensor of logits (rows may be strided)."""
    import torch

    if t is None:
        return SvRows(None, SV_F32, int(width or 1), 0)
    if not t.is_cuda or t.dim() != 2:
        raise ValueError("logits must be a 2-D CUDA tensor")
    if t.dtype == torch.bfloat16:
        code = SV_BF16
    elif t.dtype == torch.float32:
        code = SV_F32
    else:
        raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")
    if t.shape[0] > 1 and t.stride(1) != 1:
        raise ValueError("entries of a logit row must be contiguous")
    stride = t.stride(0) if t.shape[0] > 1 else t.shape[1]
    return SvRows(t.data_ptr(), code, int(width if width is not None else t.shape[1]), int(stride))


def _empty(shape, dtype, device):
    import torch

    return torch.empty(shape, dtype=dtype, device=device)


def _workspace(nbytes, device, workspace):
    import torch

    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _nbytes(t):
    return t.numel() * t.element_size()


def verify_greedy_workspace(R: int, k: int, branches: int, V: int) -> int:
    return int(load().sv_verify_greedy_workspace(R, k, branches, V))


def verify_greedy(target, R: int, k: int, branches: int, draft, out: dict | None = None, workspace=None,
                  stream=None) -> dict:
    """Greedy verification.  target: [R*rows_per_request, V] bf16/f32 CUDA
    tensor; draft: int32 [R, branches, k].  Returns accept_len [R], tokens
    [R, k+1], branch [R], status [R] (int32 CUDA tensors)."""
    import torch

    lib = load()
    dev = target.device
    if out is None:
        out = dict(accept_len=_empty(R, torch.int32, dev), tokens=_empty((R, k + 1), torch.int32, dev),
                   branch=_empty(R, torch.int32, dev), status=_empty(R, torch.int32, dev))
    ws = _workspace(lib.sv_verify_greedy_workspace(R, k, branches, target.shape[1]), dev, workspace)
    _check(lib.sv_verify_greedy(rows_of(target), R, k, branches, _ptr(draft), _ptr(out["accept_len"]),
                                _ptr(out["tokens"]), _ptr(out.get("branch")), _ptr(out.get("status")), _ptr(ws),
                                _nbytes(ws), _stream(stream)))
    return out


def verify_greedy_top2_workspace(R: int, k: int, branches: int, V: int) -> int:
    return int(load().sv_verify_greedy_top2_workspace(R, k, branches, V))


def verify_greedy_top2(target, R: int, k: int, branches: int, draft, out: dict | None = None, workspace=None,
                       stream=None) -> dict:
    """verify_greedy plus top2 [rows, 2]: per row the argmax and the runner-up id
    (logit descending, then id ascending; -1 when V == 1), from the same pass."""
    import torch

    lib = load()
    dev = target.device
    rows = target.shape[0] if R == 0 else R * (1 + branches * k)
    if out is None:
        out = dict(accept_len=_empty(R, torch.int32, dev), tokens=_empty((R, k + 1), torch.int32, dev),
                   branch=_empty(R, torch.int32, dev), status=_empty(R, torch.int32, dev),
                   top2=_empty((rows, 2), torch.int32, dev))
    ws = _workspace(lib.sv_verify_greedy_top2_workspace(R, k, branches, target.shape[1]), dev, workspace)
    _check(lib.sv_verify_greedy_top2(rows_of(target), R, k, branches, _ptr(draft), _ptr(out["accept_len"]),
                                     _ptr(out["tokens"]), _ptr(out.get("branch")), _ptr(out.get("status")),
                                     _ptr(out["top2"]), _ptr(ws), _nbytes(ws), _stream(stream)))
    return out


def infer_modality(logits, part_start, out: dict | None = None, workspace=None, stream=None) -> dict:
    """Per row of full-vocabulary logits [N, V]: amax, the partition holding it (part, -1 for
    none) and its id range (mask_lo, mask_hi), with status bits.  part_start: host ints,
    ascending, P + 1 of them."""
    import numpy as np
    import torch

    lib = load()
    dev = logits.device
    N = logits.shape[0]
    ps = np.ascontiguousarray(np.asarray(part_start, dtype=np.int32))
    if out is None:
        out = {key: _empty(N, torch.int32, dev) for key in ("amax", "part", "mask_lo", "mask_hi", "status")}
    ws = _workspace(lib.sv_infer_modality_workspace(N, logits.shape[1]), dev, workspace)
    _check(lib.sv_infer_modality(rows_of(logits), N, ps.ctypes.data, ps.size - 1, _ptr(out.get("amax")),
                                 _ptr(out["part"]), _ptr(out.get("mask_lo")), _ptr(out.get("mask_hi")),
                                 _ptr(out.get("status")), _ptr(ws), _nbytes(ws), _stream(stream)))
    return out


def verify_sample_workspace(R: int, k: int, V: int, Vd: int) -> int:
    return int(load().sv_verify_sample_workspace(R, k, V, Vd))


def d2t_plan(d2t, V: int, stream=None):
    """Build the device-side plan of a d2t map once (a uint8 CUDA tensor) for
    verify_sample(..., plan=...)."""
    import torch

    lib = load()
    Vd = d2t.numel()
    nbytes = int(lib.sv_d2t_plan_bytes(V, Vd))
    plan = torch.empty(nbytes, dtype=torch.uint8, device=d2t.device)
    _check(lib.sv_d2t_plan_build(_ptr(d2t), Vd, V, _ptr(plan), nbytes, _stream(stream)))
    return plan


def verify_sample(target, draft_logits, d2t, R: int, k: int, draft, seeds, temperature, out: dict | None = None,
                  workspace=None, stream=None, stats: bool = True, plan=None) -> dict:
    """Speculative sampling.  target [R*(k+1), V]; draft_logits [R*k, Vd];
    d2t int32 [Vd] or None; draft int32 [R, k]; seeds uint64 bits in an int64
    tensor [R]; temperature float32 [R]; plan: d2t_plan(d2t, V) or None.
    Returns accept_len, tokens, status and, with stats=True, tv / p_draft /
    q_draft [R, k]."""
    import torch

    lib = load()
    dev = target.device
    V = target.shape[1]
    if draft_logits is not None:
        Vd = draft_logits.shape[1]
    else:
        Vd = V if d2t is None else d2t.numel()
    if out is None:
        out = dict(accept_len=_empty(R, torch.int32, dev), tokens=_empty((R, k + 1), torch.int32, dev),
                   status=_empty(R, torch.int32, dev))
        if stats:
            for name in ("tv", "p_draft", "q_draft"):
                out[name] = _empty((R, k), torch.float32, dev)
    ws = _workspace(lib.sv_verify_sample_workspace(R, k, V, Vd), dev, workspace)
    _check(lib.sv_verify_sample(rows_of(target), rows_of(draft_logits, Vd), _ptr(d2t), _ptr(plan), R, k, _ptr(draft),
                                _ptr(seeds), _ptr(temperature), _ptr(out["accept_len"]), _ptr(out["tokens"]),
                                _ptr(out.get("tv")), _ptr(out.get("p_draft")), _ptr(out.get("q_draft")),
                                _ptr(out.get("status")), _ptr(ws), _nbytes(ws), _stream(stream)))
    return out


def cfg_merge_sample_workspace(R: int, k: int, S: int, W: int) -> int:
    return int(load().sv_cfg_merge_sample_workspace(R, k, S, W))


def cfg_merge_sample(cond, uncond, cb_id_base, cb_data_offset, S: int, W: int, w: float, draft_logits, R: int,
                     k: int, draft, seeds, temperature, out: dict | None = None, workspace=None, stream=None,
                     stats: bool = True) -> dict:
    """CFG merge per codebook, then verification.  cond/uncond [R*(k+1)*S, row]
    with codebook s at element cb_data_offset[s] (W entries); cb_id_base and
    cb_data_offset are host int sequences of length S; draft_logits
    [R*k*S, W] or None (greedy); draft int32 [R, k, S] absolute ids."""
    import torch

    lib = load()
    dev = cond.device
    if out is None:
        out = dict(accept_len=_empty(R, torch.int32, dev), tokens=_empty((R, k + 1, S), torch.int32, dev),
                   status=_empty(R, torch.int32, dev))
        if stats:
            out["tv"] = _empty((R, k, S), torch.float32, dev)
    base = (C.c_int32 * S)(*[int(b) for b in cb_id_base])
    off = None if cb_data_offset is None else (C.c_int32 * S)(*[int(o) for o in cb_data_offset])
    ws = _workspace(lib.sv_cfg_merge_sample_workspace(R, k, S, W), dev, workspace)
    _check(lib.sv_cfg_merge_sample(rows_of(cond, W), rows_of(uncond, W), C.cast(base, C.c_void_p),
                                   None if off is None else C.cast(off, C.c_void_p), S, float(w),
                                   rows_of(draft_logits, W), R, k, _ptr(draft), _ptr(seeds), _ptr(temperature),
                                   _ptr(out["accept_len"]), _ptr(out["tokens"]), _ptr(out.get("tv")),
                                   _ptr(out.get("status")), _ptr(ws), _nbytes(ws), _stream(stream)))
    return out


def pool_append(pool, pool_len, drafts, status=None, stream=None):
    """Insert drafts int32 [R, k] (a negative id ends a draft early) into the pools
    int32 [R, Lp] whose used lengths are pool_len int32 [R]; both are updated in
    place.  status int32 [R] (optional) gets SV_ST_POOL_FULL where a draft did not fit."""
    lib = load()
    R, Lp = pool.shape
    k = drafts.shape[1]
    _check(lib.sv_pool_append(_ptr(pool), _ptr(pool_len), Lp, _ptr(drafts), k, R, _ptr(status), _stream(stream)))
    return status


def pool_lookup(pool, pool_len, suffix, gamma: int, out: dict | None = None, stream=None) -> dict:
    """Longest n-gram of the pools int32 [R, Lp] (used lengths pool_len int32 [R])
    matching the emitted suffix int32 [R, N] (-1 padded on the left); returns
    match_len int32 [R] and the continuation cont int32 [R, gamma] (-1 padded)."""
    import torch

    lib = load()
    R, Lp = pool.shape
    N = suffix.shape[1]
    dev = pool.device
    if out is None:
        out = dict(match_len=_empty(R, torch.int32, dev), cont=_empty((R, gamma), torch.int32, dev))
    _check(lib.sv_pool_lookup(_ptr(pool), _ptr(pool_len), Lp, _ptr(suffix), N, R, gamma, _ptr(out["match_len"]),
                              _ptr(out["cont"]), _stream(stream)))
    return out


def suffix_append(suffix, tokens, accept_len, stream=None):
    """Shift a verify step's committed tokens (tokens int32 [R, k + 1], entries 0..n with
    n = accept_len[r]) into the emitted suffix int32 [R, N], in place."""
    lib = load()
    R, N = suffix.shape
    k = tokens.shape[1] - 1
    _check(lib.sv_suffix_append(_ptr(suffix), N, R, _ptr(tokens), _ptr(accept_len), k, _stream(stream)))
    return suffix


def accept_scan(accept, draft, fix, out: dict | None = None, stream=None) -> dict:
    """accept uint8 [R, k]; draft int32 [R, k]; fix int32 [R, k+1]."""
    import torch

    lib = load()
    R, k = accept.shape
    dev = accept.device
    if out is None:
        out = dict(accept_len=_empty(R, torch.int32, dev), tokens=_empty((R, k + 1), torch.int32, dev))
    _check(lib.sv_accept_scan(_ptr(accept), _ptr(draft), _ptr(fix), R, k, _ptr(out["accept_len"]),
                              _ptr(out["tokens"]), _stream(stream)))
    return out


def selftest_wait_timeout(limit_cycles: int, stream=None):
    """Make one bounded barrier wait of the library run out on purpose (sv_selftest_wait_timeout);
    returns the int32 [2] device status: [0] the timeout bit, [1] whether the real copy landed."""
    import torch

    src = torch.arange(4, dtype=torch.int32, device="cuda") + 0x5A5A0000
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    _check(load().sv_selftest_wait_timeout(_ptr(src), _ptr(status), limit_cycles, _stream(stream)))
    return status
