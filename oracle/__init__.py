"""ctypes front end of the fp64 CPU oracle (``specverify_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use this module.  The CUDA library never
imports, links or runs it, and it shares no code with the CUDA library.

Logit arrays are numpy arrays of shape ``[rows, width]`` whose rows may be
strided (``arr.strides[1]`` must equal the item size).  ``np.uint16`` arrays
hold raw bfloat16 bit patterns; ``np.float32`` arrays hold fp32 logits.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specverify_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, F32 = 0, 1
ST_TOKEN_RANGE, ST_BAD_LOGITS, ST_OFF_SUPPORT = 1, 2, 4
ST_RESIDUAL_ZERO, ST_BAD_TEMP, ST_BAD_D2T = 8, 16, 32
TAG_ACCEPT, TAG_RESIDUAL, TAG_BONUS = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (plain gcc, no OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P = C.c_void_p
            i32, i64, u32, u64, f32 = C.c_int32, C.c_int64, C.c_uint32, C.c_uint64, C.c_float
            lib.or_philox4x32_10.argtypes = [P, P, P]
            lib.or_philox4x32_10.restype = None
            lib.or_uniform.argtypes = [u64, u32, u32, u32]
            lib.or_uniform.restype = C.c_double
            lib.or_uniform_from_word.argtypes = [u32]
            lib.or_uniform_from_word.restype = C.c_double
            lib.or_race.argtypes = [P, i32, u64, u32, u32, P]
            lib.or_race.restype = i32
            lib.or_accept_scan.argtypes = [P, P, P, i32, i32, P, P]
            lib.or_accept_scan.restype = C.c_int
            lib.or_verify_greedy.argtypes = [P, C.c_int, i64, i32, i32, i32, i32, P, P, P, P, P]
            lib.or_verify_greedy.restype = C.c_int
            lib.or_top2_rows.argtypes = [P, C.c_int, i64, i64, i32, P]
            lib.or_top2_rows.restype = C.c_int
            lib.or_infer_modality.argtypes = [P, C.c_int, i64, i64, i32, P, i32, P, P, P, P]
            lib.or_infer_modality.restype = C.c_int
            lib.or_pool_append.argtypes = [P, P, i32, P, i32, i32, P]
            lib.or_pool_append.restype = C.c_int
            lib.or_pool_lookup.argtypes = [P, P, i32, P, i32, i32, i32, P, P]
            lib.or_pool_lookup.restype = C.c_int
            lib.or_suffix_append.argtypes = [P, i32, i32, P, P, i32]
            lib.or_suffix_append.restype = C.c_int
            lib.or_verify_sample.argtypes = [P, C.c_int, i64, i32, P, C.c_int, i64, i32, P, i32, i32,
                                             P, P, P, P, P, P, P, P, P, P, P]
            lib.or_verify_sample.restype = C.c_int
            lib.or_cfg_merge_sample.argtypes = [P, P, C.c_int, i64, P, P, i32, i32, f32, P, C.c_int,
                                                i64, i32, i32, P, P, P, P, P, P, P, P, P]
            lib.or_cfg_merge_sample.restype = C.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _rows(a, name):
    """(array, dtype code, row stride in elements, width) of a logit matrix."""
    a = np.asarray(a)
    if a.ndim != 2:
        raise ValueError(f"{name} must be 2-D [rows, width]")
    if a.dtype == np.uint16:
        code = BF16
    elif a.dtype == np.float32:
        code = F32
    else:
        raise TypeError(f"{name}: uint16 (bf16 bits) or float32 expected, got {a.dtype}")
    if a.shape[0] > 1 and a.strides[1] != a.itemsize:
        raise ValueError(f"{name}: elements of a row must be contiguous")
    if a.strides[1] != a.itemsize:
        a = np.ascontiguousarray(a)
    stride = a.strides[0] // a.itemsize if a.shape[0] > 1 else a.shape[1]
    return a, code, stride, a.shape[1]


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def philox4x32_10(ctr, key):
    lib = _load()
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    lib.or_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, row: int, tag: int, x: int) -> float:
    return _load().or_uniform(seed, row, tag, x)


def uniform_from_word(r: int) -> float:
    return _load().or_uniform_from_word(r)


def race(w, seed: int, row: int, tag: int):
    """(index, margin) of the exponential race over weights ``w``."""
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
    m = C.c_double(0.0)
    idx = _load().or_race(_ptr(w), w.size, seed, row, tag, C.byref(m))
    return int(idx), float(m.value)


def accept_scan(accept, draft, fix):
    accept = np.ascontiguousarray(np.asarray(accept, dtype=np.uint8))
    R, k = accept.shape
    draft, fix = _i32(draft), _i32(fix)
    acc_len = np.zeros(R, np.int32)
    tokens = np.zeros((R, k + 1), np.int32)
    _load().or_accept_scan(_ptr(accept), _ptr(draft), _ptr(fix), R, k, _ptr(acc_len), _ptr(tokens))
    return dict(accept_len=acc_len, tokens=tokens)


def verify_greedy(target, R: int, k: int, branches: int, draft):
    t, code, stride, V = _rows(target, "target")
    rows_per_req = 1 + branches * k
    if t.shape[0] < R * rows_per_req:
        raise ValueError("target has too few rows")
    draft = _i32(draft).reshape(R, branches, k) if k else np.zeros((R, branches, 0), np.int32)
    acc_len = np.zeros(R, np.int32)
    tokens = np.zeros((R, k + 1), np.int32)
    branch = np.zeros(R, np.int32)
    status = np.zeros(R, np.int32)
    rc = _load().or_verify_greedy(_ptr(t), code, stride, V, R, k, branches, _ptr(draft),
                                  _ptr(acc_len), _ptr(tokens), _ptr(branch), _ptr(status))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments ({rc})")
    return dict(accept_len=acc_len, tokens=tokens, branch=branch, status=status)


def top2_rows(rows):
    """[n, 2] int32: per row the argmax and the runner-up id (value descending, then id
    ascending; NaN read as -inf; -1 for one-id rows)."""
    t, code, stride, V = _rows(rows, "rows")
    out = np.zeros((t.shape[0], 2), np.int32)
    rc = _load().or_top2_rows(_ptr(t), code, stride, t.shape[0], V, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments ({rc})")
    return out


def infer_modality(rows, part_start):
    """Per row of full-vocabulary logits: argmax, the partition holding it (-1: none) and
    that partition's id range [lo, hi) (0, 0 when none)."""
    t, code, stride, V = _rows(rows, "rows")
    ps = _i32(part_start)
    n = t.shape[0]
    out = {key: np.zeros(n, np.int32) for key in ("amax", "part", "mask_lo", "mask_hi")}
    rc = _load().or_infer_modality(_ptr(t), code, stride, n, V, _ptr(ps), ps.size - 1, _ptr(out["amax"]),
                                   _ptr(out["part"]), _ptr(out["mask_lo"]), _ptr(out["mask_hi"]))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments ({rc})")
    return out


def pool_append(pool, pool_len, drafts):
    """Insert drafts int32 [R, k] (a negative id ends a draft early) into the pools
    int32 [R, Lp] with used lengths pool_len int32 [R].  Returns the new pool,
    pool_len and status (128 where a draft did not fit)."""
    pool = _i32(pool).copy()
    pool_len = _i32(pool_len).copy()
    drafts = _i32(drafts)
    R, Lp = pool.shape
    status = np.zeros(R, np.int32)
    rc = _load().or_pool_append(_ptr(pool), _ptr(pool_len), Lp, _ptr(drafts), drafts.shape[1], R, _ptr(status))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments ({rc})")
    return dict(pool=pool, pool_len=pool_len, status=status)


def pool_lookup(pool, pool_len, suffix, gamma: int):
    """pool int32 [R, Lp] with used lengths pool_len int32 [R]; suffix int32 [R, N]
    (the last N emitted tokens, -1 where shorter).  Returns match_len [R] and
    cont [R, gamma]."""
    pool = _i32(pool)
    pool_len = _i32(pool_len)
    suffix = _i32(suffix)
    R, Lp = pool.shape
    N = suffix.shape[1]
    match_len = np.zeros(R, np.int32)
    cont = np.zeros((R, gamma), np.int32)
    rc = _load().or_pool_lookup(_ptr(pool), _ptr(pool_len), Lp, _ptr(suffix), N, R, gamma, _ptr(match_len),
                                _ptr(cont))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments ({rc})")
    return dict(match_len=match_len, cont=cont)


def suffix_append(suffix, tokens, accept_len):
    """The emitted suffix int32 [R, N] after a step that committed tokens[r, 0..n],
    n = accept_len[r] (tokens int32 [R, k + 1]).  Returns the new suffix."""
    suffix = _i32(suffix).copy()
    tokens = _i32(tokens)
    accept_len = _i32(accept_len)
    R, N = suffix.shape
    rc = _load().or_suffix_append(_ptr(suffix), N, R, _ptr(tokens), _ptr(accept_len), tokens.shape[1] - 1)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments ({rc})")
    return suffix


def verify_sample(target, draft_logits, d2t, R: int, k: int, draft, seeds, temperature):
    t, tcode, tstride, V = _rows(target, "target")
    if draft_logits is None:
        dl, dcode, dstride, Vd = None, F32, 0, (V if d2t is None else len(d2t))
    else:
        dl, dcode, dstride, Vd = _rows(draft_logits, "draft_logits")
    d2t_a = None if d2t is None else _i32(d2t)
    draft = _i32(draft).reshape(R, k) if k else np.zeros((R, 0), np.int32)
    seeds = np.ascontiguousarray(np.asarray(seeds, dtype=np.uint64))
    temperature = np.ascontiguousarray(np.asarray(temperature, dtype=np.float32))
    acc_len = np.zeros(R, np.int32)
    tokens = np.zeros((R, k + 1), np.int32)
    tv = np.zeros((R, k)); pd = np.zeros((R, k)); qd = np.zeros((R, k))
    status = np.zeros(R, np.int32)
    am = np.zeros((R, k)); rm = np.zeros(R)
    rc = _load().or_verify_sample(_ptr(t), tcode, tstride, V, _ptr(dl), dcode, dstride, Vd, _ptr(d2t_a),
                                  R, k, _ptr(draft), _ptr(seeds), _ptr(temperature), _ptr(acc_len),
                                  _ptr(tokens), _ptr(tv), _ptr(pd), _ptr(qd), _ptr(status), _ptr(am),
                                  _ptr(rm))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments ({rc})")
    return dict(accept_len=acc_len, tokens=tokens, tv=tv, p_draft=pd, q_draft=qd, status=status,
                accept_margin=am, race_margin=rm)


def cfg_merge_sample(cond, uncond, cb_id_base, cb_data_offset, S: int, W: int, w: float,
                     draft_logits, R: int, k: int, draft, seeds, temperature):
    c, code, stride, width = _rows(cond, "cond")
    u, ucode, ustride, _ = _rows(uncond, "uncond")
    if ucode != code or ustride != stride:
        raise ValueError("cond and uncond must share dtype and row stride")
    if draft_logits is None:
        dl, dcode, dstride = None, F32, 0
    else:
        dl, dcode, dstride, _ = _rows(draft_logits, "draft_logits")
    base = _i32(cb_id_base)
    off = _i32(cb_data_offset)
    draft = _i32(draft).reshape(R, k, S) if k else np.zeros((R, 0, S), np.int32)
    seeds = np.ascontiguousarray(np.asarray(seeds, dtype=np.uint64))
    temperature = np.ascontiguousarray(np.asarray(temperature, dtype=np.float32))
    acc_len = np.zeros(R, np.int32)
    tokens = np.zeros((R, k + 1, S), np.int32)
    tv = np.zeros((R, k, S)); status = np.zeros(R, np.int32)
    am = np.zeros((R, k, S)); rm = np.zeros((R, S))
    rc = _load().or_cfg_merge_sample(_ptr(c), _ptr(u), code, stride, _ptr(base), _ptr(off), S, W, w,
                                     _ptr(dl), dcode, dstride, R, k, _ptr(draft), _ptr(seeds),
                                     _ptr(temperature), _ptr(acc_len), _ptr(tokens), _ptr(tv),
                                     _ptr(status), _ptr(am), _ptr(rm))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments ({rc})")
    return dict(accept_len=acc_len, tokens=tokens, tv=tv, status=status, accept_margin=am,
                race_margin=rm)


MARGIN = 1e-6  # decision margin below which a row is exempt from exact parity


def exempt_rows(out: dict) -> np.ndarray:
    """Boolean [R, rows per request] mask of the rows of a verify_sample / cfg_merge_sample
    result whose decision margin is below MARGIN: tested positions with |u - p/q| < MARGIN,
    and the row the race ran on (the first rejected position, or the bonus row: index
    accept_len) when its two smallest keys are within MARGIN (relative).  CFG results
    ([R, k + 1, S] tokens) give one row per (frame, codebook)."""
    n = np.asarray(out["accept_len"])
    R = len(n)
    tok = np.asarray(out["tokens"])
    k1 = tok.shape[1]
    S = tok.shape[2] if tok.ndim == 3 else 1
    mask = np.zeros((R, k1, S), bool)
    if k1 > 1:
        mask[:, : k1 - 1] |= np.asarray(out["accept_margin"]).reshape(R, k1 - 1, S) < MARGIN
    mask[np.arange(R), n] |= np.asarray(out["race_margin"]).reshape(R, S) < MARGIN
    return mask.reshape(R, -1)
