"""CPU oracle of the DSpark ragged-verification hot path — TEST INFRASTRUCTURE ONLY.

A thin ctypes wrapper over ``dspark_oracle.c``: a plain, single-threaded C implementation of
the confidence scheduler, the front-pack, greedy and stochastic verify and the compact scatter,
written from "DSpark in SGLang: Speculative Decoding with Confidence-Driven, Variable-Length
Verification" (LMSYS blog summary) and the min(1, p/q) rule of the lshu.cn DSpark article.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. The CUDA library never imports, links or calls it, and the two share no
code. Arrays are numpy; bf16 logits are passed as their raw uint16 bit patterns, fp32 logits as
float32, so the oracle widens bf16 itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

STATIC, COMPACT, CAP_ACCEPT = 0, 1, 2
BF16, F32 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_SO = os.path.join(_HERE, "libdspark_oracle.so")
_LOCK = threading.Lock()
_LIB = None

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_u64 = ctypes.c_uint64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            build()
            lib = ctypes.CDLL(_SO)
            lib.oracle_philox4x64_10.argtypes = [_p, _p, _p]
            lib.oracle_philox4x64_10.restype = None
            lib.oracle_survival_keys.argtypes = [_p, _i32, _i32, _p]
            lib.oracle_survival_keys.restype = None
            lib.oracle_schedule.argtypes = [_p, _i32, _i32, ctypes.c_double, _p, _i32, _p, _i32,
                                            _p, _p, _p, _p, _p]
            lib.oracle_schedule.restype = ctypes.c_int
            lib.oracle_pack.argtypes = [_p, _p, _i32, _i32, _p, _i32, _p, _p, _p, _p, _i32, _p, _p]
            lib.oracle_pack.restype = ctypes.c_int
            lib.oracle_row_argmax.argtypes = [_p, _i32, _i32, ctypes.c_int64]
            lib.oracle_row_argmax.restype = ctypes.c_int
            lib.oracle_row_softmax_stats.argtypes = [_p, _i32, _i32, ctypes.c_int64,
                                                     ctypes.c_double, _p, _p]
            lib.oracle_row_softmax_stats.restype = None
            lib.oracle_verify.argtypes = [_i32, _i32, _p, _i32, _p, _i32, _i32, _p, _p, _p, _i32,
                                          _i32, ctypes.c_float, _u64, _u64, _p, _p, _p, _p, _p,
                                          _p, _p, _p]
            lib.oracle_verify.restype = ctypes.c_int
            lib.oracle_scatter.argtypes = [_p, _p, _i32, _i32, _p, _p, _i32, _p]
            lib.oracle_scatter.restype = ctypes.c_int
            lib.oracle_observe.argtypes = [_p, _p, _p, _i32, _i32, _i32, _p, _p, _p]
            lib.oracle_observe.restype = ctypes.c_int
            _LIB = lib
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _logits(a):
    """(contiguous array, dtype code) for uint16 bf16 bits or float32 logits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float32:
        return a, F32
    raise TypeError(f"logits must be uint16 (bf16 bits) or float32, got {a.dtype}")


def philox4x64_10(ctr, key) -> np.ndarray:
    """Philox4x64-10 block for a 4-word counter and a 2-word key (all uint64)."""
    c = _c(ctr, np.uint64)
    k = _c(key, np.uint64)
    out = np.zeros(4, np.uint64)
    _lib().oracle_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def survival_keys(conf) -> np.ndarray:
    conf = _c(conf, np.float32)
    B, L = conf.shape
    keys = np.zeros((B, L), np.uint64)
    _lib().oracle_survival_keys(_ptr(conf), B, L + 1, _ptr(keys))
    return keys


def schedule(conf, bias, alpha, theta) -> dict:
    """Confidence scheduler: windows [B], k_star, status bits, obj [n+1], sorted keys [n]."""
    conf = _c(conf, np.float32)
    B, L = conf.shape
    alpha = _c(alpha, np.float64)
    theta = _c(theta, np.float64)
    n = B * L
    windows = np.zeros(B, np.int32)
    k_star = np.zeros(1, np.int32)
    status = np.zeros(1, np.int32)
    obj = np.zeros(n + 1, np.float64)
    skeys = np.zeros(max(n, 1), np.uint64)
    rc = _lib().oracle_schedule(_ptr(conf), B, L + 1, float(bias), _ptr(alpha), alpha.size,
                                _ptr(theta), theta.size, _ptr(windows), _ptr(k_star),
                                _ptr(status), _ptr(obj), _ptr(skeys))
    if rc != 0:
        raise ValueError("oracle_schedule: invalid arguments")
    return dict(windows=windows, k_star=int(k_star[0]), status=int(status[0]), obj=obj,
                sorted_keys=skeys[:n])


def pack(windows, tokens, tiers, packed_cap) -> dict:
    windows = _c(windows, np.int32)
    tokens = _c(tokens, np.int32)
    tiers = _c(tiers, np.int32)
    B, gamma = tokens.shape
    cu = np.zeros(B + 1, np.int32)
    cap = int(packed_cap)
    packed = np.full(max(cap, 1), -7, np.int32)
    row_req = np.full(max(cap, 1), -7, np.int32)
    row_pos = np.full(max(cap, 1), -7, np.int32)
    meta = np.zeros(2, np.int32)
    status = np.zeros(1, np.int32)
    rc = _lib().oracle_pack(_ptr(windows), _ptr(tokens), B, gamma, _ptr(tiers), tiers.size,
                            _ptr(cu), _ptr(packed), _ptr(row_req), _ptr(row_pos), cap,
                            _ptr(meta), _ptr(status))
    if rc != 0:
        raise ValueError("oracle_pack: invalid arguments")
    return dict(cu=cu, packed_ids=packed[:cap], row_req=row_req[:cap], row_pos=row_pos[:cap],
                M=int(meta[0]), tier=int(meta[1]), status=int(status[0]))


def row_argmax(logits, row: int) -> int:
    a, dt = _logits(logits)
    return int(_lib().oracle_row_argmax(_ptr(a), dt, a.shape[-1], int(row)))


def row_softmax_stats(logits, row: int, temperature: float):
    a, dt = _logits(logits)
    m = np.zeros(1, np.float64)
    z = np.zeros(1, np.float64)
    _lib().oracle_row_softmax_stats(_ptr(a), dt, a.shape[-1], int(row), float(temperature),
                                    _ptr(m), _ptr(z))
    return float(m[0]), float(z[0])


def verify(mode, stochastic, target, tokens, *, cu=None, windows=None, draft=None,
           temperature=1.0, seed=0, step=0) -> dict:
    """Verify. target: [rows, V] logits; draft: [B*(gamma-1), V] (stochastic); tokens [B, gamma]."""
    target, dt = _logits(target)
    rows, V = target.shape
    tokens = _c(tokens, np.int32)
    B, gamma = tokens.shape
    if draft is not None:
        draft, ddt = _logits(draft)
        if ddt != dt:
            raise TypeError("target and draft logits must share a dtype")
    cu = None if cu is None else _c(cu, np.int32)
    windows = None if windows is None else _c(windows, np.int32)
    accept = np.zeros(B, np.int32)
    committed = np.zeros((B, gamma), np.int32)
    ceiling = np.zeros(B, np.int32)
    row_prob = np.zeros((max(rows, 1), 2), np.float32)
    status = np.zeros(1, np.int32)
    L = gamma - 1
    ratio = np.zeros(max(B * L, 1), np.float32)
    u = np.zeros(max(B * L, 1), np.float32)
    margin = np.zeros(max(B, 1), np.float64)
    rc = _lib().oracle_verify(int(mode), int(bool(stochastic)), _ptr(target), rows, _ptr(draft),
                              dt, V, _ptr(cu), _ptr(windows), _ptr(tokens), B, gamma,
                              float(temperature), int(seed), int(step), _ptr(accept),
                              _ptr(committed), _ptr(ceiling), _ptr(row_prob), _ptr(status),
                              _ptr(ratio), _ptr(u), _ptr(margin))
    if rc != 0:
        raise ValueError("oracle_verify: invalid arguments")
    return dict(accept_len=accept, committed=committed, ceiling_len=ceiling,
                row_prob=row_prob[:rows], status=int(status[0]),
                ratio=ratio[:B * L].reshape(B, L), u=u[:B * L].reshape(B, L), margin=margin[:B])


def scatter(committed, accept_len, out_tokens, out_len) -> dict:
    committed = _c(committed, np.int32)
    accept_len = _c(accept_len, np.int32)
    out_tokens = _c(out_tokens, np.int32).copy()
    out_len = _c(out_len, np.int32).copy()
    B, gamma = committed.shape
    cap = out_tokens.shape[1]
    status = np.zeros(1, np.int32)
    rc = _lib().oracle_scatter(_ptr(committed), _ptr(accept_len), B, gamma, _ptr(out_tokens),
                               _ptr(out_len), cap, _ptr(status))
    if rc != 0:
        raise ValueError("oracle_scatter: invalid arguments")
    return dict(out_tokens=out_tokens, out_len=out_len, status=int(status[0]))


def observe(conf, accept_len, ceiling_len, n_bins, hist=None, util=None) -> dict:
    """Calibration histogram [n_bins, 3] and utilisation counters [2], accumulated."""
    conf = _c(conf, np.float32)
    accept_len = _c(accept_len, np.int32)
    ceiling_len = _c(ceiling_len, np.int32)
    B = accept_len.size
    gamma = (conf.shape[1] + 1) if conf.ndim == 2 else 1
    hist = np.zeros((n_bins, 3), np.uint64) if hist is None else _c(hist, np.uint64).copy()
    util = np.zeros(2, np.uint64) if util is None else _c(util, np.uint64).copy()
    status = np.zeros(1, np.int32)
    rc = _lib().oracle_observe(_ptr(conf), _ptr(accept_len), _ptr(ceiling_len), B, gamma,
                               int(n_bins), _ptr(hist), _ptr(util), _ptr(status))
    if rc != 0:
        raise ValueError("oracle_observe: invalid arguments")
    return dict(hist=hist, util=util, status=int(status[0]))
