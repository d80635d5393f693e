"""ctypes binding of libdspark's C ABI (include/dspark.h), same names, argument marshalling only.

Every function takes CUDA torch tensors (torch supplies device memory and streams, nothing
else), checks dtype / device / contiguity / size on the host, passes raw pointers and the
current CUDA stream, and raises DSparkError when the library returns an error code. All the
work of the hot path runs in the library's kernels; if the library is not built, the first
call raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

STATIC, COMPACT, CAP_ACCEPT = 0, 1, 2
MODES = {"static": STATIC, "compact": COMPACT, "cap_accept": CAP_ACCEPT}
BF16, F32 = 0, 1

STATUS_TIER_OVERFLOW = 0x01
STATUS_PACK_CAPACITY = 0x02
STATUS_BAD_WINDOW = 0x04
STATUS_OUT_OVERFLOW = 0x08
STATUS_BAD_COST = 0x10
STATUS_BAD_ROWS = 0x20
STATUS_BAD_TOKEN = 0x40
STATUS_BAD_LENGTH = 0x80
STATUS_STALL = 0x100

STREAM_AUTO, STREAM_REGISTER, STREAM_BULK = 0, 1, 2

MAX_GAMMA = 32
MAX_CANDIDATES = 16384
MAX_BATCH = 8192

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdspark.so")
_LOCK = threading.Lock()
_LIB = None

_p = ctypes.c_void_p
_i = ctypes.c_int
_u64 = ctypes.c_uint64


class DSparkError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


class _Cost(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_double), ("alpha", ctypes.c_void_p), ("alpha_len", ctypes.c_int32),
                ("theta", ctypes.c_void_p), ("theta_len", ctypes.c_int32)]


SYMBOLS = {
    "dspark_schedule": ([_p, _i, _i, ctypes.POINTER(_Cost), _p, _p, _p, _p], _i),
    "dspark_pack": ([_p, _p, _i, _i, _p, _i, _p, _p, _p, _p, _i, _p, _p, _p], _i),
    "dspark_verify": ([_i, _i, _p, _i, _p, _i, _i, _p, _p, _p, _i, _i, ctypes.c_float, _u64, _u64,
                       _p, _p, _p, _p, _p, ctypes.c_size_t, _p, _p], _i),
    "dspark_verify_workspace_bytes": ([_i, _i, _i, _i], ctypes.c_size_t),
    "dspark_scatter": ([_p, _p, _i, _i, _p, _p, _i, _p, _p], _i),
    "dspark_schedule_pack": ([_p, _i, _i, ctypes.POINTER(_Cost), _p, _p, _i, _p, _p, _p, _p, _p,
                              _p, _i, _p, _p, _p], _i),
    "dspark_verify_scatter": ([_i, _i, _p, _i, _p, _i, _i, _p, _p, _p, _i, _i, ctypes.c_float,
                               _u64, _u64, _p, _p, _p, _p, _p, ctypes.c_size_t, _p, _p, _i, _p,
                               _p], _i),
    "dspark_verify_noalloc": ([_i, _i, _p, _i, _p, _i, _i, _p, _p, _p, _i, _i, ctypes.c_float,
                               _u64, _u64, _p, _p, _p, _p, _p, _p], _i),
    "dspark_observe": ([_p, _p, _p, _i, _i, _i, _p, _p, _p, _p], _i),
    "dspark_graph_begin": ([_p], _i),
    "dspark_graph_end": ([_p, ctypes.POINTER(_p)], _i),
    "dspark_graph_launch": ([_p, _p], _i),
    "dspark_graph_destroy": ([_p], _i),
    "dspark_set_stream_kernel": ([_i], _i),
    "dspark_set_stream_events": ([_p, _p], _i),
    "dspark_last_error": ([], ctypes.c_char_p),
    "dspark_version": ([], _i),
}


def lib():
    """The loaded library; raises if it has not been built (no fallback exists)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built: run speculative_decoding_ragged_gb300.build.build()")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SYMBOLS.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _LIB = handle
    return _LIB


def last_error() -> str:
    return lib().dspark_last_error().decode()


def _check(fn: str, rc: int):
    if rc != 0:
        raise DSparkError(fn, rc, last_error())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, numel=None, min_numel=None,
         required=True):
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name} must have at least {min_numel} elements, got {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


class Prepared:
    """One checked, marshalled call: calling it re-issues the same C call (same pointers,
    sizes and stream) with no Python-side checks, for tight step loops."""

    __slots__ = ("name", "fn", "args")

    def __init__(self, name, args):
        self.name = name
        self.fn = getattr(lib(), name)
        self.args = args

    def __call__(self):
        rc = self.fn(*self.args)
        if rc != 0:
            raise DSparkError(self.name, rc, last_error())


def _call(name: str, args, prepare: bool):
    if prepare:
        return Prepared(name, args)
    _check(name, getattr(lib(), name)(*args))
    return None


def set_stream_kernel(which: int) -> None:
    """Which kernel streams the logits inside verify (STREAM_AUTO, STREAM_REGISTER,
    STREAM_BULK); results are bit-identical, only speed differs."""
    _check("dspark_set_stream_kernel", lib().dspark_set_stream_kernel(int(which)))


def set_stream_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]):
    """Record `start` / `stop` around the logit-streaming kernel of every later verify call
    (None, None: off). The events must have been recorded once (torch creates them lazily)."""
    def handle(ev):
        if ev is None:
            return None
        h = int(ev.cuda_event)
        if h == 0:
            raise ValueError("record the event once before handing it to the library")
        return ctypes.c_void_p(h)
    _check("dspark_set_stream_events", lib().dspark_set_stream_events(handle(start), handle(stop)))


class StepGraph:
    """Library calls captured once as a CUDA graph through the C ABI (dspark_graph_begin /
    dspark_graph_end) and replayed with one cudaGraphLaunch (dspark_graph_launch).

        s = torch.cuda.Stream()              # capture needs a stream other than the default
        with torch.cuda.stream(s):
            calls = [...]                    # prepared while s is current: bound to s
            g = StepGraph(s)
            for c in calls: c()
            g.end()
        g.launch()                           # replays on torch's current stream
    """

    def __init__(self, stream):
        self._stream = _stream(stream)
        self._h = ctypes.c_void_p()
        _check("dspark_graph_begin", lib().dspark_graph_begin(self._stream))

    def end(self):
        _check("dspark_graph_end", lib().dspark_graph_end(self._stream, ctypes.byref(self._h)))
        return self

    def prepare_launch(self, stream=None) -> "Prepared":
        """The replay as a prepared call bound to `stream` (torch's current by default)."""
        return Prepared("dspark_graph_launch", (self._h, _stream(stream)))

    def launch(self, stream=None):
        _check("dspark_graph_launch", lib().dspark_graph_launch(self._h, _stream(stream)))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _LIB is not None:
            _LIB.dspark_graph_destroy(h)
            self._h = ctypes.c_void_p()


def version() -> int:
    return lib().dspark_version()


class CostTable:
    """T(bs, K) = bias + alpha[bs] + theta[bs + K]; alpha and theta are float64 CUDA tensors."""

    def __init__(self, bias: float, alpha: torch.Tensor, theta: torch.Tensor):
        self.bias = float(bias)
        self.alpha = alpha
        self.theta = theta
        self._c = _Cost(self.bias, _ptr(alpha, "alpha", torch.float64), alpha.numel(),
                        _ptr(theta, "theta", torch.float64), theta.numel())

    @property
    def c(self):
        return self._c


def dspark_schedule(conf: torch.Tensor, cost: CostTable, windows: torch.Tensor,
                    k_star: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None,
                    prepare: bool = False):
    B = windows.numel()
    L = conf.shape[-1] if conf.dim() == 2 else 0
    gamma = L + 1
    args = (_ptr(conf, "conf", torch.float32, numel=B * L, required=L > 0 and B > 0), B, gamma,
            ctypes.byref(cost.c), _ptr(windows, "windows", torch.int32),
            _ptr(k_star, "k_star", torch.int32, min_numel=1),
            _ptr(status, "status", torch.int32, min_numel=1, required=False), _stream(stream))
    return _call("dspark_schedule", args, prepare)


def dspark_pack(windows: torch.Tensor, block_tokens: torch.Tensor, tiers: torch.Tensor,
                cu_seqlens: torch.Tensor, packed_ids: torch.Tensor, meta: torch.Tensor,
                row_req: Optional[torch.Tensor] = None, row_pos: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream=None, prepare: bool = False):
    B, gamma = block_tokens.shape
    cap = packed_ids.numel()
    args = (
        _ptr(windows, "windows", torch.int32, numel=B, required=B > 0),
        _ptr(block_tokens, "block_tokens", torch.int32, required=B > 0), B, gamma,
        _ptr(tiers, "tiers", torch.int32), tiers.numel(),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32, min_numel=B + 1),
        _ptr(packed_ids, "packed_ids", torch.int32, required=cap > 0),
        _ptr(row_req, "row_req", torch.int32, min_numel=cap, required=False),
        _ptr(row_pos, "row_pos", torch.int32, min_numel=cap, required=False), cap,
        _ptr(meta, "meta", torch.int32, min_numel=2),
        _ptr(status, "status", torch.int32, min_numel=1, required=False), _stream(stream))
    return _call("dspark_pack", args, prepare)


def dspark_schedule_pack(conf: torch.Tensor, cost: CostTable, block_tokens: torch.Tensor,
                         tiers: torch.Tensor, windows: torch.Tensor, k_star: torch.Tensor,
                         cu_seqlens: torch.Tensor, packed_ids: torch.Tensor, meta: torch.Tensor,
                         row_req: Optional[torch.Tensor] = None,
                         row_pos: Optional[torch.Tensor] = None,
                         status: Optional[torch.Tensor] = None, stream=None,
                         prepare: bool = False):
    """dspark_schedule then dspark_pack of the windows it writes, in one kernel."""
    B, gamma = block_tokens.shape
    L = gamma - 1
    if conf.dim() == 2 and tuple(conf.shape) != (B, L):
        raise ValueError(f"conf must be [{B}, {L}]")
    cap = packed_ids.numel()
    args = (
        _ptr(conf, "conf", torch.float32, numel=B * L, required=L > 0 and B > 0), B, gamma,
        ctypes.byref(cost.c), _ptr(block_tokens, "block_tokens", torch.int32, required=B > 0),
        _ptr(tiers, "tiers", torch.int32), tiers.numel(),
        _ptr(windows, "windows", torch.int32, numel=B),
        _ptr(k_star, "k_star", torch.int32, min_numel=1),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32, min_numel=B + 1),
        _ptr(packed_ids, "packed_ids", torch.int32, required=cap > 0),
        _ptr(row_req, "row_req", torch.int32, min_numel=cap, required=False),
        _ptr(row_pos, "row_pos", torch.int32, min_numel=cap, required=False), cap,
        _ptr(meta, "meta", torch.int32, min_numel=2),
        _ptr(status, "status", torch.int32, min_numel=1, required=False), _stream(stream))
    return _call("dspark_schedule_pack", args, prepare)


def dspark_verify_workspace_bytes(B: int, gamma: int, V: int, stochastic: bool) -> int:
    return int(lib().dspark_verify_workspace_bytes(B, gamma, V, int(bool(stochastic))))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise ValueError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _verify_args(mode, target, block_tokens, accept_len, committed, workspace, stochastic,
                 draft, cu_seqlens, windows, ceiling_len, row_prob, temperature, seed, step):
    mode = MODES[mode] if isinstance(mode, str) else int(mode)
    B, gamma = block_tokens.shape
    rows, V = target.shape
    dt = _dtype_code(target)
    if draft is not None:
        if draft.dtype != target.dtype or draft.shape[-1] != V:
            raise ValueError("draft logits must match the target's dtype and vocabulary")
        if draft.numel() != B * (gamma - 1) * V:
            raise ValueError(f"draft logits must hold B*(gamma-1) = {B * (gamma - 1)} rows")
    return (
        mode, int(bool(stochastic)), _ptr(target, "target"), rows,
        _ptr(draft, "draft", required=False), dt, V,
        _ptr(cu_seqlens, "cu_seqlens", torch.int32, min_numel=B + 1, required=False),
        _ptr(windows, "windows", torch.int32, min_numel=B, required=False),
        _ptr(block_tokens, "block_tokens", torch.int32), B, gamma, float(temperature),
        int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
        _ptr(accept_len, "accept_len", torch.int32, min_numel=B),
        _ptr(committed, "committed", torch.int32, min_numel=B * gamma),
        _ptr(ceiling_len, "ceiling_len", torch.int32, min_numel=B, required=False),
        _ptr(row_prob, "row_prob", torch.float32, min_numel=2 * rows, required=False),
        _ptr(workspace, "workspace", required=False),
        workspace.numel() * workspace.element_size() if workspace is not None else 0)


def dspark_verify(mode, target: torch.Tensor, block_tokens: torch.Tensor,
                  accept_len: torch.Tensor, committed: torch.Tensor, workspace: torch.Tensor, *,
                  stochastic: bool = False, draft: Optional[torch.Tensor] = None,
                  cu_seqlens: Optional[torch.Tensor] = None,
                  windows: Optional[torch.Tensor] = None,
                  ceiling_len: Optional[torch.Tensor] = None,
                  row_prob: Optional[torch.Tensor] = None, temperature: float = 1.0,
                  seed: int = 0, step: int = 0, status: Optional[torch.Tensor] = None,
                  stream=None, prepare: bool = False):
    args = _verify_args(mode, target, block_tokens, accept_len, committed, workspace,
                        stochastic, draft, cu_seqlens, windows, ceiling_len, row_prob,
                        temperature, seed, step)
    args += (_ptr(status, "status", torch.int32, min_numel=1, required=False), _stream(stream))
    return _call("dspark_verify", args, prepare)


def dspark_verify_scatter(mode, target: torch.Tensor, block_tokens: torch.Tensor,
                          accept_len: torch.Tensor, committed: torch.Tensor,
                          workspace: torch.Tensor, out_tokens: torch.Tensor,
                          out_len: torch.Tensor, *, stochastic: bool = False,
                          draft: Optional[torch.Tensor] = None,
                          cu_seqlens: Optional[torch.Tensor] = None,
                          windows: Optional[torch.Tensor] = None,
                          ceiling_len: Optional[torch.Tensor] = None,
                          row_prob: Optional[torch.Tensor] = None, temperature: float = 1.0,
                          seed: int = 0, step: int = 0, status: Optional[torch.Tensor] = None,
                          stream=None, prepare: bool = False):
    """dspark_verify then dspark_scatter of its committed tokens, without the scatter launch."""
    B = block_tokens.shape[0]
    cap = out_tokens.shape[1] if out_tokens.dim() == 2 else 0
    args = _verify_args(mode, target, block_tokens, accept_len, committed, workspace,
                        stochastic, draft, cu_seqlens, windows, ceiling_len, row_prob,
                        temperature, seed, step)
    args += (_ptr(out_tokens, "out_tokens", torch.int32, min_numel=B * cap, required=B * cap > 0),
             _ptr(out_len, "out_len", torch.int32, min_numel=B, required=B > 0), cap,
             _ptr(status, "status", torch.int32, min_numel=1, required=False), _stream(stream))
    return _call("dspark_verify_scatter", args, prepare)


def dspark_scatter(committed: torch.Tensor, accept_len: torch.Tensor, out_tokens: torch.Tensor,
                   out_len: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None,
                   prepare: bool = False):
    B, gamma = committed.shape
    cap = out_tokens.shape[1] if out_tokens.dim() == 2 else 0
    args = (
        _ptr(committed, "committed", torch.int32, required=B > 0),
        _ptr(accept_len, "accept_len", torch.int32, min_numel=B, required=B > 0), B, gamma,
        _ptr(out_tokens, "out_tokens", torch.int32, min_numel=B * cap, required=B * cap > 0),
        _ptr(out_len, "out_len", torch.int32, min_numel=B, required=B > 0), cap,
        _ptr(status, "status", torch.int32, min_numel=1, required=False), _stream(stream))
    return _call("dspark_scatter", args, prepare)


def dspark_observe(conf: torch.Tensor, accept_len: torch.Tensor, ceiling_len: torch.Tensor,
                   hist: torch.Tensor, util: torch.Tensor, status: Optional[torch.Tensor] = None,
                   stream=None, prepare: bool = False):
    """Accumulate calibration counters (hist: int64 [n_bins, 3]) and utilisation counters
    (util: int64 [2]) on the device; see ece() and utilisation() for the derived metrics."""
    B = accept_len.numel()
    L = conf.shape[-1] if conf.dim() == 2 else 0
    n_bins = hist.numel() // 3
    if hist.numel() != 3 * n_bins or n_bins < 1:
        raise ValueError("hist must hold 3 counters per bin")
    args = (_ptr(conf, "conf", torch.float32, numel=B * L, required=B > 0 and L > 0),
            _ptr(accept_len, "accept_len", torch.int32, required=B > 0),
            _ptr(ceiling_len, "ceiling_len", torch.int32, numel=B, required=B > 0), B, L + 1,
            n_bins, _ptr(hist, "hist", torch.int64), _ptr(util, "util", torch.int64, numel=2),
            _ptr(status, "status", torch.int32, min_numel=1, required=False), _stream(stream))
    return _call("dspark_observe", args, prepare)


def ece(hist) -> float:
    """Expected calibration error from dspark_observe's counters (n_bins x 3, host array)."""
    import numpy as np
    h = np.asarray(hist, dtype=np.float64).reshape(-1, 3)
    n = h[:, 0]
    N = n.sum()
    if N == 0:
        return 0.0
    nz = n > 0
    conf = h[nz, 1] / 4294967296.0 / n[nz]
    acc = h[nz, 2] / n[nz]
    return float((n[nz] / N * np.abs(acc - conf)).sum())


def utilisation(util) -> float:
    """Committed tokens over the acceptance ceiling, from dspark_observe's counters."""
    c, ceil = int(util[0]), int(util[1])
    return c / ceil if ceil else 0.0


NOALLOC_SCRATCH_BYTES = 4 << 20


def dspark_verify_noalloc(mode, target: torch.Tensor, block_tokens: torch.Tensor,
                          accept_len: torch.Tensor, committed: torch.Tensor, *,
                          stochastic: bool = False, draft: Optional[torch.Tensor] = None,
                          cu_seqlens: Optional[torch.Tensor] = None,
                          windows: Optional[torch.Tensor] = None,
                          ceiling_len: Optional[torch.Tensor] = None,
                          row_prob: Optional[torch.Tensor] = None, temperature: float = 1.0,
                          seed: int = 0, step: int = 0, status: Optional[torch.Tensor] = None,
                          stream=None):
    """dspark_verify without a workspace argument, for callers that cannot provide scratch
    memory: the library keeps a static 4 MiB device array per GPU and uses that instead.
    Calls that overlap on the GPU share the array; keep them ordered on one stream."""
    mode = MODES[mode] if isinstance(mode, str) else int(mode)
    B, gamma = block_tokens.shape
    rows, V = target.shape
    dt = _dtype_code(target)
    if draft is not None:
        if draft.dtype != target.dtype or draft.shape[-1] != V:
            raise ValueError("draft logits must match the target's dtype and vocabulary")
        if draft.numel() != B * (gamma - 1) * V:
            raise ValueError(f"draft logits must hold B*(gamma-1) = {B * (gamma - 1)} rows")
    rc = lib().dspark_verify_noalloc(
        mode, int(bool(stochastic)), _ptr(target, "target"), rows,
        _ptr(draft, "draft", required=False), dt, V,
        _ptr(cu_seqlens, "cu_seqlens", torch.int32, min_numel=B + 1, required=False),
        _ptr(windows, "windows", torch.int32, min_numel=B, required=False),
        _ptr(block_tokens, "block_tokens", torch.int32), B, gamma, float(temperature),
        int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
        _ptr(accept_len, "accept_len", torch.int32, min_numel=B),
        _ptr(committed, "committed", torch.int32, min_numel=B * gamma),
        _ptr(ceiling_len, "ceiling_len", torch.int32, min_numel=B, required=False),
        _ptr(row_prob, "row_prob", torch.float32, min_numel=2 * rows, required=False),
        _ptr(status, "status", torch.int32, min_numel=1, required=False), _stream(stream))
    _check("dspark_verify_noalloc", rc)
