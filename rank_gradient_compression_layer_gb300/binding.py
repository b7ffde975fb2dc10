"""ctypes binding of libpsgd.so (the C ABI in include/psgd.h).

Argument marshalling only: every step of the compression runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  There
is no fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpsgd.so")

PSGD_OK = 0
PSGD_ERR_INVALID = -1
PSGD_ERR_OOM = -2
PSGD_ERR_CUDA = -3
PSGD_ERR_TIMEOUT = -4
PSGD_ERR_STATE = -5

# every symbol include/psgd.h declares
EXPORTS = (
    "psgd_create", "psgd_create_ex", "psgd_destroy", "psgd_set_stream", "psgd_step", "psgd_step_host",
    "psgd_sync", "psgd_get_PQ", "psgd_get_Qw", "psgd_get_error", "psgd_set_state", "psgd_get_stats",
    "psgd_layer_info", "psgd_plan_layout", "psgd_count_sent", "psgd_last_error", "psgd_version",
    "psgd_get_phase_times", "psgd_step_noalloc", "psgd_step_momentum", "psgd_set_timing", "psgd_get_sparse",
    "psgd_plan_queue", "psgd_exchange_sizes", "psgd_step_begin", "psgd_step_mid", "psgd_step_end",
    "psgd_layer_flags", "psgd_plan_one_pass",
)

PSGD_POWERSGD = 0
PSGD_RTOPK = 1

PHASES = ("project", "orthonormalise", "back_project", "decompress")


class PsgdError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"psgd error {code}: {msg}")
        self.code = code


class Stats(ctypes.Structure):
    _fields_ = [
        ("steps", ctypes.c_int64),
        ("floats_sent", ctypes.c_int64),
        ("floats_uncompressed", ctypes.c_int64),
        ("floats_sent_per_step", ctypes.c_int64),
        ("floats_uncompressed_per_step", ctypes.c_int64),
        ("matrix_elements", ctypes.c_int64),
        ("vector_elements", ctypes.c_int64),
        ("buffer_elements", ctypes.c_int64),
        ("tiles", ctypes.c_int64 * 4),
        ("kernel_rank", ctypes.c_int32),
        ("launches_per_step", ctypes.c_int32),
        ("tile_rows", ctypes.c_int32 * 3),
        ("fused_step", ctypes.c_int32),
        ("message_floats", ctypes.c_int64),
        ("one_pass_project", ctypes.c_int32),
        ("reserved_", ctypes.c_int32),
    ]


class Options(ctypes.Structure):
    _fields_ = [("timing", ctypes.c_int32), ("project_rows", ctypes.c_int32), ("unbiased", ctypes.c_int32),
                ("compressor", ctypes.c_int32), ("rtopk_top_div", ctypes.c_int32),
                ("rtopk_sample_div", ctypes.c_int32), ("fused", ctypes.c_int32), ("wait_ms", ctypes.c_int32),
                ("queue_lag_kb", ctypes.c_int32), ("test_stall", ctypes.c_int32),
                ("total_workers", ctypes.c_int32), ("one_pass", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I64P = ctypes.POINTER(ctypes.c_int64)


def lib() -> ctypes.CDLL:
    """Load libpsgd.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libpsgd.so not built (expected at {LIB_PATH}); run the package's build()")
    L = ctypes.CDLL(LIB_PATH)
    sig = {
        "psgd_create": ([ctypes.POINTER(_P), ctypes.c_int, _I64P, _I64P, ctypes.c_int, ctypes.c_int,
                         ctypes.c_uint64, _P], ctypes.c_int),
        "psgd_create_ex": ([ctypes.POINTER(_P), ctypes.c_int, _I64P, _I64P, ctypes.c_int, ctypes.c_int,
                            ctypes.c_uint64, _P, ctypes.POINTER(Options)], ctypes.c_int),
        "psgd_destroy": ([_P], None),
        "psgd_set_stream": ([_P, _P], ctypes.c_int),
        "psgd_step": ([_P, ctypes.POINTER(_P), _P], ctypes.c_int),
        "psgd_step_host": ([_P, ctypes.POINTER(_P), _P, _P], ctypes.c_int),
        "psgd_step_momentum": ([_P, ctypes.POINTER(_P), _P, _P, ctypes.c_float, ctypes.c_float, _P], ctypes.c_int),
        "psgd_sync": ([_P], ctypes.c_int),
        "psgd_get_PQ": ([_P, ctypes.c_int, _P, _P], ctypes.c_int),
        "psgd_get_Qw": ([_P, ctypes.c_int, ctypes.c_int, _P], ctypes.c_int),
        "psgd_get_error": ([_P, ctypes.c_int, ctypes.c_int, _P], ctypes.c_int),
        "psgd_set_state": ([_P, ctypes.c_int, _P, ctypes.POINTER(_P)], ctypes.c_int),
        "psgd_get_stats": ([_P, ctypes.POINTER(Stats)], ctypes.c_int),
        "psgd_layer_info": ([_P, ctypes.c_int, _I64P, _I64P, _I64P, _I64P], ctypes.c_int),
        "psgd_layer_flags": ([_P, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
        "psgd_plan_layout": ([ctypes.c_int, _I64P, _I64P, _I64P, _I64P, _I64P], ctypes.c_int),
        "psgd_count_sent": ([ctypes.c_int, _I64P, _I64P, ctypes.c_int, _I64P, _I64P], ctypes.c_int),
        "psgd_exchange_sizes": ([_P, _I64P, _I64P], ctypes.c_int),
        "psgd_step_begin": ([_P, ctypes.POINTER(_P), _P], ctypes.c_int),
        "psgd_step_mid": ([_P, _P, _P], ctypes.c_int),
        "psgd_step_end": ([_P, _P, _P], ctypes.c_int),
        "psgd_plan_one_pass": ([ctypes.c_int, _I64P, _I64P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), _I64P], ctypes.c_int),
        "psgd_plan_queue": ([ctypes.c_int, _I64P, _I64P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                             ctypes.c_int, ctypes.POINTER(ctypes.c_int32), _I64P], ctypes.c_int),
        "psgd_last_error": ([], ctypes.c_char_p),
        "psgd_version": ([], ctypes.c_char_p),
        "psgd_get_phase_times": ([_P, ctypes.POINTER(ctypes.c_float)], ctypes.c_int),
        "psgd_set_timing": ([_P, ctypes.c_int], ctypes.c_int),
        "psgd_get_sparse": ([_P, ctypes.c_int, ctypes.c_int, _P, _P, _I64P], ctypes.c_int),
        "psgd_step_noalloc": ([ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_P),
                               _P, _P, _P, _P, _P, ctypes.c_int, _P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def _check(rc: int) -> None:
    if rc != PSGD_OK:
        raise PsgdError(rc, lib().psgd_last_error().decode(errors="replace"))


def _i64(values: Sequence[int]):
    return (ctypes.c_int64 * len(values))(*[int(v) for v in values])


def _shapes(shapes: Sequence[Tuple[int, int]]):
    return _i64([s[0] for s in shapes]), _i64([s[1] for s in shapes])


# ----------------------------------------------------------- host-only -----

def psgd_plan_layout(shapes: Sequence[Tuple[int, int]]) -> Tuple[List[int], List[int], int]:
    """(offsets, row strides, floats per packed buffer); needs no GPU."""
    n, m = _shapes(shapes)
    L = len(shapes)
    off, ld, tot = (ctypes.c_int64 * L)(), (ctypes.c_int64 * L)(), ctypes.c_int64()
    _check(lib().psgd_plan_layout(L, n, m, off, ld, ctypes.byref(tot)))
    return list(off), list(ld), tot.value


def psgd_count_sent(shapes: Sequence[Tuple[int, int]], rank: int) -> Tuple[int, int]:
    """Floats one worker sends per step (compressed, uncompressed); needs no GPU."""
    n, m = _shapes(shapes)
    c, u = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().psgd_count_sent(len(shapes), n, m, rank, ctypes.byref(c), ctypes.byref(u)))
    return c.value, u.value


def psgd_plan_queue(shapes: Sequence[Tuple[int, int]], rank: int, workers: int, project_rows: int = 0,
                    lag_bytes: int = 0, with_update: bool = True) -> List[Tuple[int, int, int, int, int]]:
    """The fused step's queue for a layer set, needs no GPU: a list of
    (phase, matrix or vector index, a, b, c) in queue order (see
    psgd_plan_queue in include/psgd.h)."""
    n, m = _shapes(shapes)
    cnt = ctypes.c_int64()
    _check(lib().psgd_plan_queue(len(shapes), n, m, rank, workers, project_rows, lag_bytes, int(with_update), None,
                                 ctypes.byref(cnt)))
    buf = (ctypes.c_int32 * (4 * cnt.value))()
    _check(lib().psgd_plan_queue(len(shapes), n, m, rank, workers, project_rows, lag_bytes, int(with_update), buf,
                                 ctypes.byref(cnt)))
    out = []
    for i in range(cnt.value):
        lay, a, b, c = buf[4 * i:4 * i + 4]
        out.append((lay >> 24, lay & 0xFFFFFF, a, b, c))
    return out


def psgd_plan_one_pass(shapes: Sequence[Tuple[int, int]], rank: int, workers: int, clusters: int):
    """The one-pass project's plan for a layer set, needs no GPU (see
    psgd_plan_one_pass in include/psgd.h): (per matrix layer (cw, yfc, yr,
    nys), per cluster its segments [(matrix index, first block, end block,
    slot), ...])."""
    n, m = _shapes(shapes)
    mats = sum(1 for _, b in shapes if b)
    cnt = ctypes.c_int64()
    _check(lib().psgd_plan_one_pass(len(shapes), n, m, rank, workers, clusters, None, None, ctypes.byref(cnt)))
    plan = (ctypes.c_int32 * (4 * max(mats, 1)))()
    buf = (ctypes.c_int32 * (4 * cnt.value))()
    _check(lib().psgd_plan_one_pass(len(shapes), n, m, rank, workers, clusters, plan, buf, ctypes.byref(cnt)))
    layers = [tuple(plan[4 * i:4 * i + 4]) for i in range(mats)]
    tiles = [tuple(buf[4 * i:4 * i + 4]) for i in range(cnt.value)]
    runs = []
    for c in range(clusters):
        _, first, segs, _ = tiles[c]
        runs.append(tiles[clusters + first:clusters + first + segs])
    return layers, runs


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


# ------------------------------------------------------------- context -----

class PowerSGD:
    """One compression context: layer shapes, rank r, W simulated workers.

    ``shapes`` lists (n, m) per layer; m == 0 marks a vector (averaged, not
    compressed).  Gradients are passed as packed float32 device buffers (see
    ``layout``/``pack``), one per worker.
    """

    def __init__(self, shapes: Sequence[Tuple[int, int]], rank: int, workers: int, seed: int = 0,
                 stream=None, timing: bool = False, project_rows: int = 0, unbiased: bool = False,
                 compressor: str = "powersgd", top_div: int = 100, sample_div: int = 4,
                 fused: bool = False, wait_ms: int = 0, queue_lag_kb: int = 0, test_stall: int = 0,
                 total_workers: int = 0, one_pass: bool = False):
        import torch

        if not torch.cuda.is_available():
            raise RuntimeError("PowerSGD needs a CUDA device")
        self.shapes = [(int(a), int(b)) for a, b in shapes]
        self.rank, self.workers, self.seed = int(rank), int(workers), int(seed)
        self.device = torch.device("cuda", torch.cuda.current_device())
        self._stream = stream
        n, m = _shapes(self.shapes)
        if compressor not in ("powersgd", "rtopk"):
            raise ValueError(f"unknown compressor {compressor!r}")
        opt = Options(int(bool(timing)), int(project_rows), int(bool(unbiased)),
                      PSGD_RTOPK if compressor == "rtopk" else PSGD_POWERSGD, int(top_div), int(sample_div),
                      int(bool(fused)), int(wait_ms), int(queue_lag_kb), int(test_stall),
                      int(total_workers), int(bool(one_pass)))
        h = _P()
        _check(lib().psgd_create_ex(ctypes.byref(h), len(self.shapes), n, m, self.rank, self.workers,
                                    ctypes.c_uint64(self.seed), _stream_ptr(stream), ctypes.byref(opt)))
        self._h = h
        self.offsets, self.lds, self.total = psgd_plan_layout(self.shapes)

    # -- lifetime
    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().psgd_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_stream(self, stream) -> None:
        self._stream = stream
        _check(lib().psgd_set_stream(self._h, _stream_ptr(stream)))

    # -- packed layout helpers (plain tensor copies, outside the step)
    def empty_buffer(self):
        import torch
        return torch.zeros(self.total, dtype=torch.float32, device=self.device)

    def layer_view(self, buf, layer: int):
        n, m = self.shapes[layer]
        off, ld = self.offsets[layer], self.lds[layer]
        if m == 0:
            return buf[off:off + n]
        return buf[off:off + n * ld].view(n, ld)[:, :m]

    def pack(self, tensors: Sequence, out=None):
        """Copy per-layer gradients ((n, m) or (n,)) into one packed buffer."""
        buf = self.empty_buffer() if out is None else out
        for li, t in enumerate(tensors):
            self.layer_view(buf, li).copy_(t)
        return buf

    def unpack(self, buf) -> List:
        return [self.layer_view(buf, li) for li in range(len(self.shapes))]

    # -- the step
    def step(self, grads: Sequence, out_update=None) -> None:
        if len(grads) != self.workers:
            raise ValueError(f"expected {self.workers} gradient buffers, got {len(grads)}")
        ptrs = (_P * self.workers)(*[_ptr(g) for g in grads])
        _check(lib().psgd_step(self._h, ptrs, _ptr(out_update)))

    def step_momentum(self, grads: Sequence, params, momentum, lr: float, beta: float, out_update=None) -> None:
        """One step, then momentum <- beta momentum + U; params <- params - lr (U + momentum).

        ``params`` and ``momentum`` are packed device buffers, updated in place.
        """
        if len(grads) != self.workers:
            raise ValueError(f"expected {self.workers} gradient buffers, got {len(grads)}")
        ptrs = (_P * self.workers)(*[_ptr(g) for g in grads])
        _check(lib().psgd_step_momentum(self._h, ptrs, _ptr(params), _ptr(momentum), float(lr), float(beta),
                                        _ptr(out_update)))

    def step_host(self, grads_host: Sequence, msg_host, update_host=None) -> None:
        ptrs = (_P * self.workers)(*[_ptr(g) for g in grads_host])
        _check(lib().psgd_step_host(self._h, ptrs, _ptr(msg_host), _ptr(update_host)))

    # -- the split step (workers spread over processes)
    def exchange_sizes(self) -> Tuple[int, int]:
        """Floats of the two exchange buffers of a split step (P, then Q + vectors)."""
        p, q = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().psgd_exchange_sizes(self._h, ctypes.byref(p), ctypes.byref(q)))
        return p.value, q.value

    def step_begin(self, grads: Sequence, p_out) -> None:
        if len(grads) != self.workers:
            raise ValueError(f"expected {self.workers} gradient buffers, got {len(grads)}")
        self._split_grads = list(grads)  # kept alive until step_end
        ptrs = (_P * self.workers)(*[_ptr(g) for g in grads])
        _check(lib().psgd_step_begin(self._h, ptrs, _ptr(p_out)))

    def step_mid(self, p_sum, q_out) -> None:
        _check(lib().psgd_step_mid(self._h, _ptr(p_sum), _ptr(q_out)))

    def step_end(self, q_sum, out_update=None) -> None:
        _check(lib().psgd_step_end(self._h, _ptr(q_sum), _ptr(out_update)))
        self._split_grads = None

    def step_split(self, grads: Sequence, out_update=None, all_reduce=None) -> None:
        """One step whose workers span processes: all_reduce(t) must sum the
        float32 device tensor t in place over the processes (for example
        torch.distributed.all_reduce); None means one process.  Runs on the
        context's stream, which must be the one the collectives follow (the
        current stream when the context was made with stream=None)."""
        import torch
        if getattr(self, "_xbufs", None) is None:
            p, q = self.exchange_sizes()
            self._xbufs = (torch.empty(max(p, 1), dtype=torch.float32, device=self.device),
                           torch.empty(max(q, 1), dtype=torch.float32, device=self.device))
        xp, xq = self._xbufs
        p, q = self.exchange_sizes()
        self.step_begin(grads, xp)
        if all_reduce is not None and p:
            all_reduce(xp[:p])
        self.step_mid(xp, xq)
        if all_reduce is not None and q:
            all_reduce(xq[:q])
        self.step_end(xq, out_update)

    def sync(self) -> None:
        _check(lib().psgd_sync(self._h))

    # -- state access
    def _shape(self, layer: int):
        # out-of-range layers are passed through so that the library reports them
        return self.shapes[layer] if 0 <= layer < len(self.shapes) else (1, 1)

    def get_PQ(self, layer: int):
        import torch
        n, m = self._shape(layer)
        P = torch.empty(n, self.rank, dtype=torch.float32, device=self.device)
        Q = torch.empty(m, self.rank, dtype=torch.float32, device=self.device)
        _check(lib().psgd_get_PQ(self._h, layer, _ptr(P), _ptr(Q)))
        return P, Q

    def get_sparse(self, layer: int, worker: int):
        """rTop-k: (indices int32, values float32) of worker's message for a matrix layer."""
        import torch
        cnt = ctypes.c_int64()
        _check(lib().psgd_get_sparse(self._h, layer, worker, None, None, ctypes.byref(cnt)))
        idx = torch.empty(cnt.value, dtype=torch.int32, device=self.device)
        val = torch.empty(cnt.value, dtype=torch.float32, device=self.device)
        _check(lib().psgd_get_sparse(self._h, layer, worker, _ptr(idx), _ptr(val), None))
        return idx, val

    def layer_flags(self, layer: int) -> dict:
        """How the last step treated matrix layer ``layer``: ``one_pass_qr`` (one
        Cholesky-QR pass sufficed) and ``q_from_y`` (Q_w formed from the one-pass
        project's partials, M not read again)."""
        f = ctypes.c_int32(0)
        _check(lib().psgd_layer_flags(self._h, layer, ctypes.byref(f)))
        return {"one_pass_qr": bool(f.value & 1), "q_from_y": bool(f.value & 2)}

    def get_Qw(self, layer: int, worker: int):
        import torch
        n, m = self._shape(layer)
        Q = torch.empty(m, self.rank, dtype=torch.float32, device=self.device)
        _check(lib().psgd_get_Qw(self._h, layer, worker, _ptr(Q)))
        return Q

    def get_error(self, layer: int, worker: int):
        import torch
        n, m = self._shape(layer)
        E = torch.empty(n, m, dtype=torch.float32, device=self.device)
        _check(lib().psgd_get_error(self._h, layer, worker, _ptr(E)))
        return E

    def set_state(self, layer: int, Q, E: Optional[Sequence] = None) -> None:
        Q = Q.contiguous()
        if E is not None:
            E = [e.contiguous() for e in E]
            arr = (_P * self.workers)(*[_ptr(e) for e in E])
        else:
            arr = None
        _check(lib().psgd_set_state(self._h, layer, _ptr(Q), arr))

    def stats(self) -> dict:
        s = Stats()
        _check(lib().psgd_get_stats(self._h, ctypes.byref(s)))
        out = {f: getattr(s, f) for f, _ in Stats._fields_}
        out["tiles"] = dict(zip(PHASES, list(s.tiles)))
        out["tile_rows"] = list(s.tile_rows)
        return out

    def set_timing(self, on: bool) -> None:
        """Per-phase events on or off for the following steps."""
        _check(lib().psgd_set_timing(self._h, 1 if on else 0))

    def phase_times(self) -> dict:
        """Device milliseconds of each phase, averaged over the steps since the
        last call (timing on); a fused step gives {"step": ms of the launch}."""
        ms = (ctypes.c_float * 4)()
        _check(lib().psgd_get_phase_times(self._h, ms))
        if self.fused:
            return {"step": ms[0]}
        return dict(zip(PHASES, list(ms)))

    @property
    def fused(self) -> bool:
        """True when each step is one fused launch."""
        return bool(self.stats()["fused_step"])

    @property
    def one_pass(self) -> bool:
        """True when each step runs the one-pass project (no second read of M)."""
        return bool(self.stats()["one_pass_project"])

    @property
    def message_floats(self) -> int:
        """Floats step_host writes to its message buffer (the library's count)."""
        return int(self.stats()["message_floats"])


# ------------------------------------------------------ no-allocation step --

def step_noalloc(n: int, m: int, rank: int, grads: Sequence, B, Phat, Qbar, Qw, out_update=None,
                 has_prev: bool = False, stream=None) -> None:
    """One step of one n x m layer with caller-owned state; nothing is allocated.

    ``grads`` holds one (n, ld) float32 device tensor per worker (ld = m
    rounded up to 4); ``B`` (W, n, ld), ``Phat`` (n, rank), ``Qbar`` (ld,
    rank) and ``Qw`` (W, ld, rank) are the state tensors and ``out_update``
    an (n, ld) tensor or None; see psgd_step_noalloc in include/psgd.h for
    what each holds before and after.  Asynchronous on ``stream`` (torch's
    current stream by default).
    """
    W = len(grads)
    arr = (_P * W)(*[_ptr(g) for g in grads])
    _check(lib().psgd_step_noalloc(int(n), int(m), int(rank), W, arr, _ptr(B), _ptr(Phat), _ptr(Qbar), _ptr(Qw),
                                   _ptr(out_update), 1 if has_prev else 0, _stream_ptr(stream)))
