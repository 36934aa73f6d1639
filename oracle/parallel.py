"""Row-parallel runner of the CPU oracle over this host's cores.

TEST AND BASELINE INFRASTRUCTURE ONLY, like the rest of ``oracle/``: used by
the full-size parity tests and by the benchmark's CPU legs, never by the
product path.  It holds none of the method's arithmetic.  It cuts a problem
into row slices, runs the unchanged functions of ``fp8_oracle`` on each
slice in worker processes, and pastes the slices back together.

Why slicing is exact, from the grouping of "The Definitive Information To
Deepseek" (paragraph 3, "Figure 7 (a)"):
  * 1x128 activation groups lie within one row, so the codes and scales of a
    row slice of X are those rows of the whole result;
  * 128x128 weight blocks lie within one 128-row slab of W, so slices cut on
    multiples of 128 rows quantise exactly as the whole matrix;
  * an output row of the block-scaled GEMM needs only its own row of codes
    and scales and all of the weights, and a grouped GEMM's rows use their
    group's weights.
The oracle pins check row independence and grouped = concatenated dense.

Workers are started with the "spawn" method (safe in a process that already
holds a CUDA context) and with one BLAS thread each, so that the pool uses
each core once.  Arrays travel through shared memory, not pickles.
"""
from __future__ import annotations

import contextlib
import os
import sys
import types
from multiprocessing import get_context, shared_memory

import numpy as np

from . import fp8_oracle as _o

_BLAS_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def host_cores() -> int:
    """Cores this process may run on (its affinity mask)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# Shared arrays
# ---------------------------------------------------------------------------
class _Shared:
    """A numpy array in a named shared-memory block."""

    def __init__(self, shape, dtype, fill=None):
        dtype = np.dtype(dtype)
        nbytes = max(1, int(np.prod(shape)) * dtype.itemsize)
        self.shm = shared_memory.SharedMemory(create=True, size=nbytes)
        self.desc = (self.shm.name, tuple(int(s) for s in shape), dtype.str)
        self.array = np.ndarray(shape, dtype=dtype, buffer=self.shm.buf)
        if fill is not None:
            self.array[...] = fill

    def close(self):
        self.array = None
        self.shm.close()
        self.shm.unlink()


_ATTACHED = {}


def _view(desc):
    name, shape, dtype = desc
    shm = _ATTACHED.get(name)
    if shm is None:
        shm = shared_memory.SharedMemory(name=name)
        _ATTACHED[name] = shm
    return np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)


def _detach(names):
    for name in names:
        shm = _ATTACHED.pop(name, None)
        if shm is not None:
            shm.close()


def _as_f32(a):
    """float32 values of BF16 inputs given as float32, or as raw BF16 bit
    patterns (uint16/int16): a BF16 value is the top half of its float32."""
    a = np.asarray(a)
    if a.dtype in (np.uint16, np.int16):
        return (a.view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32, copy=False)


# ---------------------------------------------------------------------------
# Worker tasks: each runs an unchanged oracle function on one slice.
# ---------------------------------------------------------------------------
def _task_quant_act(x, qa, sa, r0, r1):
    q, s = _o.quant_act_1x128(_as_f32(_view(x)[r0:r1]))
    _view(qa)[r0:r1] = q
    _view(sa)[:, r0:r1] = s


def _task_quant_weight(w, qw, sw, r0, r1):
    q, s = _o.quant_weight_128x128(_as_f32(_view(w)[r0:r1]))
    _view(qw)[r0:r1] = q
    _view(sw)[r0 // _o.GROUP:r1 // _o.GROUP] = s


def _task_gemm(qa, sa, qw, sw, y, r0, r1):
    _view(y)[r0:r1] = _o.blockscaled_gemm(_view(qa)[r0:r1], _view(sa)[:, r0:r1], _view(qw), _view(sw))


def _task_grouped_gemm(qa, sa, qw, sw, y, g, r0, r1):
    _view(y)[r0:r1] = _o.blockscaled_gemm(_view(qa)[r0:r1], _view(sa)[:, r0:r1], _view(qw)[g], _view(sw)[g])


def _run(task, args):
    try:
        task(*args)
    finally:
        _detach([a[0] for a in args if isinstance(a, tuple) and len(a) == 3 and isinstance(a[0], str)])


def _init_worker():
    # spawn children start from a fresh interpreter: nothing to reset but the
    # BLAS pools, already limited through the environment
    pass


@contextlib.contextmanager
def _spawn_environment():
    """One BLAS thread per worker, and a bare __main__ so that a spawned
    worker imports only numpy and the oracle, not the launching script."""
    saved_env = {k: os.environ.get(k) for k in _BLAS_ENV}
    saved_main = sys.modules.get("__main__")
    for k in _BLAS_ENV:
        os.environ[k] = "1"
    sys.modules["__main__"] = types.ModuleType("__main__")
    try:
        yield
    finally:
        sys.modules["__main__"] = saved_main
        for k, v in saved_env.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _slices(n, parts, align=1):
    """[r0, r1) slices of range(n) with boundaries on multiples of `align`."""
    units = -(-n // align)
    parts = max(1, min(parts, units))
    bounds = [min(n, (units * i // parts) * align) for i in range(parts + 1)]
    return [(bounds[i], bounds[i + 1]) for i in range(parts) if bounds[i + 1] > bounds[i]]


class OraclePool:
    """Process pool that runs the oracle on row slices.

        with OraclePool() as pool:
            qa, sa = pool.quant_act_1x128(x)          # x float32 or BF16 bits
            qw, sw = pool.quant_weight_128x128(w)
            y = pool.blockscaled_gemm(qa, sa, qw, sw)

    Results equal those of the same functions in ``oracle`` called on the
    whole arrays."""

    def __init__(self, workers=None):
        self.workers = int(workers or host_cores())
        with _spawn_environment():
            self._pool = get_context("spawn").Pool(self.workers, initializer=_init_worker)
        self._shared = []

    # -- plumbing --
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def close(self):
        if self._pool is not None:
            self._pool.terminate()
            self._pool.join()
            self._pool = None
        self._release()

    def _share(self, a):
        a = np.ascontiguousarray(a)
        s = _Shared(a.shape, a.dtype)
        s.array[...] = a
        self._shared.append(s)
        return s

    def _out(self, shape, dtype):
        s = _Shared(shape, dtype)
        self._shared.append(s)
        return s

    def _release(self):
        for s in self._shared:
            s.close()
        self._shared = []

    def _map(self, jobs):
        results = [self._pool.apply_async(_run, (task, args)) for task, args in jobs]
        for r in results:
            r.get()

    def _parts(self):
        return 4 * self.workers

    # -- the oracle, row-parallel --
    def quant_act_1x128(self, x):
        """oracle.quant_act_1x128 over row slices: (qa [M, K], sa [K/128, M])."""
        M, K = np.shape(x)
        try:
            xs = self._share(x)
            qa = self._out((M, K), np.uint8)
            sa = self._out((K // _o.GROUP, M), np.float32)
            self._map([(_task_quant_act, (xs.desc, qa.desc, sa.desc, r0, r1))
                       for r0, r1 in _slices(M, self._parts())])
            return qa.array.copy(), sa.array.copy()
        finally:
            self._release()

    def quant_weight_128x128(self, w):
        """oracle.quant_weight_128x128 over 128-row slabs: (qw [N, K], sw [N/128, K/128])."""
        N, K = np.shape(w)
        try:
            ws = self._share(w)
            qw = self._out((N, K), np.uint8)
            sw = self._out((N // _o.GROUP, K // _o.GROUP), np.float32)
            self._map([(_task_quant_weight, (ws.desc, qw.desc, sw.desc, r0, r1))
                       for r0, r1 in _slices(N, self._parts(), align=_o.GROUP)])
            return qw.array.copy(), sw.array.copy()
        finally:
            self._release()

    def blockscaled_gemm(self, qa, sa, qw, sw):
        """oracle.blockscaled_gemm over row slices: float64 [M, N]."""
        M = np.shape(qa)[0]
        N = np.shape(qw)[0]
        try:
            args = [self._share(a).desc for a in (qa, np.asarray(sa)[:, :M], qw, sw)]
            y = self._out((M, N), np.float64)
            self._map([(_task_gemm, (*args, y.desc, r0, r1)) for r0, r1 in _slices(M, self._parts())])
            return y.array.copy()
        finally:
            self._release()

    def blockscaled_grouped_gemm(self, offsets, qa, sa, qw, sw):
        """oracle.blockscaled_grouped_gemm over row slices of each group:
        float64 [offsets[G], N]."""
        offsets = [int(o) for o in offsets]
        G = len(offsets) - 1
        N = np.shape(qw)[1]
        M = offsets[-1]
        try:
            args = [self._share(a).desc for a in (qa, np.asarray(sa)[:, :M], qw, sw)]
            y = self._out((M, N), np.float64)
            per_group = max(1, -(-self._parts() // max(G, 1)))
            jobs = []
            for g in range(G):
                r0, r1 = offsets[g], offsets[g + 1]
                for a, b in _slices(r1 - r0, per_group):
                    jobs.append((_task_grouped_gemm, (*args, y.desc, g, r0 + a, r0 + b)))
            self._map(jobs)
            return y.array.copy()
        finally:
            self._release()
