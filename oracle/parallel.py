"""The C oracle run on every host core at once -- TEST INFRASTRUCTURE ONLY.

Only the tests and the benchmark's CPU-baseline leg use this module.  It holds
none of the quantizer's arithmetic: it splits a tensor into row stripes whose
heights are multiples of 16 (a columnwise block, a 16x16 tile and a
columnwise Hadamard vector each lie inside one stripe), runs the unmodified C
oracle (``oracle.amax`` and ``oracle.quantize`` with ``row0``/``row1``) on
each stripe in its own process, and assembles the results:

* the tensor amax per copy is the largest stripe amax (every element, and
  every Hadamard vector of either copy, lies in exactly one stripe);
* each stripe's quantize call writes its own rows of the rowwise outputs and
  its own byte range of every row of the columnwise outputs, so the stripes
  fill disjoint parts of shared output buffers.

Processes are started with the ``spawn`` method, so the pool is safe to use
after CUDA has been initialised in the parent.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import time
from multiprocessing import shared_memory

import numpy as np

__all__ = ["stripes", "amax_parallel", "quantize_parallel"]


def stripes(M: int, parts: int):
    """Row bounds [r0, r1) of up to `parts` stripes; every r0 is a multiple of 16."""
    blocks = (M + 15) // 16
    parts = max(1, min(parts, blocks))
    bounds = [min(M, 16 * (blocks * i // parts)) for i in range(parts)] + [M]
    return [(bounds[i], bounds[i + 1]) for i in range(parts) if bounds[i] < bounds[i + 1]]


def _nproc(nproc):
    return max(1, nproc or len(os.sched_getaffinity(0)))


class _Shared:
    """A numpy array in a shared-memory block (created by the parent)."""

    def __init__(self, shape, dtype, fill=None):
        self.shape, self.dtype = tuple(shape), np.dtype(dtype)
        n = int(np.prod(self.shape)) * self.dtype.itemsize
        self.shm = shared_memory.SharedMemory(create=True, size=max(n, 1))
        self.array = np.ndarray(self.shape, self.dtype, buffer=self.shm.buf)
        if fill is not None:
            self.array[...] = fill

    def spec(self):
        return (self.shm.name, self.shape, self.dtype.str)

    def close(self):
        del self.array
        self.shm.close()
        self.shm.unlink()


def _attach(spec):
    name, shape, dtype = spec
    shm = shared_memory.SharedMemory(name=name)
    return shm, np.ndarray(shape, np.dtype(dtype), buffer=shm.buf)


def _amax_worker(x_spec, N, r0, r1, flags, rht_seed):
    import oracle
    shm, x = _attach(x_spec)
    try:
        st, am = oracle.amax(x[r0:r1], flags, rht_seed, N=N)
        return st, (float(am[0]), float(am[1]))
    finally:
        del x
        shm.close()


def _quant_worker(x_spec, out_specs, N, r0, r1, amax2, flags, sel, sr_seed, rht_seed, counter_offset):
    import oracle
    shm, x = _attach(x_spec)
    att = [None if s is None else _attach(s) for s in out_specs]
    try:
        outs = tuple(None if a is None else a[1] for a in att)
        t0 = time.monotonic()
        r = oracle.quantize(x, N, np.asarray(amax2, np.float32), flags, sel=sel, sr_seed=sr_seed,
                            rht_seed=rht_seed, counter_offset=counter_offset, row0=r0, row1=r1, outs=outs)
        return r["status"], t0, time.monotonic(), [float(v) for v in r["alpha"]]
    finally:
        del x
        shm.close()
        for a in att:
            if a is not None:
                a[0].close()


def _pool(n):
    return mp.get_context("spawn").Pool(n)


def amax_parallel(bits: np.ndarray, flags: int, rht_seed: int = 0, nproc: int | None = None, N: int | None = None):
    """(status, float32[2]) of oracle.amax over the whole tensor, computed per stripe."""
    M, ld = bits.shape
    N = ld if N is None else N
    xs = _Shared(bits.shape, np.uint16, bits)
    try:
        with _pool(_nproc(nproc)) as pool:
            res = pool.starmap(_amax_worker, [(xs.spec(), N, r0, r1, flags, rht_seed)
                                              for r0, r1 in stripes(M, _nproc(nproc))])
    finally:
        xs.close()
    for st, _ in res:
        if st != 0:
            return st, np.zeros(2, np.float32)
    am = np.array([max(r[1][0] for r in res), max(r[1][1] for r in res)], np.float32) if res else np.zeros(2, np.float32)
    return 0, am


def quantize_parallel(bits: np.ndarray, flags: int, sel: int = 0, sr_seed: int = 0, rht_seed: int = 0,
                      counter_offset: int = 0, amax2=None, nproc: int | None = None):
    """oracle.quantize of the whole tensor, one process per stripe.

    Returns dict(status, amax, alpha, q_row, s_row, q_col, s_col, seconds, procs):
    `seconds` runs from the first stripe's start to the last one's finish
    (the quantize calls only; the amax is taken first, also in parallel,
    unless `amax2` is given)."""
    import oracle
    M, N = bits.shape
    n = _nproc(nproc)
    if amax2 is None:
        st, amax2 = amax_parallel(bits, flags, rht_seed, n)
        if st != 0:
            return dict(status=st)
    amax2 = np.asarray(amax2, np.float32)
    shapes = oracle.output_buffers(M, N, flags)
    xs = _Shared(bits.shape, np.uint16, bits)
    outs = [None if a is None else _Shared(a.shape, np.uint8, 0) for a in shapes]
    try:
        parts = stripes(M, n)
        with _pool(n) as pool:
            res = pool.starmap(_quant_worker,
                               [(xs.spec(), [None if o is None else o.spec() for o in outs], N, r0, r1,
                                 amax2.tolist(), flags, sel, sr_seed, rht_seed, counter_offset) for r0, r1 in parts])
        status = next((r[0] for r in res if r[0] != 0), 0)
        result = [None if o is None else o.array.copy() for o in outs]
        seconds = (max(r[2] for r in res) - min(r[1] for r in res)) if res else 0.0
        alpha = np.array(res[0][3] if res else [0.0, 0.0], np.float32)
    finally:
        xs.close()
        for o in outs:
            if o is not None:
                o.close()
    return dict(status=status, amax=amax2, alpha=alpha, q_row=result[0], s_row=result[1], q_col=result[2],
                s_col=result[3], seconds=seconds, procs=len(parts))
