"""Parallel runs of the CPU oracle for parity checks at full size.

The oracle is plain single-threaded C; a full-size comparison (billions of
elements) runs it on every host core instead: a pool of spawned worker
processes (spawn, never fork, because the parent has a CUDA context), each
running the oracle as it stands on a block of rows.  The matrices travel
through shared memory: the parent copies the input and the outputs under
test into it (straight from the GPU tensors), and each worker compares its
block of the oracle's result with the outputs byte for byte, returning only
counts, the first differing index and the block's amax.  Nothing here does
any of the method's arithmetic; it only splits rows and compares bytes.

Used by the -m gpu parity tests (the 48-tensor list, the FP8 conversion over
every fp32 bit pattern) and, with the oracle's own output planted as the
"device" result, by CPU tests of this module.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np


def _attach(name, shape, dtype):
    shm = shared_memory.SharedMemory(name=name)   # owned (and unlinked) by the parent
    return shm, np.ndarray(shape, dtype=dtype, buffer=shm.buf)


def _first_bad(a, b):
    bad = np.flatnonzero(a.reshape(-1) != b.reshape(-1))
    return int(bad.size), (int(bad[0]) if bad.size else -1)


def _worker(conn):
    """Serve tasks until None arrives.  Shared-memory segments are attached
    per task by name (the parent may grow them between tasks)."""
    import oracle
    while True:
        task = conn.recv()
        if task is None:
            break
        kind = task[0]
        try:
            if kind == "cast_transpose":
                _, names, rows, cols, r0, r1, scale, fmt, check_qt = task
                shx, x = _attach(names[0], (rows, cols), np.uint16)
                shq, q = _attach(names[1], (rows, cols), np.uint8)
                shqt, qt = _attach(names[2], (cols, rows), np.uint8) if check_qt else (None, None)
                try:
                    ref = oracle.cast_transpose(x[r0:r1], scale, fmt, want_qt=check_qt)
                    nq, fq = _first_bad(q[r0:r1], ref["q"])
                    nqt, fqt = (0, -1)
                    if check_qt:
                        nqt, fqt = _first_bad(np.ascontiguousarray(qt[:, r0:r1]), ref["qt"])
                    res = {"bad_q": nq, "first_q": (fq // cols + r0, fq % cols) if nq else None,
                           "bad_qt": nqt,
                           "first_qt": (fqt // (r1 - r0), fqt % (r1 - r0) + r0) if nqt else None,
                           "amax": float(ref["amax"])}
                    del x, q, qt
                finally:
                    for s in (shx, shq, shqt):
                        if s is not None:
                            s.close()
                conn.send(res)
            elif kind == "encode_patterns":
                _, name, n, p0, i0, i1, fmt = task
                sh, codes = _attach(name, (n,), np.uint8)
                try:
                    pats = np.arange(p0 + i0, p0 + i1, dtype=np.uint64).astype(np.uint32)
                    ref = oracle.fp8_encode(pats.view(np.float32), fmt)
                    nb, fb = _first_bad(codes[i0:i1], ref)
                    res = {"bad": nb, "first_pattern": (p0 + i0 + fb) if nb else None,
                           "got": int(codes[i0 + fb]) if nb else None,
                           "want": int(ref[fb]) if nb else None}
                    del codes
                finally:
                    sh.close()
                conn.send(res)
            elif kind == "encode_vs_search":
                # the oracle's encode against the exhaustive nearest-code search
                # over the fp32 bit patterns p0 .. p1 - 1 (< 2^31: sign clear)
                # and the same patterns with the sign bit set (no device involved)
                import fp8_search
                _, p0, p1, fmt = task
                pos = np.arange(p1 - p0, dtype=np.uint32) + np.uint32(p0)
                ref = fp8_search.nearest_code_by_search(pos.view(np.float32), fmt)
                res = {"bad": 0, "first_pattern": None, "got": None, "want": None}
                for pats, want in ((pos, ref),
                                   (pos | np.uint32(0x80000000),
                                    np.where(ref == 0x7F, ref, ref | 0x80).astype(np.uint8))):
                    # (the search gives 0x7F for NaN; a negative value's code is the
                    # positive one with the sign bit, NaN stays 0x7F)
                    mine = oracle.fp8_encode(pats.view(np.float32), fmt)
                    nb, fb = _first_bad(mine, want)
                    if nb and res["first_pattern"] is None:
                        res.update(first_pattern=int(pats[fb]), got=int(mine[fb]), want=int(want[fb]))
                    res["bad"] += nb
                conn.send(res)
            else:
                conn.send({"error": f"unknown task {kind!r}"})
        except Exception as e:   # reported to the parent, which raises
            conn.send({"error": repr(e)})


class _Segment:
    """A growable shared-memory segment owned by the parent."""

    def __init__(self):
        self.shm = None

    def ensure(self, nbytes):
        nbytes = max(int(nbytes), 1)
        if self.shm is None or self.shm.size < nbytes:
            self.close()
            self.shm = shared_memory.SharedMemory(create=True, size=nbytes)
        return self.shm

    def view(self, shape, dtype):
        return np.ndarray(shape, dtype=dtype, buffer=self.shm.buf)

    def close(self):
        if self.shm is not None:
            try:
                self.shm.close()
            except BufferError:   # a caller's view is still alive: unmapped when it dies
                pass
            self.shm.unlink()
            self.shm = None


class OraclePool:
    """Spawned oracle workers plus the shared segments they read.

    Use as a context manager.  `workers` defaults to every host core."""

    def __init__(self, workers: int | None = None):
        self.workers = max(1, workers or os.cpu_count() or 1)
        self.ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        self.seg = [_Segment() for _ in range(3)]

    def __enter__(self):
        for _ in range(self.workers):
            a, b = self.ctx.Pipe()
            p = self.ctx.Process(target=_worker, args=(b,), daemon=True)
            p.start()
            self.procs.append(p)
            self.conns.append(a)
        return self

    def __exit__(self, *exc):
        for c in self.conns:
            try:
                c.send(None)
            except Exception:
                pass
        for p in self.procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
        for s in self.seg:
            s.close()
        return False

    def _run(self, tasks):
        """Send tasks round-robin, at most one outstanding per worker."""
        results = [None] * len(tasks)
        pending = {}   # worker -> task index
        it = iter(enumerate(tasks))
        for w in range(self.workers):
            nxt = next(it, None)
            if nxt is None:
                break
            self.conns[w].send(nxt[1])
            pending[w] = nxt[0]
        while pending:
            for w in list(pending):
                c = self.conns[w]
                if not c.poll(0.005):
                    continue
                r = c.recv()
                if "error" in r:
                    raise RuntimeError(f"oracle worker failed: {r['error']}")
                results[pending.pop(w)] = r
                nxt = next(it, None)
                if nxt is not None:
                    c.send(nxt[1])
                    pending[w] = nxt[0]
        return results

    # ---- buffers the caller fills (numpy views into shared memory) -------
    def input_bf16(self, rows, cols):
        self.seg[0].ensure(2 * rows * cols)
        return self.seg[0].view((rows, cols), np.uint16)

    def output_q(self, rows, cols):
        self.seg[1].ensure(rows * cols)
        return self.seg[1].view((rows, cols), np.uint8)

    def output_qt(self, rows, cols):
        self.seg[2].ensure(rows * cols)
        return self.seg[2].view((cols, rows), np.uint8)

    def codes(self, n):
        self.seg[1].ensure(n)
        return self.seg[1].view((n,), np.uint8)

    # ---- checks -----------------------------------------------------------
    def check_cast_transpose(self, rows, cols, scale, fmt, check_qt=True, block_rows=None):
        """Compare the q (and qT) views filled by the caller with the oracle's
        cast-transpose of the input view, all rows.  Returns totals, the
        first differing (row, col) of q and of qT, and the oracle's amax."""
        if block_rows is None:
            block_rows = max(1, -(-rows // (4 * self.workers)))
        names = (self.seg[0].shm.name, self.seg[1].shm.name,
                 self.seg[2].shm.name if check_qt else None)
        tasks = [("cast_transpose", names, rows, cols, r0, min(rows, r0 + block_rows),
                  float(np.float32(scale)), fmt, check_qt)
                 for r0 in range(0, rows, block_rows)]
        res = self._run(tasks)
        out = {"bad_q": sum(r["bad_q"] for r in res), "bad_qt": sum(r["bad_qt"] for r in res),
               "first_q": next((r["first_q"] for r in res if r["bad_q"]), None),
               "first_qt": next((r["first_qt"] for r in res if r["bad_qt"]), None)}
        # amax: the largest IEEE magnitude pattern over the blocks (all >= 0)
        bits = np.array([r["amax"] for r in res], dtype=np.float32).view(np.uint32)
        out["amax"] = np.uint32(bits.max()).view(np.float32) if len(bits) else np.float32(0)
        return out

    def check_encode_against_search(self, p0, p1, fmt, chunk=1 << 18):
        """The oracle's encode of the fp32 patterns p0 .. p1 - 1 (p1 <= 2^31,
        the sign-clear half) and of the same patterns with the sign bit set,
        against the exhaustive nearest-code search (tests/fp8_search.py)."""
        assert 0 <= p0 <= p1 <= (1 << 31)
        tasks = [("encode_vs_search", a, min(p1, a + chunk), fmt) for a in range(p0, p1, chunk)]
        res = self._run(tasks)
        bad = [r for r in res if r["bad"]]
        return {"bad": sum(r["bad"] for r in res),
                "first": (bad[0]["first_pattern"], bad[0]["got"], bad[0]["want"]) if bad else None}

    def check_encode_patterns(self, p0, n, fmt, chunk=None):
        """Compare the codes view (filled by the caller with the conversion of
        the fp32 bit patterns p0 .. p0+n-1) with the oracle's encode."""
        if chunk is None:
            chunk = max(1, -(-n // (4 * self.workers)))
        name = self.seg[1].shm.name
        tasks = [("encode_patterns", name, n, p0, i0, min(n, i0 + chunk), fmt)
                 for i0 in range(0, n, chunk)]
        res = self._run(tasks)
        bad = [r for r in res if r["bad"]]
        return {"bad": sum(r["bad"] for r in res),
                "first": (bad[0]["first_pattern"], bad[0]["got"], bad[0]["want"]) if bad else None}
