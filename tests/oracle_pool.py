"""Parallel evaluation of the oracle for the full-size parity tests.

The oracle is unchanged: every task is one call of its own functions
(``sampled_forward``, ``sampled_dq``, ``attention_backward``) on a slice of
the query rows, in fp64 on the host cores. The pieces are put back together
here, using only what the definitions give:
* the forward and dQ of a query row depend on that row alone, so rows are
  split freely;
* dK and dV of a key are sums over the query rows that see it, so the sums
  over a partition of those rows add up to the whole;
* query heads are independent given their KV head (query head h uses KV
  head h // G), so each task handles one KV head and its G query heads.
Keys that no row of a task can see (after the task's last position, or
before the document of its first row) are left out of the task, as the
oracle itself skips them.

Workers are started with the ``spawn`` method (the parent holds a CUDA
context) and one BLAS thread each. K and V, in natural token order as bf16
bit patterns, go to temporary .npy files that the workers map read-only;
query-side rows travel with the tasks.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS",
                "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS")


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def host_memory_bytes() -> int:
    """Memory this process may still use: MemAvailable, capped by a cgroup
    limit when there is one."""
    avail = 1 << 60
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    for path in ("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory/memory.limit_in_bytes"):
        try:
            with open(path) as f:
                v = f.read().strip()
            if v.isdigit():
                avail = min(avail, int(v))
        except OSError:
            pass
    return avail


# largest host memory one task takes (a million-key prefix of K and V in fp64
# plus a 32-row block of scores and its temporaries)
TASK_BYTES = 4 << 30


# ---------------------------------------------------------------- workers
_MAPS = {}


def _mapped(path):
    a = _MAPS.get(path)
    if a is None:
        a = np.load(path, mmap_mode="r")
        _MAPS[path] = a
    return a


def _widen(bits):
    from workloads import bf16_bits_to_f64
    return bf16_bits_to_f64(np.ascontiguousarray(bits))


def _key_span(spec, qp_min, qp_max):
    """[ka, kb): the keys any row with positions in [qp_min, qp_max] can see
    (natural key index = position)."""
    cu = spec["cu"]
    ka = 0
    if cu is not None:
        ka = int(cu[np.searchsorted(cu, qp_min, side="right") - 1])
    return ka, int(qp_max) + 1


def _run_task(task):
    import oracle
    spec, kind, g, qbits, dbits, qp, extra = task
    k_all, v_all = _mapped(spec["k"]), _mapped(spec["v"])
    cu = spec["cu"]
    ka, kb = _key_span(spec, qp.min(), qp.max())
    kk = _widen(k_all[ka:kb, g:g + 1])
    vv = _widen(v_all[ka:kb, g:g + 1])
    kp = np.arange(ka, kb)
    qq = _widen(qbits)
    sub = np.arange(len(qp))
    if kind == "forward":
        return oracle.sampled_forward(qq, kk, vv, sub, qp, kp, cu)
    if kind == "dq":
        return oracle.sampled_dq(qq, kk, vv, _widen(dbits), sub, qp, kp, cu)
    O, L = oracle.sampled_forward(qq, kk, vv, sub, qp, kp, cu)
    if kind == "dkdv":  # the share of these rows in dK/dV of keys [a, b)
        a, b = extra
        dq, dk, dv = oracle.attention_backward(
            qq, _widen(k_all[a:b, g:g + 1]), _widen(v_all[a:b, g:g + 1]), _widen(dbits),
            O, L, qp, np.arange(a, b), cu)
        return dk, dv
    if kind == "backward":  # O, LSE, dQ of these rows, their share of dK/dV
        dq, dk, dv = oracle.attention_backward(qq, kk, vv, _widen(dbits), O, L, qp, kp, cu)
        return O, L, dq, ka, dk, dv
    raise ValueError(kind)


# ---------------------------------------------------------------- parent
class OraclePool:
    """A pool of spawned worker processes running the oracle."""

    def __init__(self, n_workers: int | None = None):
        by_memory = max(1, int(0.6 * host_memory_bytes() // TASK_BYTES))
        self.n = max(1, min(n_workers or host_cores(), by_memory, 32))
        saved = {k: os.environ.get(k) for k in _THREAD_VARS}
        for k in _THREAD_VARS:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.n)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.tmp = tempfile.mkdtemp(prefix="cp_attn_oracle_")
        self._count = 0

    def close(self):
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.tmp, ignore_errors=True)

    def problem(self, inp, kv_prefix_len: int = 0):
        """Register one workload's inputs (bf16 bits, natural order)."""
        paths = []
        for x in (inp.k, inp.v):
            self._count += 1
            p = os.path.join(self.tmp, f"a{self._count}.npy")
            np.save(p, np.ascontiguousarray(x))
            paths.append(p)
        G = inp.q.shape[1] // inp.k.shape[1]
        cu = None if inp.cu_seqlens is None else np.asarray(inp.cu_seqlens, dtype=np.int64)
        return {"k": paths[0], "v": paths[1], "G": G, "Hkv": inp.k.shape[1],
                "P": int(kv_prefix_len), "cu": cu, "q": inp.q, "dout": inp.dout}

    # -- task construction
    def _chunks(self, spec, rows, n_chunks):
        """Split sorted natural query rows into about n_chunks pieces of
        similar oracle work (visible keys per row)."""
        rows = np.asarray(rows, dtype=np.int64)
        if len(rows) == 0:
            return []
        qp = spec["P"] + rows
        cu = spec["cu"]
        start = np.zeros_like(qp) if cu is None else cu[np.searchsorted(cu, qp, side="right") - 1]
        work = np.cumsum((qp - start + 1).astype(np.float64))
        cuts = np.searchsorted(work, np.linspace(0, work[-1], n_chunks + 1)[1:-1])
        return [c for c in np.split(rows, np.unique(cuts)) if len(c)]

    def _tasks(self, spec, kind, rows, heads_of, extra=None, per_worker=4):
        G = spec["G"]
        tasks, index = [], []
        for g in heads_of:
            hs = slice(g * G, (g + 1) * G)
            for r in self._chunks(spec, rows, per_worker * self.n):
                qb = np.ascontiguousarray(spec["q"][r][:, hs])
                db = None
                if kind != "forward":
                    db = np.ascontiguousarray(spec["dout"][r][:, hs])
                tasks.append(({k: spec[k] for k in ("k", "v", "cu")}, kind, g, qb, db,
                              spec["P"] + r, extra))
                index.append((g, r))
        return tasks, index

    # -- public calls; each returns a handle whose .get() gives the result
    def forward_rows(self, spec, rows):
        """O [len(rows), Hq, d] and LSE [Hq, len(rows)] at natural rows."""
        rows = np.asarray(rows, dtype=np.int64)
        tasks, index = self._tasks(spec, "forward", rows, range(spec["Hkv"]))
        res = self.pool.map_async(_run_task, tasks, chunksize=1)
        Hq, d = spec["q"].shape[1], spec["q"].shape[2]
        G = spec["G"]

        def get():
            O = np.zeros((len(rows), Hq, d))
            L = np.zeros((Hq, len(rows)))
            pos = {int(r): i for i, r in enumerate(rows)}
            for (g, r), (o, l) in zip(index, res.get()):
                at = np.array([pos[int(x)] for x in r])
                O[at, g * G:(g + 1) * G] = o
                L[g * G:(g + 1) * G, at] = l
            return O, L
        return _Handle(get)

    def dq_rows(self, spec, rows):
        """dQ [len(rows), Hq, d] at natural rows."""
        rows = np.asarray(rows, dtype=np.int64)
        tasks, index = self._tasks(spec, "dq", rows, range(spec["Hkv"]))
        res = self.pool.map_async(_run_task, tasks, chunksize=1)
        Hq, d = spec["q"].shape[1], spec["q"].shape[2]
        G = spec["G"]

        def get():
            out = np.zeros((len(rows), Hq, d))
            pos = {int(r): i for i, r in enumerate(rows)}
            for (g, r), dq in zip(index, res.get()):
                out[np.array([pos[int(x)] for x in r]), g * G:(g + 1) * G] = dq
            return out
        return _Handle(get)

    def dkdv_keys(self, spec, a: int, b: int):
        """dK, dV [b - a, Hkv, d] of the natural keys [a, b): the sums over
        every query row that sees one of them."""
        P, cu = spec["P"], spec["cu"]
        n_new = spec["q"].shape[0]
        # rows that can see a key in [a, b): positions from a up to the end
        # of the last key's document
        hi = P + n_new if cu is None else int(cu[np.searchsorted(cu, b - 1, side="right")])
        rows = np.arange(max(a, P), hi) - P
        Hkv, d = spec["Hkv"], spec["q"].shape[2]
        tasks, index = self._tasks(spec, "dkdv", rows, range(Hkv), extra=(a, b))
        res = self.pool.map_async(_run_task, tasks, chunksize=1)

        def get():
            dk = np.zeros((b - a, Hkv, d))
            dv = np.zeros((b - a, Hkv, d))
            for (g, _), (k_, v_) in zip(index, res.get()):
                dk[:, g] += k_[:, 0]
                dv[:, g] += v_[:, 0]
            return dk, dv
        return _Handle(get)

    def backward_head(self, spec, g: int):
        """Whole forward and backward of KV head g and its G query heads:
        O [N, G, d], LSE [G, N], dQ [N, G, d], dK and dV [P + N, d]."""
        n_new = spec["q"].shape[0]
        rows = np.arange(n_new)
        tasks, index = self._tasks(spec, "backward", rows, [g], per_worker=3)
        res = self.pool.map_async(_run_task, tasks, chunksize=1)
        G, d = spec["G"], spec["q"].shape[2]
        n_kv = spec["P"] + n_new

        def get():
            O = np.zeros((n_new, G, d))
            L = np.zeros((G, n_new))
            dq = np.zeros((n_new, G, d))
            dk = np.zeros((n_kv, d))
            dv = np.zeros((n_kv, d))
            for (_, r), (o, l, q_, ka, k_, v_) in zip(index, res.get()):
                O[r], L[:, r], dq[r] = o, l, q_
                dk[ka:ka + len(k_)] += k_[:, 0]
                dv[ka:ka + len(v_)] += v_[:, 0]
            return O, L, dq, dk, dv
        return _Handle(get)


class _Handle:
    def __init__(self, fn):
        self._fn = fn
        self._val = None
        self._done = False

    def get(self):
        if not self._done:
            self._val = self._fn()
            self._done = True
        return self._val
