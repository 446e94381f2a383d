"""Process pool for oracle checks on large workloads -- TEST INFRASTRUCTURE.

Each (b, h) head is independent, so sampled-row checks fan the heads out to
worker processes started with the ``spawn`` method (never ``fork``: a pool
forked after CUDA has been initialised hangs).  Workers run BLAS with
``cores // workers`` threads each, so the total thread count equals the
number of cores available.  Arithmetic is the
oracle's own (``usp_oracle.attention_rows`` / ``attention_bwd_sampled``).
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np


def default_workers() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _rows_job(args):
    from oracle.usp_oracle import attention_rows
    qh, kh, vh, rows, scale = args
    return attention_rows(qh, kh, vh, rows, scale, row_block=512)


def _bwd_job(args):
    from oracle.usp_oracle import attention_bwd_sampled
    qh, kh, vh, doh, scale, qrows, krows = args
    return attention_bwd_sampled(qh, kh, vh, doh, scale, qrows, krows, row_block=512)


def _executor(workers: int, threads_each: int = 1):
    old = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")}
    os.environ["OPENBLAS_NUM_THREADS"] = str(threads_each)
    os.environ["OMP_NUM_THREADS"] = str(threads_each)
    try:
        ex = cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))
        # start the workers now, while the single-thread environment is set
        list(ex.map(int, range(workers)))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return ex


def sampled_attention(q, k, v, rows, scale, workers: int | None = None):
    """Oracle O and LSE at query ``rows`` for every head.

    q, k, v: float32/float64 numpy arrays [BH, N, D] holding the exact input
    values (bf16 inputs widened).  Returns (O [BH, R, D], L [BH, R]) fp64.
    """
    workers = workers or default_workers()
    BH = q.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    jobs = split_row_jobs(q, k, v, rows, scale, workers)
    if workers == 1:
        res = [_rows_job(j) for j in jobs]
    else:
        with _executor(min(workers, len(jobs))) as ex:
            res = list(ex.map(_rows_job, jobs))
    return join_row_results(res, BH)


def split_row_jobs(q, k, v, rows, scale, workers: int):
    """One job per (head, slice of ``rows``): the rows of a head are cut into
    as many slices as it takes to give every worker a job (rows are
    independent, so this changes no arithmetic)."""
    BH = q.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    per_head = max(1, min(len(rows), -(-workers // BH)))
    cuts = np.array_split(np.arange(len(rows)), per_head)
    return [(q[h][rows[c]], k[h], v[h], np.arange(len(c)), scale) for h in range(BH) for c in cuts if len(c)]


def join_row_results(res, BH: int):
    """Reassemble the per-(head, slice) results of :func:`split_row_jobs`."""
    per = len(res) // BH
    O = [np.concatenate([r[0] for r in res[h * per:(h + 1) * per]]) for h in range(BH)]
    L = [np.concatenate([r[1] for r in res[h * per:(h + 1) * per]]) for h in range(BH)]
    return np.stack(O), np.stack(L)


def rows_executor(workers: int):
    """A spawn pool of ``workers`` single-threaded oracle workers, started."""
    return _executor(workers, 1)


def rows_job(job):
    """Run one job of :func:`split_row_jobs` (in a worker or in-process)."""
    return _rows_job(job)


def sampled_backward(q, k, v, dout, scale, heads, qrows, krows, workers: int | None = None):
    """Oracle dq at ``qrows`` and dk, dv at ``krows`` for the listed heads.

    q, k, v, dout: numpy [BH, N, D]; ``heads`` indexes the BH axis.
    Returns (dq [len(heads), Rq, D], dk [len(heads), Rk, D], dv [...]) fp64.
    """
    workers = workers or default_workers()
    jobs = [(q[h], k[h], v[h], dout[h], scale, qrows, krows) for h in heads]
    if workers == 1:
        res = [_bwd_job(j) for j in jobs]
    else:
        nw = min(workers, len(jobs))
        with _executor(nw, max(1, workers // nw)) as ex:
            res = list(ex.map(_bwd_job, jobs))
    return (np.stack([r[0] for r in res]), np.stack([r[1] for r in res]),
            np.stack([r[2] for r in res]))
