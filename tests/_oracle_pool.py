"""The oracle's output for every decode row of a full-size workload, computed
in a pool of spawned worker processes.

Test infrastructure only: each worker replays the workload on the oracle's own
allocator model (``oracle.replay``) and, per row, takes the branch's logical
token sequence and runs the oracle on it (``oracle.attention`` for bf16;
``oracle.fp8.quantize_sequence`` then ``oracle.attention`` for e4m3).  Nothing
here touches the CUDA library.  Workers are spawned (not forked), so the pool
can start after the GPU has been used.
"""

from __future__ import annotations

import multiprocessing as mp
import os

# One BLAS thread per worker process (the workers inherit this environment
# and load their BLAS after it is set); the pool supplies the parallelism.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ[_v] = "1"

import numpy as np  # noqa: E402

_W = None
_REF = None
_BIG: dict = {}      # the most recent long source node's rows (a shared root)


def _init(name):
    global _W, _REF
    from oracle import replay as rp
    from paged_kv_cache_attn_gb300 import workloads as W
    _W = W.CONFIGS[name]()
    _REF = rp.replay(_W, with_data=False)


def _source(src):
    n = _W.nodes[src].n_tokens
    if n < 2048:
        return _W.node_kv(src)
    if src not in _BIG:
        _BIG.clear()
        _BIG[src] = _W.node_kv(src)
    return _BIG[src]


def _branch(nid):
    ks, vs, lens = [], [], []
    for src, lo, hi in _REF.logical[nid]:
        k, v = _source(src)
        ks.append(k[:, lo:hi])
        vs.append(v[:, lo:hi])
        lens.append(hi - lo)
    return np.concatenate(ks, axis=1), np.concatenate(vs, axis=1), lens


def _rows(task):
    from oracle import attention as att
    from oracle import fp8
    rows, q, kv_dtype = task
    w, out = _W, []
    G = w.Hq // w.Hkv
    for b, qb in zip(rows, q):
        kb, vb, lens = _branch(_REF.decode_ids[b])
        if kv_dtype == "bf16":
            out.append(att.decode_branch_contiguous(qb, kb[0], vb[0], w.Hkv,
                                                    w.scale))
            continue
        kq = fp8.quantize_sequence(lens, kb)[0]
        vq = fp8.quantize_sequence(lens, vb)[0]
        o = np.empty((w.Hq, w.d), dtype=np.float64)
        for g in range(w.Hkv):
            qr = att.bf16_to_f64(qb[g * G:(g + 1) * G])
            o[g * G:(g + 1) * G] = att.attention(qr, kq[:, g], vq[:, g],
                                                 w.scale)
        out.append(o)
    return rows, out


def decode_ids(name):
    """The rows' branch ids as the oracle's replay produces them."""
    from oracle import replay as rp
    from paged_kv_cache_attn_gb300 import workloads as W
    return rp.replay(W.CONFIGS[name](), with_data=False).decode_ids


def all_rows(name, q, kv_dtype="bf16", procs=None):
    """float64 [nb][Hq][d]: the oracle's output for every row of workload
    `name` with queries q (bf16 bits [nb][Hq][d])."""
    nb = q.shape[0]
    procs = procs or max(1, min(16, os.cpu_count() or 1))
    # Contiguous runs of rows, so that a worker meets a shared root's
    # branches one after another.
    per = max(1, -(-nb // (4 * procs)))
    tasks = [(list(range(s, min(s + per, nb))), q[s:s + per], kv_dtype)
             for s in range(0, nb, per)]
    out = np.empty(q.shape, dtype=np.float64)
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs, initializer=_init, initargs=(name,)) as pool:
        for rows, res in pool.imap_unordered(_rows, tasks):
            for b, o in zip(rows, res):
                out[b] = o
    return out
