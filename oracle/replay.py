"""Replay a synthetic workload on the oracle's own allocator model.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Produces, with no help from the CUDA library: the allocator state (tables,
refcounts, free stack), optionally the oracle's own host copy of the pools,
the ids evicted by the importance score, the surviving leaves that the decode
step runs over, and each branch's logical token sequence -- the parent's
tokens at the moment of the fork followed by the branch's own appends
("The Reasoning Engine Meltdown", §5: a child starts from its parent's pages).
"""

from __future__ import annotations

import numpy as np

from . import attention as att
from .allocator import STOP_EVICTED_LEAVES, PoolData, PoolModel
from .fp8 import Fp8PoolData, decode_step_fp8


class Replayed:
    def __init__(self, w, with_data: bool, kv_dtype: str = "bf16"):
        self.w = w
        self.kv_dtype = kv_dtype
        self.model = PoolModel(w.num_blocks, w.block_size,
                               w.initial_free_order())
        if kv_dtype not in ("bf16", "e4m3"):
            raise ValueError(kv_dtype)
        kind = PoolData if kv_dtype == "bf16" else Fp8PoolData
        self.data = (kind(w.num_layers, w.num_blocks, w.Hkv, w.block_size,
                          w.d) if with_data else None)
        # logical[nid] = list of (source node, lo, hi): the node's tokens are
        # tokens [lo, hi) of the source node's own appended rows, in order.
        self.logical: dict[int, list] = {}
        self.evicted: list = []
        self.decode_ids: list = []
        self._kv_cache: dict = {}

    def node_kv(self, nid):
        if nid not in self._kv_cache:
            if len(self._kv_cache) > 8:
                self._kv_cache.clear()
            self._kv_cache[nid] = self.w.node_kv(nid)
        return self._kv_cache[nid]

    def branch_kv(self, nid):
        """Contiguous K, V of a branch: uint16 [L][seq_len][Hkv][d]."""
        ks, vs = [], []
        for src, lo, hi in self.logical[nid]:
            k, v = self.node_kv(src)
            ks.append(k[:, lo:hi])
            vs.append(v[:, lo:hi])
        return np.concatenate(ks, axis=1), np.concatenate(vs, axis=1)


def replay(w, with_data: bool = True, kv_dtype: str = "bf16") -> Replayed:
    """``kv_dtype``: "bf16" (pool copy of bf16 bits) or "e4m3" (FP8 codes and
    per-block scales, ``oracle.fp8``)."""
    r = Replayed(w, with_data, kv_dtype)
    m = r.model
    own_appended = {}
    for op in w.ops:
        if op[0] == "create":
            nid = m.create()
            r.logical[nid] = []
            own_appended[nid] = 0
        elif op[0] == "append":
            nid = op[1]
            n = w.nodes[nid].n_tokens
            writes = m.append(nid, n)
            if r.data is not None:
                k, v = w.node_kv(nid)
                r.data.write(writes, k, v)
            lo = own_appended[nid]
            r.logical[nid].append((nid, lo, lo + n))
            own_appended[nid] = lo + n
        elif op[0] == "fork":
            parent, count = op[1], op[2]
            for cid, cow in m.fork_many(parent, count):
                if cow is not None and r.data is not None:
                    r.data.copy_block(*cow)
                r.logical[cid] = list(r.logical[parent])
                own_appended[cid] = 0
        else:
            raise ValueError(op)
    if w.evict_target_leaves() > 0:
        cand = w.evict_candidates()
        r.evicted = m.evict(cand, [w.evict_scores[i] for i in cand],
                            STOP_EVICTED_LEAVES, w.evict_target_leaves())
    r.decode_ids = [i for i in w.leaves() if m.nodes[i].live]
    return r


def decode_rows(r: Replayed, q: np.ndarray, rows, scale: float) -> dict:
    """Oracle output for the listed batch rows from each branch's logical
    (contiguous) token sequence: {row: [Hq][d] float64}.  Needs no pool copy,
    so it runs at any size."""
    out = {}
    for b in rows:
        nid = r.decode_ids[b]
        k, v = r.branch_kv(nid)
        out[b] = att.decode_branch_contiguous(q[b], k[0], v[0], r.w.Hkv, scale)
    return out


def decode_all_from_pool(r: Replayed, q: np.ndarray, scale: float,
                         layer: int = 0) -> np.ndarray:
    """Oracle output for the whole batch, gathered through the oracle's own
    block tables from the oracle's own pool copy (one layer)."""
    assert r.data is not None
    m = r.model
    tables = [m.nodes[i].table for i in r.decode_ids]
    lens = [m.nodes[i].seq_len for i in r.decode_ids]
    if r.kv_dtype == "e4m3":
        return decode_step_fp8(q, r.data, tables, lens, scale,
                               r.w.block_size, layer=layer)
    return att.decode_step(q, r.data.k[layer], r.data.v[layer], tables, lens, scale,
                           r.w.block_size)
