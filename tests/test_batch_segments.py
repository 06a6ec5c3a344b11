"""The batch builder's shared-prefix segments over pools shaped by random
operations -- forks, appends, frees, spills and restores through the host
tier, and branches made from the radix index (which share blocks with no
common fork ancestor) -- checked against the tables themselves: every
segment is valid (its rows hold the same full blocks over its range, the
oracle's check) and the segments are maximal (two adjacent rows never share
a full block beyond their deepest common segment).  Metadata-only pools."""

import random

import numpy as np
import pytest

from oracle import attention as att
from paged_kv_cache_attn_gb300 import binding as B


def check_batch(h, ids):
    tables, lens, groups = B.kv_build_batch(h, ids)
    tl = [row[row >= 0].tolist() for row in tables]
    att.validate_prefix_groups(groups, tl, lens, 16)
    ends = np.zeros(len(ids), dtype=int)
    for bb, bc, kb, kc in groups:
        ends[bb:bb + bc] = np.maximum(ends[bb:bb + bc], kb + kc)
    for i in range(len(ids) - 1):
        lim = min(lens[i], lens[i + 1]) // 16
        j = 0
        while j < lim and tl[i][j] == tl[i + 1][j]:
            j += 1
        assert min(ends[i], ends[i + 1]) >= j, (i, j, ends[i], ends[i + 1])
    return len(groups)


@pytest.mark.parametrize("seed", range(8))
def test_segments_after_random_operations(seed):
    rnd = random.Random(900 + seed)
    nblocks, slots = 400, 200
    order = list(range(nblocks))
    rnd.shuffle(order)
    h = B.kv_pool_create(nblocks, 1, 1, 64, None, None, order)
    B.kv_offload_attach(h, None, None, slots)
    r = B.kv_radix_create(h)
    ids, spilled, nodes = [], set(), []
    tokens = {}             # branch -> its token ids (for the radix index)
    n_groups = 0

    def live():
        out = []
        for i in ids:
            try:
                if B.kv_branch_info(h, i)["live"]:
                    out.append(i)
            except B.KVError:
                pass
        return out

    for step in range(250):
        lv = live()
        x = rnd.choice(lv) if lv else None
        op = rnd.random()
        try:
            if x is None or op < 0.08:
                b = B.kv_branch_create(h)
                ids.append(b)
                tokens[b] = []
            elif op < 0.35 and x not in spilled:
                n = rnd.randint(1, 70)
                B.kv_append(h, x, n)
                tokens[x] += [rnd.randrange(50) for _ in range(n)]
            elif op < 0.55 and x not in spilled:
                kids = B.kv_fork_branches(h, x, rnd.randint(1, 3))
                for c in kids:
                    tokens[c] = list(tokens[x])
                ids += kids
            elif op < 0.65:
                xs = rnd.sample(lv, min(len(lv), 2))
                B.kv_spill(h, xs)
                spilled |= set(xs)
            elif op < 0.75:
                xs = [i for i in lv if i in spilled][:2]
                if xs:
                    B.kv_restore(h, xs)
                    spilled -= set(xs)
            elif op < 0.83 and x not in spilled and len(tokens[x]) >= 16:
                nodes.append(B.kv_radix_insert(r, x, tokens[x]))
            elif op < 0.9 and nodes:
                node = rnd.choice(nodes)
                b = B.kv_radix_fork(r, node)
                ids.append(b)
                t, n_tok = B.kv_get_block_table(h, b)
                tokens[b] = [0] * n_tok   # its cached tokens (not re-indexed)
            elif op < 0.97:
                B.kv_free(h, x)
                spilled.discard(x)
        except B.KVError:
            pass                 # out of blocks or host slots, or a bad op
        if step % 10 == 9:
            batch = [i for i in live()
                     if i not in spilled and B.kv_get_block_table(h, i)[1] > 0]
            if len(batch) >= 2:
                n_groups += check_batch(h, batch)              # id order
                rnd.shuffle(batch)
                n_groups += check_batch(h, batch)              # any order
    assert n_groups > 0
    B.kv_radix_destroy(r)
    B.kv_pool_destroy(h)
