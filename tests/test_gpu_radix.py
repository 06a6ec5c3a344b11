"""Branches adopted from the radix prefix index, decoded on the GPU
("Dismantling the Memory Wall", RadixAttention section: a token-keyed tree
whose nodes hold cached KV blocks; requests start from the longest cached
prefix; lock_ref pins a path in use; unlocked leaves are evicted least
recently used first).

Two system prompts are cached through the index; requests start from them
with kv_radix_fork, append the prompt's uncached tail and their own suffix,
and one decode step runs over all of them through paged_decode_attn with the
shared-prefix segments the batch builder finds (a 96-row tcgen05 segment and
a 24-row split-KV segment).  The output is compared with the oracle over each
branch's logical token sequence (prompt rows, then its own rows), which does
not depend on the pool at all.  The tables and refcounts are compared bit for
bit with the oracle's pool and radix models driven by the same operations.
Then the first prompt's requests finish and unlock their node, a new turn is
indexed, an eviction releases exactly the least recently used unlocked leaf,
and a second step (a request that finds its prompt evicted and re-appends it,
beside the surviving requests grown by one token) is checked again.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import allocator as al  # noqa: E402
from oracle import attention as att  # noqa: E402
from oracle import radix as rx  # noqa: E402
from paged_kv_cache_attn_gb300 import binding as B  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2
HQ, HKV, D, NBLK = 64, 8, 128, 600
SCALE = 1.0 / np.sqrt(D)


def _rows(rng, n):
    """n tokens' K or V rows: bf16 bits [n][Hkv][d]."""
    return W.f32_to_bf16_bits(rng.standard_normal((n, HKV, D),
                                                  dtype=np.float32))


def _prompt(rng, n):
    """(K rows, V rows, token ids) of an n-token prompt."""
    return _rows(rng, n), _rows(rng, n), rng.integers(0, 32000, n).tolist()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits[None]).view(np.int16)) \
        .cuda().view(torch.bfloat16)


class Both:
    """The library's pool and index, and the oracle's models, driven by the
    same operations; each branch's logical K/V sequence is kept beside."""

    def __init__(self):
        self.k = torch.empty((1, NBLK, HKV, 16, D), dtype=torch.bfloat16,
                             device="cuda")
        self.v = torch.empty_like(self.k)
        order = np.random.default_rng(7).permutation(NBLK).astype(np.int32)
        self.h = B.kv_pool_create(NBLK, 1, HKV, D, self.k, self.v, order)
        self.r = B.kv_radix_create(self.h)
        self.m = al.PoolModel(NBLK, 16, order)
        self.rm = rx.RadixModel(self.m)
        self.kv = {}        # branch -> (K bits [L][Hkv][d], V bits, tokens)

    def append(self, b, k, v, toks):
        B.kv_append(self.h, b, len(toks), _dev(k), _dev(v))
        self.m.append(b, len(toks))
        K, V, T = self.kv.get(b, (k[:0], v[:0], []))
        self.kv[b] = (np.concatenate([K, k]), np.concatenate([V, v]),
                      T + list(toks))

    def new_branch(self, k, v, toks):
        b = B.kv_branch_create(self.h)
        assert b == self.m.create()
        self.append(b, k, v, toks)
        return b

    def insert(self, b):
        toks = self.kv[b][2]
        n = B.kv_radix_insert(self.r, b, toks)
        assert n == self.rm.insert(b, toks)
        return n

    def match(self, toks):
        got = B.kv_radix_match(self.r, toks)
        assert got == self.rm.match(toks)
        return got

    def fork(self, node, kv_of, n_tokens):
        b = B.kv_radix_fork(self.r, node)
        assert b == self.rm.fork(node)
        K, V, T = kv_of
        self.kv[b] = (K[:n_tokens], V[:n_tokens], T[:n_tokens])
        return b

    def lock(self, node):
        B.kv_radix_lock(self.r, node)
        self.rm.lock(node)

    def unlock(self, node):
        B.kv_radix_unlock(self.r, node)
        self.rm.unlock(node)

    def free(self, b):
        B.kv_free(self.h, b)
        self.m.free_node(b)

    def evict(self, target):
        got = B.kv_radix_evict(self.r, target)
        assert got == self.rm.evict(target)
        return got

    def check_state(self, ids):
        assert B.kv_get_refcounts(self.h, NBLK).tolist() == self.m.ref
        assert B.kv_get_free_stack(self.h).tolist() == self.m.free_stack()
        for b in ids:
            t, L = B.kv_get_block_table(self.h, b)
            assert t.tolist() == self.m.nodes[b].table
            assert L == self.m.nodes[b].seq_len == len(self.kv[b][2])

    def step(self, ids, seed):
        """One decode step over `ids` in this order; returns the segments."""
        tables, lens, groups = B.kv_build_batch(self.h, ids)
        nb = len(ids)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        plan, info = B.paged_decode_plan(nb, HQ, HKV, D, tables.shape[1], lens,
                                         groups, sms)
        q_bits = W.f32_to_bf16_bits(np.random.default_rng(seed).standard_normal(
            (nb, HQ, D), dtype=np.float32))
        q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
        out = torch.empty_like(q)
        ws = torch.empty(max(info.workspace_bytes, 256), dtype=torch.uint8,
                         device="cuda")
        g = torch.from_numpy(np.ascontiguousarray(groups.reshape(-1))
                             if len(groups) else np.zeros(4, np.int32)).cuda()
        B.paged_decode_attn(q, self.k[0], self.v[0], NBLK,
                            torch.from_numpy(tables).cuda(),
                            torch.from_numpy(lens).cuda(), g, len(groups), nb,
                            tables.shape[1], HQ, HKV, D, SCALE, out,
                            torch.from_numpy(plan).cuda(), info, ws,
                            ws.numel())
        torch.cuda.synchronize()
        assert B.kv_check_device_status(ws) == (0, 0)
        gpu = att.bf16_to_f64(out.view(torch.int16).cpu().numpy()
                              .view(np.uint16))
        for row, b in enumerate(ids):
            K, V, _ = self.kv[b]
            want = att.decode_branch_contiguous(q_bits[row], K, V, HKV, SCALE)
            err = np.abs(gpu[row] - want)
            bad = err > ATOL + RTOL * np.abs(want)
            assert not bad.any(), (row, b, err.max())
        return groups, info


def test_radix_adopted_branches_decode_and_survive_eviction():
    rng = np.random.default_rng(2024)
    s = Both()
    # Two system prompts, each cached through a branch that then ends (the
    # index keeps its full blocks alive).
    p1, p2 = [_prompt(rng, n) for n in (16 * 40 + 5, 16 * 9 + 3)]
    a1 = s.new_branch(*p1)
    n1 = s.insert(a1)
    s.free(a1)
    a2 = s.new_branch(*p2)
    n2 = s.insert(a2)
    s.free(a2)

    # Requests: 12 on the first prompt, 3 on the second.  Each matches its
    # prompt, adopts the cached blocks, pins the node, and appends the
    # prompt's uncached tail and its own suffix.
    reqs = []
    for prompt, node_want, count in ((p1, n1, 12), (p2, n2, 3)):
        for _ in range(count):
            suffix = rng.integers(0, 32000, int(rng.integers(1, 300))).tolist()
            node, matched = s.match(prompt[2] + suffix)
            assert node == node_want and matched == len(prompt[2]) // 16 * 16
            b = s.fork(node, prompt, matched)
            s.lock(node)
            tail = slice(matched, len(prompt[2]))
            s.append(b, prompt[0][tail], prompt[1][tail], prompt[2][tail])
            s.append(b, _rows(rng, len(suffix)), _rows(rng, len(suffix)),
                     suffix)
            reqs.append((b, node))
    ids = [b for b, _ in reqs]
    s.check_state(ids)
    groups, info = s.step(ids, seed=1)
    # The adopted branches share the cached blocks: one segment per prompt
    # (96 rows on tcgen05, 24 rows through the split-KV kernel).
    segs = sorted(map(tuple, groups.tolist()))
    assert segs == [(0, 12, 0, 40), (12, 3, 0, 9)]
    assert info.n_tile_items > 0

    # The first prompt's requests end: their branches are freed and the node
    # unlocked.  A new conversation turn is indexed (a newer leaf).
    for b, node in reqs[:12]:
        s.free(b)
        s.unlock(node)
    turn = rng.integers(0, 32000, 16 * 6).tolist()
    a3 = s.new_branch(_rows(rng, len(turn)), _rows(rng, len(turn)), turn)
    n3 = s.insert(a3)
    s.free(a3)
    # Ask for exactly the first prompt's blocks back: the least recently
    # used unlocked leaf is n1 (n2 is locked, n3 is newer).
    target = len(B.kv_get_free_stack(s.h)) + 40
    assert s.evict(target) == [n1]
    assert len(B.kv_get_free_stack(s.h)) == target
    assert B.kv_radix_node_info(s.r, n3)["live"]

    # Second step: a new request on the first prompt finds nothing cached and
    # appends it all; the second prompt's requests grow by one token.
    node, matched = s.match(p1[2] + [5, 6, 7])
    assert (node, matched) == (0, 0)
    fresh = s.new_branch(p1[0], p1[1], p1[2])
    for b, _ in reqs[12:]:
        s.append(b, _rows(rng, 1), _rows(rng, 1), [9])
    ids2 = [fresh] + [b for b, _ in reqs[12:]]
    s.check_state(ids2)
    groups2, _ = s.step(ids2, seed=2)
    assert sorted(map(tuple, groups2.tolist())) == [(1, 3, 0, 9)]
    B.kv_radix_destroy(s.r)
    B.kv_pool_destroy(s.h)
