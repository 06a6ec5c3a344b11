"""Radix prefix index: the pages' behaviour, and the library against the
oracle model bit-exactly (node structure, blocks, lock_ref, recency, pool
refcounts and free stack)."""

import random

import pytest

from oracle import allocator as al
from oracle import radix as rx
from paged_kv_cache_attn_gb300 import binding as B


def _pool(n=400):
    return B.kv_pool_create(n, 1, 1, 64), al.PoolModel(n, 16)


def _branch(h, m, n_tokens):
    b = B.kv_branch_create(h)
    B.kv_append(h, b, n_tokens)
    mb = m.create()
    m.append(mb, n_tokens)
    assert b == mb
    return b


def test_shared_system_prompt_is_kept_and_leaves_are_evicted_lru():
    """A 64-token system prompt used by three requests stays cached; the
    least recently used unlocked conversation leaf goes first; a locked leaf
    is never evicted; the root never is."""
    h, m = _pool(64)
    r = B.kv_radix_create(h)
    prompt = list(range(1000, 1064))
    convs = [prompt + [i] * 32 for i in range(3)]
    leaves = []
    for c in convs:
        b = _branch(h, m, len(c))
        leaves.append(B.kv_radix_insert(r, b, c))
        B.kv_free(h, b)                     # the index keeps the KV alive
    node, n = B.kv_radix_match(r, prompt + [7] * 40)
    assert n == 64                          # the shared prompt, 4 blocks
    shared = node
    assert B.kv_radix_node_info(r, shared)["n_children"] == 3
    # Turn 2 of conversation 1 reuses its whole history.
    node, n = B.kv_radix_match(r, convs[1] + [9] * 20)
    assert n == 96 and node == leaves[1]
    B.kv_radix_lock(r, leaves[2])
    free0 = len(B.kv_get_free_stack(h))
    ev = B.kv_radix_evict(r, free0 + 2)     # one leaf (2 blocks) is enough
    assert ev == [leaves[0]]                # least recently used, unlocked
    ev = B.kv_radix_evict(r, 64)            # evict all that may go
    assert leaves[2] not in ev and shared not in ev
    assert B.kv_radix_node_info(r, leaves[2])["live"] == 1
    B.kv_radix_unlock(r, leaves[2])
    assert B.kv_radix_evict(r, 64)[-1] == shared    # then the prompt goes
    B.kv_radix_destroy(r)
    assert len(B.kv_get_free_stack(h)) == 64
    B.kv_pool_destroy(h)


def test_fork_from_cached_prefix_shares_blocks():
    h, m = _pool(64)
    r = B.kv_radix_create(h)
    toks = list(range(50))
    b = _branch(h, m, 50)
    leaf = B.kv_radix_insert(r, b, toks)
    assert B.kv_radix_node_info(r, leaf)["n_blocks"] == 3   # full blocks only
    node, n = B.kv_radix_match(r, toks[:40])                # ends inside: split
    assert n == 32 and node != leaf
    assert B.kv_radix_node_info(r, leaf)["parent"] == node
    c = B.kv_radix_fork(r, node)
    t, L = B.kv_get_block_table(h, c)
    assert L == 32 and t.tolist() == B.kv_get_block_table(h, b)[0][:2].tolist()
    ref = B.kv_get_refcounts(h, 64)
    assert ref[t[0]] == 3                                   # branch, index, fork
    B.kv_radix_destroy(r)
    B.kv_pool_destroy(h)


def _state(h, r, nblocks):
    nodes = []
    for i in range(B.kv_radix_num_nodes(r)):
        info = B.kv_radix_node_info(r, i)
        blocks = B.kv_radix_node_blocks(r, i) if info["live"] else []
        nodes.append((info["live"], info["parent"], info["n_blocks"],
                      info["lock_ref"], info["n_children"],
                      info["last_access"], blocks))
    return (nodes, B.kv_get_refcounts(h, nblocks).tolist(),
            B.kv_get_free_stack(h).tolist())


def _model_state(m, rm):
    nodes = []
    for n in rm.nodes:
        nodes.append((int(n.live), n.parent, len(n.blocks), n.lock_ref,
                      len(n.children), n.last_access,
                      list(n.blocks) if n.live else []))
    return nodes, list(m.ref), m.free_stack()


@pytest.mark.parametrize("seed", range(5))
def test_random_ops_match_oracle_model(seed):
    rnd = random.Random(seed)
    nblocks = 300
    h, m = _pool(nblocks)
    r = B.kv_radix_create(h)
    rm = rx.RadixModel(m)
    vocab = [list(range(100 * k, 100 * k + 16)) for k in range(5)]
    branches, node_ids = [], [0]
    for step in range(150):
        op = rnd.random()
        # Token sequences built from a few 16-token chunks, so prefixes recur.
        toks = sum((rnd.choice(vocab) for _ in range(rnd.randint(0, 6))), [])
        toks += [7] * rnd.randint(0, 20)
        if op < 0.35 and len(m.free) > 20:
            b = _branch(h, m, max(len(toks), 1))
            branches.append((b, toks))
            got = B.kv_radix_insert(r, b, toks)
            want = rm.insert(b, toks)
            assert got == want
            node_ids.append(got)
        elif op < 0.6:
            assert B.kv_radix_match(r, toks) == rm.match(toks)
        elif op < 0.7 and len(node_ids) > 1:
            x = rnd.choice(node_ids)
            if rm.nodes[x].live:
                B.kv_radix_lock(r, x); rm.lock(x)
        elif op < 0.8:
            locked = [i for i, n in enumerate(rm.nodes) if n.live and i > 0
                      and n.lock_ref > sum(rm.nodes[c].lock_ref
                                           for c in n.children)]
            if locked:
                x = rnd.choice(locked)
                B.kv_radix_unlock(r, x); rm.unlock(x)
        elif op < 0.88:
            target = len(m.free) + rnd.randint(0, 30)
            assert B.kv_radix_evict(r, target) == rm.evict(target)
        elif op < 0.94 and len(node_ids) > 1:
            x = rnd.choice(node_ids)
            if rm.nodes[x].live:
                assert B.kv_radix_fork(r, x) == rm.fork(x)
        elif branches:
            b, _ = branches.pop(rnd.randrange(len(branches)))
            B.kv_free(h, b); m.free_node(b)
        assert _state(h, r, nblocks) == _model_state(m, rm), step
    B.kv_radix_destroy(r)
    rm.destroy()
    assert B.kv_get_refcounts(h, nblocks).tolist() == m.ref
    B.kv_pool_destroy(h)


def test_oracle_model_follows_the_pages_scenario():
    """The same hand-derived expectations, on the oracle model: shared prompt
    kept, whole-history reuse, LRU unlocked leaves first, locked leaf and
    (until unlocked leaves are gone) the shared prompt kept."""
    m = al.PoolModel(64, 16)
    rm = rx.RadixModel(m)
    prompt = list(range(1000, 1064))
    convs = [prompt + [i] * 32 for i in range(3)]
    leaves = []
    for c in convs:
        b = m.create()
        m.append(b, len(c))
        leaves.append(rm.insert(b, c))
        m.free_node(b)
    node, n = rm.match(prompt + [7] * 40)
    assert n == 64 and len(rm.nodes[node].children) == 3
    shared = node
    node, n = rm.match(convs[1] + [9] * 20)
    assert n == 96 and node == leaves[1]
    rm.lock(leaves[2])
    assert rm.evict(m.free_count() + 2) == [leaves[0]]
    ev = rm.evict(64)
    assert leaves[2] not in ev and shared not in ev
    rm.unlock(leaves[2])
    assert rm.evict(64)[-1] == shared
    rm.destroy()
    assert m.free_count() == 64
