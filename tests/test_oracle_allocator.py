"""Pins for the oracle's allocator model: the pages' worked examples and rules."""

import json
import os
import random

import pytest

from oracle import allocator as al
from oracle import replay as rp
from paged_kv_cache_attn_gb300 import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "pages_worked_examples.json")))


def test_kv_bytes_worked_example():
    g = GOLDEN["kv_bytes_per_token_70b"]
    a = g["args"]
    per_tok = al.kv_bytes_per_token(a["num_layers"], a["num_heads"],
                                    a["head_dim"], a["elem_bytes"])
    assert per_tok == g["bytes_per_token"]
    total = per_tok * g["tokens"]
    assert total == 21_474_836_480
    assert round(total / 1e9, 2) == g["quoted_total_gb"]


def test_page_counts_round_up():
    assert [al.blocks_for(t, 16) for t in (0, 1, 15, 16, 17, 100)] == \
        [0, 1, 1, 1, 2, 7]


def _diagram_pool():
    g = GOLDEN["page_table_diagram"]
    f = g["frames"]
    order = [f["root_block_0"], f["branch_a_block_1"], f["branch_b_block_2"]]
    order += [b for b in range(128) if b not in order]
    m = al.PoolModel(128, g["block_size_tokens"], order)
    root = m.create()
    m.append(root, 16)
    a, _ = m.fork(root)
    b, _ = m.fork(root)
    m.append(a, 16)
    m.append(b, 16)
    return g, m, root, a, b


def test_page_table_diagram_state():
    g, m, root, a, b = _diagram_pool()
    f = g["frames"]
    assert m.nodes[a].table == [f["root_block_0"], f["branch_a_block_1"]]
    assert m.nodes[b].table == [f["root_block_0"], f["branch_b_block_2"]]
    # With the root handle still held, the rules give three references.
    assert m.ref[f["root_block_0"]] == 3
    m.free_node(root)
    for blk, ref in g["ref_counts"].items():
        assert m.ref[int(blk)] == ref
    m.check_invariants()


def test_fork_shares_full_blocks_and_copies_partial():
    m = al.PoolModel(64, 16)
    r = m.create()
    m.append(r, 100)                   # 6 full blocks + 4-token tail
    c, cow = m.fork(r)
    pt = m.nodes[r].table
    assert cow == (pt[6], m.nodes[c].table[6])
    assert m.nodes[c].table[:6] == pt[:6]
    assert all(m.ref[b] == 2 for b in pt[:6])
    assert m.ref[pt[6]] == 1 and m.ref[cow[1]] == 1
    assert m.nodes[c].seq_len == 100 and m.nodes[c].depth == 1
    # Aligned parent: no copy.
    r2 = m.create()
    m.append(r2, 32)
    _, cow2 = m.fork(r2)
    assert cow2 is None
    m.check_invariants()


def test_appends_only_write_owned_blocks():
    rnd = random.Random(11)
    m = al.PoolModel(4096, 16)
    ids = [m.create()]
    m.append(ids[0], 37)
    for _ in range(300):
        op = rnd.random()
        live = [i for i in ids if m.nodes[i].live]
        x = rnd.choice(live)
        if op < 0.4:
            for t, blk, slot in m.append(x, rnd.randint(0, 40)):
                assert m.ref[blk] == 1
        elif op < 0.7:
            ids += [c for c, _ in m.fork_many(x, rnd.randint(1, 3))]
        elif op < 0.85 and x != ids[0]:
            m.free_node(x)
        elif x != ids[0]:
            m.free_subtree(x)
        m.check_invariants()
        for i in ids:
            nd = m.nodes[i]
            if nd.live:
                assert len(nd.table) * 16 - nd.seq_len <= \
                    GOLDEN["internal_fragmentation"]["max_unused_slots_per_sequence"]


def test_oom_leaves_state_unchanged():
    m = al.PoolModel(4, 16)
    r = m.create()
    m.append(r, 40)                     # 3 blocks
    before = (list(m.ref), list(m.free), list(m.nodes[r].table))
    with pytest.raises(al.OutOfBlocks):
        m.append(r, 40)                 # needs 3 more, 1 free
    with pytest.raises(al.OutOfBlocks):
        m.fork_many(r, 2)               # partial tail: 2 copies, 1 free
    assert (list(m.ref), list(m.free), list(m.nodes[r].table)) == before
    assert len(m.nodes) == 1


def test_unknown_handles_raise():
    m = al.PoolModel(8, 16)
    with pytest.raises(KeyError):
        m.fork(3)
    r = m.create()
    m.free_node(r)
    with pytest.raises(KeyError):
        m.free_node(r)
    with pytest.raises(KeyError):
        m.append(r, 1)


def test_free_pushes_lifo_in_table_order():
    m = al.PoolModel(10, 16, [9, 8, 7, 6, 5, 4, 3, 2, 1, 0])
    r = m.create()
    m.append(r, 48)
    assert m.nodes[r].table == [9, 8, 7]
    m.free_node(r)
    # Walk 9, 8, 7: 7 was pushed last, so it is popped first.
    assert m.free_stack()[:3] == [7, 8, 9]


def test_omega_order_and_ties():
    m = al.PoolModel(64, 16)
    r = m.create()                                  # depth 0
    m.append(r, 16)
    (a, _), (b, _) = m.fork_many(r, 2)              # depth 1
    (c, _), = m.fork_many(a, 1)                     # depth 2
    # omega: r 0.9/1 = 0.9, a 0.5/2 = 0.25, b 0.5/2 = 0.25, c 0.6/3 = 0.2
    order = m.evict_order([r, a, b, c], [0.9, 0.5, 0.5, 0.6])
    assert order == [c, a, b, r]
    with pytest.raises(ValueError):
        m.evict_order([r], [float("nan")])


def test_evict_stop_rules():
    m = al.PoolModel(64, 16)
    r = m.create()
    m.append(r, 32)
    kids = [c for c, _ in m.fork_many(r, 3)]
    for k in kids:
        m.append(k, 16)
    free0 = m.free_count()
    ev = m.evict(kids, [0.3, 0.1, 0.2], al.STOP_FREE_BLOCKS, free0 + 2)
    assert ev == [kids[1], kids[2]]
    assert m.free_count() == free0 + 2
    ev2 = m.evict([r] + kids, [0.0, 0.3, 0.1, 0.2], al.STOP_EVICTED_LEAVES, 1)
    assert ev2 == [r]                   # frees the root and its last child
    assert all(not n.live for n in m.nodes)
    assert m.free_count() == 64
    m.check_invariants()


def test_deep_tree_eviction_reaches_target():
    w = W.deep_tree()
    r = rp.replay(w, with_data=False)
    assert len(w.leaves()) == 243
    assert 243 - len(r.decode_ids) >= w.evict_target_leaves() == 73
    r.model.check_invariants()


# ---- host tier ("Dismantling the Memory Wall", cross-tier offloading) -------

def _host_tier_scenario(ops):
    """A scenario worked by hand from the host-tier reading (blocks a branch
    owns alone move to host slots in branch and table order; freed device
    blocks and emptied host slots are pushed on their LIFO stacks as they are
    freed; a spilled entry is -(slot + 2); a restore pops device blocks in
    branch and table order).  `ops` supplies create / append / fork / spill /
    restore / free and the state readers, so the same script runs on the
    oracle's model and on the library."""
    a = ops.create()
    ops.append(a, 40)                 # blocks 0, 1, 2 (8 tokens in 2)
    b = ops.fork(a)                   # COW block 3 <- copy of 2; shares 0, 1
    ops.append(b, 20)                 # 8 more tokens into 3, then block 4
    got = {"b0": ops.table(b)}
    got["spill_b"] = ops.spill([b])   # 3 -> slot 0, 4 -> slot 1
    got["b1"] = ops.table(b)
    got["free1"] = ops.free_stack()
    got["host1"] = ops.host_free()
    got["spill_a"] = ops.spill([a])   # only 2 is a's alone -> slot 2
    got["a1"] = ops.table(a)
    got["restore"] = ops.restore([b, a])
    got["a2"], got["b2"] = ops.table(a), ops.table(b)
    got["free2"] = ops.free_stack()
    got["host2"] = ops.host_free()
    ops.spill([a])                    # a's block 3 -> slot 2 (top of host)
    got["a3"] = ops.table(a)
    ops.free(a)                       # 0, 1 drop to refcount 1; slot 2 back
    got["ref"] = ops.ref()
    got["free3"] = ops.free_stack()
    got["host3"] = ops.host_free()
    return got


HOST_TIER_WANT = {
    "b0": [0, 1, 3, 4],
    "spill_b": 2,
    "b1": [0, 1, -2, -3],
    "free1": [4, 3, 5, 6, 7, 8, 9],
    "host1": [2, 3],
    "spill_a": 1,
    "a1": [0, 1, -4],
    "restore": 3,
    # b's slot 0 -> block 2 (top of the device stack), slot 1 -> block 4;
    # a's slot 2 -> block 3; each slot pushed back as it empties.
    "b2": [0, 1, 2, 4],
    "a2": [0, 1, 3],
    "free2": [5, 6, 7, 8, 9],
    "host2": [2, 1, 0, 3],
    "a3": [0, 1, -4],
    "ref": [1, 1, 1, 0, 1, 0, 0, 0, 0, 0],
    "free3": [3, 5, 6, 7, 8, 9],
    "host3": [2, 1, 0, 3],
}


class _ModelOps:
    def __init__(self):
        self.m = al.PoolModel(10, 16)
        self.m.attach_host(4)

    def create(self):
        return self.m.create()

    def append(self, i, n):
        self.m.append(i, n)

    def fork(self, i):
        return self.m.fork(i)[0]

    def spill(self, ids):
        return len(self.m.spill(ids))

    def restore(self, ids):
        return len(self.m.restore(ids))

    def free(self, i):
        self.m.free_node(i)

    def table(self, i):
        return list(self.m.nodes[i].table)

    def free_stack(self):
        return self.m.free_stack()

    def host_free(self):
        return self.m.host_free_stack()

    def ref(self):
        return list(self.m.ref)


def test_host_tier_hand_worked_scenario():
    got = _host_tier_scenario(_ModelOps())
    assert got == HOST_TIER_WANT


def test_host_tier_pairs_name_the_copies():
    """The copies a spill or restore returns: (device block, host slot) in
    branch and table order, then (host slot, device block)."""
    m = al.PoolModel(10, 16)
    m.attach_host(4)
    a = m.create()
    m.append(a, 40)
    b = m.fork(a)[0]
    m.append(b, 20)
    assert m.spill([b]) == [(3, 0), (4, 1)]
    assert m.spill([a]) == [(2, 2)]
    assert m.restore([b, a]) == [(0, 2), (1, 4), (2, 3)]
    m.check_invariants()


def test_host_tier_refusals_leave_the_model_unchanged():
    m = al.PoolModel(4, 16)
    m.attach_host(1)
    a = m.create()
    m.append(a, 40)                    # three blocks of a's own
    before = (list(m.nodes[a].table), m.free_stack(), m.host_free_stack())
    with pytest.raises(al.OutOfBlocks):
        m.spill([a])                   # three blocks, one host slot
    assert (list(m.nodes[a].table), m.free_stack(),
            m.host_free_stack()) == before
    with pytest.raises(ValueError):
        m.restore([a, a])
