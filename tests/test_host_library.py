"""The library's host logic (allocator, tree, eviction, batch builder, plan)
against the oracle's allocator model, bit-exact, on metadata-only pools (no
GPU, no kernels)."""

import json
import os
import random

import numpy as np
import pytest

from oracle import allocator as al
from oracle import attention as att
from oracle import replay as rp
from paged_kv_cache_attn_gb300 import binding as B
from paged_kv_cache_attn_gb300 import harness as H
from paged_kv_cache_attn_gb300 import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "pages_worked_examples.json")))

SMALL = {
    "tiny_tree": lambda: W.tiny_tree(),
    "independent": lambda: W.independent(),
    "fanout": lambda: W.fanout(),
    "deep_tree": lambda: W.deep_tree(),
    "long_context": lambda: W.long_context(),
}


def model_tables(m):
    return {i: (n.table, n.seq_len) for i, n in enumerate(m.nodes) if n.live}


@pytest.mark.parametrize("name", list(SMALL))
def test_workload_state_matches_oracle_bit_exact(name):
    w = SMALL[name]()
    lib = H.Cache(w, with_data=False)
    ref = rp.replay(w, with_data=False)
    assert lib.tables() == model_tables(ref.model)
    assert lib.refcounts() == ref.model.ref
    assert lib.free_stack() == ref.model.free_stack()
    assert lib.evicted == ref.evicted
    assert lib.decode_ids == ref.decode_ids


def test_page_table_diagram_through_the_library():
    g = GOLDEN["page_table_diagram"]
    f = g["frames"]
    order = [f["root_block_0"], f["branch_a_block_1"], f["branch_b_block_2"]]
    order += [b for b in range(128) if b not in order]
    h = B.kv_pool_create(128, 1, 1, 128, None, None, order)
    root = B.kv_branch_create(h)
    B.kv_append(h, root, 16)
    a = B.kv_fork_branch(h, root)
    b = B.kv_fork_branch(h, root)
    B.kv_append(h, a, 16)
    B.kv_append(h, b, 16)
    assert B.kv_get_refcounts(h, 128)[f["root_block_0"]] == 3
    B.kv_free(h, root)
    ref = B.kv_get_refcounts(h, 128)
    for blk, n in g["ref_counts"].items():
        assert ref[int(blk)] == n
    assert B.kv_get_block_table(h, a)[0].tolist() == [42, 87]
    assert B.kv_get_block_table(h, b)[0].tolist() == [42, 103]
    B.kv_pool_destroy(h)


def _apply(lib_h, m, op):
    """Run one op on both sides; return (lib outcome, model outcome)."""
    kind = op[0]

    def lib_call():
        if kind == "create":
            return B.kv_branch_create(lib_h)
        if kind == "append":
            return B.kv_append(lib_h, op[1], op[2])
        if kind == "fork":
            return B.kv_fork_branches(lib_h, op[1], op[2])
        if kind == "free":
            return B.kv_free(lib_h, op[1])
        if kind == "subtree":
            return B.kv_free_subtree(lib_h, op[1])
        if kind == "evict":
            return B.kv_evict(lib_h, op[1], op[2], op[3], op[4])
        raise ValueError(kind)

    def model_call():
        if kind == "create":
            return m.create()
        if kind == "append":
            m.append(op[1], op[2])
            return None
        if kind == "fork":
            return [c for c, _ in m.fork_many(op[1], op[2])]
        if kind == "free":
            m.free_node(op[1])
            return None
        if kind == "subtree":
            return m.free_subtree(op[1])
        if kind == "evict":
            return m.evict(op[1], op[2], op[3], op[4])
        raise ValueError(kind)

    def outcome(fn):
        try:
            return ("ok", fn())
        except al.OutOfBlocks:
            return ("oom", None)
        except KeyError:
            return ("notfound", None)
        except B.KVError as e:
            return ({B.KV_ERR_OOM: "oom", B.KV_ERR_NOT_FOUND: "notfound"}
                    .get(e.code, f"err{e.code}"), None)

    return outcome(lib_call), outcome(model_call)


@pytest.mark.parametrize("seed", range(6))
def test_random_ops_match_oracle(seed):
    rnd = random.Random(seed)
    nblocks = rnd.choice([8, 40, 300])
    order = list(range(nblocks))
    rnd.shuffle(order)
    h = B.kv_pool_create(nblocks, 2, 2, 64, None, None, order)
    m = al.PoolModel(nblocks, 16, order)
    ids = []
    for step in range(250):
        r = rnd.random()
        if not ids or r < 0.08:
            op = ("create",)
        elif r < 0.45:
            op = ("append", rnd.choice(ids + [len(ids) + 3]), rnd.randint(0, 50))
        elif r < 0.7:
            op = ("fork", rnd.choice(ids), rnd.randint(1, 4))
        elif r < 0.82:
            op = ("free", rnd.choice(ids))
        elif r < 0.9:
            op = ("subtree", rnd.choice(ids))
        else:
            cand = rnd.sample(ids, min(len(ids), 5))
            scores = [rnd.random() for _ in cand]
            op = ("evict", cand, scores, rnd.choice([0, 1]), rnd.randint(0, 6))
        got, want = _apply(h, m, op)
        assert got == want, (step, op)
        if op[0] == "create" and got[0] == "ok":
            ids.append(got[1])
        if op[0] == "fork" and got[0] == "ok":
            ids += got[1]
        # Full state after every op.
        assert B.kv_get_refcounts(h, nblocks).tolist() == m.ref
        assert B.kv_get_free_stack(h).tolist() == m.free_stack()
        for i in ids:
            info = B.kv_branch_info(h, i)
            nd = m.nodes[i]
            assert info["live"] == int(nd.live)
            assert info["depth"] == nd.depth and info["parent"] == nd.parent
            if nd.live:
                t, L = B.kv_get_block_table(h, i)
                assert t.tolist() == nd.table and L == nd.seq_len
        m.check_invariants()
    B.kv_pool_destroy(h)


def test_error_codes_and_atomicity():
    h = B.kv_pool_create(4, 1, 1, 64)
    r = B.kv_branch_create(h)
    B.kv_append(h, r, 40)
    before = (B.kv_get_refcounts(h, 4).tolist(), B.kv_get_free_stack(h).tolist())
    with pytest.raises(B.KVError) as e:
        B.kv_append(h, r, 40)
    assert e.value.code == B.KV_ERR_OOM
    with pytest.raises(B.KVError) as e:
        B.kv_fork_branches(h, r, 2)
    assert e.value.code == B.KV_ERR_OOM
    assert (B.kv_get_refcounts(h, 4).tolist(),
            B.kv_get_free_stack(h).tolist()) == before
    assert B.kv_num_branches(h) == 1
    with pytest.raises(B.KVError) as e:
        B.kv_fork_branch(h, 9)
    assert e.value.code == B.KV_ERR_NOT_FOUND
    with pytest.raises(B.KVError) as e:
        B.kv_evict_order(h, [r], [float("nan")])
    assert e.value.code == B.KV_ERR_INVALID_ARG
    with pytest.raises(B.KVError) as e:
        B.kv_pool_create(8, 1, 1, 64, None, None, [0, 1, 2, 3, 4, 5, 6, 6])
    assert e.value.code == B.KV_ERR_INVALID_ARG
    B.kv_pool_destroy(h)


def test_evict_order_matches_oracle():
    w = W.deep_tree()
    lib = H.Cache(w, with_data=False, evict=False)
    ref = rp.replay(w, with_data=False)
    cand = w.evict_candidates()
    scores = [w.evict_scores[i] for i in cand]
    assert B.kv_evict_order(lib.h, cand, scores) == \
        ref.model.evict_order(cand, scores)


# ---- batch builder --------------------------------------------------------------

def test_tiny_tree_has_one_segment():
    lib = H.Cache(W.tiny_tree(), with_data=False)
    tables, lens, groups = B.kv_build_batch(lib.h, lib.decode_ids)
    assert lens.tolist() == [120, 127, 133, 140]
    assert groups.tolist() == [[0, 4, 0, 6]]
    assert (tables[0, 8:] == -1).all()       # 120 tokens = 8 blocks


@pytest.mark.parametrize("name", list(SMALL))
def test_segments_are_valid_and_maximal(name):
    w = SMALL[name]()
    lib = H.Cache(w, with_data=False)
    tables, lens, groups = B.kv_build_batch(lib.h, lib.decode_ids)
    tl = [row[row >= 0].tolist() for row in tables]
    att.validate_prefix_groups(groups, tl, lens, 16)
    # Maximal: consecutive rows never share a full block beyond their
    # deepest common segment.
    ends = np.zeros(len(lens), dtype=int)
    for bb, bc, kb, kc in groups:
        ends[bb:bb + bc] = np.maximum(ends[bb:bb + bc], kb + kc)
    for i in range(len(lens) - 1):
        lim = min(lens[i], lens[i + 1]) // 16
        j = 0
        while j < lim and tl[i][j] == tl[i + 1][j]:
            j += 1
        assert min(ends[i], ends[i + 1]) >= j
    if name == "fanout":
        assert groups.tolist() == [[64 * r, 64, 0, 128] for r in range(8)]
    if name == "long_context":
        assert groups.tolist() == [[128 + 16 * r, 16, 0, 2048]
                                   for r in range(16)]
    if name == "independent":
        assert len(groups) == 0


# ---- decode plan ----------------------------------------------------------------

def decode_plan(plan, info, nb, Hq, Hkv):
    """Read the plan format documented in csrc/internal.h."""
    hdr = plan[:16]
    assert hdr[0] == 0x31564B50
    nr, nt = int(hdr[5]), int(hdr[6])
    rows = plan[int(hdr[8]):int(hdr[8]) + 8 * nr].reshape(-1, 8)
    tiles = plan[int(hdr[9]):int(hdr[9]) + 8 * nt].reshape(-1, 8)
    ptr = plan[int(hdr[10]):int(hdr[10]) + nb + 1]
    ent = plan[int(hdr[11]):int(hdr[11]) + 4 * int(hdr[7])].reshape(-1, 4)
    return rows, tiles, ptr, ent


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("flags", [0, B.KV_PLAN_IGNORE_GROUPS])
def test_plan_covers_every_token_once(name, flags):
    w = SMALL[name]()
    lib = H.Cache(w, with_data=False)
    bt = lib.batch(flags=flags, num_sms=152)
    nb, G = bt.nb, w.Hq // w.Hkv
    rows, tiles, ptr, ent = decode_plan(bt.plan, bt.info, nb, w.Hq, w.Hkv)
    nblk = (bt.seq_lens + 15) // 16
    # cover[b][g] counts how often each logical block is read for each row.
    cover = {}
    written = np.zeros(bt.info.partial_rows, dtype=int)
    for it in np.concatenate([rows, tiles]):
        b0, g, row0, nr, lo, hi, pbase, masked = [int(x) for x in it]
        assert 0 <= lo < hi <= nblk[b0] and nr >= 1
        written[pbase:pbase + nr] += 1
        for r in range(row0, row0 + nr):
            b, qr = b0 + r // G, r % G
            key = (b, g, qr)
            cover.setdefault(key, np.zeros(nblk[b], dtype=int))
            cover[key][lo:hi] += 1
    assert (written == 1).all()
    for b in range(nb):
        for g in range(w.Hkv):
            for qr in range(G):
                assert (cover[(b, g, qr)] == 1).all()
    # The merge list of each (branch, q-head) names one partial row per item
    # covering it, and those rows' item covers that branch.
    row_owner = {}
    for it in np.concatenate([rows, tiles]):
        b0, g, row0, nr, lo, hi, pbase, masked = [int(x) for x in it]
        for r in range(nr):
            row_owner[pbase + r] = (b0 + (row0 + r) // G, g, (row0 + r) % G,
                                    hi - lo)
    for b in range(nb):
        for h in range(w.Hq):
            g, qr = h // G, h % G
            total = 0
            for base, stride, lo, hi in ent[ptr[b]:ptr[b + 1]]:
                if lo <= qr < hi:
                    owner = row_owner[int(base + g * stride + qr - lo)]
                    assert owner[:3] == (b, g, qr)
                    total += owner[3]
            assert total == nblk[b]
    if flags & B.KV_PLAN_IGNORE_GROUPS:
        assert (rows[:, 7] == 1).all()
    # The split-KV items of at most 16 blocks come last; when there are more
    # than two waves of split-KV CTAs of them (3 CTAs per SM), the info
    # counts them as per-warp items.
    nw = bt.info.n_row_warp_items
    span = rows[:, 5] - rows[:, 4]
    n_short = int((span <= 16).sum())
    assert (span[len(rows) - n_short:] <= 16).all()
    assert (span[:len(rows) - n_short] > 16).all()
    assert nw == (n_short if n_short > 2 * 3 * 152 else 0)


@pytest.mark.parametrize("name", ["deep_tree", "independent", "fanout"])
def test_split_items_longest_first(name):
    """The short items are moved behind the long ones, and within each group
    the items run longest first (the hardware hands out CTAs in list order:
    longest-processing-time-first scheduling).  Among items of equal length
    the order of generation is kept (a stable sort), and every item is still
    there."""
    w = W.make(name)
    bt = H.Cache(w, with_data=False).batch(num_sms=152)
    rows, _, _, _ = decode_plan(bt.plan, bt.info, bt.nb, w.Hq, w.Hkv)
    span = rows[:, 5] - rows[:, 4]
    short = span <= 16
    n_short = int(short.sum())
    groups = (slice(0, len(rows) - n_short), slice(len(rows) - n_short, None))
    if name == "deep_tree":
        assert bt.info.n_row_warp_items > 1000   # most items are short
    # Partial-row bases were handed out in generation order.
    base = rows[:, 6]
    for g in groups:
        sp, b = span[g], base[g]
        assert (np.diff(sp) <= 0).all()          # longest first
        same = np.diff(sp) == 0
        assert (np.diff(b)[same] > 0).all()      # stable among equal lengths
    assert sorted(base.tolist()) == sorted(set(base.tolist()))
    if name == "independent":
        # units of more than 128 blocks are cut into shorter items, so the
        # generation order was not longest first: the sort moved items
        assert (np.diff(base[groups[0]]) < 0).any()


@pytest.mark.parametrize("fan,flags,want", [
    (40, 0, [(0, 128), (128, 128), (256, 64)]),        # 320 rows
    (30, 0, [(0, 240)]),                                # one two-M-tile item
    (30, B.KV_PLAN_NARROW_TILES, [(0, 128), (128, 112)]),
])
def test_multi_tile_segments_split_into_row_tiles(fan, flags, want):
    # fan branches x 8 q-heads, over every block range and kv-head of the
    # segment: a segment of 129-256 rows is one two-M-tile item (listed first,
    # counted in n_tile_wide_items) unless the plan asks for narrow tiles; a
    # larger one is cut into 128-row tiles.
    w = W.fanout(n_roots=1, root_tokens=512, fan=fan, min_suffix=1,
                 max_suffix=50, Hq=64, Hkv=8)
    bt = H.Cache(w, with_data=False).batch(num_sms=152, flags=flags)
    rows, tiles, ptr, ent = decode_plan(bt.plan, bt.info, bt.nb, w.Hq, w.Hkv)
    assert bt.info.n_tile_wide_items == (len(tiles) if len(want) == 1 else 0)
    ranges = {(int(t[4]), int(t[5])) for t in tiles}
    assert len(tiles) == len(want) * 8 * len(ranges)
    for lo, hi in ranges:
        for g in range(8):
            got = sorted((int(t[2]), int(t[3])) for t in tiles
                         if (t[4], t[5]) == (lo, hi) and t[1] == g)
            assert got == want


def test_plan_rejects_bad_input():
    with pytest.raises(B.KVError):
        B.paged_decode_plan(2, 8, 2, 128, 4, [10, 0], [])
    with pytest.raises(B.KVError):
        B.paged_decode_plan(2, 8, 2, 128, 4, [10, 80], [])        # > 4 blocks
    with pytest.raises(B.KVError):      # segment block not full for row 0
        B.paged_decode_plan(2, 8, 2, 128, 4, [20, 40], [[0, 2, 0, 2]])
    with pytest.raises(B.KVError):      # gap: row's segments start at 1
        B.paged_decode_plan(2, 8, 2, 128, 4, [40, 40], [[0, 2, 1, 1]])
    with pytest.raises(B.KVError):      # overlap
        B.paged_decode_plan(2, 8, 2, 128, 4, [40, 40],
                            [[0, 2, 0, 2], [0, 2, 1, 1]])
    plan, info = B.paged_decode_plan(2, 8, 2, 128, 4, [40, 40], [[0, 2, 0, 2]])
    assert info.partial_rows > 0 and len(plan) == info.plan_ints


# ---- batched append and reservation ------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_batched_append_equals_sequential(seed):
    rnd = random.Random(100 + seed)
    nblocks = 200
    order = list(range(nblocks))
    rnd.shuffle(order)
    hb = B.kv_pool_create(nblocks, 1, 2, 64, None, None, order)
    hr = B.kv_pool_create(nblocks, 1, 2, 64, None, None, order)
    m = al.PoolModel(nblocks, 16, order)
    roots = []
    for _ in range(3):
        roots.append(B.kv_branch_create(hb))
        B.kv_branch_create(hr)
        m.create()
    for r in roots:
        n = rnd.randint(1, 40)
        B.kv_append(hb, r, n); B.kv_append(hr, r, n); m.append(r, n)
    kids = B.kv_fork_branches(hb, roots[0], 3)
    B.kv_fork_branches(hr, roots[0], 3)
    m.fork_many(roots[0], 3)
    ids = kids + roots + [kids[0]]          # a branch may repeat
    n_tok = [rnd.randint(0, 35) for _ in ids]
    B.kv_append_batch(hb, ids, n_tok)
    B.kv_reserve(hr, ids, n_tok)
    for i, n in zip(ids, n_tok):
        m.append(i, n)
    for h in (hb, hr):
        assert B.kv_get_refcounts(h, nblocks).tolist() == m.ref
        assert B.kv_get_free_stack(h).tolist() == m.free_stack()
        for i in range(len(m.nodes)):
            t, L = B.kv_get_block_table(h, i)
            assert t.tolist() == m.nodes[i].table and L == m.nodes[i].seq_len
    B.kv_pool_destroy(hb)
    B.kv_pool_destroy(hr)


def test_batched_append_is_all_or_nothing():
    h = B.kv_pool_create(6, 1, 1, 64)
    a = B.kv_branch_create(h)
    b = B.kv_branch_create(h)
    B.kv_append(h, a, 20)
    before = (B.kv_get_refcounts(h, 6).tolist(), B.kv_get_free_stack(h).tolist())
    with pytest.raises(B.KVError) as e:
        B.kv_append_batch(h, [a, b], [20, 60])     # needs 1 + 4 > 4 free
    assert e.value.code == B.KV_ERR_OOM
    with pytest.raises(B.KVError) as e:
        B.kv_reserve(h, [a, 99], [1, 1])
    assert e.value.code == B.KV_ERR_NOT_FOUND
    assert (B.kv_get_refcounts(h, 6).tolist(),
            B.kv_get_free_stack(h).tolist()) == before
    assert B.kv_get_block_table(h, a)[1] == 20
    B.kv_pool_destroy(h)


def test_tile_items_as_long_as_the_step_allows():
    """With split-KV items in the step, a segment's tile items are as long as
    the step's block work per SM (every tile and split item moves its blocks
    into one SM), cut evenly; a step made of segments only halves them from
    256 blocks until there are two items per SM."""
    nb, mb, sms = 16, 600, 152
    lens = np.full(nb, 600 * 16, dtype=np.int32)
    for seg in (512, 64):
        # 16 branches x 8 q-heads = 128 rows (one 128-row tile) sharing `seg`
        # full blocks; each branch keeps 600 - seg blocks of its own.
        shared = np.array([[0, nb, 0, seg]], dtype=np.int32)
        plan, info = B.paged_decode_plan(nb, 64, 8, 128, mb, lens, shared, sms)
        rows, tiles, _, _ = decode_plan(plan, info, nb, 64, 8)
        assert info.n_row_items > 0
        work = seg * 8 + nb * (600 - seg) * 8          # block work of all items
        chunk = max(8, work // sms)
        pieces = -(-seg // chunk)
        span = (tiles[:, 5] - tiles[:, 4]).tolist()
        assert len(span) == pieces * 8
        assert set(span) <= {seg // pieces, -(-seg // pieces)}
    # the whole table shared: no split-KV item at all
    full = np.array([[0, nb, 0, 600]], dtype=np.int32)
    plan2, only_tiles = B.paged_decode_plan(nb, 64, 8, 128, mb, lens, full, sms)
    _, tiles2, _, _ = decode_plan(plan2, only_tiles, nb, 64, 8)
    assert only_tiles.n_row_items == 0
    assert (tiles2[:, 5] - tiles2[:, 4]).max() < 256
    assert only_tiles.n_tile_items >= 2 * sms
