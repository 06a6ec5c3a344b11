"""Pure-Python model of the refcounted block pool for tree-shaped decoding.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Rules, with the passage each one follows:

* Physical blocks carry a reference count; a fork points the child at the
  parent's blocks and adds one reference to each; a prune drops one
  reference per block and a block whose count reaches zero returns to the
  free pool at once ("The Reasoning Engine Meltdown", §5, the four numbered
  fork rules, and §6 ``fork_node`` / ``free_node``).
* A request asks for ceil(tokens / page size) pages and fails with an
  out-of-memory error if the pool cannot supply them (same page, §6
  ``allocate_root`` and ``_allocate_single_page``).  Reading taken: every
  state change is all-or-nothing -- on error nothing changes.
* Writes go only to pages the branch owns alone (§5 rule 3, copy-on-write;
  "Dismantling the Memory Wall", copy-on-write for beam search: a new block
  only where branches diverge).  Reading taken: the divergence point is the
  fork itself.  If the parent's last block is partial at the fork, the child
  receives a fresh block holding a copy of that whole block (every layer, K
  and V); the parent keeps its own partial block.  Full blocks are shared.
  The page's own ``append_tokens`` listing replaces a shared page with an
  empty one and never copies its contents, which would lose tokens; that is
  not reproduced.
* The free pool is a set on the page (``free_page_ids``, popped in no
  defined order).  Reading taken: a LIFO stack.  Its initial order is the
  caller's ``initial_free_order`` (first element popped first), else
  ascending ids.  Allocation pops; a block whose count reaches zero is pushed
  at that moment.  Freeing a branch walks its table from logical index 0
  upward.  A fork allocates its copy-on-write block; an append allocates its
  new blocks in logical order.
* Branch handles are integers 0, 1, 2, ... in creation order and are never
  reused.  A root has depth 0; a fork's child has its parent's depth + 1.
* Eviction: blocks are evicted in ascending order of
  omega = branch_score / (depth + 1) (RKSC summary, §2.C RSBCM).  Reading
  taken: omega is per branch node, computed in binary64, ties broken by the
  smaller id; evicting a node frees its whole subtree (post-order, children
  in creation order), since dropping a block in the middle of a path would
  corrupt every descendant.  Eviction stops once a target is met: a number
  of free blocks, or a number of evicted leaf nodes.
"""

from __future__ import annotations

from dataclasses import dataclass, field

STOP_FREE_BLOCKS = 0
STOP_EVICTED_LEAVES = 1


class OutOfBlocks(MemoryError):
    """The pool cannot supply the blocks an operation needs (nothing changed)."""


def kv_bytes_per_token(num_layers: int, num_heads: int, head_dim: int,
                       elem_bytes: int) -> int:
    """KV bytes per cached token: 2 (K and V) x L x H x d_h x P.

    "The Reasoning Engine Meltdown", §2.1, the Memory_KV formula with
    S = 1 (its 70B worked example gives 2,621,440 bytes per token).
    """
    return 2 * num_layers * num_heads * head_dim * elem_bytes


def blocks_for(tokens: int, block_size: int) -> int:
    """ceil(tokens / block_size) ("The Reasoning Engine Meltdown", §6
    ``allocate_root``)."""
    return (tokens + block_size - 1) // block_size


@dataclass
class Node:
    parent: int
    depth: int
    table: list = field(default_factory=list)
    seq_len: int = 0
    live: bool = True
    children: list = field(default_factory=list)


class PoolModel:
    """Block pool + per-branch block tables + fork tree."""

    def __init__(self, num_blocks: int, block_size: int = 16,
                 initial_free_order=None):
        if num_blocks < 1 or block_size < 1:
            raise ValueError("empty pool")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = (list(range(num_blocks)) if initial_free_order is None
                 else [int(x) for x in initial_free_order])
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("initial_free_order must be a permutation")
        self.ref = [0] * num_blocks
        self.free = list(reversed(order))     # top of the stack = last element
        self.nodes: list[Node] = []

    # -- queries -----------------------------------------------------------
    def node(self, nid: int) -> Node:
        if not (0 <= nid < len(self.nodes)):
            raise KeyError(nid)
        return self.nodes[nid]

    def live_node(self, nid: int) -> Node:
        n = self.node(nid)
        if not n.live:
            raise KeyError(nid)
        return n

    def free_stack(self) -> list:
        """Free blocks, next-to-be-popped first."""
        return list(reversed(self.free))

    def free_count(self) -> int:
        return len(self.free)

    # -- allocation primitives ----------------------------------------------
    def _pop(self) -> int:
        blk = self.free.pop()
        assert self.ref[blk] == 0
        self.ref[blk] = 1
        return blk

    def _release(self, blk: int) -> None:
        self.ref[blk] -= 1
        assert self.ref[blk] >= 0
        if self.ref[blk] == 0:
            self.free.append(blk)

    # -- operations ----------------------------------------------------------
    def create(self) -> int:
        self.nodes.append(Node(parent=-1, depth=0))
        return len(self.nodes) - 1

    def append(self, nid: int, n_tokens: int):
        """Append n tokens; returns their (token index, block, slot) list."""
        nd = self.live_node(nid)
        if n_tokens < 0:
            raise ValueError("negative token count")
        B = self.block_size
        if nd.seq_len % B != 0:
            # The partial last block is always owned alone (see the fork rule).
            assert self.ref[nd.table[-1]] == 1
        need = blocks_for(nd.seq_len + n_tokens, B) - len(nd.table)
        if need > len(self.free):
            raise OutOfBlocks(f"append needs {need} blocks, {len(self.free)} free")
        for _ in range(need):
            nd.table.append(self._pop())
        writes = []
        for i in range(n_tokens):
            t = nd.seq_len + i
            writes.append((t, nd.table[t // B], t % B))
        nd.seq_len += n_tokens
        return writes

    def fork_many(self, parent: int, n: int):
        """Fork n children of ``parent``; returns [(child id, cow pair or None)].

        A cow pair ``(src, dst)`` means: copy the whole physical block src
        (every layer, K and V) into dst.
        """
        p = self.live_node(parent)
        if n < 1:
            raise ValueError("fork count must be positive")
        B = self.block_size
        full = p.seq_len // B
        partial = p.seq_len % B != 0
        if partial and len(self.free) < n:
            raise OutOfBlocks(f"fork needs {n} copy-on-write blocks, "
                              f"{len(self.free)} free")
        out = []
        for _ in range(n):
            child = Node(parent=parent, depth=p.depth + 1, seq_len=p.seq_len)
            cow = None
            if partial:
                dst = self._pop()
                cow = (p.table[full], dst)
            for blk in p.table[:full]:
                self.ref[blk] += 1
            child.table = list(p.table[:full]) + ([cow[1]] if cow else [])
            self.nodes.append(child)
            cid = len(self.nodes) - 1
            p.children.append(cid)
            out.append((cid, cow))
        return out

    def fork(self, parent: int):
        return self.fork_many(parent, 1)[0]

    # -- host tier ("Dismantling the Memory Wall", cross-tier offloading) -------
    # Reading taken: a branch's blocks that only it references move to host
    # slots (a LIFO stack, slot 0 first) in branch order and table order and
    # are freed on the device in that order; shared blocks stay.  A spilled
    # table entry is -(slot + 2).  Restoring pops device blocks in branch and
    # table order and pushes each host slot back as it is emptied.

    def attach_host(self, slots: int) -> None:
        self.host_free = list(reversed(range(slots)))

    def host_free_stack(self) -> list:
        return list(reversed(self.host_free))

    def spill(self, ids) -> list:
        """Returns the (device block, host slot) copies."""
        moved, seen = [], set()
        for i in ids:
            for b in self.live_node(i).table:
                if b >= 0 and self.ref[b] == 1 and b not in seen:
                    seen.add(b)
                    moved.append(b)
        if len(moved) > len(self.host_free):
            raise OutOfBlocks("host tier full")
        pairs = []
        for i in ids:
            nd = self.nodes[i]
            for j, b in enumerate(nd.table):
                if len(pairs) < len(moved) and b == moved[len(pairs)]:
                    slot = self.host_free.pop()
                    self.ref[b] = 0
                    self.free.append(b)
                    nd.table[j] = -(slot + 2)
                    pairs.append((b, slot))
        return pairs

    def restore(self, ids) -> list:
        """Returns the (host slot, device block) copies."""
        ids = list(ids)
        if len(set(ids)) != len(ids):
            raise ValueError("branch listed twice")
        need = sum(1 for i in ids for b in self.live_node(i).table if b < 0)
        if need > len(self.free):
            raise OutOfBlocks("restore needs more device blocks")
        pairs = []
        for i in ids:
            nd = self.nodes[i]
            for j, b in enumerate(nd.table):
                if b < 0:
                    blk = self._pop()
                    slot = -b - 2
                    self.host_free.append(slot)
                    nd.table[j] = blk
                    pairs.append((slot, blk))
        return pairs

    def adopt(self, blocks) -> int:
        """New root branch whose table is the given (full, cached) blocks,
        +1 reference each: a request starting from a cached prefix."""
        nd = Node(parent=-1, depth=0, table=list(blocks),
                  seq_len=len(blocks) * self.block_size)
        for b in blocks:
            self.ref[b] += 1
        self.nodes.append(nd)
        return len(self.nodes) - 1

    def free_node(self, nid: int) -> None:
        nd = self.live_node(nid)
        for blk in nd.table:
            if blk < 0:                     # spilled: its host slot is freed
                self.host_free.append(-blk - 2)
                continue
            self._release(blk)
        nd.table = []
        nd.seq_len = 0
        nd.live = False

    def free_subtree(self, nid: int) -> list:
        """Free every live node of nid's subtree, post-order, children in
        creation order.  Returns the freed ids in freeing order."""
        self.node(nid)
        freed = []

        def walk(x):
            for c in self.nodes[x].children:
                walk(c)
            if self.nodes[x].live:
                self.free_node(x)
                freed.append(x)

        walk(nid)
        return freed

    def omega(self, nid: int, score: float) -> float:
        """Importance score omega = branch_score / (depth + 1), in binary64
        (RKSC summary, §2.C)."""
        return float(score) / float(self.node(nid).depth + 1)

    def evict_order(self, ids, scores) -> list:
        """Candidate ids sorted by ascending omega, ties by ascending id."""
        ids = [int(i) for i in ids]
        scores = [float(s) for s in scores]
        if len(ids) != len(scores):
            raise ValueError("one score per candidate")
        for i in ids:
            self.node(i)
        for s in scores:
            if s != s:
                raise ValueError("NaN score")
        keyed = [(self.omega(i, s), i) for i, s in zip(ids, scores)]
        return [i for _, i in sorted(keyed)]

    def evict(self, ids, scores, stop_kind: int, target: int) -> list:
        """Evict whole subtrees in ascending omega until the target holds.

        ``stop_kind`` STOP_FREE_BLOCKS: stop once at least ``target`` blocks
        are free.  STOP_EVICTED_LEAVES: stop once at least ``target`` leaf
        nodes (nodes without children) have been freed.  A candidate whose
        subtree holds no live node is skipped.  Returns the evicted ids.
        """
        if stop_kind not in (STOP_FREE_BLOCKS, STOP_EVICTED_LEAVES):
            raise ValueError("unknown stop rule")
        evicted, leaves = [], 0
        for nid in self.evict_order(ids, scores):
            if stop_kind == STOP_FREE_BLOCKS and len(self.free) >= target:
                break
            if stop_kind == STOP_EVICTED_LEAVES and leaves >= target:
                break
            freed = self.free_subtree(nid)
            if freed:
                evicted.append(nid)
                leaves += sum(1 for x in freed if not self.nodes[x].children)
        return evicted

    # -- invariants ------------------------------------------------------------
    def check_invariants(self) -> None:
        """Refcount = number of live tables holding the block; free stack =
        blocks with refcount 0, each once; only a table's last block may be
        partial (at most block_size - 1 unused slots per branch)."""
        count = [0] * self.num_blocks
        for nd in self.nodes:
            if not nd.live:
                assert nd.table == []
                continue
            assert len(nd.table) == blocks_for(nd.seq_len, self.block_size)
            for blk in nd.table:
                if blk >= 0:
                    count[blk] += 1
        assert count == self.ref
        assert len(set(self.free)) == len(self.free)
        assert sorted(self.free) == [b for b in range(self.num_blocks)
                                     if self.ref[b] == 0]


class PoolData:
    """The oracle's own host copy of the K and V pools, written by replaying
    the model's appends and copy-on-write copies.

    Layout ``[num_layers][num_blocks][Hkv][block_size][d]`` uint16 (bf16
    bits).  Slots never written stay zero; only slots below a live branch's
    length are meaningful.
    """

    def __init__(self, num_layers, num_blocks, Hkv, block_size, d):
        import numpy as np
        shape = (num_layers, num_blocks, Hkv, block_size, d)
        self.k = np.zeros(shape, dtype=np.uint16)
        self.v = np.zeros(shape, dtype=np.uint16)

    def write(self, writes, k_new, v_new) -> None:
        """k_new, v_new: [L][n][Hkv][d] bf16 bits for the appended tokens."""
        for i, (_t, blk, slot) in enumerate(writes):
            self.k[:, blk, :, slot, :] = k_new[:, i, :, :]
            self.v[:, blk, :, slot, :] = v_new[:, i, :, :]

    def copy_block(self, src: int, dst: int) -> None:
        self.k[:, dst] = self.k[:, src]
        self.v[:, dst] = self.v[:, src]
