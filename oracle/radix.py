"""Model of a token-keyed radix prefix index over the block pool.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

From "Dismantling the Memory Wall", RadixAttention section: a compressed
prefix tree (nodes with a single child are merged into their parent); each
node holds a token sequence (its key), the KV of those tokens (its value), a
lock_ref and a last-access time; a request using a prefix increments lock_ref
on that node and all its ancestors, so they cannot be overwritten; under
memory pressure the least-recently-used leaves with lock_ref 0 are evicted,
which keeps shared roots (system prompts) cached.

Readings taken for the paged pool:
* the sharing unit is a full 16-token block: keys are whole blocks, the value
  of a node is the physical block of each of its 16-token chunks, and the
  index holds one reference on every block it stores;
* recency is a logical clock that ticks once per match or insert; every node
  on the matched path takes the current tick;
* a match that ends inside a node splits it: the new node (next id) takes the
  prefix and the node's place under its parent, the old node keeps its id and
  the rest of its key and hangs below the new one (same lock_ref and time);
* eviction picks, repeatedly, the leaf (no children, not the root) with
  lock_ref 0 and the smallest (last-access, id), releases its blocks in key
  order and removes it; a parent left without children is a leaf in turn; it
  stops once the pool holds the target number of free blocks or no leaf
  qualifies.
"""

from __future__ import annotations

from dataclasses import dataclass, field

BLOCK = 16


@dataclass
class RNode:
    parent: int
    key: list = field(default_factory=list)      # tokens
    blocks: list = field(default_factory=list)   # one per 16 tokens
    children: list = field(default_factory=list)
    lock_ref: int = 0
    last_access: int = 0
    live: bool = True


class RadixModel:
    def __init__(self, pool):
        self.pool = pool                 # oracle.allocator.PoolModel
        self.nodes = [RNode(parent=-1)]
        self.clock = 0

    def _child(self, node, chunk):
        for c in self.nodes[node].children:
            if self.nodes[c].key[:BLOCK] == chunk:
                return c
        return None

    def _split(self, x, m):
        X = self.nodes[x]
        y = RNode(parent=X.parent, key=X.key[:m * BLOCK], blocks=X.blocks[:m],
                  children=[x], lock_ref=X.lock_ref, last_access=X.last_access)
        self.nodes.append(y)
        yid = len(self.nodes) - 1
        X.key = X.key[m * BLOCK:]
        X.blocks = X.blocks[m:]
        sib = self.nodes[y.parent].children
        sib[sib.index(x)] = yid
        X.parent = yid
        return yid

    def _walk(self, tokens, nfull):
        cur, pos = 0, 0
        self.nodes[0].last_access = self.clock
        while pos < nfull:
            c = self._child(cur, list(tokens[pos * BLOCK:(pos + 1) * BLOCK]))
            if c is None:
                break
            C = self.nodes[c]
            m = 1
            while (m < len(C.blocks) and pos + m < nfull and
                   C.key[m * BLOCK:(m + 1) * BLOCK] ==
                   list(tokens[(pos + m) * BLOCK:(pos + m + 1) * BLOCK])):
                m += 1
            hit = self._split(c, m) if m < len(C.blocks) else c
            self.nodes[hit].last_access = self.clock
            cur = hit
            pos += m
        return cur, pos

    def match(self, tokens):
        self.clock += 1
        node, blocks = self._walk(list(tokens), len(tokens) // BLOCK)
        return node, blocks * BLOCK

    def insert(self, branch, tokens):
        br = self.pool.live_node(branch)
        tokens = list(tokens)
        nfull = min(len(tokens), br.seq_len) // BLOCK
        self.clock += 1
        cur, pos = self._walk(tokens, nfull)
        if pos < nfull:
            leaf = RNode(parent=cur, key=tokens[pos * BLOCK:nfull * BLOCK],
                         blocks=list(br.table[pos:nfull]),
                         last_access=self.clock)
            for b in leaf.blocks:
                self.pool.ref[b] += 1
            self.nodes.append(leaf)
            cur_id = len(self.nodes) - 1
            self.nodes[cur].children.append(cur_id)
            cur = cur_id
        return cur

    def _path(self, node):
        out = []
        while node != -1:
            out.append(node)
            node = self.nodes[node].parent
        return out

    def fork(self, node):
        if not self.nodes[node].live:
            raise KeyError(node)
        blocks = []
        for x in reversed(self._path(node)):
            blocks += self.nodes[x].blocks
        return self.pool.adopt(blocks)

    def lock(self, node):
        if not self.nodes[node].live:
            raise KeyError(node)
        for x in self._path(node):
            self.nodes[x].lock_ref += 1

    def unlock(self, node):
        if not self.nodes[node].live:
            raise KeyError(node)
        path = self._path(node)
        if any(self.nodes[x].lock_ref < 1 for x in path):
            raise ValueError("not locked")
        for x in path:
            self.nodes[x].lock_ref -= 1

    def evict(self, target_free_blocks):
        evicted = []
        while self.pool.free_count() < target_free_blocks:
            cand = [(n.last_access, i) for i, n in enumerate(self.nodes)
                    if i > 0 and n.live and not n.children and n.lock_ref == 0]
            if not cand:
                break
            _, i = min(cand)
            n = self.nodes[i]
            for b in n.blocks:
                self.pool._release(b)
            n.blocks, n.key, n.live = [], [], False
            self.nodes[n.parent].children.remove(i)
            evicted.append(i)
        return evicted

    def destroy(self):
        for n in self.nodes:
            if n.live:
                for b in n.blocks:
                    self.pool._release(b)
