"""Seeded synthetic workloads: tree shapes, segment lengths, KV and query values.

This module is the only thing the CUDA path and the CPU oracle both consume.
It holds none of the method's arithmetic -- no attention, no allocator, no
block translation: it only says which branch nodes exist (parent, tokens each
node appends after its fork), in which order they are created, the seeded
bf16 values of each node's K/V rows and of the decode queries, the seeded
physical free-block order and the seeded eviction scores.  It imports numpy
only.

Five workload families, after the decode-attention configurations the
reasoning-tree setting calls for:

1. ``tiny_tree``: 4 q-heads / 2 kv-heads, head_dim 64; a 100-token root forked
   into 4 branches that append 20/27/33/40 tokens.
2. ``independent``: 32 / 8 / 128 (Llama-3-8B attention shape); 64 independent
   sequences, lengths uniform in [512, 4096].
3. ``fanout``: 32 / 8 / 128; 8 roots of 2048 tokens, each forked into 64
   branches with suffixes uniform in [128, 1024].
4. ``deep_tree``: 64 / 8 / 128 (70B shape); a 4096-token root, branching factor
   3 to depth 5 (243 leaves), per-node segments uniform in [64, 256]; before
   the step, whole subtrees are evicted by the importance score until 30% of
   the leaves are gone (scores uniform in (0, 1)).
5. ``long_context``: 64 / 8 / 128; 128 sequences of 8192 tokens plus 16 roots
   of 32768 tokens each forked into 16 branches of 512 suffix tokens.

All use block size 16, one layer, values ~ N(0, 1) drawn in fp32 and rounded
to bf16 (round to nearest even), scale 1/sqrt(head_dim), and a seeded random
permutation of the physical block ids as the pool's initial free order.  Each
generator takes size arguments so tests can build a smaller case of the same
structure.  Integer uniforms are inclusive of both ends.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


@dataclass
class NodeSpec:
    parent: int        # -1 for a root
    n_tokens: int      # tokens the node appends after it is created/forked


@dataclass
class Workload:
    """A tree of branch nodes plus the seeds of every value they hold.

    ``ops`` is the exact creation order: ``("create",)`` makes a root,
    ``("fork", parent, count)`` makes ``count`` children, ``("append", nid)``
    appends ``nodes[nid].n_tokens`` tokens.  Handles are assigned 0, 1, 2, ...
    in the order roots and children are made, which is the order of
    ``nodes``.
    """
    name: str
    Hq: int
    Hkv: int
    d: int
    seed: int
    nodes: list = field(default_factory=list)
    ops: list = field(default_factory=list)
    block_size: int = BLOCK_SIZE
    num_layers: int = 1
    num_blocks: int = 0
    evict_scores: np.ndarray | None = None     # float64 per node (roots unused)
    evict_leaf_fraction: float = 0.0
    q_gain: float = 1.0
    description: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def children(self, nid: int) -> list:
        return [i for i, n in enumerate(self.nodes) if n.parent == nid]

    def leaves(self) -> list:
        has_child = {n.parent for n in self.nodes}
        return [i for i in range(len(self.nodes)) if i not in has_child]

    def initial_free_order(self) -> np.ndarray:
        rng = np.random.default_rng([self.seed, 7])
        return rng.permutation(self.num_blocks).astype(np.int32)

    def node_kv(self, nid: int):
        """K and V rows a node appends: two uint16 arrays [L][n][Hkv][d]."""
        n = self.nodes[nid].n_tokens
        rng = np.random.default_rng([self.seed, 1, nid])
        shape = (self.num_layers, n, self.Hkv, self.d)
        k = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        v = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        return k, v

    def queries(self, nb: int, salt: int = 0) -> np.ndarray:
        """Decode queries for a batch of nb branches: uint16 [nb][Hq][d]."""
        rng = np.random.default_rng([self.seed, 2, salt])
        q = rng.standard_normal((nb, self.Hq, self.d), dtype=np.float32)
        return f32_to_bf16_bits(q * np.float32(self.q_gain))

    def total_node_tokens(self) -> int:
        return sum(n.n_tokens for n in self.nodes)

    def evict_target_leaves(self) -> int:
        """How many leaves the pre-step eviction must remove (0: none)."""
        if self.evict_scores is None or self.evict_leaf_fraction <= 0:
            return 0
        return math.ceil(self.evict_leaf_fraction * len(self.leaves()))

    def evict_candidates(self) -> list:
        """Every non-root node is an eviction candidate."""
        return [i for i, n in enumerate(self.nodes) if n.parent >= 0]


def _pool_blocks(nodes, block_size, slack=1.02):
    # Upper bound on what the tree can hold: each node's own tokens plus one
    # copied block per fork, with a little slack so the pool is never exact.
    bound = sum((n.n_tokens + block_size - 1) // block_size + 1 for n in nodes)
    return int(bound * slack) + 16


def _finish(w: Workload) -> Workload:
    w.num_blocks = _pool_blocks(w.nodes, w.block_size)
    return w


def tiny_tree(seed: int = 1001, root_tokens: int = 100,
              suffixes=(20, 27, 33, 40), Hq: int = 4, Hkv: int = 2,
              d: int = 64, q_gain: float = 1.0) -> Workload:
    w = Workload("tiny_tree", Hq, Hkv, d, seed, q_gain=q_gain,
                 description=f"root {root_tokens} tokens forked into "
                             f"{len(suffixes)} branches {list(suffixes)}")
    w.nodes.append(NodeSpec(-1, root_tokens))
    w.ops += [("create",), ("append", 0), ("fork", 0, len(suffixes))]
    for s in suffixes:
        w.nodes.append(NodeSpec(0, int(s)))
    for i in range(1, len(suffixes) + 1):
        w.ops.append(("append", i))
    return _finish(w)


def independent(seed: int = 1002, n_seqs: int = 64, min_len: int = 512,
                max_len: int = 4096, Hq: int = 32, Hkv: int = 8,
                d: int = 128) -> Workload:
    rng = np.random.default_rng([seed, 0])
    lens = rng.integers(min_len, max_len, size=n_seqs, endpoint=True)
    w = Workload("independent", Hq, Hkv, d, seed,
                 description=f"{n_seqs} independent sequences, lengths "
                             f"U[{min_len}, {max_len}]")
    for i, L in enumerate(lens):
        w.nodes.append(NodeSpec(-1, int(L)))
        w.ops += [("create",), ("append", i)]
    return _finish(w)


def fanout(seed: int = 1003, n_roots: int = 8, root_tokens: int = 2048,
           fan: int = 64, min_suffix: int = 128, max_suffix: int = 1024,
           Hq: int = 32, Hkv: int = 8, d: int = 128) -> Workload:
    rng = np.random.default_rng([seed, 0])
    w = Workload("fanout", Hq, Hkv, d, seed,
                 description=f"{n_roots} roots x {root_tokens} tokens, each "
                             f"forked into {fan} branches, suffixes "
                             f"U[{min_suffix}, {max_suffix}]")
    for _ in range(n_roots):
        r = len(w.nodes)
        w.nodes.append(NodeSpec(-1, root_tokens))
        w.ops += [("create",), ("append", r), ("fork", r, fan)]
        suffix = rng.integers(min_suffix, max_suffix, size=fan, endpoint=True)
        first = len(w.nodes)
        for s in suffix:
            w.nodes.append(NodeSpec(r, int(s)))
        for i in range(first, first + fan):
            w.ops.append(("append", i))
    return _finish(w)


def deep_tree(seed: int = 1004, root_tokens: int = 4096, branching: int = 3,
              depth: int = 5, min_seg: int = 64, max_seg: int = 256,
              evict_leaf_fraction: float = 0.3, Hq: int = 64, Hkv: int = 8,
              d: int = 128) -> Workload:
    rng = np.random.default_rng([seed, 0])
    w = Workload("deep_tree", Hq, Hkv, d, seed,
                 evict_leaf_fraction=evict_leaf_fraction,
                 description=f"root {root_tokens} tokens, branching "
                             f"{branching} to depth {depth}, segments "
                             f"U[{min_seg}, {max_seg}], "
                             f"{int(evict_leaf_fraction * 100)}% of leaves "
                             "evicted by importance score")
    w.nodes.append(NodeSpec(-1, root_tokens))
    w.ops += [("create",), ("append", 0)]
    level = [0]
    for _ in range(depth):
        nxt = []
        for p in level:
            w.ops.append(("fork", p, branching))
            first = len(w.nodes)
            seg = rng.integers(min_seg, max_seg, size=branching, endpoint=True)
            for s in seg:
                w.nodes.append(NodeSpec(p, int(s)))
            for i in range(first, first + branching):
                w.ops.append(("append", i))
                nxt.append(i)
        level = nxt
    w.evict_scores = np.random.default_rng([seed, 3]).random(len(w.nodes))
    return _finish(w)


def long_context(seed: int = 1005, n_indep: int = 128, indep_tokens: int = 8192,
                 n_roots: int = 16, root_tokens: int = 32768, fan: int = 16,
                 suffix_tokens: int = 512, Hq: int = 64, Hkv: int = 8,
                 d: int = 128) -> Workload:
    w = Workload("long_context", Hq, Hkv, d, seed,
                 description=f"{n_indep} x {indep_tokens} independent + "
                             f"{n_roots} roots x {root_tokens} forked into "
                             f"{fan} x {suffix_tokens} suffixes")
    for i in range(n_indep):
        w.nodes.append(NodeSpec(-1, indep_tokens))
        w.ops += [("create",), ("append", i)]
    for _ in range(n_roots):
        r = len(w.nodes)
        w.nodes.append(NodeSpec(-1, root_tokens))
        w.ops += [("create",), ("append", r), ("fork", r, fan)]
        first = len(w.nodes)
        for _ in range(fan):
            w.nodes.append(NodeSpec(r, suffix_tokens))
        for i in range(first, first + fan):
            w.ops.append(("append", i))
    return _finish(w)


def long_context_quarter(seed: int = 1005) -> Workload:
    """long_context at a quarter of the trees (for profiler captures)."""
    w = long_context(seed=seed, n_indep=32, n_roots=4)
    w.name = "long_context_quarter"
    return w


CONFIGS = {
    "tiny_tree": tiny_tree,
    "independent": independent,
    "fanout": fanout,
    "deep_tree": deep_tree,
    "long_context": long_context,
    "long_context_quarter": long_context_quarter,
}


def make(name: str, rank: int = 0, **sizes) -> Workload:
    """Workload ``name`` for one rank of a multi-GPU run.  Every rank gets its
    own trees (the default seed offset by 1000 x rank) of the same shape, so
    ranks share nothing and need no exchange."""
    import inspect
    fn = CONFIGS[name]
    seed = inspect.signature(fn).parameters["seed"].default + 1000 * rank
    return fn(seed=seed, **sizes)

