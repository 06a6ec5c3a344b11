"""The bench's byte accounting, checked on the CPU against figures that follow
from each workload's own definition (the roofline and the sharing criterion
are computed from these counts):

* unique KV bytes: every distinct physical block once, weighted by its valid
  tokens, x Hkv x d x 2 bytes x 2 (K and V) -- against the token counts the
  workload specifies (its sequences, roots and suffixes);
* a plan that reads every block once (no segment of more than 128 rows)
  requests exactly the unique bytes; the per-branch re-read plan requests
  each branch's whole sequence;
* prefix bytes: the segment items read each shared prefix once, the re-read
  arm once per branch (the branch-sharing factor);
* the kernels a step launches.
"""

import numpy as np
import pytest

import bench
from paged_kv_cache_attn_gb300 import binding as B
from paged_kv_cache_attn_gb300 import harness as H
from paged_kv_cache_attn_gb300 import workloads as W


def _plan(w, flags=0):
    return H.Cache(w, with_data=False).batch(num_sms=152, flags=flags)


def _per_token(w):
    return w.Hkv * w.d * 2 * 2


def _own_tokens(w):
    """Tokens each node adds on top of its parent (the workload's spec)."""
    return [n.n_tokens for n in w.nodes]


def test_unique_bytes_follow_the_workload_definition():
    # long_context: 128 sequences of 8192 tokens, 16 roots of 32768 tokens
    # each forked into 16 branches of 512 (every boundary block-aligned, so
    # no copy-on-write block)
    w = W.make("long_context")
    bt = _plan(w)
    want = (128 * 8192 + 16 * 32768 + 16 * 16 * 512) * _per_token(w)
    assert want == 6_979_321_856
    assert bench.unique_kv_bytes(bt.tables, bt.seq_lens, w.Hkv, w.d) == want
    # tiny_tree: a 100-token root (6 full blocks and 4 tokens) forked into
    # 4 branches; each fork copies the 4-token partial block, then appends
    # 20 / 27 / 33 / 40 tokens: 96 + 4 x 4 + 120 = 232 tokens
    w = W.make("tiny_tree")
    bt = _plan(w)
    assert bench.unique_kv_bytes(bt.tables, bt.seq_lens, w.Hkv, w.d) == \
        232 * _per_token(w) == 118_784
    # independent and fanout: the specified tokens, each stored once (the
    # fan-out roots are 2048 tokens, block-aligned)
    for name in ("independent", "fanout"):
        w = W.make(name)
        bt = _plan(w)
        got = bench.unique_kv_bytes(bt.tables, bt.seq_lens, w.Hkv, w.d)
        assert got == sum(_own_tokens(w)) * _per_token(w), name


@pytest.mark.parametrize("name", ["long_context", "independent", "fanout"])
def test_a_shared_plan_requests_the_unique_bytes(name):
    w = W.make(name)
    bt = _plan(w)
    uniq = bench.unique_kv_bytes(bt.tables, bt.seq_lens, w.Hkv, w.d)
    got = sum(bench.item_bytes(bt.plan, bt.info, w.Hkv, w.d, bt.seq_lens, k)
              for k in ("row", "tile"))
    assert got == uniq
    # re-read arm: every branch reads its whole sequence
    br = _plan(w, B.KV_PLAN_IGNORE_GROUPS)
    assert br.info.n_tile_items == 0
    assert bench.item_bytes(br.plan, br.info, w.Hkv, w.d, br.seq_lens, "row") \
        == int(np.sum(br.seq_lens)) * _per_token(w)


def test_deep_tree_requests_its_root_once_per_m_tile():
    # 1360 rows over the 4096-token root: 11 M-tiles of 128 rows each read
    # the root, so the step requests more than its unique bytes
    w = W.make("deep_tree")
    bt = _plan(w)
    uniq = bench.unique_kv_bytes(bt.tables, bt.seq_lens, w.Hkv, w.d)
    got = sum(bench.item_bytes(bt.plan, bt.info, w.Hkv, w.d, bt.seq_lens, k)
              for k in ("row", "tile"))
    assert got > uniq
    root = 4096 * _per_token(w)
    tiles = bench.plan_items(bt.plan, bt.info, "tile")
    root_items = tiles[(tiles[:, 4] == 0) & (tiles[:, 5] == 256)]
    assert len(root_items) == 11 * w.Hkv
    assert bench.item_bytes(bt.plan, bt.info, w.Hkv, w.d, bt.seq_lens,
                            "tile", segments_only=True) >= 11 * root


@pytest.mark.parametrize("name,roots,root_tokens,fan", [
    ("long_context", 16, 32768, 16),
    ("fanout", 8, 2048, 64),
])
def test_prefix_bytes_shared_once_reread_once_per_branch(name, roots,
                                                         root_tokens, fan):
    w = W.make(name)
    bt = _plan(w)
    prefix = roots * root_tokens * _per_token(w)
    shared = sum(bench.item_bytes(bt.plan, bt.info, w.Hkv, w.d, bt.seq_lens, k,
                                  segments_only=True)
                 for k in ("row", "tile"))
    assert shared == prefix
    # the re-read arm's prefix: each branch's segment blocks, as the bench
    # counts them from the segments
    kvb = 2 * w.d * 2 * w.Hkv * 16
    reread = int(sum(int(g[1]) * int(g[3]) for g in bt.groups)) * kvb
    assert reread == fan * prefix
    assert reread // shared == fan


@pytest.mark.parametrize("name,kernels,launches", [
    ("long_context", "tile_decode_kernel", 3),
    ("fanout", "tile_wide_kernel", 3),
    ("deep_tree", "tile_wide_kernel+tile_decode_kernel", 4),
    ("independent", "", 2),
])
def test_kernels_a_step_launches(name, kernels, launches):
    bt = _plan(W.make(name))
    assert bench.tile_kernel_name(bt.info) == kernels
    assert bench.kernels_per_step(bt.info) == launches
