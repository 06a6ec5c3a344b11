"""Host-side rules of e4m3 pools, checked on the CPU: argument validation at
pool creation and host-tier attach, the plan flag and its effect on the work
split, and the decode entry points refusing a plan made for the other
element type before any device work (fake, aligned addresses are passed
where a device pointer is required; nothing dereferences them)."""

import numpy as np
import pytest

from paged_kv_cache_attn_gb300 import binding as B
from paged_kv_cache_attn_gb300 import workloads as W

FAKE = 0x10000      # 16-byte aligned stand-in for a device address
FAKE2 = 0x20000
FAKE3 = 0x30000


def create(**kw):
    args = dict(num_blocks=64, num_layers=1, num_kv_heads=2, head_dim=128)
    args.update(kw)
    return B.kv_pool_create(args.pop("num_blocks"), args.pop("num_layers"),
                            args.pop("num_kv_heads"), args.pop("head_dim"),
                            **args)


def code(fn):
    with pytest.raises(B.KVError) as e:
        fn()
    return e.value.code


def test_pool_create_validates_dtype_and_scales():
    # metadata-only e4m3 pool: fine
    B.kv_pool_destroy(create(kv_dtype=B.KV_DTYPE_E4M3))
    # e4m3 data pool with its scale records: fine (nothing is touched)
    B.kv_pool_destroy(create(k_pool=FAKE, v_pool=FAKE2,
                             kv_dtype=B.KV_DTYPE_E4M3, kv_scales=FAKE3))
    assert code(lambda: create(kv_dtype=7)) == B.KV_ERR_INVALID_ARG
    # an e4m3 data pool needs kv_scales
    assert code(lambda: create(k_pool=FAKE, v_pool=FAKE2,
                               kv_dtype=B.KV_DTYPE_E4M3)) == B.KV_ERR_INVALID_ARG
    # kv_scales only for e4m3 data pools, 16-byte aligned
    assert code(lambda: create(k_pool=FAKE, v_pool=FAKE2,
                               kv_scales=FAKE3)) == B.KV_ERR_INVALID_ARG
    assert code(lambda: create(kv_dtype=B.KV_DTYPE_E4M3,
                               kv_scales=FAKE3)) == B.KV_ERR_INVALID_ARG
    assert code(lambda: create(k_pool=FAKE, v_pool=FAKE2,
                               kv_dtype=B.KV_DTYPE_E4M3,
                               kv_scales=FAKE3 + 8)) == B.KV_ERR_INVALID_ARG


def test_host_tier_attach_rules_for_e4m3():
    h = create(k_pool=FAKE, v_pool=FAKE2, kv_dtype=B.KV_DTYPE_E4M3,
               kv_scales=FAKE3)
    # the scale records need a host copy too
    assert code(lambda: B.kv_offload_attach(h, FAKE, FAKE2, 8)) == \
        B.KV_ERR_INVALID_ARG
    B.kv_offload_attach(h, FAKE, FAKE2, 8, host_scales=FAKE3)
    B.kv_pool_destroy(h)
    h = create(k_pool=FAKE, v_pool=FAKE2)          # bf16 data pool
    assert code(lambda: B.kv_offload_attach(h, FAKE, FAKE2, 8,
                                            host_scales=FAKE3)) == \
        B.KV_ERR_INVALID_ARG
    B.kv_pool_destroy(h)


def segment_plan(flags):
    """One shared-prefix segment of 40 branches x 8 heads (320 rows, three
    128-row tiles) over 32 full blocks, and a 4-block suffix per branch."""
    nb, mb = 40, 36
    lens = np.full(nb, 36 * 16, dtype=np.int32)
    groups = np.array([[0, nb, 0, 32]], dtype=np.int32)
    return B.paged_decode_plan(nb, 64, 8, 128, mb, lens, groups, 152, flags)


def test_plan_records_its_flags_and_keeps_e4m3_tiles_narrow():
    _, bf = segment_plan(0)
    _, e8 = segment_plan(B.KV_PLAN_KV_E4M3)
    assert bf.flags == 0 and e8.flags == B.KV_PLAN_KV_E4M3
    # 320 rows: three 128-row tiles per block range and kv-head either way
    assert bf.n_tile_wide_items == 0 == e8.n_tile_wide_items
    assert e8.n_tile_items == bf.n_tile_items > 0
    assert e8.n_tile_items == 3 * 8 * (e8.n_tile_items // 24)
    # 256 rows: one two-M-tile item in bf16 (not in e4m3, nor in a narrow
    # plan)
    nb, mb = 32, 36
    lens = np.full(nb, 36 * 16, dtype=np.int32)
    groups = np.array([[0, nb, 0, 32]], dtype=np.int32)
    plans = {f: B.paged_decode_plan(nb, 64, 8, 128, mb, lens, groups, 152, f)[1]
             for f in (0, B.KV_PLAN_NARROW_TILES, B.KV_PLAN_KV_E4M3)}
    w = plans[0]
    assert w.n_tile_items == w.n_tile_wide_items > 0
    for f in (B.KV_PLAN_NARROW_TILES, B.KV_PLAN_KV_E4M3):
        assert plans[f].n_tile_wide_items == 0
        assert plans[f].n_tile_items == 2 * w.n_tile_items
    _, nt = segment_plan(B.KV_PLAN_KV_E4M3 | B.KV_PLAN_NO_TENSOR_CORES)
    assert nt.n_tile_items == 0
    assert code(lambda: segment_plan(64)) == B.KV_ERR_INVALID_ARG


def test_decode_refuses_a_plan_for_the_other_element_type():
    nb, mb = 40, 36
    lens = np.full(nb, 36 * 16, dtype=np.int32)
    plan_bf, info_bf = segment_plan(0)
    plan_e8, info_e8 = segment_plan(B.KV_PLAN_KV_E4M3)
    common = dict(num_blocks=4096, block_tables=FAKE, seq_lens=FAKE,
                  prefix_groups=FAKE, n_groups=1, nb=nb, max_blocks=mb, Hq=64,
                  Hkv=8, head_dim=128, scale=0.088, out=FAKE, plan=FAKE)
    ws = info_bf.workspace_bytes
    assert code(lambda: B.paged_decode_attn_e4m3(
        FAKE, FAKE, FAKE, FAKE3, common["num_blocks"], FAKE, FAKE, FAKE, 1,
        nb, mb, 64, 8, 128, 0.088, FAKE, FAKE, info_bf, 0x100000, ws)) == \
        B.KV_ERR_INVALID_ARG
    assert code(lambda: B.paged_decode_attn(
        FAKE, FAKE, FAKE, common["num_blocks"], FAKE, FAKE, FAKE, 1, nb, mb,
        64, 8, 128, 0.088, FAKE, FAKE, info_e8, 0x100000,
        info_e8.workspace_bytes)) == B.KV_ERR_INVALID_ARG
    # and the scale records are required by the e4m3 entry point
    assert code(lambda: B.paged_decode_attn_e4m3(
        FAKE, FAKE, FAKE, None, common["num_blocks"], FAKE, FAKE, FAKE, 1,
        nb, mb, 64, 8, 128, 0.088, FAKE, FAKE, info_e8, 0x100000,
        info_e8.workspace_bytes)) == B.KV_ERR_INVALID_ARG


def test_decode_refuses_a_bad_short_item_count():
    """The count of short split items (run one per warp) must lie within the
    plan's split items; decode checks it before any device work."""
    nb, mb = 40, 36
    _, info = segment_plan(0)
    for bad in (-1, info.n_row_items + 1):
        info.n_row_warp_items = bad
        with pytest.raises(B.KVError) as e:
            B.paged_decode_attn(FAKE, FAKE, FAKE, 4096, FAKE, FAKE, FAKE, 1, nb,
                                mb, 64, 8, 128, 0.088, FAKE, FAKE, info,
                                0x100000, info.workspace_bytes)
        assert e.value.code == B.KV_ERR_INVALID_ARG
        assert "n_row_warp_items" in str(e.value)   # this check, no other


def test_e4m3_metadata_pool_replays_like_bf16():
    """The allocator does not depend on the element type."""
    from paged_kv_cache_attn_gb300 import harness as H
    w = W.make("deep_tree")
    a = H.Cache(w, with_data=False)
    b = H.Cache(w, with_data=False, kv_dtype="e4m3")
    assert a.tables() == b.tables()
    assert a.refcounts() == b.refcounts()
    assert a.free_stack() == b.free_stack()
    assert a.decode_ids == b.decode_ids
    a.close()
    b.close()
