"""Shared-prefix segment lengths at the edges of the tensor-core tile kernels'
pipelines, in both element types: one block, one 128-token tile, exactly
three tiles (the depth of the bf16 kernel's K/V rings and of the e4m3
kernel's K code ring), three tiles and a block, eight tiles and a block, and
a long segment (40 tiles and a ragged tail) that wraps every ring many times.
Each tree has 20 branches x 8 q-heads per kv-head = 160 rows: in bf16 one
256-row item whose second M-tile is ragged (or, in a narrow-tile plan, two
128-row tiles, the second one ragged), in e4m3 two 128-row tiles; the
branches' own suffixes go to the split-KV pass.  The plan is made for one SM
(the split sizes do not change the result), so that each tile item covers
its whole segment instead of a chunk of it.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import attention as att  # noqa: E402
from oracle import replay as rp  # noqa: E402
from paged_kv_cache_attn_gb300 import binding as B  # noqa: E402
from paged_kv_cache_attn_gb300 import harness as H  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2

# Full blocks of the shared root (its tokens past the last full block are
# copied into each branch on the fork and read by the split-KV pass).
ROOT_BLOCKS = [1, 8, 24, 25, 65, 325]


@pytest.mark.parametrize("kv_dtype", ["bf16", "bf16-narrow", "e4m3"])
@pytest.mark.parametrize("blocks", ROOT_BLOCKS)
def test_segment_lengths_at_ring_edges(blocks, kv_dtype):
    narrow = kv_dtype == "bf16-narrow"
    kv_dtype = "bf16" if narrow else kv_dtype
    w = W.fanout(n_roots=1, root_tokens=16 * blocks + 3, fan=20, min_suffix=1,
                 max_suffix=40, Hq=64, Hkv=8)
    cache = H.Cache(w, kv_dtype=kv_dtype)
    ref = rp.replay(w, with_data=True, kv_dtype=kv_dtype)
    q = w.queries(len(cache.decode_ids))
    bt = cache.batch(num_sms=1,
                     flags=B.KV_PLAN_NARROW_TILES if narrow else 0).upload()
    # planned for one SM, every tile item covers its whole segment (the
    # 325-block one in a single item of 40 tiles and a ragged tail)
    per_head = 1 if kv_dtype == "bf16" and not narrow else 2
    assert bt.info.n_tile_items == 8 * per_head
    assert bt.info.n_tile_wide_items == (bt.info.n_tile_items
                                         if per_head == 1 else 0)
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty_like(qd)
    bt.decode(qd, out)
    torch.cuda.synchronize()
    assert bt.device_status() == (0, 0)
    gpu = att.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    want = rp.decode_all_from_pool(ref, q, w.scale)
    err = np.abs(gpu - want)
    bad = err > ATOL + RTOL * np.abs(want)
    assert not bad.any(), (f"{blocks} blocks {kv_dtype}: {bad.sum()} outside, "
                           f"max err {err.max():.3g}")
    cache.close()
