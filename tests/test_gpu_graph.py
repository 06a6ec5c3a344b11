"""The decode step captured into a CUDA graph and replayed: the side-stream
fork / join of the tile pass, the status-word clear and every kernel are
captured; replays with new query values give the oracle's answer."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import attention as att  # noqa: E402
from oracle import replay as rp  # noqa: E402
from paged_kv_cache_attn_gb300 import harness as H  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2

CASES = {
    "long_context": lambda: W.long_context(n_indep=3, indep_tokens=1000,
                                           n_roots=2, root_tokens=2048,
                                           fan=16, suffix_tokens=37),
    "deep_tree": lambda: W.deep_tree(root_tokens=300, depth=3, min_seg=5,
                                     max_seg=40),
    # a 696-row root (128-row tiles) and depth-1 segments of 80-176 rows
    # (256-row items beside 128-row ones): both tile kernels, on two side
    # streams, inside the capture
    "wide_tree": lambda: W.deep_tree(root_tokens=300, depth=3, branching=5,
                                     min_seg=20, max_seg=50),
}


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("name", list(CASES))
def test_captured_step_replays(name, kv_dtype):
    w = CASES[name]()
    cache = H.Cache(w, kv_dtype=kv_dtype)
    ref = rp.replay(w, with_data=True, kv_dtype=kv_dtype)
    nb = len(cache.decode_ids)
    bt = cache.batch().upload()
    assert bt.info.n_tile_items > 0 and bt.info.n_row_items > 0  # both passes
    if name == "wide_tree" and kv_dtype == "bf16":
        assert 0 < bt.info.n_tile_wide_items < bt.info.n_tile_items
    q = torch.empty((nb, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    # Warm up outside the capture (first-use function attributes, streams).
    q.copy_(torch.from_numpy(w.queries(nb).view(np.int16)).cuda().view(torch.bfloat16))
    bt.decode(q, out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bt.decode(q, out)
    for salt in (11, 12, 13):
        qh = w.queries(nb, salt=salt)
        q.copy_(torch.from_numpy(qh.view(np.int16)).cuda().view(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        gpu = att.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        want = rp.decode_all_from_pool(ref, qh, w.scale)
        err = np.abs(gpu - want)
        assert (err <= ATOL + RTOL * np.abs(want)).all(), (salt, err.max())
    assert bt.device_status() == (0, 0)
    cache.close()
