"""The bounded-wait timeout path, exercised without a fault or a hang: a
wait on an mbarrier that nothing completes runs out after its bound,
records KV_ERR_TIMEOUT in the status word, the host reads it back, and the
context stays usable for a normal decode step."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import attention as att  # noqa: E402
from oracle import replay as rp  # noqa: E402
from paged_kv_cache_attn_gb300 import binding as B  # noqa: E402
from paged_kv_cache_attn_gb300 import harness as H  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402


def test_timeout_is_recorded_and_the_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    B.kv_selftest_timeout(ws, 1 << 22)          # a few milliseconds
    code, detail = B.kv_check_device_status(ws)
    assert (code, detail) == (B.KV_ERR_TIMEOUT, 99)
    assert B.kv_check_device_status(ws) == (0, 0)   # read clears it
    with pytest.raises(B.KVError):
        B.kv_selftest_timeout(ws, 0)
    # a normal step afterwards
    w = W.tiny_tree()
    cache = H.Cache(w)
    ref = rp.replay(w, with_data=True)
    q = w.queries(len(cache.decode_ids))
    bt = cache.batch().upload()
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty_like(qd)
    bt.decode(qd, out)
    torch.cuda.synchronize()
    assert bt.device_status() == (0, 0)
    gpu = att.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    want = rp.decode_all_from_pool(ref, q, w.scale)
    assert np.all(np.abs(gpu - want) <= 2e-3 + 1e-2 * np.abs(want))
    cache.close()
