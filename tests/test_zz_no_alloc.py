"""paged_decode_attn_noalloc: the decode step for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).

It must give the same output as paged_decode_attn with a caller workspace,
within the parity tolerance used throughout (|a - b| <= 2e-3 + 1e-2 |b|), on
two calls in a row -- the second one runs over the scratch the first left
behind.  This file is collected last so that a run stopping at its first
failure has already run every other test.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from paged_kv_cache_attn_gb300 import binding as B  # noqa: E402
from paged_kv_cache_attn_gb300 import harness as H  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("make", [
    lambda: W.long_context(n_indep=3, indep_tokens=1000, n_roots=2,
                           root_tokens=2048, fan=16, suffix_tokens=37),
    lambda: W.tiny_tree(),
])
def test_noalloc_matches_workspace_entry(make):
    w = make()
    cache = H.Cache(w)
    bt = cache.batch().upload()
    d = bt.dev
    out_ref = torch.empty((bt.nb, w.Hq, w.d), dtype=torch.bfloat16,
                          device="cuda")
    for call in range(2):
        q = torch.from_numpy(w.queries(bt.nb, salt=call).view(np.int16)) \
            .cuda().view(torch.bfloat16)
        bt.decode(q, out_ref)
        out = torch.full_like(out_ref, float("nan"))
        B.paged_decode_attn_noalloc(
            q, cache.k[0], cache.v[0], w.num_blocks, d["tables"],
            d["seq_lens"], d["groups"], len(bt.groups), bt.nb,
            bt.tables.shape[1], w.Hq, w.Hkv, w.d, w.scale, out, d["plan"],
            bt.info)
        torch.cuda.synchronize()
        a, b = _f64(out), _f64(out_ref)
        assert np.isfinite(a).all()
        assert (np.abs(a - b) <= ATOL + RTOL * np.abs(b)).all(), call
    cache.close()


def test_noalloc_rejects_steps_beyond_its_scratch():
    w = W.tiny_tree()
    cache = H.Cache(w)
    bt = cache.batch().upload()
    info = B.kv_decode_plan_info()
    for f, _ in info._fields_:
        setattr(info, f, getattr(bt.info, f))
    info.workspace_bytes = (64 << 20) + 256
    q = torch.zeros((bt.nb, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.KVError) as e:
        B.paged_decode_attn_noalloc(
            q, cache.k[0], cache.v[0], w.num_blocks, bt.dev["tables"],
            bt.dev["seq_lens"], bt.dev["groups"], len(bt.groups), bt.nb,
            bt.tables.shape[1], w.Hq, w.Hkv, w.d, w.scale, torch.empty_like(q),
            bt.dev["plan"], info)
    assert e.value.code == B.KV_ERR_INVALID_ARG and "64 MiB" in str(e.value)
    cache.close()
