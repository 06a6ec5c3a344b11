"""paged_decode_attn_noalloc: the decode step for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).

It runs the same plan and kernels as paged_decode_attn, only with the
library's scratch in place of a caller workspace, so its output must equal
paged_decode_attn's bit for bit (which also puts it inside the parity
tolerance used throughout, |a - b| <= 2e-3 + 1e-2 |b|), on two calls in a row
-- the second one runs over the scratch the first left behind -- and its
status word, read through kv_check_noalloc_status, must stay 0.  A bad block
id in a table must show up in that status word.  This file is collected last
so that a run stopping at its first failure has already run every other test.
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


def _noalloc(cache, bt, q, out):
    w, d = cache.w, bt.dev
    B.paged_decode_attn_noalloc(
        q, cache.k[0], cache.v[0], w.num_blocks, d["tables"], d["seq_lens"],
        d["groups"], len(bt.groups), bt.nb, bt.tables.shape[1], w.Hq, w.Hkv,
        w.d, w.scale, out, d["plan"], bt.info)


@pytest.mark.parametrize("make", [
    lambda: W.long_context(n_indep=3, indep_tokens=1000, n_roots=2,
                           root_tokens=2048, fan=16, suffix_tokens=37),
    lambda: W.tiny_tree(),
])
def test_noalloc_matches_workspace_entry(make):
    w = make()
    cache = H.Cache(w)
    bt = cache.batch().upload()
    out_ref = torch.empty((bt.nb, w.Hq, w.d), dtype=torch.bfloat16,
                          device="cuda")
    for call in range(2):
        q = torch.from_numpy(w.queries(bt.nb, salt=call).view(np.int16)) \
            .cuda().view(torch.bfloat16)
        bt.decode(q, out_ref)
        out = torch.full_like(out_ref, float("nan"))
        _noalloc(cache, bt, q, out)
        torch.cuda.synchronize()
        assert B.kv_check_noalloc_status() == (0, 0), call
        assert bt.device_status() == (0, 0), call
        a, b = _f64(out), _f64(out_ref)
        assert np.isfinite(a).all()
        assert np.array_equal(out.view(torch.int16).cpu().numpy(),
                              out_ref.view(torch.int16).cpu().numpy()), call
        assert (np.abs(a - b) <= ATOL + RTOL * np.abs(b)).all(), call
    cache.close()


def test_noalloc_reports_a_bad_block_id():
    """A table entry past the pool is recorded in the built-in scratch's
    status word and its access skipped; the reader returns it and clears it."""
    w = W.independent(n_seqs=6, min_len=1, max_len=700)
    cache = H.Cache(w)
    bt = cache.batch().upload()
    bt.dev["tables"][1, 2] = w.num_blocks + 5
    q = torch.zeros((bt.nb, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    _noalloc(cache, bt, q, out)
    assert B.kv_check_noalloc_status() == (B.KV_ERR_DEVICE, w.num_blocks + 5)
    assert B.kv_check_noalloc_status() == (0, 0)      # cleared by the read
    bt.dev["tables"][1, 2] = int(bt.tables[1, 2])
    _noalloc(cache, bt, q, out)
    assert B.kv_check_noalloc_status() == (0, 0)
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
