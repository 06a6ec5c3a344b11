"""Head-grouping extremes and a very long branch, in both element types:

* multi-query attention (one kv-head for all q-heads, G = 8) and plain
  multi-head attention (G = 1, so a 128-row tensor-core tile carries 128
  different branches);
* one branch of 2^19 tokens (32,768 blocks: long block-table windows, many
  split items merged), checked on every q-head against the oracle reading
  the branch's logical token sequence.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import attention as att  # noqa: E402
from oracle import fp8  # noqa: E402
from oracle import replay as rp  # noqa: E402
from paged_kv_cache_attn_gb300 import harness as H  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def close(gpu, want, what):
    err = np.abs(gpu - want)
    bad = err > ATOL + RTOL * np.abs(want)
    assert not bad.any(), f"{what}: {bad.sum()} outside, max err {err.max():.3g}"


def decode(cache, q):
    bt = cache.batch().upload()
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty_like(qd)
    bt.decode(qd, out)
    torch.cuda.synchronize()
    assert bt.device_status() == (0, 0)
    return att.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16)), bt


SHAPES = {
    # 2 roots x 64 branches; G = 8 with a single kv-head
    "mqa": lambda: W.fanout(n_roots=2, root_tokens=300, fan=64, min_suffix=1,
                            max_suffix=60, Hq=8, Hkv=1),
    # G = 1: 128 branches of one root -> one full 128-row tile per kv-head
    "mha": lambda: W.fanout(n_roots=1, root_tokens=520, fan=128, min_suffix=1,
                            max_suffix=40, Hq=8, Hkv=8),
}


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("name", list(SHAPES))
def test_head_grouping_extremes(name, kv_dtype):
    w = SHAPES[name]()
    cache = H.Cache(w, kv_dtype=kv_dtype)
    ref = rp.replay(w, with_data=True, kv_dtype=kv_dtype)
    q = w.queries(len(cache.decode_ids))
    gpu, bt = decode(cache, q)
    if name == "mha":
        assert bt.info.n_tile_items > 0       # 128 rows of 128 branches
    close(gpu, rp.decode_all_from_pool(ref, q, w.scale), f"{name} {kv_dtype}")
    cache.close()


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_one_very_long_branch(kv_dtype):
    w = W.independent(n_seqs=1, min_len=1 << 19, max_len=1 << 19, Hq=16,
                      Hkv=2)
    cache = H.Cache(w, kv_dtype=kv_dtype)
    ref = rp.replay(w, with_data=False)
    q = w.queries(1)
    gpu, bt = decode(cache, q)
    assert bt.info.n_row_items >= 2 * 16    # many chunks merged per head
    k, v = ref.branch_kv(cache.decode_ids[0])
    if kv_dtype == "e4m3":
        lens = [hi - lo for _s, lo, hi in ref.logical[cache.decode_ids[0]]]
        kq = fp8.quantize_sequence(lens, k)[0]
        vq = fp8.quantize_sequence(lens, v)[0]
        G = w.Hq // w.Hkv
        want = np.empty((w.Hq, w.d))
        for g in range(w.Hkv):
            qr = att.bf16_to_f64(q[0, g * G:(g + 1) * G])
            want[g * G:(g + 1) * G] = att.attention(qr, kq[:, g], vq[:, g],
                                                    w.scale)
    else:
        want = att.decode_branch_contiguous(q[0], k[0], v[0], w.Hkv, w.scale)
    close(gpu[0], want, f"2^19 tokens {kv_dtype}")
    cache.close()
