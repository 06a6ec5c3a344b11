"""Pools with several layers: every layer's K/V land in their own slots
through appends and copy-on-write forks, and the decode step of each layer
reads only that layer (bf16 and e4m3)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import attention as att  # noqa: E402
from oracle import replay as rp  # noqa: E402
from paged_kv_cache_attn_gb300 import harness as H  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2
LAYERS = 3


def workload(name):
    w = {"tiny_tree": lambda: W.tiny_tree(),
         "deep_tree": lambda: W.deep_tree(root_tokens=300, depth=3, min_seg=5,
                                          max_seg=40),
         "long_context": lambda: W.long_context(n_indep=3, indep_tokens=1000,
                                                n_roots=2, root_tokens=2048,
                                                fan=16, suffix_tokens=37)}[name]()
    w.num_layers = LAYERS
    return w


def bits_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda() \
        .view(torch.bfloat16)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("name", ["tiny_tree", "deep_tree", "long_context"])
def test_every_layer_decodes_its_own_kv(name, kv_dtype):
    w = workload(name)
    cache = H.Cache(w, kv_dtype=kv_dtype)
    ref = rp.replay(w, with_data=True, kv_dtype=kv_dtype)
    assert cache.decode_ids == ref.decode_ids
    nb = len(cache.decode_ids)
    bt = cache.batch().upload()
    outs = []
    for layer in range(LAYERS):
        q = w.queries(nb, salt=layer)
        out = torch.empty((nb, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
        bt.decode(bits_to_dev(q), out, layer=layer)
        torch.cuda.synchronize()
        assert bt.device_status() == (0, 0)
        gpu = att.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        want = rp.decode_all_from_pool(ref, q, w.scale, layer=layer)
        err = np.abs(gpu - want)
        assert (err <= ATOL + RTOL * np.abs(want)).all(), (layer, err.max())
        outs.append(gpu)
    # the layers hold different data, so their outputs differ
    assert not np.allclose(outs[0], outs[1])
    cache.close()


def test_bf16_pool_bytes_of_every_layer():
    w = workload("deep_tree")
    cache = H.Cache(w)
    ref = rp.replay(w, with_data=True)
    torch.cuda.synchronize()
    k = cache.k.view(torch.int16).cpu().numpy().view(np.uint16)
    v = cache.v.view(torch.int16).cpu().numpy().view(np.uint16)
    for n in ref.model.nodes:
        if not n.live or n.seq_len == 0:
            continue
        t = np.arange(n.seq_len)
        blk = np.asarray(n.table)[t // 16]
        for layer in range(LAYERS):
            assert np.array_equal(k[layer][blk, :, t % 16],
                                  ref.data.k[layer][blk, :, t % 16])
            assert np.array_equal(v[layer][blk, :, t % 16],
                                  ref.data.v[layer][blk, :, t % 16])
    cache.close()
