"""Spill to pinned host memory and restore, on the GPU: bytes round-trip
bit-exactly and decoding after a restore matches the oracle."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import attention as att  # noqa: E402
from oracle import replay as rp  # noqa: E402
from paged_kv_cache_attn_gb300 import binding as B  # noqa: E402
from paged_kv_cache_attn_gb300 import harness as H  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_spill_restore_round_trip():
    w = W.fanout(n_roots=2, root_tokens=256, fan=8, min_suffix=1,
                 max_suffix=100)
    w.num_blocks += 64
    cache = H.Cache(w)
    slots = 256
    shape = (w.num_layers, slots, w.Hkv, w.block_size, w.d)
    hk = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    hv = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    B.kv_offload_attach(cache.h, hk, hv, slots)
    ids = cache.decode_ids
    victims = ids[::2]
    torch.cuda.synchronize()
    before = {i: B.kv_get_block_table(cache.h, i)[0].tolist() for i in victims}
    k0, v0 = _bits(cache.k), _bits(cache.v)
    n = B.kv_spill(cache.h, victims)
    torch.cuda.synchronize()
    assert n > 0
    hkb, hvb = _bits(hk), _bits(hv)
    for i in victims:
        now = B.kv_get_block_table(cache.h, i)[0].tolist()
        for old, code in zip(before[i], now):
            if code < 0:                       # moved: the whole block copied
                slot = -code - 2
                assert np.array_equal(hkb[:, slot], k0[:, old])
                assert np.array_equal(hvb[:, slot], v0[:, old])
            else:
                assert code == old             # shared blocks stay
    # Overwrite the freed device blocks with other data.
    filler = B.kv_branch_create(cache.h)
    free = len(B.kv_get_free_stack(cache.h))
    junk = torch.randn((w.num_layers, free * 16, w.Hkv, w.d), device="cuda") \
        .to(torch.bfloat16)
    B.kv_append(cache.h, filler, free * 16, junk, junk)
    B.kv_free(cache.h, filler)
    B.kv_restore(cache.h, victims)
    torch.cuda.synchronize()
    k1, v1 = _bits(cache.k), _bits(cache.v)
    for i in victims:
        now = B.kv_get_block_table(cache.h, i)[0].tolist()
        for old, new in zip(before[i], now):
            assert new >= 0
            assert np.array_equal(k1[:, new], k0[:, old])
            assert np.array_equal(v1[:, new], v0[:, old])
    # Decoding after the restore still matches the oracle.
    ref = rp.replay(w, with_data=True)
    q = w.queries(len(ids))
    bt = cache.batch().upload()
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty_like(qd)
    bt.decode(qd, out)
    gpu = att.bf16_to_f64(_bits(out))
    want = rp.decode_rows(ref, q, range(len(ids)), w.scale)
    for b in range(len(ids)):
        err = np.abs(gpu[b] - want[b])
        assert (err <= 2e-3 + 1e-2 * np.abs(want[b])).all()
    cache.close()


def test_restore_as_prefetch_beside_decode():
    """Spilled branches come back on a side stream while the step keeps
    decoding the branches still resident (a prefetch: the restore pops device
    blocks that no batch built before it references).  Both the steps that
    run beside the restore and a step over every branch after it match the
    oracle."""
    w = W.fanout(n_roots=2, root_tokens=256, fan=8, min_suffix=1,
                 max_suffix=100)
    w.num_blocks += 64
    cache = H.Cache(w)
    slots = 256
    shape = (w.num_layers, slots, w.Hkv, w.block_size, w.d)
    hk = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    hv = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    B.kv_offload_attach(cache.h, hk, hv, slots)
    ids = cache.decode_ids
    victims, others = ids[::2], ids[1::2]
    assert B.kv_spill(cache.h, victims) > 0
    torch.cuda.synchronize()
    ref = rp.replay(w, with_data=False)
    q = w.queries(len(ids))
    # The resident branches' batch, built before the restore.
    bo = cache.batch(ids=others).upload()
    qo = torch.from_numpy(np.ascontiguousarray(q[1::2]).view(np.int16)).cuda() \
        .view(torch.bfloat16)
    outs = [torch.empty_like(qo) for _ in range(3)]
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    done = torch.cuda.Event()
    with torch.cuda.stream(side):
        assert B.kv_restore(cache.h, victims, stream=side) > 0
        done.record(side)
    for o in outs:                       # on the current stream, beside it
        bo.decode(qo, o)
    torch.cuda.current_stream().wait_event(done)
    want = rp.decode_rows(ref, q, range(len(ids)), w.scale)
    for o in outs:
        gpu = att.bf16_to_f64(_bits(o))
        for k in range(len(others)):
            err = np.abs(gpu[k] - want[2 * k + 1])
            assert (err <= 2e-3 + 1e-2 * np.abs(want[2 * k + 1])).all()
    # Every branch, restored ones included, after the restore.
    bt = cache.batch().upload()
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty_like(qd)
    bt.decode(qd, out)
    gpu = att.bf16_to_f64(_bits(out))
    for b in range(len(ids)):
        err = np.abs(gpu[b] - want[b])
        assert (err <= 2e-3 + 1e-2 * np.abs(want[b])).all()
    cache.close()
