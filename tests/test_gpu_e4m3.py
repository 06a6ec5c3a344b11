"""e4m3 pools through the C ABI against the oracle's FP8 model.

* Pool contents (codes and per-tile scales) after appends, batched appends,
  copy-on-write forks, the decode step's own append, spill and restore:
  bit-exact against the oracle, reading the device tiles through the byte
  layouts pagedkv.h declares.
* Decode output: element-wise |gpu - oracle| <= 2e-3 + 1e-2 |oracle|, the
  oracle attending in fp64 over the dequantised values.  The bound is the
  bf16 path's: the kernel widens codes to f16 exactly, carries q in f16 after
  a power-of-two row scaling (11-bit significands, finer than bf16's 8) and
  P in f16, and accumulates in fp32.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import attention as att  # noqa: E402
from oracle import fp8  # noqa: E402
from oracle import replay as rp  # noqa: E402
from oracle.allocator import PoolModel  # noqa: E402
from paged_kv_cache_attn_gb300 import binding as B  # noqa: E402
from paged_kv_cache_attn_gb300 import harness as H  # noqa: E402
from paged_kv_cache_attn_gb300 import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2

SMALL = {
    "tiny_tree": lambda: W.tiny_tree(),
    "tiny_tree_peaked": lambda: W.tiny_tree(q_gain=4.0),
    "independent": lambda: W.independent(n_seqs=6, min_len=1, max_len=700),
    "fanout": lambda: W.fanout(n_roots=2, root_tokens=256, fan=8,
                               min_suffix=1, max_suffix=100),
    "deep_tree": lambda: W.deep_tree(root_tokens=300, depth=3, min_seg=5,
                                     max_seg=40),
    "long_context": lambda: W.long_context(n_indep=3, indep_tokens=1000,
                                           n_roots=2, root_tokens=2048,
                                           fan=16, suffix_tokens=37),
    "fanout_3tiles": lambda: W.fanout(n_roots=1, root_tokens=512, fan=40,
                                      min_suffix=1, max_suffix=50, Hq=64,
                                      Hkv=8),
    "gqa_2": lambda: W.independent(n_seqs=3, min_len=17, max_len=300, Hq=8,
                                   Hkv=4, d=64),
    "gqa_16": lambda: W.fanout(n_roots=1, root_tokens=64, fan=3,
                               min_suffix=1, max_suffix=30, Hq=32, Hkv=2),
}


# ---- the tile byte layouts of pagedkv.h, restated -----------------------------

def k_offsets(d):
    t = np.arange(16)[:, None]
    c = np.arange(d)[None, :]
    if d == 128:
        return t * 128 + (((c >> 4) ^ (t & 7)) << 4) + (c & 15)
    return t * d + c


def v_offsets(d):
    t = np.arange(16)[:, None]
    c = np.arange(d)[None, :]
    return c * 16 + t


def logical_codes(raw, d, kind):
    """[..., 16 * d] device tile bytes -> [..., 16, d] codes by (slot, dim)."""
    off = k_offsets(d) if kind == "k" else v_offsets(d)
    return raw[..., off]


def device_state(cache):
    torch.cuda.synchronize()
    d = cache.w.d
    k = logical_codes(cache.k.cpu().numpy(), d, "k")
    v = logical_codes(cache.v.cpu().numpy(), d, "v")
    s = cache.scales.cpu().numpy()
    return k, v, s


def check_live_blocks(cache, ref, what):
    """Codes of every valid slot and the scales of every block in a live
    table equal the oracle's replay."""
    k, v, s = device_state(cache)
    m = ref.model
    for i, n in enumerate(m.nodes):
        if not n.live or n.seq_len == 0:
            continue
        t = np.arange(n.seq_len)
        blk = np.asarray(n.table)[t // 16]
        slot = t % 16
        assert np.array_equal(k[:, blk, :, slot], ref.data.k[:, blk, :, slot]), \
            f"{what}: K codes of branch {i}"
        assert np.array_equal(v[:, blk, :, slot], ref.data.v[:, blk, :, slot]), \
            f"{what}: V codes of branch {i}"
        ub = np.unique(blk)
        assert np.array_equal(s[..., 0][:, ub], np.exp2(ref.data.ek[:, ub])), \
            f"{what}: K scales of branch {i}"
        assert np.array_equal(s[..., 1][:, ub], np.exp2(ref.data.ev[:, ub])), \
            f"{what}: V scales of branch {i}"


def assert_close(gpu, ref, what=""):
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside "
                           f"tolerance; max abs err {err.max():.3g}")


def bits_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda() \
        .view(torch.bfloat16)


def bf16_out(t):
    return att.bf16_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


def run_decode(cache, q_bits, flags=0):
    bt = cache.batch(flags=flags).upload()
    q = bits_to_dev(q_bits)
    out = torch.empty_like(q)
    bt.decode(q, out)
    torch.cuda.synchronize()
    assert bt.device_status() == (0, 0)
    return bf16_out(out), bt


# ---- tests ---------------------------------------------------------------------

def deep_tree_3_layers():
    w = SMALL["deep_tree"]()
    w.num_layers = 3
    return w


@pytest.mark.parametrize("name", ["tiny_tree", "deep_tree", "fanout", "gqa_2",
                                  "deep_tree_3_layers"])
def test_e4m3_pool_bit_exact(name):
    w = deep_tree_3_layers() if name == "deep_tree_3_layers" else SMALL[name]()
    cache = H.Cache(w, kv_dtype="e4m3")
    ref = rp.replay(w, with_data=True, kv_dtype="e4m3")
    assert cache.tables() == {i: (n.table, n.seq_len)
                              for i, n in enumerate(ref.model.nodes) if n.live}
    check_live_blocks(cache, ref, name)
    cache.close()


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("flags", [0, B.KV_PLAN_IGNORE_GROUPS,
                                   B.KV_PLAN_NO_TENSOR_CORES])
def test_e4m3_decode_matches_oracle(name, flags):
    """Segments of more than 64 rows (head_dim 128) run on the tcgen05 e4m3
    tile kernel unless the plan says otherwise; the rest on the split-KV
    kernel."""
    w = SMALL[name]()
    cache = H.Cache(w, kv_dtype="e4m3")
    ref = rp.replay(w, with_data=True, kv_dtype="e4m3")
    assert cache.decode_ids == ref.decode_ids
    q = w.queries(len(cache.decode_ids))
    gpu, bt = run_decode(cache, q, flags)
    assert bt.info.flags & B.KV_PLAN_KV_E4M3
    if flags or w.d != 128:
        assert bt.info.n_tile_items == 0
    assert_close(gpu, rp.decode_all_from_pool(ref, q, w.scale), name)
    cache.close()


def test_e4m3_poisoned_slots_do_not_leak():
    """Free and unwritten slots hold NaN codes and NaN scales."""
    w = SMALL["long_context"]()
    cache = H.Cache(w, kv_dtype="e4m3", poison=True)
    ref = rp.replay(w, with_data=True, kv_dtype="e4m3")
    q = w.queries(len(cache.decode_ids))
    gpu, _ = run_decode(cache, q)
    assert np.isfinite(gpu).all()
    assert_close(gpu, rp.decode_all_from_pool(ref, q, w.scale), "poisoned")
    cache.close()


def test_e4m3_scale_growth_and_batch_order():
    """Writes into one block that need ever larger scales re-encode the rows
    already stored; two writes to one block in a batch apply in order."""
    d, Hkv, nblocks = 128, 2, 8
    rng = np.random.default_rng(11)

    def rows(n, gain):
        return W.f32_to_bf16_bits(
            (rng.standard_normal((1, n, Hkv, d)) * gain).astype(np.float32))

    w = W.Workload(name="growth", Hq=2 * Hkv, Hkv=Hkv, d=d, seed=0,
                   num_blocks=nblocks)
    w.initial_free_order = lambda: np.arange(nblocks, dtype=np.int32)
    cache = H.Cache(w, kv_dtype="e4m3", poison=True, replay=False)
    model = PoolModel(nblocks, 16, np.arange(nblocks, dtype=np.int32))
    data = fp8.Fp8PoolData(1, nblocks, Hkv, 16, d)
    b = B.kv_branch_create(cache.h)
    assert model.create() == b
    a = rows(5, 2.0 ** -6)
    B.kv_append(cache.h, b, 5, bits_to_dev(a), bits_to_dev(a))
    data.write(model.append(b, 5), a, a)
    # one batch holding the branch twice: (3 rows, gain 1) then (2, 2^5)
    k1, k2 = rows(3, 1.0), rows(2, 2.0 ** 5)
    v1, v2 = rows(3, 2.0 ** 4), rows(2, 2.0 ** -2)
    B.kv_append_batch(cache.h, [b, b], [3, 2],
                      bits_to_dev(np.concatenate([k1, k2], axis=1)),
                      bits_to_dev(np.concatenate([v1, v2], axis=1)))
    data.write(model.append(b, 3), k1, v1)
    data.write(model.append(b, 2), k2, v2)
    # a single small row, then 20 rows crossing into the next block
    k3, v3 = rows(1, 2.0 ** -3), rows(1, 2.0 ** 6)
    B.kv_append(cache.h, b, 1, bits_to_dev(k3), bits_to_dev(v3))
    data.write(model.append(b, 1), k3, v3)
    k4, v4 = rows(20, 3.0), rows(20, 0.5)
    B.kv_append(cache.h, b, 20, bits_to_dev(k4), bits_to_dev(v4))
    data.write(model.append(b, 20), k4, v4)

    class Ref:
        pass
    ref = Ref()
    ref.model, ref.data = model, data
    check_live_blocks(cache, ref, "growth")
    # the first block's scale did grow past its first write's
    assert data.ek[0, 0, 0] > fp8.exponent_for(
        np.abs(att.bf16_to_f64(a[0, :, 0])).max())
    cache.close()


@pytest.mark.parametrize("name", ["long_context", "deep_tree", "tiny_tree"])
def test_e4m3_decode_append(name):
    """The newest token is quantised into its reserved slot (re-encoding its
    block if needed) and attended to, in one call; a later plain step reads
    the same values."""
    w = SMALL[name]()
    cache = H.Cache(w, kv_dtype="e4m3")
    ref = rp.replay(w, with_data=False)
    ids = cache.decode_ids
    nb = len(ids)
    B.kv_reserve(cache.h, ids, [1] * nb)
    rng = np.random.default_rng(9)
    ks = W.f32_to_bf16_bits(
        (rng.standard_normal((nb, w.Hkv, w.d)) * 4).astype(np.float32))
    vs = W.f32_to_bf16_bits(
        (rng.standard_normal((nb, w.Hkv, w.d)) * 4).astype(np.float32))
    q = w.queries(nb, salt=5)
    bt = cache.batch().upload()
    out = torch.empty((nb, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    bt.decode_append(bits_to_dev(q), bits_to_dev(ks), bits_to_dev(vs), out)
    torch.cuda.synchronize()
    assert bt.device_status() == (0, 0)
    gpu = bf16_out(out)
    kd, vd, sd = device_state(cache)
    for b in range(nb):
        kb, vb = ref.branch_kv(ids[b])
        kb = np.concatenate([kb, ks[b][None, None]], axis=1)
        vb = np.concatenate([vb, vs[b][None, None]], axis=1)
        lens = [hi - lo for _s, lo, hi in ref.logical[ids[b]]] + [1]
        kq = fp8.quantize_sequence(lens, kb)[0]
        vq = fp8.quantize_sequence(lens, vb)[0]
        G = w.Hq // w.Hkv
        want = np.empty((w.Hq, w.d))
        for g in range(w.Hkv):
            qr = att.bf16_to_f64(q[b, g * G:(g + 1) * G])
            want[g * G:(g + 1) * G] = att.attention(qr, kq[:, g], vq[:, g],
                                                    w.scale)
        assert_close(gpu[b], want, f"{name} row {b}")
        # the last block's stored values (codes x scale) equal the oracle's
        L = int(bt.seq_lens[b])
        lb = (L - 1) // 16
        blk = int(bt.tables[b][lb])
        n_in = L - 16 * lb
        got_k = fp8.decode(kd[0, blk, :, :n_in]) * sd[0, blk, :, 0][:, None, None]
        got_v = fp8.decode(vd[0, blk, :, :n_in]) * sd[0, blk, :, 1][:, None, None]
        assert np.array_equal(got_k, kq[16 * lb:L].transpose(1, 0, 2))
        assert np.array_equal(got_v, vq[16 * lb:L].transpose(1, 0, 2))
    q2 = w.queries(nb, salt=6)
    out2 = torch.empty_like(out)
    bt.decode(bits_to_dev(q2), out2)
    torch.cuda.synchronize()
    gpu2 = bf16_out(out2)
    for b in range(min(nb, 4)):
        kb, vb = ref.branch_kv(ids[b])
        kb = np.concatenate([kb, ks[b][None, None]], axis=1)
        vb = np.concatenate([vb, vs[b][None, None]], axis=1)
        lens = [hi - lo for _s, lo, hi in ref.logical[ids[b]]] + [1]
        kq = fp8.quantize_sequence(lens, kb)[0]
        vq = fp8.quantize_sequence(lens, vb)[0]
        G = w.Hq // w.Hkv
        for g in range(w.Hkv):
            qr = att.bf16_to_f64(q2[b, g * G:(g + 1) * G])
            assert_close(gpu2[b, g * G:(g + 1) * G],
                         att.attention(qr, kq[:, g], vq[:, g], w.scale),
                         f"{name} later row {b}")
    cache.close()


def test_e4m3_spill_restore_round_trip():
    w = W.fanout(n_roots=2, root_tokens=256, fan=8, min_suffix=1,
                 max_suffix=100)
    w.num_blocks += 64
    cache = H.Cache(w, kv_dtype="e4m3")
    slots = 256
    hk = torch.empty((w.num_layers, slots, w.Hkv, 16 * w.d),
                     dtype=torch.uint8).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    hs = torch.empty((w.num_layers, slots, w.Hkv, 4),
                     dtype=torch.float32).pin_memory()
    B.kv_offload_attach(cache.h, hk, hv, slots, hs)
    ids = cache.decode_ids
    victims = ids[::2]
    torch.cuda.synchronize()
    before = {i: B.kv_get_block_table(cache.h, i)[0].tolist() for i in victims}
    k0, v0, s0 = cache.k.cpu().numpy(), cache.v.cpu().numpy(), \
        cache.scales.cpu().numpy()
    assert B.kv_spill(cache.h, victims) > 0
    torch.cuda.synchronize()
    hkb, hvb, hsb = hk.numpy(), hv.numpy(), hs.numpy()
    moved = 0
    for i in victims:
        now = B.kv_get_block_table(cache.h, i)[0].tolist()
        for old, code in zip(before[i], now):
            if code < 0:
                slot = -code - 2
                assert np.array_equal(hkb[:, slot], k0[:, old])
                assert np.array_equal(hvb[:, slot], v0[:, old])
                assert np.array_equal(hsb[:, slot, :, :2], s0[:, old, :, :2])
                moved += 1
    assert moved > 0
    free = B.kv_get_free_stack(cache.h)
    for blk in free:                     # freed device blocks hold garbage
        cache.k[:, blk] = 0x7F
        cache.v[:, blk] = 0x7F
        cache.scales[:, blk] = float("nan")
    B.kv_restore(cache.h, victims)
    torch.cuda.synchronize()
    ref = rp.replay(w, with_data=True, kv_dtype="e4m3")
    q = w.queries(len(cache.decode_ids))
    gpu, _ = run_decode(cache, q)
    assert_close(gpu, rp.decode_all_from_pool(ref, q, w.scale), "restored")
    cache.close()


@pytest.mark.parametrize("name", ["independent", "fanout", "deep_tree",
                                  "long_context"])
def test_e4m3_full_size_every_row(name):
    """The benchmarked workloads over e4m3 pools at full size: every output
    element against the oracle quantising each branch from its own token
    sequence (in worker processes spawned after the GPU step)."""
    import _oracle_pool
    w = W.CONFIGS[name]()
    cache = H.Cache(w, kv_dtype="e4m3")
    assert cache.decode_ids == _oracle_pool.decode_ids(name)
    nb = len(cache.decode_ids)
    q = w.queries(nb)
    gpu, bt = run_decode(cache, q)
    cache.close()
    want = _oracle_pool.all_rows(name, q, "e4m3")
    assert_close(gpu, want, f"{name} e4m3 ({nb} branches, every row)")


def test_e4m3_stale_shared_memory_does_not_leak():
    """Shared memory left behind by an earlier kernel must not reach the
    output.  A step over a pool whose every byte is 0xC0 (each 32-bit word
    reads as -6.02) runs on every SM first; then a step whose segment tiles
    end part-way through (deep_tree: ranges that are not a multiple of 8
    blocks) must still match the oracle."""
    junk_w = W.independent(n_seqs=64, min_len=1500, max_len=2500)
    junk = H.Cache(junk_w, kv_dtype="e4m3")
    junk.k.fill_(0xC0)
    junk.v.fill_(0xC0)
    junk.scales.view(torch.uint8).fill_(0xC0)
    jq = junk_w.queries(len(junk.decode_ids))
    jb = junk.batch().upload()
    jout = torch.empty((len(junk.decode_ids), junk_w.Hq, junk_w.d),
                       dtype=torch.bfloat16, device="cuda")
    w = SMALL["deep_tree"]()
    cache = H.Cache(w, kv_dtype="e4m3")
    ref = rp.replay(w, with_data=True, kv_dtype="e4m3")
    q = w.queries(len(cache.decode_ids))
    bt = cache.batch().upload()
    assert bt.info.n_tile_items > 0
    out = torch.empty((len(cache.decode_ids), w.Hq, w.d), dtype=torch.bfloat16,
                      device="cuda")
    want = rp.decode_all_from_pool(ref, q, w.scale)
    for _ in range(3):
        jb.decode(bits_to_dev(jq), jout)
        bt.decode(bits_to_dev(q), out)
        torch.cuda.synchronize()
        gpu = bf16_out(out)
        assert np.isfinite(gpu).all()
        assert_close(gpu, want, "after a junk step")
    junk.close()
    cache.close()
