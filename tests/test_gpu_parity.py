"""CUDA path vs the fp64 oracle, through the C ABI.

Tolerance (the bound stated for this path: bf16 inputs, fp32 accumulation):
element-wise |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|.
Allocator state and pool bytes: bit-exact.
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


def bf16_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_decode(cache, q_bits, flags=0):
    bt = cache.batch(flags=flags).upload()
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty_like(q)
    bt.decode(q, out)
    torch.cuda.synchronize()
    code, detail = bt.device_status()
    assert code == 0, (code, detail)
    return att.bf16_to_f64(bf16_bits(out)), bt


def assert_close(gpu, ref, what=""):
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside "
                           f"tolerance; max abs err {err.max():.3g}")


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
    "fanout_256": lambda: W.fanout(n_roots=2, root_tokens=777, fan=64,
                                   min_suffix=1, max_suffix=90),
    "wide_tree": lambda: W.deep_tree(root_tokens=300, depth=3, branching=5,
                                     min_seg=20, max_seg=50),
    "gqa_2": lambda: W.independent(n_seqs=3, min_len=17, max_len=300, Hq=8,
                                   Hkv=4, d=64),
    "gqa_16": lambda: W.fanout(n_roots=1, root_tokens=64, fan=3,
                               min_suffix=1, max_suffix=30, Hq=32, Hkv=2),
}


@pytest.fixture(scope="module")
def built():
    assert torch.cuda.is_available()
    return True


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("flags", [0, B.KV_PLAN_IGNORE_GROUPS,
                                   B.KV_PLAN_NO_TENSOR_CORES,
                                   B.KV_PLAN_NARROW_TILES])
def test_decode_matches_oracle(built, name, flags):
    w = SMALL[name]()
    cache = H.Cache(w)
    ref = rp.replay(w, with_data=True)
    assert cache.decode_ids == ref.decode_ids
    q = w.queries(len(cache.decode_ids))
    gpu, _ = run_decode(cache, q, flags)
    want = rp.decode_all_from_pool(ref, q, w.scale)
    assert_close(gpu, want, name)


@pytest.mark.parametrize("name", ["tiny_tree", "deep_tree", "fanout"])
def test_pool_bytes_bit_exact(built, name):
    """Appends and copy-on-write copies put every valid token's K/V rows in
    the slot the oracle's own replay puts them."""
    w = SMALL[name]()
    cache = H.Cache(w)
    ref = rp.replay(w, with_data=True)
    torch.cuda.synchronize()
    k = bf16_bits(cache.k)
    v = bf16_bits(cache.v)
    assert cache.tables() == {i: (n.table, n.seq_len)
                              for i, n in enumerate(ref.model.nodes) if n.live}
    for i, n in enumerate(ref.model.nodes):
        if not n.live:
            continue
        t = np.arange(n.seq_len)
        blk = np.asarray(n.table)[t // 16]
        slot = t % 16
        assert np.array_equal(k[:, blk, :, slot], ref.data.k[:, blk, :, slot])
        assert np.array_equal(v[:, blk, :, slot], ref.data.v[:, blk, :, slot])


def test_poisoned_free_slots_do_not_leak(built):
    """Slots past a branch's length hold NaN: the output must not see them."""
    w = SMALL["long_context"]()
    cache = H.Cache(w, poison=True)
    ref = rp.replay(w, with_data=True)
    q = w.queries(len(cache.decode_ids))
    gpu, _ = run_decode(cache, q)
    assert np.isfinite(gpu).all()
    assert_close(gpu, rp.decode_all_from_pool(ref, q, w.scale), "poisoned")


def test_physical_layout_does_not_change_the_output(built):
    w1 = SMALL["fanout"]()
    w2 = SMALL["fanout"]()
    w2.initial_free_order = lambda: np.arange(w2.num_blocks, dtype=np.int32)
    q = w1.queries(len(w1.leaves()))
    a, _ = run_decode(H.Cache(w1), q)
    b, _ = run_decode(H.Cache(w2), q)
    assert np.array_equal(a, b)


def test_bad_block_id_is_reported(built):
    w = SMALL["independent"]()
    cache = H.Cache(w)
    bt = cache.batch().upload()
    bt.dev["tables"][1, 2] = w.num_blocks + 5
    q = torch.zeros((bt.nb, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    bt.decode(q, out)
    code, detail = bt.device_status()
    assert code == B.KV_ERR_DEVICE and detail == w.num_blocks + 5
    # The status word is cleared by the read; a clean step reports 0.
    bt.dev["tables"][1, 2] = int(bt.tables[1, 2])
    bt.decode(q, out)
    assert bt.device_status() == (0, 0)


# ---- full sizes: every row against the oracle --------------------------------

FULL = ["independent", "fanout", "deep_tree", "long_context"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(built, name):
    """The benchmarked workloads at their full sizes, in the launch
    configuration the benchmark times: every output element of every branch
    against the oracle run on that branch's logical token sequence (in worker
    processes spawned after the GPU step)."""
    import _oracle_pool
    w = W.CONFIGS[name]()
    cache = H.Cache(w)
    assert cache.decode_ids == _oracle_pool.decode_ids(name)
    nb = len(cache.decode_ids)
    q = w.queries(nb)
    gpu, bt = run_decode(cache, q)
    cache.close()
    want = _oracle_pool.all_rows(name, q, "bf16")
    assert_close(gpu, want, f"{name} ({nb} branches, every row)")


# ---- batched append and the fused append + decode step -----------------------

def _bits_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda() \
        .view(torch.bfloat16)


def test_batched_append_pool_bytes(built):
    """Children's first segments appended in one kv_append_batch land where
    the oracle's sequential appends put them."""
    w = SMALL["fanout"]()
    cache = H.Cache(w, replay=False)
    pending = []                        # consecutive appends -> one batch

    def flush():
        if not pending:
            return
        ks, vs = zip(*[w.node_kv(i) for i in pending])
        k = np.concatenate(ks, axis=1)
        v = np.concatenate(vs, axis=1)
        B.kv_append_batch(cache.h, pending,
                          [w.nodes[i].n_tokens for i in pending],
                          _bits_to_dev(k), _bits_to_dev(v))
        pending.clear()

    for op in w.ops:
        if op[0] == "append":
            pending.append(op[1])
            continue
        flush()
        if op[0] == "create":
            B.kv_branch_create(cache.h)
        else:
            B.kv_fork_branches(cache.h, op[1], op[2])
    flush()
    torch.cuda.synchronize()
    ref = rp.replay(w, with_data=True)
    k = bf16_bits(cache.k)
    v = bf16_bits(cache.v)
    for i, n in enumerate(ref.model.nodes):
        t = np.arange(n.seq_len)
        blk = np.asarray(n.table)[t // 16]
        assert np.array_equal(k[:, blk, :, t % 16], ref.data.k[:, blk, :, t % 16])
        assert np.array_equal(v[:, blk, :, t % 16], ref.data.v[:, blk, :, t % 16])
    cache.close()


@pytest.mark.parametrize("name", ["long_context", "deep_tree", "tiny_tree",
                                  "fanout_3tiles"])
def test_fused_append_decode(built, name):
    """Each branch's newest token is reserved, then written and attended to in
    one step; the result matches the oracle over the sequence with the token
    appended, the slot holds the token, and a later plain step sees it."""
    w = SMALL[name]()
    cache = H.Cache(w)
    ref = rp.replay(w, with_data=False)
    ids = cache.decode_ids
    nb = len(ids)
    B.kv_reserve(cache.h, ids, [1] * nb)
    rng = np.random.default_rng(9)
    ks = W.f32_to_bf16_bits(rng.standard_normal((nb, w.Hkv, w.d), dtype=np.float32))
    vs = W.f32_to_bf16_bits(rng.standard_normal((nb, w.Hkv, w.d), dtype=np.float32))
    q = w.queries(nb, salt=5)
    bt = cache.batch().upload()
    out = torch.empty((nb, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    bt.decode_append(_bits_to_dev(q), _bits_to_dev(ks), _bits_to_dev(vs), out)
    torch.cuda.synchronize()
    assert bt.device_status() == (0, 0)
    gpu = att.bf16_to_f64(bf16_bits(out))
    for b in range(nb):
        k, v = ref.branch_kv(ids[b])
        k = np.concatenate([k[0], ks[b][None]], axis=0)
        v = np.concatenate([v[0], vs[b][None]], axis=0)
        want = att.decode_branch_contiguous(q[b], k, v, w.Hkv, w.scale)
        assert_close(gpu[b], want, f"{name} fused row {b}")
    # The slot now holds the token.
    kp, vp = bf16_bits(cache.k), bf16_bits(cache.v)
    for b in range(nb):
        L = int(bt.seq_lens[b])
        blk = int(bt.tables[b][(L - 1) // 16])
        assert np.array_equal(kp[0, blk, :, (L - 1) % 16], ks[b])
        assert np.array_equal(vp[0, blk, :, (L - 1) % 16], vs[b])
    # A plain step afterwards reads it from the pool.
    q2 = w.queries(nb, salt=6)
    out2 = torch.empty_like(out)
    bt.decode(_bits_to_dev(q2), out2)
    gpu2 = att.bf16_to_f64(bf16_bits(out2))
    for b in range(min(nb, 6)):
        k, v = ref.branch_kv(ids[b])
        k = np.concatenate([k[0], ks[b][None]], axis=0)
        v = np.concatenate([v[0], vs[b][None]], axis=0)
        want = att.decode_branch_contiguous(q2[b], k, v, w.Hkv, w.scale)
        assert_close(gpu2[b], want, f"{name} later row {b}")
    cache.close()
