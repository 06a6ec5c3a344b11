"""Pins for the oracle's attention: closed forms, invariants, brute force.

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (a dropped max subtraction that overflows, a missing
normalisation, a wrong scale, a transposed operand, a wrong GQA head, a wrong
block/slot translation) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import attention as att
from oracle import brute
from oracle import replay as rp
from paged_kv_cache_attn_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "pages_worked_examples.json")


def bf16(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_bf16_decode_exact():
    # 1.0 = 0x3F80, -2.0 = 0xC000, 0.15625 = 0x3E20, smallest normal 2^-126.
    bits = np.array([0x3F80, 0xC000, 0x3E20, 0x0080], dtype=np.uint16)
    assert list(att.bf16_to_f64(bits)) == [1.0, -2.0, 0.15625, 2.0 ** -126]


def test_single_token_returns_its_value():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((3, 8))
    K = rng.standard_normal((1, 8)) * 50.0
    V = rng.standard_normal((1, 5))
    out = att.attention(q, K, V, 0.3)
    assert np.array_equal(out, np.repeat(V, 3, axis=0))


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 16))
    K = np.repeat(rng.standard_normal((1, 16)), 37, axis=0)
    V = rng.standard_normal((37, 16))
    out = att.attention(q, K, V, 1.0 / 4.0)
    assert np.allclose(out, np.repeat(V.mean(axis=0, keepdims=True), 2, 0),
                       rtol=0, atol=1e-13)


def test_two_tokens_follow_the_logistic_function():
    # Two keys: weight of token 1 = 1 / (1 + exp(-(s1 - s0))), the logistic
    # function; with q=[1,0], k0=[0,0], k1=[2,0], scale 0.5: s1 - s0 = 1.
    q = np.array([[1.0, 0.0]])
    K = np.array([[0.0, 0.0], [2.0, 0.0]])
    V = np.array([[1.0, 0.0], [0.0, 1.0]])
    w1 = 1.0 / (1.0 + math.exp(-1.0))
    out = att.attention(q, K, V, 0.5)
    assert out[0, 0] == pytest.approx(1.0 - w1, abs=1e-15)
    assert out[0, 1] == pytest.approx(w1, abs=1e-15)
    # The scale matters: scale 1.0 doubles the logit gap.
    w1b = 1.0 / (1.0 + math.exp(-2.0))
    assert att.attention(q, K, V, 1.0)[0, 1] == pytest.approx(w1b, abs=1e-15)


def test_dominant_key_returns_its_value_within_bound():
    rng = np.random.default_rng(2)
    d, L, j = 64, 50, 17
    q = rng.standard_normal((1, d))
    K = rng.standard_normal((L, d)) * 0.1
    K[j] = 8.0 * q[0] / np.linalg.norm(q[0]) * math.sqrt(d)
    V = rng.standard_normal((L, d))
    scale = 1.0 / math.sqrt(d)
    s = (q @ K.T)[0] * scale
    gap = s[j] - np.max(np.delete(s, j))
    assert gap > 20
    out = att.attention(q, K, V, scale)[0]
    bound = (L - 1) * math.exp(-gap) * np.max(np.abs(V - V[j]))
    assert np.max(np.abs(out - V[j])) <= bound + 1e-15


def test_huge_scores_do_not_overflow():
    # Scores near 1e4: exp() without the max subtraction would overflow.
    q = np.array([[100.0]])
    K = np.array([[100.0], [99.0]])
    V = np.array([[1.0], [0.0]])
    out = att.attention(q, K, V, 1.0)
    w0 = 1.0 / (1.0 + math.exp(-100.0))
    assert np.isfinite(out).all() and out[0, 0] == pytest.approx(w0, abs=1e-15)


def test_key_order_does_not_matter():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 32))
    K = rng.standard_normal((29, 32))
    V = rng.standard_normal((29, 32))
    perm = rng.permutation(29)
    a = att.attention(q, K, V, 0.2)
    b = att.attention(q, K[perm], V[perm], 0.2)
    assert np.allclose(a, b, rtol=0, atol=1e-13)


def test_score_shift_and_value_affinity():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 16))
    K = rng.standard_normal((20, 16))
    V = rng.standard_normal((20, 16))
    base = att.attention(q, K, V, 0.25)
    # Adding the same vector u to every key shifts every score by q.u.
    u = rng.standard_normal((1, 16))
    assert np.allclose(att.attention(q, K + u, V, 0.25), base, atol=1e-13)
    # Weights sum to one: adding c to every value adds c to the output.
    assert np.allclose(att.attention(q, K, V + 3.5, 0.25), base + 3.5,
                       atol=1e-13)
    # Linear in V.
    V2 = rng.standard_normal((20, 16))
    assert np.allclose(att.attention(q, K, V + V2, 0.25),
                       base + att.attention(q, K, V2, 0.25), atol=1e-13)


def test_matches_scalar_brute_force():
    rng = np.random.default_rng(5)
    for L in (1, 2, 5, 23):
        q = rng.standard_normal((3, 8))
        K = rng.standard_normal((L, 8))
        V = rng.standard_normal((L, 6))
        out = att.attention(q, K, V, 0.35)
        for r in range(3):
            ref = brute.single_query(list(q[r]), K.tolist(), V.tolist(), 0.35)
            assert np.allclose(out[r], ref, rtol=0, atol=1e-13)


def test_block_translation_matches_pages_examples():
    g = json.load(open(GOLDEN))["block_translation"]
    table = [900 + 7 * i for i in range(600)]
    for c in g["cases"]:
        blk, slot = att.token_slot(table, c["token"], g["block_size"])
        assert blk == table[c["logical_block"]] and slot == c["slot"]


def test_gather_reads_each_token_from_its_slot():
    # Token t's value row holds t in column 0 (exact in bf16 for t < 256).
    B, Hkv, d, L = 16, 2, 8, 70
    table = [5, 2, 7, 0, 3]
    pool = np.zeros((8, Hkv, B, d), dtype=np.uint16)
    for t in range(L):
        pool[table[t // B], 1, t % B, 0] = bf16([float(t)])[0]
    col = att.gather_branch(pool, table, L, 1, B)[:, 0]
    assert list(col) == [float(t) for t in range(L)]
    # A dominant key at token j returns row j.
    kpool = np.zeros_like(pool)
    j = 41
    kpool[table[j // B], 1, j % B, 0] = bf16([30.0])[0]
    q = bf16(np.zeros((4, d)))
    q[:, 0] = bf16([30.0])[0]
    out = att.decode_branch_from_pool(q, kpool, pool, table, L, 1.0, B)
    assert out[2, 0] == pytest.approx(j, abs=1e-9)
    assert out[3, 0] == pytest.approx(j, abs=1e-9)


def test_gqa_head_mapping():
    # kv-head g holds value g + 1 everywhere; q-head h must read h // G.
    Hq, Hkv, d, L = 8, 2, 4, 9
    K = bf16(np.random.default_rng(6).standard_normal((L, Hkv, d)))
    V = np.zeros((L, Hkv, d), dtype=np.uint16)
    for g in range(Hkv):
        V[:, g, :] = bf16([float(g + 1)])[0]
    q = bf16(np.random.default_rng(7).standard_normal((Hq, d)))
    out = att.decode_branch_contiguous(q, K, V, Hkv, 0.5)
    for h in range(Hq):
        assert np.allclose(out[h], float(h // (Hq // Hkv) + 1), atol=1e-12)


def _tiny_replay(seed=1001):
    w = W.tiny_tree(seed=seed)
    return w, rp.replay(w, with_data=True)


def test_pool_path_equals_contiguous_path():
    w, r = _tiny_replay()
    q = w.queries(len(r.decode_ids))
    a = rp.decode_all_from_pool(r, q, w.scale)
    b = rp.decode_rows(r, q, range(len(r.decode_ids)), w.scale)
    for i in range(len(r.decode_ids)):
        assert np.array_equal(a[i], b[i])


def test_physical_block_permutation_invariance():
    w, r = _tiny_replay()
    q = w.queries(len(r.decode_ids))
    base = rp.decode_all_from_pool(r, q, w.scale)
    perm = np.random.default_rng(8).permutation(w.num_blocks)
    kp = np.empty_like(r.data.k[0])
    vp = np.empty_like(r.data.v[0])
    kp[perm] = r.data.k[0]
    vp[perm] = r.data.v[0]
    tables = [[int(perm[b]) for b in r.model.nodes[i].table]
              for i in r.decode_ids]
    lens = [r.model.nodes[i].seq_len for i in r.decode_ids]
    moved = att.decode_step(q, kp, vp, tables, lens, w.scale, w.block_size)
    assert np.array_equal(base, moved)


def test_shared_prefix_equals_private_copies():
    # The same branches laid out with every block private (no sharing).
    w, r = _tiny_replay()
    q = w.queries(len(r.decode_ids))
    shared = rp.decode_all_from_pool(r, q, w.scale)
    B = w.block_size
    blocks = []
    tables = []
    for nid in r.decode_ids:
        k, v = r.branch_kv(nid)
        L = k.shape[1]
        tab = []
        for j in range(0, L, B):
            kb = np.zeros((w.Hkv, B, w.d), dtype=np.uint16)
            vb = np.zeros_like(kb)
            n = min(B, L - j)
            kb[:, :n] = k[0, j:j + n].transpose(1, 0, 2)
            vb[:, :n] = v[0, j:j + n].transpose(1, 0, 2)
            tab.append(len(blocks))
            blocks.append((kb, vb))
        tables.append(tab)
    kp = np.stack([b[0] for b in blocks])
    vp = np.stack([b[1] for b in blocks])
    lens = [r.model.nodes[i].seq_len for i in r.decode_ids]
    private = att.decode_step(q, kp, vp, tables, lens, w.scale, B)
    assert np.array_equal(shared, private)


def test_branch_order_permutes_outputs():
    w, r = _tiny_replay()
    q = w.queries(len(r.decode_ids))
    base = rp.decode_all_from_pool(r, q, w.scale)
    order = [2, 0, 3, 1]
    tables = [r.model.nodes[r.decode_ids[i]].table for i in order]
    lens = [r.model.nodes[r.decode_ids[i]].seq_len for i in order]
    out = att.decode_step(q[order], r.data.k[0], r.data.v[0], tables, lens,
                          w.scale, w.block_size)
    assert np.array_equal(out, base[order])


def test_prefix_group_validation():
    w, r = _tiny_replay()
    tables = [r.model.nodes[i].table for i in r.decode_ids]
    lens = [r.model.nodes[i].seq_len for i in r.decode_ids]
    att.validate_prefix_groups([[0, 4, 0, 6]], tables, lens, 16)
    with pytest.raises(ValueError):       # block 6 is each branch's COW copy
        att.validate_prefix_groups([[0, 4, 0, 7]], tables, lens, 16)
    with pytest.raises(ValueError):
        att.validate_prefix_groups([[0, 5, 0, 6]], tables, lens, 16)


def test_seq_len_zero_rejected():
    with pytest.raises(ValueError):
        att.gather_branch(np.zeros((1, 1, 16, 4), np.uint16), [0], 0, 0, 16)
