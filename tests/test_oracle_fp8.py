"""Pins for the oracle's FP8 (E4M3) KV storage model (``oracle.fp8``).

Each pin checks the oracle against something other than itself: the E4M3
format as PyTorch's independent float8_e4m3fn type implements it, hand-worked
codes, the defining inequalities of the scale exponent, the rounding error
bound of a 3-bit mantissa, exactness of a power-of-two rescale, and a
derived bound on how far attention may move under the quantisation.
"""

import math

import numpy as np
import pytest

from oracle import attention as att
from oracle import fp8
from oracle import replay as rp
from paged_kv_cache_attn_gb300 import workloads as wl

torch = pytest.importorskip("torch")


def torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode_f32(x32):
    """PyTorch's float32 -> float8_e4m3fn conversion (round to nearest even);
    inputs must be within +-448."""
    t = torch.from_numpy(np.asarray(x32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_table_matches_torch():
    ours = fp8.DECODE
    theirs = torch_e4m3_values()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], theirs[~nan])
    # signed zeros
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_hand_worked_codes():
    assert fp8.e4m3_value(0x38) == 1.0                # exp 7, man 0
    assert fp8.e4m3_value(0x7E) == 448.0              # largest finite
    assert fp8.e4m3_value(0x08) == 2.0 ** -6          # smallest normal
    assert fp8.e4m3_value(0x01) == 2.0 ** -9          # smallest subnormal
    assert fp8.e4m3_value(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert fp8.e4m3_value(0xB9) == -1.125             # sign, exp 7, man 1
    assert math.isnan(fp8.e4m3_value(0x7F))


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(fp8.encode(fp8.DECODE[codes]), codes.astype(np.uint8))


def test_encode_ties_go_to_even_mantissa():
    # halfway between 1.0 (0x38) and 1.125 (0x39) -> 0x38
    assert fp8.encode(np.array([1.0625]))[0] == 0x38
    # halfway between 1.125 (0x39) and 1.25 (0x3A) -> 0x3A
    assert fp8.encode(np.array([1.1875]))[0] == 0x3A
    # halfway between 1.875 (0x3F, man 7) and 2.0 (0x40) -> 0x40
    assert fp8.encode(np.array([1.9375]))[0] == 0x40
    # halfway between 0 and the smallest subnormal -> 0
    assert fp8.encode(np.array([2.0 ** -10]))[0] == 0x00
    # just above it -> smallest subnormal
    assert fp8.encode(np.array([2.0 ** -10 * (1 + 2 ** -20)]))[0] == 0x01
    # halfway between the largest subnormal and the smallest normal
    assert fp8.encode(np.array([7.5 * 2.0 ** -9]))[0] == 0x08


def test_encode_saturates_and_keeps_sign():
    assert fp8.encode(np.array([1e6]))[0] == 0x7E
    assert fp8.encode(np.array([-1e6]))[0] == 0xFE
    assert fp8.encode(np.array([-0.0]))[0] == 0x80
    assert fp8.encode(np.array([-1e-9]))[0] == 0x80
    with pytest.raises(ValueError):
        fp8.encode(np.array([np.nan]))


def test_encode_matches_torch_on_float32_values():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000) * 40,
        rng.uniform(-2.0 ** -5, 2.0 ** -5, 20000),    # subnormal range
        (fp8.DECODE[:0x7E] + fp8.DECODE[1:0x7F]) / 2,  # every midpoint
    ]).astype(np.float32)
    x = np.clip(x, -448, 448)
    assert np.array_equal(fp8.encode(x.astype(np.float64)), torch_encode_f32(x))


@pytest.mark.parametrize("amax", [0.0, 1e-300, 2.0 ** -133, 1.0, 3.9, 448.0,
                                  448.0 * (1 + 2 ** -20), 449.0, 896.0, 1e30,
                                  3.3895e38])
def test_exponent_is_smallest_that_avoids_saturation(amax):
    e = fp8.exponent_for(amax)
    assert fp8.E_MIN <= e <= fp8.E_MAX
    assert amax <= 448.0 * 2.0 ** e
    if e > fp8.E_MIN:
        assert amax > 448.0 * 2.0 ** (e - 1)


def test_exponent_on_exact_boundaries():
    for k in range(-100, 100, 7):
        assert fp8.exponent_for(448.0 * 2.0 ** k) == k
        assert fp8.exponent_for(448.0 * 2.0 ** k * (1 + 2 ** -30)) == k + 1
    assert fp8.exponent_for(0.0) == fp8.E_MIN


def bf16_rows(rng, shape, sigma=1.0):
    bits = wl.f32_to_bf16_bits((rng.standard_normal(shape) * sigma)
                               .astype(np.float32))
    return att.bf16_to_f64(bits)


def test_quantisation_error_bound():
    """|x - deq(q(x))| <= max(2^-4 |x|, 2^(e-10)): half a unit in the last
    place of a 3-bit mantissa, or half the subnormal spacing 2^(e-9)."""
    rng = np.random.default_rng(3)
    for sigma in (1e-3, 1.0, 50.0):
        x = bf16_rows(rng, (16, 128), sigma)
        e = fp8.exponent_for(np.abs(x).max())
        deq = fp8.decode(fp8.quantize_rows(x, e)) * 2.0 ** e
        err = np.abs(deq - x)
        bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** (e - 10))
        assert np.all(err <= bound)
        # the largest magnitude does not saturate
        assert np.abs(deq).max() <= 448 * 2.0 ** e


def test_block_write_fresh_then_extend_without_growth():
    rng = np.random.default_rng(4)
    x = bf16_rows(rng, (16, 64))
    codes = np.zeros((16, 64), np.uint8)
    e = fp8.block_write(codes, 999, 0, x[:5])          # e_old ignored at s0=0
    assert e == fp8.exponent_for(np.abs(x[:5]).max())
    small = x[5:9] * 2.0 ** -3
    e2 = fp8.block_write(codes, e, 5, small)
    assert e2 == e                                      # no growth
    # rows 0..4 untouched, rows 5..8 coded under e
    assert np.array_equal(codes[:5], fp8.quantize_rows(x[:5], e))
    assert np.array_equal(codes[5:9], fp8.quantize_rows(small, e))


def test_block_write_growth_reencodes_by_exponent_shift():
    rng = np.random.default_rng(5)
    x = bf16_rows(rng, (16, 128))
    codes = np.zeros((16, 128), np.uint8)
    e = fp8.block_write(codes, 0, 0, x[:8])
    before = codes[:8].copy()
    big = x[8:10] * 2.0 ** 5
    e2 = fp8.block_write(codes, e, 8, big)
    assert e2 == fp8.exponent_for(np.abs(big).max()) and e2 > e
    shift = e2 - e
    # stored values re-encoded from their decoded values; for codes that
    # stay normal after the shift this is exact (same value).
    old_vals = fp8.decode(before) * 2.0 ** e
    new_vals = fp8.decode(codes[:8]) * 2.0 ** e2
    normal = np.abs(fp8.decode(before)) * 2.0 ** -shift >= 2.0 ** -6
    assert np.array_equal(old_vals[normal], new_vals[normal])
    assert np.all(np.abs(old_vals - new_vals) <= 2.0 ** (e2 - 10))


def test_fp8_pool_replay_is_close_to_bf16_pool():
    w = wl.make("tiny_tree")
    r16 = rp.replay(w, with_data=True)
    r8 = rp.replay(w, with_data=True, kv_dtype="e4m3")
    assert r8.model.free_stack() == r16.model.free_stack()
    k16 = att.bf16_to_f64(r16.data.k[0])
    v16 = att.bf16_to_f64(r16.data.v[0])
    k8, v8 = r8.data.values(0)
    m = r8.model
    for nid in r8.decode_ids:
        node = m.nodes[nid]
        for t in range(node.seq_len):
            blk, slot = node.table[t // 16], t % 16
            for h in range(w.Hkv):
                for a16, a8, e in ((k16, k8, r8.data.ek), (v16, v8, r8.data.ev)):
                    x = a16[blk, h, slot]
                    err = np.abs(a8[blk, h, slot] - x)
                    bound = np.maximum(np.abs(x) * 2.0 ** -4,
                                       2.0 ** (e[0, blk, h] - 10))
                    assert np.all(err <= bound)


def test_attention_error_bound_holds_and_catches_a_wrong_scale():
    """The FP8 oracle's output stays within the derived bound of the bf16
    oracle's; a decode that forgot the V scale would not."""
    w = wl.make("tiny_tree")
    r16 = rp.replay(w, with_data=True)
    r8 = rp.replay(w, with_data=True, kv_dtype="e4m3")
    q = w.queries(len(r8.decode_ids))
    k16 = att.bf16_to_f64(r16.data.k[0])
    v16 = att.bf16_to_f64(r16.data.v[0])
    k8, v8 = r8.data.values(0)
    G = w.Hq // w.Hkv
    checked = 0
    for b, nid in enumerate(r8.decode_ids):
        node = r8.model.nodes[nid]
        L = node.seq_len
        for g in range(w.Hkv):
            K = fp8.gather_values(k16, node.table, L, g, 16)
            V = fp8.gather_values(v16, node.table, L, g, 16)
            Kq = fp8.gather_values(k8, node.table, L, g, 16)
            Vq = fp8.gather_values(v8, node.table, L, g, 16)
            qr = att.bf16_to_f64(q[b, g * G:(g + 1) * G])
            o = att.attention(qr, K, V, w.scale)
            oq = att.attention(qr, Kq, Vq, w.scale)
            bound = fp8.attention_error_bound(qr, K, Kq, V, Vq, w.scale)
            assert np.all(np.abs(oq - o).max(axis=1) <= bound)
            # V decoded without its per-block scale: far outside the bound
            Vbad = fp8.gather_values(fp8.decode(r8.data.v[0]), node.table, L,
                                     g, 16)
            obad = att.attention(qr, Kq, Vbad, w.scale)
            assert np.any(np.abs(obad - o).max(axis=1) > bound)
            checked += 1
    assert checked == len(r8.decode_ids) * w.Hkv


def test_decode_step_fp8_equals_attention_on_dequantised_values():
    w = wl.make("tiny_tree")
    r8 = rp.replay(w, with_data=True, kv_dtype="e4m3")
    q = w.queries(len(r8.decode_ids))
    out = rp.decode_all_from_pool(r8, q, w.scale)
    k8, v8 = r8.data.values(0)
    # brute force: one (branch, head) at a time through the scalar path
    from oracle import brute
    b = 1
    node = r8.model.nodes[r8.decode_ids[b]]
    h = 3
    g = att.kv_head_of(h, w.Hq, w.Hkv)
    K = fp8.gather_values(k8, node.table, node.seq_len, g, 16)
    V = fp8.gather_values(v8, node.table, node.seq_len, g, 16)
    ref = brute.single_query(att.bf16_to_f64(q[b, h]).tolist(), K.tolist(),
                             V.tolist(), w.scale)
    assert np.allclose(out[b, h], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name", ["tiny_tree", "deep_tree"])
def test_sequence_route_equals_pool_route(name):
    """Quantising a branch from its logical token sequence and its append
    history gives, bit for bit, the values the replayed pool holds for it
    (through forks with copy-on-write and multi-block appends)."""
    w = (wl.make("tiny_tree") if name == "tiny_tree"
         else wl.deep_tree(root_tokens=300, depth=3, min_seg=5, max_seg=40))
    r8 = rp.replay(w, with_data=True, kv_dtype="e4m3")
    kf, vf = r8.data.values(0)
    for nid in r8.decode_ids:
        node = r8.model.nodes[nid]
        kb, vb = r8.branch_kv(nid)
        lens = [hi - lo for _src, lo, hi in r8.logical[nid]]
        kq = fp8.quantize_sequence(lens, kb)
        vq = fp8.quantize_sequence(lens, vb)
        for g in range(w.Hkv):
            K = fp8.gather_values(kf, node.table, node.seq_len, g, 16)
            V = fp8.gather_values(vf, node.table, node.seq_len, g, 16)
            assert np.array_equal(K, kq[0, :, g])
            assert np.array_equal(V, vq[0, :, g])
