"""FP8 (E4M3) KV storage with one power-of-two scale per block and kv-head.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages name FP8 only in passing: FP4/FP8 quantisation is listed among the
memory-architecture skills of a reasoning engine, beside virtual paging and
cache locality ("The Reasoning Engine Meltdown", §9, the competency table),
and an FP8 evaluator cluster sits in its §4 architecture diagram.  They fix
no format.  The readings taken here, stated once:

* Element format: E4M3 in the form with no infinities -- a sign bit, four
  exponent bits with bias 7 and three mantissa bits; exponent field 0 holds
  the subnormals m/8 * 2^-6; exponent field 15 with mantissa 7 is NaN; the
  largest finite magnitude is 1.75 * 2^8 = 448.
* A stored value is ``value(code) * 2^e``.  There is one integer exponent e
  for each (layer, physical block, kv-head) and each of K and V: the block's
  scale.  A power of two makes the stored value exact to decode and makes a
  change of scale a pure exponent shift.
* e is the smallest integer in [E_MIN, E_MAX] with max|x| <= 448 * 2^e over
  the values written, so nothing saturates.  A write into a block either
  starts it (it writes slot 0: the block was just allocated, e comes from the
  new rows alone) or extends it; then e = max(e_old, e_required(new rows)),
  and when e grows the rows already stored are re-encoded from their stored
  values.  Each value is encoded as the finite code nearest to x * 2^-e,
  ties to the even mantissa (round to nearest even), magnitudes above 448
  clamped to 448.  Writes are applied in program order.
* Copy-on-write and the host tier copy codes and scales verbatim.

Everything is done in float64 or exact integer arithmetic.  x * 2^-e is exact
in float64 for every bf16 input x and every e in range.
"""

from __future__ import annotations

import math

import numpy as np

from . import attention as att

E_MIN = -126
E_MAX = 120
MAX_FINITE = 448.0


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 15 and man == 7:
        return math.nan
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


# Value of every code, and the 127 non-negative finite codes in value order.
DECODE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
_POS_CODES = np.arange(0x7F, dtype=np.int64)          # 0x00 .. 0x7E
_POS_VALUES = DECODE[:0x7F]
assert np.all(np.diff(_POS_VALUES) > 0)


def encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code to each value of ``x`` (float64), ties to the
    code with the even mantissa; magnitudes above 448 give 448; the sign is
    kept (so -0.0 and negatives that round to zero give 0x80).  NaN input is
    rejected."""
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN has no E4M3 encoding here")
    mag = np.minimum(np.abs(x), MAX_FINITE)
    hi = np.searchsorted(_POS_VALUES, mag, side="left")   # first value >= mag
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - mag
    d_lo = mag - _POS_VALUES[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    code = np.where(mag == _POS_VALUES[hi], _POS_CODES[hi], code)
    sign = np.signbit(x)
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8)


def decode(codes: np.ndarray) -> np.ndarray:
    """float64 value of each code."""
    return DECODE[np.asarray(codes, dtype=np.uint8)]


def exponent_for(amax: float) -> int:
    """Smallest integer e in [E_MIN, E_MAX] with amax <= 448 * 2^e.

    With amax = m * 2^k, m in [0.5, 1) (exact decomposition) and
    448 = 0.875 * 2^9: amax <= 0.875 * 2^(9 + e) holds iff e >= k - 9 when
    m <= 0.875, else iff e >= k - 8."""
    amax = float(amax)
    if not math.isfinite(amax) or amax < 0:
        raise ValueError("amax must be finite and >= 0")
    if amax == 0.0:
        return E_MIN
    m, k = math.frexp(amax)
    e = k - 9 if m <= 0.875 else k - 8
    return max(E_MIN, min(E_MAX, e))


def quantize_rows(x: np.ndarray, e: int) -> np.ndarray:
    """Codes of float64 values ``x`` under the scale 2^e."""
    return encode(np.asarray(x, dtype=np.float64) * 2.0 ** (-e))


def block_write(codes: np.ndarray, e_old: int, s0: int,
                new_rows: np.ndarray) -> int:
    """Write float64 ``new_rows`` [n][d] into slots [s0, s0 + n) of one
    (block, kv-head) tile ``codes`` [16][d] (uint8, updated in place) whose
    scale exponent is ``e_old`` (ignored when s0 == 0).  Returns the tile's
    new exponent."""
    n = new_rows.shape[0]
    amax = float(np.max(np.abs(new_rows))) if n else 0.0
    e_req = exponent_for(amax)
    if s0 == 0:
        e = e_req
    else:
        e = max(e_old, e_req)
        if e > e_old:
            old = decode(codes[:s0]) * 2.0 ** e_old
            codes[:s0] = quantize_rows(old, e)
    codes[s0:s0 + n] = quantize_rows(new_rows, e)
    return e


class Fp8PoolData:
    """The oracle's own host copy of FP8 K and V pools with their scales.

    ``k``, ``v``: uint8 codes ``[L][num_blocks][Hkv][16][d]`` in logical
    (slot, dim) order; ``ek``, ``ev``: int64 exponents ``[L][num_blocks][Hkv]``.
    Fed with the same writes and copies as the bf16 ``PoolData``.
    """

    def __init__(self, num_layers, num_blocks, Hkv, block_size, d):
        shape = (num_layers, num_blocks, Hkv, block_size, d)
        self.k = np.zeros(shape, dtype=np.uint8)
        self.v = np.zeros(shape, dtype=np.uint8)
        self.ek = np.zeros(shape[:3], dtype=np.int64)
        self.ev = np.zeros(shape[:3], dtype=np.int64)

    @staticmethod
    def segments(writes):
        """Group per-token writes [(t, blk, slot)] into per-block runs
        (blk, s0, s1, first row), keeping their order."""
        runs = []
        for i, (_t, blk, slot) in enumerate(writes):
            if runs and runs[-1][0] == blk and runs[-1][2] == slot:
                b, s0, s1, r0 = runs[-1]
                runs[-1] = (b, s0, s1 + 1, r0)
            else:
                runs.append((blk, slot, slot + 1, i))
        return runs

    def write(self, writes, k_new, v_new) -> None:
        """k_new, v_new: [L][n][Hkv][d] bf16 bits of the appended tokens."""
        kf = att.bf16_to_f64(k_new)
        vf = att.bf16_to_f64(v_new)
        L, _n, Hkv, _d = kf.shape
        for blk, s0, s1, r0 in self.segments(writes):
            for layer in range(L):
                for h in range(Hkv):
                    rows = slice(r0, r0 + s1 - s0)
                    self.ek[layer, blk, h] = block_write(
                        self.k[layer, blk, h], int(self.ek[layer, blk, h]), s0,
                        kf[layer, rows, h, :])
                    self.ev[layer, blk, h] = block_write(
                        self.v[layer, blk, h], int(self.ev[layer, blk, h]), s0,
                        vf[layer, rows, h, :])

    def copy_block(self, src: int, dst: int) -> None:
        for a in (self.k, self.v, self.ek, self.ev):
            a[:, dst] = a[:, src]

    def values(self, layer: int = 0):
        """Dequantised float64 K, V of one layer: [num_blocks][Hkv][16][d]."""
        k = decode(self.k[layer]) * np.exp2(self.ek[layer].astype(np.float64))[..., None, None]
        v = decode(self.v[layer]) * np.exp2(self.ev[layer].astype(np.float64))[..., None, None]
        return k, v


def quantize_sequence(seg_lens, rows_bits: np.ndarray) -> np.ndarray:
    """Stored (dequantised) values of one branch's logical token sequence.

    ``rows_bits``: bf16 bits [L][T][Hkv][d] of the branch's tokens, oldest
    first; ``seg_lens``: the lengths of the appends that wrote them, in order
    (they sum to T).  Token t sits in the branch's logical block t // 16;
    each append writes its tokens of every block it touches as one write, in
    append order, and a block's first write starts at slot 0 -- also for a
    copy-on-write block, whose copy carries the parent's codes and scale.
    Returns float64 [L][T][Hkv][d].  Needs no pool, so it runs for a few
    sampled branches of any workload."""
    x = att.bf16_to_f64(rows_bits)
    L, T, Hkv, d = x.shape
    bounds = np.cumsum([0] + [int(n) for n in seg_lens])
    if bounds[-1] != T:
        raise ValueError("segment lengths do not add up to the sequence")
    out = np.empty_like(x)
    for lb in range((T + 15) // 16):
        lo, hi = 16 * lb, min(16 * lb + 16, T)
        writes = [(max(a, lo) - lo, min(b, hi) - lo)
                  for a, b in zip(bounds[:-1], bounds[1:]) if a < hi and b > lo]
        for layer in range(L):
            for h in range(Hkv):
                codes = np.zeros((16, d), np.uint8)
                e = 0
                for s0, s1 in writes:
                    e = block_write(codes, e, s0, x[layer, lo + s0:lo + s1, h])
                out[layer, lo:hi, h] = decode(codes[:hi - lo]) * 2.0 ** e
    return out


def gather_values(pool_f64: np.ndarray, table, seq_len: int, kv_head: int,
                  block_size: int) -> np.ndarray:
    """Like ``attention.gather_branch`` for a pool already in float64."""
    if seq_len < 1:
        raise ValueError("a decode branch holds at least one token")
    t = np.arange(seq_len)
    blocks = np.asarray(table, dtype=np.int64)[t // block_size]
    if blocks.min() < 0 or blocks.max() >= pool_f64.shape[0]:
        raise IndexError("block table entry outside the pool")
    return pool_f64[blocks, kv_head, t % block_size, :]


def decode_step_fp8(q: np.ndarray, data: Fp8PoolData, tables, seq_lens,
                    scale: float, block_size: int, rows=None,
                    layer: int = 0) -> np.ndarray:
    """Decode step over the dequantised FP8 pool: for each branch and q-head,
    ``attention.attention`` on the branch's dequantised K and V (gathered
    through its block table).  Returns [nb][Hq][d] float64 (unlisted rows
    NaN)."""
    kf, vf = data.values(layer)
    nb, Hq, d = q.shape
    Hkv = kf.shape[1]
    out = np.full((nb, Hq, d), np.nan, dtype=np.float64)
    for b in (range(nb) if rows is None else rows):
        qf = att.bf16_to_f64(q[b])
        L = int(seq_lens[b])
        for g in range(Hkv):
            K = gather_values(kf, tables[b], L, g, block_size)
            V = gather_values(vf, tables[b], L, g, block_size)
            heads = [h for h in range(Hq) if att.kv_head_of(h, Hq, Hkv) == g]
            out[b, heads] = att.attention(qf[heads], K, V, scale)
    return out


def attention_error_bound(q_rows: np.ndarray, K: np.ndarray, Kq: np.ndarray,
                          V: np.ndarray, Vq: np.ndarray,
                          scale: float) -> np.ndarray:
    """Per-row bound on |attention(q, Kq, Vq) - attention(q, K, V)| (max over
    the output's columns), from the two quantisation errors alone.

    With s_t = scale q.k_t and p = softmax(s): a score error of at most
    delta = max_t |s'_t - s_t| multiplies every weight by a factor within
    [e^-2delta, e^2delta], so sum_t |p'_t - p_t| <= e^(2 delta) - 1; then
    |o' - o| <= max_t |v'_t - v_t| + (e^(2 delta) - 1) max_t |v_t|.
    Returns [R] float64."""
    ds = np.abs(q_rows @ (Kq - K).T) * float(scale)        # [R][L]
    delta = ds.max(axis=1)
    dv = np.abs(Vq - V).max()
    vmax = np.abs(V).max()
    return dv + np.expm1(2.0 * delta) * vmax
