"""fp64 decode attention over a paged KV pool -- the oracle's definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What is computed, and where the pages define it:

* Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
  ("The Reasoning Engine Meltdown", §2.1, the attention equation).  The
  decode step attends the one new query of a branch to every cached key and
  value of that branch (same section, the paragraph on step t+1).  ``scale``
  is passed in; the workloads use 1/sqrt(d).
* A token's KV lives in physical block ``table[t // B]`` at slot ``t % B``
  ("Dismantling the Memory Wall", PagedAttention section,
  ``BlockTable.get_block_for_token``: logical block = token index // block
  size; the offset inside the block is the remainder).
* Grouped-query heads: the pages never mention GQA.  Reading taken: q-head h
  reads kv-head ``h // (Hq // Hkv)`` (consecutive q-heads share a kv-head).

Data layouts (one layer):

* ``k_pool``, ``v_pool``: uint16 bf16 bit patterns ``[num_blocks][Hkv][B][d]``.
* ``q``: uint16 bf16 bit patterns ``[nb][Hq][d]``.
* ``tables``: int ``[nb][max_blocks]`` (entries past the branch's blocks are
  ignored), ``seq_lens``: int ``[nb]``.

Everything is converted to float64 before any arithmetic; bf16 -> fp64 is
exact.  No blocking, no online softmax, no split: a plain gather, one matrix
product for the scores, a max-subtracted exponential, a normalisation and one
matrix product for the output.
"""

from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64, exactly.

    A bf16 value is the upper 16 bits of an IEEE binary32 value, so shifting
    the pattern into the high half of a 32-bit word gives that binary32 value;
    binary32 -> binary64 is exact.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    as_f32 = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return as_f32.astype(np.float64)


def token_slot(table, t: int, block_size: int) -> tuple[int, int]:
    """Logical token index -> (physical block id, slot inside the block).

    "Dismantling the Memory Wall", PagedAttention section: the block table
    maps logical block ``t // block_size`` to a physical block; the token sits
    at offset ``t % block_size`` inside it.
    """
    return int(table[t // block_size]), t % block_size


def gather_branch(pool: np.ndarray, table, seq_len: int, kv_head: int,
                  block_size: int) -> np.ndarray:
    """Gather one branch's tokens for one kv-head into a contiguous fp64 array.

    Returns ``[seq_len][d]`` float64: row t is the pool row at
    ``token_slot(table, t)``.
    """
    if seq_len < 1:
        raise ValueError("a decode branch holds at least one token")
    t = np.arange(seq_len)
    blocks = np.asarray(table, dtype=np.int64)[t // block_size]
    if blocks.min() < 0 or blocks.max() >= pool.shape[0]:
        raise IndexError("block table entry outside the pool")
    slots = t % block_size
    return bf16_to_f64(pool[blocks, kv_head, slots, :])


def attention(q_rows: np.ndarray, K: np.ndarray, V: np.ndarray,
              scale: float) -> np.ndarray:
    """softmax(q K^T * scale) V in float64 for a few query rows.

    ``q_rows``: [R][d], ``K``: [L][d], ``V``: [L][dv], all float64.
    Returns [R][dv].  The row maximum is subtracted before the exponential
    (the result is the same real number; it only keeps exp() finite).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    scores = (q_rows @ K.T) * float(scale)            # [R][L]
    scores = scores - scores.max(axis=1, keepdims=True)
    weights = np.exp(scores)
    weights = weights / weights.sum(axis=1, keepdims=True)
    return weights @ V                                 # [R][dv]


def kv_head_of(h: int, Hq: int, Hkv: int) -> int:
    """GQA mapping (reading taken where the pages are silent): q-head h reads
    kv-head h // (Hq // Hkv)."""
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (Hq // Hkv)


def decode_branch_contiguous(q_b: np.ndarray, K_b: np.ndarray, V_b: np.ndarray,
                             Hkv: int, scale: float) -> np.ndarray:
    """One branch's decode output from contiguous per-token KV.

    ``q_b``: [Hq][d] bf16 bits; ``K_b``, ``V_b``: [L][Hkv][d] bf16 bits (the
    branch's logical token sequence, oldest first).  Returns [Hq][d] float64.
    """
    Hq = q_b.shape[0]
    G = Hq // Hkv
    out = np.empty((Hq, q_b.shape[1]), dtype=np.float64)
    qf = bf16_to_f64(q_b)
    for g in range(Hkv):
        Kg = bf16_to_f64(K_b[:, g, :])
        Vg = bf16_to_f64(V_b[:, g, :])
        heads = [h for h in range(Hq) if kv_head_of(h, Hq, Hkv) == g]
        out[heads] = attention(qf[heads], Kg, Vg, scale)
    assert G * Hkv == Hq
    return out


def decode_branch_from_pool(q_b: np.ndarray, k_pool: np.ndarray,
                            v_pool: np.ndarray, table, seq_len: int,
                            scale: float, block_size: int) -> np.ndarray:
    """One branch's decode output, gathering its tokens through its block
    table.  Returns [Hq][d] float64."""
    Hq = q_b.shape[0]
    Hkv = k_pool.shape[1]
    qf = bf16_to_f64(q_b)
    out = np.empty((Hq, v_pool.shape[3]), dtype=np.float64)
    for g in range(Hkv):
        Kg = gather_branch(k_pool, table, seq_len, g, block_size)
        Vg = gather_branch(v_pool, table, seq_len, g, block_size)
        heads = [h for h in range(Hq) if kv_head_of(h, Hq, Hkv) == g]
        out[heads] = attention(qf[heads], Kg, Vg, scale)
    return out


def decode_step(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                tables, seq_lens, scale: float, block_size: int,
                rows=None) -> np.ndarray:
    """Decode step for every branch of a batch (or the listed ``rows``).

    Returns ``[nb][Hq][d]`` float64; rows not listed are left as NaN.
    """
    nb, Hq, d = q.shape
    out = np.full((nb, Hq, v_pool.shape[3]), np.nan, dtype=np.float64)
    for b in (range(nb) if rows is None else rows):
        out[b] = decode_branch_from_pool(q[b], k_pool, v_pool, tables[b],
                                         int(seq_lens[b]), scale, block_size)
    return out


def validate_prefix_groups(groups, tables, seq_lens, block_size: int) -> None:
    """Check that each shared-prefix segment really is shared.

    A segment ``(branch_begin, branch_count, blk_begin, blk_count)`` claims
    that branches [branch_begin, branch_begin + branch_count) hold the same
    physical block at every logical index in [blk_begin, blk_begin +
    blk_count), and that those blocks are full for every branch (their tokens
    are all below the branch's length).  The oracle never uses segments to
    compute; it only checks the claim, since sharing does not change the
    mathematics ("The Reasoning Engine Meltdown", §5: a fork points at the
    parent's pages without copying them).
    """
    for (bb, bc, kb, kc) in np.asarray(groups, dtype=np.int64).reshape(-1, 4):
        if bc < 1 or kc < 1 or bb < 0 or kb < 0 or bb + bc > len(seq_lens):
            raise ValueError(f"malformed segment {(bb, bc, kb, kc)}")
        for b in range(bb, bb + bc):
            if (kb + kc) * block_size > int(seq_lens[b]):
                raise ValueError(f"segment {(bb, bc, kb, kc)} covers a block "
                                 f"that is not full for branch {b}")
            if list(tables[b][kb:kb + kc]) != list(tables[bb][kb:kb + kc]):
                raise ValueError(f"segment {(bb, bc, kb, kc)}: branch {b} "
                                 "does not share the segment's blocks")
