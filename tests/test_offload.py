"""Host tier (spill / restore) against the oracle's pool model, bit-exact,
on metadata-only pools; the data round trip is in test_gpu_offload."""

import random

import pytest

from oracle import allocator as al
from paged_kv_cache_attn_gb300 import binding as B


def _outcome(fn):
    try:
        return ("ok", fn())
    except al.OutOfBlocks:
        return ("oom", None)
    except KeyError:
        return ("notfound", None)
    except ValueError:
        return ("invalid", None)
    except B.KVError as e:
        return ({B.KV_ERR_OOM: "oom", B.KV_ERR_NOT_FOUND: "notfound",
                 B.KV_ERR_INVALID_ARG: "invalid"}.get(e.code, e.code), None)


@pytest.mark.parametrize("seed", range(6))
def test_spill_restore_matches_model(seed):
    rnd = random.Random(300 + seed)
    nblocks, slots = 120, 60
    order = list(range(nblocks))
    rnd.shuffle(order)
    h = B.kv_pool_create(nblocks, 1, 1, 64, None, None, order)
    B.kv_offload_attach(h, None, None, slots)
    m = al.PoolModel(nblocks, 16, order)
    m.attach_host(slots)
    ids = []
    spilled = set()
    for step in range(300):
        r = rnd.random()
        live = [i for i in ids if m.nodes[i].live]
        if not live or r < 0.1:
            got = _outcome(lambda: B.kv_branch_create(h))
            want = _outcome(m.create)
            if got[0] == "ok":
                ids.append(got[1])
        elif r < 0.35:
            x, n = rnd.choice(live), rnd.randint(0, 40)

            def model_append():
                if x in spilled:
                    raise ValueError("spilled")
                m.append(x, n)

            got = _outcome(lambda: B.kv_append(h, x, n))
            want = _outcome(model_append)
        elif r < 0.5:
            x, n = rnd.choice(live), rnd.randint(1, 3)

            def model_fork():
                if x in spilled:
                    raise ValueError("spilled")
                return [c for c, _ in m.fork_many(x, n)]

            got = _outcome(lambda: B.kv_fork_branches(h, x, n))
            want = _outcome(model_fork)
            if got[0] == "ok":
                ids += got[1]
        elif r < 0.7:
            xs = rnd.sample(live, min(len(live), rnd.randint(1, 3)))
            got = _outcome(lambda: B.kv_spill(h, xs))
            want = _outcome(lambda: len(m.spill(xs)))
            if got[0] == "ok":
                spilled |= {x for x in xs if any(b < 0 for b in m.nodes[x].table)}
        elif r < 0.85:
            xs = list(dict.fromkeys(rnd.sample(live, min(len(live), 2))))
            got = _outcome(lambda: B.kv_restore(h, xs))
            want = _outcome(lambda: len(m.restore(xs)))
            if got[0] == "ok":
                spilled -= set(xs)
        else:
            x = rnd.choice(live)
            got = _outcome(lambda: B.kv_free(h, x))
            want = _outcome(lambda: m.free_node(x))
            spilled.discard(x)
        assert got == want, (step, got, want)
        assert B.kv_get_refcounts(h, nblocks).tolist() == m.ref
        assert B.kv_get_free_stack(h).tolist() == m.free_stack()
        assert B.kv_get_host_free(h).tolist() == m.host_free_stack()
        for i in ids:
            if m.nodes[i].live:
                t, L = B.kv_get_block_table(h, i)
                assert t.tolist() == m.nodes[i].table and L == m.nodes[i].seq_len
        m.check_invariants()
    B.kv_pool_destroy(h)


def test_spilled_branch_is_guarded():
    h = B.kv_pool_create(16, 1, 1, 64)
    B.kv_offload_attach(h, None, None, 8)
    a = B.kv_branch_create(h)
    B.kv_append(h, a, 40)
    assert B.kv_spill(h, [a]) == 3
    t, _ = B.kv_get_block_table(h, a)
    assert t.tolist() == [-2, -3, -4]           # host slots 0, 1, 2
    for fn in (lambda: B.kv_append(h, a, 1), lambda: B.kv_fork_branch(h, a),
               lambda: B.kv_build_batch(h, [a])):
        with pytest.raises(B.KVError) as e:
            fn()
        assert e.value.code == B.KV_ERR_INVALID_ARG
    assert B.kv_restore(h, [a]) == 3
    B.kv_append(h, a, 1)
    B.kv_free(h, a)
    assert len(B.kv_get_free_stack(h)) == 16 and len(B.kv_get_host_free(h)) == 8
    B.kv_pool_destroy(h)


class _LibOps:
    """The host-tier scenario's operations on the library (metadata-only
    pool of 10 blocks, ascending free order, 4 host slots)."""

    def __init__(self):
        self.h = B.kv_pool_create(10, 1, 1, 64)
        B.kv_offload_attach(self.h, None, None, 4)

    def create(self):
        return B.kv_branch_create(self.h)

    def append(self, i, n):
        B.kv_append(self.h, i, n)

    def fork(self, i):
        return B.kv_fork_branch(self.h, i)

    def spill(self, ids):
        return B.kv_spill(self.h, ids)

    def restore(self, ids):
        return B.kv_restore(self.h, ids)

    def free(self, i):
        B.kv_free(self.h, i)

    def table(self, i):
        return B.kv_get_block_table(self.h, i)[0].tolist()

    def free_stack(self):
        return B.kv_get_free_stack(self.h).tolist()

    def host_free(self):
        return B.kv_get_host_free(self.h).tolist()

    def ref(self):
        return B.kv_get_refcounts(self.h, 10).tolist()


def test_host_tier_hand_worked_scenario_on_the_library():
    from test_oracle_allocator import HOST_TIER_WANT, _host_tier_scenario
    ops = _LibOps()
    assert _host_tier_scenario(ops) == HOST_TIER_WANT
    B.kv_pool_destroy(ops.h)
