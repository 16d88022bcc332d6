"""Differential fuzz of the host block manager against the oracle's model,
every operation interleaved: plain and prefix-cached admission, forks, single
and batched appends (with copy-on-write), block keying, frees and moves
between two pools (a device pool and a host pool).  After every operation both
pools' free and cached counts agree; at the end every block table and every
refcount agrees, id for id.  Failures (pool exhausted, shared blocks on a
move) must happen on the same operations and leave both sides unchanged."""
import numpy as np
import pytest

from oracle.block_manager_ref import BlockManagerModel, NoBlocks


@pytest.fixture(scope="module")
def binding():
    from paged_kv_cache_237_gb300 import binding
    return binding


def _expect_same(binding, lib_call, model_call):
    """Run both; they must both succeed (same result) or fail the same way."""
    try:
        want = model_call()
    except NoBlocks:
        with pytest.raises(binding.PAError) as e:
            lib_call()
        assert e.value.code == binding.PA_ERR_NO_BLOCKS
        return None, False
    except ValueError:
        with pytest.raises(binding.PAError) as e:
            lib_call()
        assert e.value.code == binding.PA_ERR_REFCOUNT
        return None, False
    got = lib_call()
    assert got == want
    return got, True


@pytest.mark.parametrize("seed", range(6))
def test_every_operation_interleaved_matches_the_model(binding, seed):
    rng = np.random.default_rng(100 + seed)
    bs = 16
    sizes = {"dev": 96, "host": 160}
    lib = {k: binding.BlockManager(n, bs) for k, n in sizes.items()}
    mod = {k: BlockManagerModel(n, bs) for k, n in sizes.items()}
    prompts = [rng.integers(0, 30000, size=int(rng.integers(16, 120))).tolist() for _ in range(4)]
    where, tokens, salt = {}, {}, {}          # live sequence -> pool, its token ids, its salt
    nxt = 0

    def live(pool=None):
        return [s for s, w in where.items() if pool is None or w == pool]

    for _ in range(1200):
        r = rng.random()
        if r < 0.15:                                                   # prefix-cached admission
            p = int(rng.integers(0, len(prompts)))
            toks = prompts[p][:int(rng.integers(1, len(prompts[p]) + 1))] + \
                rng.integers(0, 30000, size=int(rng.integers(0, 30))).tolist()
            sl = 7 + p % 2
            _, ok = _expect_same(binding, lambda: lib["dev"].add_seq_cached(nxt, toks, sl),
                                 lambda: mod["dev"].add_seq_cached(nxt, toks, sl))
            if ok:
                where[nxt], tokens[nxt], salt[nxt] = "dev", list(toks), sl
            nxt += 1
        elif r < 0.25:                                                 # plain admission
            n = int(rng.integers(0, 90))
            _, ok = _expect_same(binding, lambda: lib["dev"].add_seq(nxt, n), lambda: mod["dev"].add_seq(nxt, n))
            if ok:
                where[nxt], tokens[nxt], salt[nxt] = "dev", rng.integers(0, 30000, size=n).tolist(), 0
            nxt += 1
        elif r < 0.35 and live("dev"):                                 # fork (parallel sampling)
            par = int(rng.choice(live("dev")))
            _expect_same(binding, lambda: lib["dev"].fork(par, nxt), lambda: mod["dev"].fork(par, nxt))
            where[nxt], tokens[nxt], salt[nxt] = "dev", list(tokens[par]), salt[par]
            nxt += 1
        elif r < 0.55 and live():                                      # one append
            sid = int(rng.choice(live()))
            pool = where[sid]
            _, ok = _expect_same(binding, lambda: lib[pool].append_slot(sid), lambda: mod[pool].append_slot(sid))
            if ok:
                tokens[sid].append(int(rng.integers(0, 30000)))
        elif r < 0.62 and live("dev"):                                 # batched append (a decode step)
            ids = [int(s) for s in rng.permutation(live("dev"))[:int(rng.integers(1, 6))]]
            want, fail = [], False
            for sid in ids:
                try:
                    want.append(mod["dev"].append_slot(sid))
                except NoBlocks:
                    fail = True
                    break
            if fail:
                with pytest.raises(binding.PAError):
                    lib["dev"].append_slots(ids)
            else:
                slots, pairs = lib["dev"].append_slots(ids)
                assert slots.tolist() == [w[0] for w in want]
                assert pairs.tolist() == [[w[1], w[2]] for w in want if w[1] >= 0]
            for sid in ids[:len(want)]:
                tokens[sid].append(int(rng.integers(0, 30000)))
        elif r < 0.68 and live("dev"):                                 # key full blocks
            sid = int(rng.choice(live("dev")))
            assert lib["dev"].register_blocks(sid, tokens[sid], salt[sid]) == \
                mod["dev"].register_blocks(sid, tokens[sid], salt[sid])
        elif r < 0.80 and live():                                      # move to the other pool
            sid = int(rng.choice(live()))
            src = where[sid]
            dst = "host" if src == "dev" else "dev"
            try:
                want = mod[src].move_seq(mod[dst], sid)
            except (NoBlocks, ValueError) as e:
                code = binding.PA_ERR_NO_BLOCKS if isinstance(e, NoBlocks) else binding.PA_ERR_REFCOUNT
                with pytest.raises(binding.PAError) as err:
                    lib[src].move_seq(lib[dst], sid)
                assert err.value.code == code
            else:
                got = lib[src].move_seq(lib[dst], sid)
                assert [tuple(x) for x in got.tolist()] == want
                where[sid] = dst
        elif live():                                                   # free
            sid = int(rng.choice(live()))
            lib[where[sid]].free_seq(sid)
            mod[where[sid]].free_seq(sid)
            del where[sid]
        for k in lib:
            assert lib[k].num_free() == mod[k].num_free(), k
            assert lib[k].num_cached() == mod[k].num_cached(), k
    for sid, pool in where.items():
        assert lib[pool].block_table(sid) == mod[pool].block_table(sid)
        assert lib[pool].num_tokens(sid) == mod[pool].num_tokens(sid)
    for k, n in sizes.items():
        assert [lib[k].refcount(b) for b in range(n)] == [mod[k].refcount(b) for b in range(n)]
