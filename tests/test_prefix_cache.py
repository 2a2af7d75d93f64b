"""Prefix cache (hash chain, tutorial page "LLM 推理服务引擎深度拆解", sections
4.2-4.3) and the shared-prefix block-manager calls.  CPU only: the oracle is
pinned by hand-derived values of the page's agent demo, the chain property and
a hand-traced eviction order; the native pd_pc_* / pd_bm_* must then match the
oracle key for key, hit for hit, eviction for eviction."""
import random

import pytest

import oracle
from oracle import BlockManager, Sequence


def _agent_demo(cache, turns=7):
    """The page's multi-turn agent scenario: a fixed 1000-token system prompt,
    60 new user tokens per turn, 120 model tokens appended after each turn.
    Returns (prompt length, hit tokens) per turn."""
    sys_prompt = list(range(1000))
    history = list(sys_prompt)
    next_id = 0
    out = []
    for turn in range(1, turns + 1):
        user = list(range(90000 + turn * 100, 90000 + turn * 100 + 60))
        prompt = history + user
        hit, keys, _ = cache.lookup(prompt)
        cache.insert(keys, list(range(next_id, next_id + len(keys))))
        next_id += len(keys)
        out.append((len(prompt), hit))
        history = prompt + list(range(80000 + turn * 50, 80000 + turn * 50 + 120))
    return out


def test_oracle_agent_demo_closed_form():
    """Prompt t is 1060 + 180 (t - 1) tokens; every full block of prompt t-1
    is a prefix of prompt t, so turn t >= 2 hits 16 * floor(len_{t-1} / 16)."""
    got = _agent_demo(oracle.PrefixCache(4096, 16))
    lens = [1060 + 180 * (t - 1) for t in range(1, 8)]
    want = [(lens[0], 0)] + [(lens[t], 16 * (lens[t - 1] // 16)) for t in range(1, 7)]
    assert got == want
    assert [h for _, h in got] == [0, 1056, 1232, 1408, 1600, 1776, 1952]
    rates = [h / n for n, h in got]
    assert all(b > a for a, b in zip(rates[1:], rates[2:]))   # rises every turn
    assert rates[5] > 0.9                                     # above 90% by turn 6


def test_oracle_chain_property():
    """A key names its whole prefix: changing one token of block i changes
    keys i.. and leaves keys ..i-1; the hits then end at block i."""
    S = 8
    toks = list(range(100, 100 + 5 * S + 3))
    c = oracle.PrefixCache(64, S)
    _, keys, _ = c.lookup(toks)
    assert len(keys) == 5                       # full blocks only
    c.insert(keys, [10, 11, 12, 13, 14])
    alt = list(toks)
    alt[2 * S + 1] += 1
    hit, keys2, blocks = c.lookup(alt)
    assert keys2[:2] == keys[:2] and all(a != b for a, b in zip(keys2[2:], keys[2:]))
    assert hit == 2 * S and blocks == [10, 11]
    hit, _, blocks = c.lookup(toks)
    assert hit == 5 * S and blocks == [10, 11, 12, 13, 14]
    # the extra string separates equal token ids
    hit, keys3, _ = c.lookup(toks, extra="image:7")
    assert hit == 0 and keys3[0] != keys[0]
    assert (c.hits, c.misses) == (2, 2)


def test_oracle_lru_eviction_hand_traced():
    S = 2
    c = oracle.PrefixCache(3, S)
    _, ka, _ = c.lookup([1, 2, 3, 4])           # keys a0 a1
    assert c.insert(ka, [100, 101]) == []
    _, kb, _ = c.lookup([9, 9])                 # key b0
    assert c.insert(kb, [200]) == []            # table full: a0 a1 b0 (LRU order)
    hit, _, _ = c.lookup([1, 2, 7, 7])          # touches a0 -> order a1 b0 a0
    assert hit == 2
    _, kc, _ = c.lookup([5, 5])
    assert c.insert(kc, [300]) == [101]         # evicts a1
    assert set(c.table.values()) == {100, 200, 300}
    _, kd, _ = c.lookup([6, 6])
    assert c.insert(kd, [400]) == [200]         # then b0


def test_oracle_shared_sequence_refcounts():
    m = BlockManager(8, 4)
    a = Sequence(m, 0)
    for _ in range(8):
        a.append_slot()
    assert a.block_table == [7, 6]
    b = Sequence.shared(m, 1, a.block_table, 8)
    assert [m.ref_count[i] for i in (7, 6)] == [2, 2]
    slot, copy = b.append_slot()                # starts a new block, no copy
    assert copy is None and b.block_table == [7, 6, 5] and slot == 5 * 4
    c = Sequence.shared(m, 2, [7, 6], 6)        # ends inside the shared block 6
    slot, copy = c.append_slot()
    assert copy == (6, 4) and c.block_table == [7, 4] and slot == 4 * 4 + 2
    with pytest.raises(ValueError):
        Sequence.shared(m, 3, [0], 1)           # block 0 is free: holds nothing


# ---- native against the oracle -------------------------------------------------

@pytest.fixture(scope="module")
def pd():
    import paged_kv_attention_26_gb300 as pd
    pd.load()
    return pd


def test_native_agent_demo(pd):
    assert _agent_demo(pd.PrefixCache(4096, 16)) == _agent_demo(oracle.PrefixCache(4096, 16))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_native_matches_oracle_random_sessions(pd, seed):
    rng = random.Random(seed)
    S = rng.choice([4, 8, 16])
    cap = rng.choice([5, 17, 64])
    nat, ref = pd.PrefixCache(cap, S), oracle.PrefixCache(cap, S)
    bases = [[rng.randrange(50000) for _ in range(rng.randrange(0, 6 * S))] for _ in range(4)]
    next_id = 0
    for _ in range(60):
        toks = list(rng.choice(bases)) + [rng.randrange(50000) for _ in range(rng.randrange(8 * S))]
        extra = rng.choice(["", "", "img:3"])
        got, want = nat.lookup(toks, extra), ref.lookup(toks, extra)
        assert got == want
        ids = list(range(next_id, next_id + len(want[1])))
        next_id += len(ids)
        assert nat.insert(want[1], ids) == ref.insert(want[1], ids)
        assert len(nat) == len(ref.table)
    assert (nat.hits, nat.misses) == (ref.hits, ref.misses)


def test_native_shared_sequences_match_oracle(pd):
    S = 4
    nat, ref = pd.BlockManager(16, S), BlockManager(16, S)
    nat.add_seq(0)
    a = Sequence(ref, 0)
    for _ in range(10):
        assert nat.append_slot(0) == a.append_slot()
    nat.add_seq_shared(1, [a.block_table[0], a.block_table[1]], 8)
    b = Sequence.shared(ref, 1, a.block_table[:2], 8)
    nat.add_seq_shared(2, a.block_table[:3], 10)
    c = Sequence.shared(ref, 2, a.block_table[:3], 10)
    for _ in range(7):
        assert nat.append_slot(1) == b.append_slot()
        assert nat.append_slot(2) == c.append_slot()
    assert nat.block_table(1) == b.block_table and nat.block_table(2) == c.block_table
    nat.retain(a.block_table[0])
    ref.incref(a.block_table[0])
    for i in range(16):
        assert nat.ref_count(i) == ref.ref_count[i]
    nat.drop(a.block_table[0])
    ref.free(a.block_table[0])
    free = next(i for i in range(16) if ref.ref_count[i] == 0)
    with pytest.raises(pd.PDError):
        nat.add_seq_shared(3, [free], 1)        # a free block holds nothing
    with pytest.raises(pd.PDError):
        nat.retain(free)
    assert nat.usage == ref.usage
