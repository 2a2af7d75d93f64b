"""Pins of the float64 oracle against things other than itself: values the
pages print, closed forms, special cases with a textbook answer, and brute
force on tiny inputs.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from oracle import BlockManager, Sequence
from tests import brute_force as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---- 16-bit float decoding ----------------------------------------------

@pytest.mark.parametrize("dtype,tdt", [(oracle.F16, torch.float16), (oracle.BF16, torch.bfloat16)])
def test_all_16bit_patterns_decode_like_torch(dtype, tdt):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(tdt).to(torch.float64).numpy()
    got = oracle.to_double(bits.numpy(), dtype)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---- KV-bytes formula ----------------------------------------------------

def test_kv_bytes_printed_values():
    g = _load("kv_bytes.json")
    for c in g["cases"]:
        args = {k: c[k] for k in ("layers", "kv_heads", "head_dim", "seq_len", "dtype_bytes", "batch")}
        assert oracle.kv_cache_bytes(**args) == c["bytes"], c["cite"]
    for c in g["lower_bounds"]:
        args = {k: c[k] for k in ("layers", "kv_heads", "head_dim", "seq_len", "dtype_bytes", "batch")}
        assert oracle.kv_cache_bytes(**args) > c["more_than_bytes"], c["cite"]
    r = g["ratios"]
    assert oracle.kv_cache_bytes(1, r[0]["kv_heads_from"], 128, 1) == \
        r[0]["ratio"] * oracle.kv_cache_bytes(1, r[0]["kv_heads_to"], 128, 1)
    assert oracle.kv_cache_bytes(1, 8, 128, 1, r[1]["dtype_from"]) == \
        r[1]["ratio"] * oracle.kv_cache_bytes(1, 8, 128, 1, r[1]["dtype_to"])
    # the transfer of one 8K request equals the per-request cache size
    assert oracle.pd_transfer_bytes(8192, 32, 8, 128, 2) == 1 << 30


# ---- block manager --------------------------------------------------------

def test_block_manager_fork_demo():
    g = _load("block_manager_fork_demo.json")
    mgr = BlockManager(g["num_blocks"], g["block_size"])
    s = Sequence(mgr, 0)
    copies = [s.append_slot()[1] for _ in range(g["prompt_len"])]
    assert all(c is None for c in copies)
    assert s.block_table == g["prompt_blocks"]
    assert mgr.usage == g["usage_after_prompt"]
    kids = [s.fork(i + 1) for i in range(g["n_children"])]
    assert mgr.usage == g["usage_after_fork"]
    assert all(mgr.ref_count[b] == g["ref_count_shared_after_fork"] for b in s.block_table)
    res = [k.append_slot() for k in kids]
    assert [list(c) for _, c in res] == g["child_cow_copies"]
    assert [slot for slot, _ in res] == g["child_slots"]
    assert mgr.usage == g["usage_after_child_appends"]
    for b, rc in g["ref_count_after_appends"].items():
        assert mgr.ref_count[int(b)] == rc


@pytest.mark.parametrize("S", [8, 16, 32, 64])
def test_block_manager_invariants_random(S):
    rng = np.random.default_rng(S)
    mgr = BlockManager(400, S)
    seqs = {0: Sequence(mgr, 0)}
    next_id = 1
    for _ in range(3000):
        op = rng.integers(0, 10)
        sid = int(rng.choice(list(seqs)))
        s = seqs[sid]
        if op < 7:
            try:
                slot, copy = s.append_slot()
            except MemoryError:
                continue
            # the slot lies in the last block of the table at offset (len-1) % S
            assert slot == s.block_table[-1] * S + (s.length - 1) % S
            if copy is not None:
                assert copy[1] == s.block_table[-1] and mgr.ref_count[copy[1]] == 1
        elif op < 9 and len(seqs) < 12:
            used = mgr.num_blocks - len(mgr.free_ids)
            seqs[next_id] = s.fork(next_id)
            next_id += 1
            assert mgr.num_blocks - len(mgr.free_ids) == used  # fork copies nothing
        elif len(seqs) > 1:
            s.release()
            del seqs[sid]
        # waste <= S - 1 per sequence; ref counts equal table references
        for t in seqs.values():
            assert len(t.block_table) * S - t.length <= S - 1
            assert len(t.block_table) == (t.length + S - 1) // S
        refs = np.zeros(mgr.num_blocks, dtype=np.int64)
        for t in seqs.values():
            for b in t.block_table:
                refs[b] += 1
        assert np.array_equal(refs, np.array(mgr.ref_count))
        assert sorted(mgr.free_ids) == [b for b in range(mgr.num_blocks) if refs[b] == 0]
    # a block written by one sequence is never referenced by another
    # (the property copy-on-write exists for)


def test_block_manager_last_writer_in_place():
    mgr = BlockManager(32, 16)
    p = Sequence(mgr, 0)
    for _ in range(20):
        p.append_slot()
    kids = [p.fork(i) for i in range(1, 4)]
    p.release()
    res = [k.append_slot()[1] for k in kids]
    assert res[0] is not None and res[1] is not None and res[2] is None


def test_block_manager_exhaustion_raises():
    mgr = BlockManager(2, 4)
    s = Sequence(mgr, 0)
    for _ in range(8):
        s.append_slot()
    with pytest.raises(MemoryError):
        s.append_slot()


# ---- store and copy -----------------------------------------------------

def _u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def test_store_then_gather_returns_the_token():
    c = pd_inputs.tiny_decode()
    kc, vc = _u16(c.pool.key_cache), _u16(c.pool.value_cache)
    S = c.pool.S
    assert oracle.reshape_and_cache(c.new_key, c.new_value, kc, vc, c.slot_mapping, S) == 0
    bt = c.pool.block_tables.numpy()
    for n, i in enumerate(range(c.B)):
        t = int(c.pool.context_lens[i]) - 1
        slot = oracle.slot_of(bt[i], t, S)
        assert slot == int(c.slot_mapping[n])
        blk, off = bt[i][t // S], t % S
        assert np.array_equal(kc[blk, :, off, :], _u16(c.new_key[n]))
        assert np.array_equal(vc[blk, :, off, :], _u16(c.new_value[n]))
    # everything else is untouched (bit compare, NaN payloads included)
    mask = np.ones(kc.shape[:3], dtype=bool)
    for n, s in enumerate(c.slot_mapping.tolist()):
        mask[s // S, :, s % S] = False
    assert np.array_equal(kc[mask], _u16(c.pool.key_cache)[mask])


def test_store_skips_negative_and_counts_out_of_range():
    kc = np.zeros((4, 2, 8, 16), dtype=np.uint16)
    vc = kc.copy()
    key = torch.ones(3, 2, 16, dtype=torch.float16)
    slots = torch.tensor([-1, 4 * 8, 5], dtype=torch.int64)
    assert oracle.reshape_and_cache(key, key, kc, vc, slots, 8) == 1
    assert kc.sum() == 2 * 16 * 0x3C00
    assert (kc[0, :, 5, :] == 0x3C00).all()


def test_copy_blocks_brute_force():
    rng = np.random.default_rng(1)
    L, NB, Hk, S, D = 3, 10, 2, 8, 16
    kcs = [rng.integers(0, 65535, (NB, Hk, S, D), dtype=np.uint16) for _ in range(L)]
    vcs = [rng.integers(0, 65535, (NB, Hk, S, D), dtype=np.uint16) for _ in range(L)]
    ref_k = [k.copy() for k in kcs]
    ref_v = [v.copy() for v in vcs]
    pairs = np.array([[1, 7], [2, 3], [9, 0]], dtype=np.int64)
    assert oracle.copy_blocks(kcs, vcs, pairs) == 0
    for l in range(L):
        for s, d in pairs:
            ref_k[l][d] = ref_k[l][s]
            ref_v[l][d] = ref_v[l][s]
        assert np.array_equal(kcs[l], ref_k[l]) and np.array_equal(vcs[l], ref_v[l])


def _coded_pools(L, NB, Hk, S, D):
    """Pools whose every element encodes its own (layer, K/V, block, head,
    offset, dim) coordinates, so a wrong index shows up as a wrong code."""
    idx = np.arange(L * 2 * NB * Hk * S * D, dtype=np.int64).reshape(L, 2, NB, Hk, S, D)
    assert idx.max() < 65536
    code = idx.astype(np.uint16)
    return [code[l, 0].copy() for l in range(L)], [code[l, 1].copy() for l in range(L)], code


def test_kv_pack_closed_form():
    """staging[l][kv][i] is block ids[i] of layer l's K (kv 0) or V (kv 1) pool,
    element for element: a closed form of the layer-major layout."""
    L, NB, Hk, S, D = 3, 7, 2, 4, 8
    kcs, vcs, code = _coded_pools(L, NB, Hk, S, D)
    ids = np.array([5, 0, 3, 6], dtype=np.int32)
    st, bad = oracle.kv_pack(kcs, vcs, ids)
    assert bad == 0 and st.shape == (L, 2, len(ids), Hk, S, D)
    for l in range(L):
        for kv in range(2):
            for i, b in enumerate(ids):
                base = (((l * 2 + kv) * NB + int(b)) * Hk) * S * D
                expect = base + np.arange(Hk * S * D).reshape(Hk, S, D)
                assert np.array_equal(st[l, kv, i].astype(np.int64), expect)
    # layer l's part is one contiguous run starting at l * 2 * nblk * Hk*S*D
    flat = st.reshape(-1)
    run = 2 * len(ids) * Hk * S * D
    assert np.array_equal(flat[run:2 * run], st[1].reshape(-1))


def test_kv_pack_unpack_moves_blocks_between_pools():
    """Pack from one pool's blocks, unpack into another pool's different
    blocks: the receiving blocks hold the sender's data bit for bit, every
    other receiving block is untouched, and out-of-range ids are skipped."""
    rng = np.random.default_rng(3)
    L, NB, Hk, S, D = 2, 9, 2, 8, 16
    src_k = [rng.integers(0, 65535, (NB, Hk, S, D), dtype=np.uint16) for _ in range(L)]
    src_v = [rng.integers(0, 65535, (NB, Hk, S, D), dtype=np.uint16) for _ in range(L)]
    dst_k = [rng.integers(0, 65535, (NB, Hk, S, D), dtype=np.uint16) for _ in range(L)]
    dst_v = [rng.integers(0, 65535, (NB, Hk, S, D), dtype=np.uint16) for _ in range(L)]
    before_k = [k.copy() for k in dst_k]
    before_v = [v.copy() for v in dst_v]
    send = np.array([4, 1, 8], dtype=np.int32)
    recv = np.array([0, 7, 2], dtype=np.int32)
    st, bad = oracle.kv_pack(src_k, src_v, send)
    assert bad == 0
    assert oracle.kv_unpack(st, dst_k, dst_v, recv) == 0
    for l in range(L):
        for b in range(NB):
            if b in recv:
                j = list(recv).index(b)
                assert np.array_equal(dst_k[l][b], src_k[l][send[j]])
                assert np.array_equal(dst_v[l][b], src_v[l][send[j]])
            else:
                assert np.array_equal(dst_k[l][b], before_k[l][b])
                assert np.array_equal(dst_v[l][b], before_v[l][b])
    st2, bad2 = oracle.kv_pack(src_k, src_v, np.array([2, -1, NB], dtype=np.int32))
    assert bad2 == 2
    for l in range(L):
        assert np.array_equal(st2[l, 0, 0], src_k[l][2]) and np.array_equal(st2[l, 1, 0], src_v[l][2])
    assert not st2[:, :, 1:].any()               # skipped slabs stay as allocated (zeros)


# ---- decode attention -----------------------------------------------------

def _stored(c):
    """A decode case with its new tokens stored, as uint16 numpy pools."""
    kc, vc = _u16(c.pool.key_cache), _u16(c.pool.value_cache)
    oracle.reshape_and_cache(c.new_key, c.new_value, kc, vc, c.slot_mapping, c.pool.S)
    return kc, vc


def _as_tensor(a, dtype):
    return torch.from_numpy(a.view(np.int16)).view(dtype)


def test_decode_matches_brute_force_tiny():
    c = pd_inputs.tiny_decode()
    kc, vc = _stored(c)
    dt = oracle.F16
    got = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale, dt)
    ref = bf.decode(c.q, _as_tensor(kc, c.dtype), _as_tensor(vc, c.dtype),
                    c.pool.block_tables, c.pool.context_lens, c.scale)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_decode_matches_brute_force_bf16_gqa_variants():
    for (H, Hk, S) in [(4, 4, 8), (8, 1, 32), (6, 2, 64), (8, 2, 16)]:
        c = pd_inputs.decode_case("v", 3, [5, 64, 65, 130], H, Hk, 64, S, torch.bfloat16)
        kc, vc = _stored(c)
        got = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens,
                            c.scale, oracle.BF16)
        ref = bf.decode(c.q, _as_tensor(kc, c.dtype), _as_tensor(vc, c.dtype),
                        c.pool.block_tables, c.pool.context_lens, c.scale)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_ctx1_returns_v_exactly():
    c = pd_inputs.decode_case("one", 5, [1, 1, 1], 8, 2, 64, 16, torch.float16)
    kc, vc = _stored(c)
    got = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                        oracle.F16)
    v = c.new_value.to(torch.float64).numpy()          # [B, Hk, D]
    for h in range(8):
        assert np.array_equal(got[:, h], v[:, h // 4])


def test_equal_keys_give_mean_of_v_and_equal_values_give_that_row():
    c = pd_inputs.decode_case("eq", 6, [40, 3], 4, 2, 64, 8, torch.float16, poison=False,
                              store_last=False)
    kc, vc = _u16(c.pool.key_cache), _u16(c.pool.value_cache)
    kc[:] = kc[0, 0, 0]                       # every key identical
    out = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                        oracle.F16)
    v64 = _as_tensor(vc, c.dtype).to(torch.float64).numpy()
    for i in range(2):
        n = int(c.pool.context_lens[i])
        V = bf.gather(v64, c.pool.block_tables[i].numpy(), n)
        for h in range(4):
            np.testing.assert_allclose(out[i, h], V[:, h // 2].mean(0), rtol=1e-12, atol=1e-13)
    kc2, vc2 = _u16(c.pool.key_cache), _u16(c.pool.value_cache)
    vc2[:] = vc2[3, 1, 2]                     # every value row identical
    out = oracle.decode(c.q, kc2, vc2, c.pool.block_tables, c.pool.context_lens, c.scale,
                        oracle.F16)
    row = _as_tensor(vc2[3, 1, 2], c.dtype).to(torch.float64).numpy()
    np.testing.assert_allclose(out, np.broadcast_to(row, out.shape), rtol=1e-14, atol=1e-14)


def test_mha_and_mqa_reductions():
    """G = H/Hk grouping: MQA (Hk=1) equals MHA over a pool in which every kv
    head holds the same data; MHA head h reads kv head h."""
    c = pd_inputs.decode_case("mqa", 7, [9, 50], 4, 1, 64, 16, torch.bfloat16, poison=False,
                              store_last=False)
    kc, vc = _u16(c.pool.key_cache), _u16(c.pool.value_cache)
    mqa = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                        oracle.BF16)
    kc4, vc4 = np.repeat(kc, 4, axis=1), np.repeat(vc, 4, axis=1)
    mha = oracle.decode(c.q, kc4, vc4, c.pool.block_tables, c.pool.context_lens, c.scale,
                        oracle.BF16)
    assert np.array_equal(mqa, mha)
    # MHA with distinct kv heads: head h must follow kv head h
    kc4[:, 2] = kc4[:, 0]
    vc4[:, 2] = vc4[:, 0] * 0 + vc4[:, 1]
    mha2 = oracle.decode(c.q, kc4, vc4, c.pool.block_tables, c.pool.context_lens, c.scale,
                         oracle.BF16)
    ref = bf.decode(c.q, _as_tensor(kc4, c.dtype), _as_tensor(vc4, c.dtype),
                    c.pool.block_tables, c.pool.context_lens, c.scale)
    np.testing.assert_allclose(mha2, ref, rtol=1e-12, atol=1e-12)


def test_block_permutation_invariance():
    c = pd_inputs.decode_case("perm", 8, [7, 100, 31], 8, 2, 64, 8, torch.float16)
    kc, vc = _stored(c)
    out = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                        oracle.F16)
    NB = kc.shape[0]
    perm = np.random.default_rng(0).permutation(NB)      # new id of old block b
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = torch.from_numpy(perm[c.pool.block_tables.numpy()].astype(np.int32))
    out2 = oracle.decode(c.q, kc2, vc2, bt2, c.pool.context_lens, c.scale, oracle.F16)
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("part", [16, 48, 64, 512])
def test_split_partitions_merge_to_unsplit(part):
    c = pd_inputs.decode_case("split", 9, [1, 15, 16, 17, 200, 513], 8, 2, 64, 16,
                              torch.bfloat16, key_outlier_frac=0.05)
    kc, vc = _stored(c)
    a = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale, oracle.BF16)
    b = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                      oracle.BF16, split_part=part)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_zero_context_gives_zeros():
    c = pd_inputs.decode_case("z", 10, [0, 5], 4, 2, 64, 16, torch.float16)
    kc, vc = _stored(c)
    out = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                        oracle.F16)
    assert (out[0] == 0).all() and np.isfinite(out[1]).all()


def test_bad_block_id_is_reported():
    c = pd_inputs.decode_case("bad", 11, [20], 4, 2, 64, 16, torch.float16)
    kc, vc = _stored(c)
    bt = c.pool.block_tables.clone()
    bt[0, 1] = kc.shape[0]
    with pytest.raises(ValueError):
        oracle.decode(c.q, kc, vc, bt, c.pool.context_lens, c.scale, oracle.F16)


# ---- chunked prefill ------------------------------------------------------

def _mixed_small(seed=12, S=16, dtype=torch.bfloat16):
    return pd_inputs.mixed_case(seed, [0, 5, 40], [1, 19, 33], [3, 70], 8, 2, 64, S, dtype)


def _stored_mixed(m):
    kc, vc = _u16(m.pool.key_cache), _u16(m.pool.value_cache)
    oracle.reshape_and_cache(m.new_key, m.new_value, kc, vc, m.slot_mapping, m.pool.S)
    return kc, vc


def test_prefill_matches_brute_force():
    m = _mixed_small()
    kc, vc = _stored_mixed(m)
    bt = m.pool.block_tables[: m.Bp]
    cl = m.pool.context_lens[: m.Bp]
    got = oracle.prefill(m.q_prefill, m.cu_q_lens, kc, vc, bt, cl, m.scale, oracle.BF16)
    ref = bf.prefill(m.q_prefill, m.cu_q_lens, _as_tensor(kc, m.dtype), _as_tensor(vc, m.dtype),
                     bt, cl, m.scale)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # sampled rows agree with the full evaluation
    rows = np.array([0, 5, 17, 8 * 20 + 3, got.shape[0] * 8 - 1])
    part = oracle.prefill(m.q_prefill, m.cu_q_lens, kc, vc, bt, cl, m.scale, oracle.BF16,
                          rows=rows)
    assert np.array_equal(part, got.reshape(-1, 64)[rows])


def test_prefill_special_cases_reduce_to_decode():
    m = _mixed_small()
    kc, vc = _stored_mixed(m)
    bt = m.pool.block_tables[: m.Bp]
    cl = m.pool.context_lens[: m.Bp]
    pre = oracle.prefill(m.q_prefill, m.cu_q_lens, kc, vc, bt, cl, m.scale, oracle.BF16)
    cu = m.cu_q_lens.tolist()
    for i in range(m.Bp):
        # the chunk's last query row is a decode step at ctx = P + C
        q_last = m.q_prefill[cu[i + 1] - 1].unsqueeze(0)
        dec = oracle.decode(q_last, kc, vc, bt[i:i + 1], cl[i:i + 1], m.scale, oracle.BF16)
        assert np.array_equal(pre[cu[i + 1] - 1], dec[0])
    # sequence 0 has P = 0, C = 1: attention to its single key returns V exactly
    v = m.new_value[0].to(torch.float64).numpy()
    for h in range(8):
        assert np.array_equal(pre[0, h], v[h // 4])


def test_prefill_causality():
    """Changing the keys/values at positions after query j leaves row j as is."""
    m = _mixed_small(seed=13)
    kc, vc = _stored_mixed(m)
    bt = m.pool.block_tables[: m.Bp]
    cl = m.pool.context_lens[: m.Bp]
    a = oracle.prefill(m.q_prefill, m.cu_q_lens, kc, vc, bt, cl, m.scale, oracle.BF16)
    i, S = 2, m.pool.S
    P = int(cl[i]) - 33
    j = 10
    for t in range(P + j + 1, int(cl[i])):
        blk, off = int(bt[i, t // S]), t % S
        kc[blk, :, off] ^= 0x0100
        vc[blk, :, off] ^= 0x0100
    b = oracle.prefill(m.q_prefill, m.cu_q_lens, kc, vc, bt, cl, m.scale, oracle.BF16)
    row = int(m.cu_q_lens[i]) + j
    assert np.array_equal(a[: row + 1], b[: row + 1])
    assert not np.array_equal(a[row + 1:int(m.cu_q_lens[i + 1])], b[row + 1:int(m.cu_q_lens[i + 1])])


def test_prefill_scale_enters_once():
    """softmax(scale * s): with scale -> 0 the output is the mean of V."""
    m = _mixed_small(seed=14)
    kc, vc = _stored_mixed(m)
    bt = m.pool.block_tables[: m.Bp]
    cl = m.pool.context_lens[: m.Bp]
    out = oracle.prefill(m.q_prefill, m.cu_q_lens, kc, vc, bt, cl, 0.0, oracle.BF16)
    v64 = _as_tensor(vc, m.dtype).to(torch.float64).numpy()
    i = 2
    P = int(cl[i]) - 33
    V = bf.gather(v64, bt[i].numpy(), int(cl[i]))
    for j in (0, 32):
        np.testing.assert_allclose(out[int(m.cu_q_lens[i]) + j, 5], V[: P + j + 1, 1].mean(0),
                                   rtol=1e-12, atol=1e-13)
    assert math.isclose(m.scale, 1 / 8)


# ---- FP8 (E4M3) KV cache -----------------------------------------------------

def test_e4m3_codes_decode_like_torch():
    """All 256 codes against torch's float8_e4m3fn (a library decoder), plus
    the format's fixed points: +-0, NaN at S.1111.111, largest 448, smallest
    subnormal 2^-9."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan]) and np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and np.isnan(got).sum() == 2
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0 and got[1] == 2.0 ** -9
    assert got[0] == 0.0 and math.copysign(1, got[0x80]) == -1


def test_e4m3_encode_round_trip_ties_and_saturation():
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    for c in finite:                                    # every value maps to its own code
        assert oracle.e4m3_encode(oracle.e4m3_to_double(c)) == c, c
    for c in range(0x7E):                               # midpoints go to the even code
        lo, hi = oracle.e4m3_to_double(c), oracle.e4m3_to_double(c + 1)
        mid = np.float32((lo + hi) / 2)
        if float(mid) != (lo + hi) / 2:
            continue                                    # midpoint not a float32: no tie
        assert oracle.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1), (c, lo, hi)
    assert oracle.e4m3_encode(1e6) == 0x7E and oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E and oracle.e4m3_encode(float("nan")) == 0x7F
    # within range, rounding agrees with torch's float32 -> float8_e4m3fn cast
    g = torch.Generator().manual_seed(11)
    y = (torch.randn(4000, generator=g) * torch.exp2(torch.randint(-12, 9, (4000,), generator=g).float()))
    y = y.clamp(-448, 448)
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in y.numpy()], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_fp8_store_matches_torch_quantisation():
    """Stored code = the float32 product x * (1 / scale[h]) cast to E4M3 (torch
    as the reference cast), at the slot the paging rule names."""
    g = torch.Generator().manual_seed(12)
    T, Hk, D, S, NB = 10, 3, 16, 8, 6
    key = torch.randn(T, Hk, D, generator=g).to(torch.bfloat16)
    value = (3 * torch.randn(T, Hk, D, generator=g)).to(torch.bfloat16)
    ks = torch.tensor([0.01, 0.5, 2.0], dtype=torch.float32)
    vs = torch.tensor([0.03, 0.125, 1.0], dtype=torch.float32)
    slots = torch.randperm(NB * S, generator=g)[:T].to(torch.int64)
    slots[4] = -1
    kc = np.zeros((NB, Hk, S, D), dtype=np.uint8)
    vc = np.zeros_like(kc)
    assert oracle.reshape_and_cache_fp8(key, value, oracle.BF16, kc, vc, slots, ks, vs, S) == 0
    for n in range(T):
        s = int(slots[n])
        if s < 0:
            continue
        for h in range(Hk):
            for x, sc, pool in ((key, ks, kc), (value, vs, vc)):
                y = x[n, h].float() * (torch.tensor(1.0) / sc[h])
                ref = y.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                assert np.array_equal(pool[s // S, h, s % S], ref)


def test_fp8_decode_reduces_to_bf16_decode():
    """With scales 1 every E4M3 value is exactly a bf16 value: FP8 decode must
    equal the 16-bit decode oracle over the same values; a K scale of 2 equals
    doubling q, a V scale of 2 doubles the output."""
    c = pd_inputs.decode_case("fp8pin", 3, [1, 9, 40, 70], 8, 2, 16, 8, torch.bfloat16,
                              poison=False, store_last=False)
    g = torch.Generator().manual_seed(13)
    NB, Hk, S, D = c.pool.key_cache.shape
    kc8 = torch.randint(0, 256, (NB, Hk, S, D), generator=g, dtype=torch.int32).to(torch.uint8)
    vc8 = torch.randint(0, 256, (NB, Hk, S, D), generator=g, dtype=torch.int32).to(torch.uint8)
    for t in (kc8, vc8):
        t[(t & 0x7F) == 0x7F] = 0x38                    # no NaN codes
    kb = kc8.view(torch.float8_e4m3fn).to(torch.bfloat16)
    vb = vc8.view(torch.float8_e4m3fn).to(torch.bfloat16)
    assert torch.equal(kb.float(), kc8.view(torch.float8_e4m3fn).float())   # exact in bf16
    one = np.ones(Hk, dtype=np.float32)
    bt, cl = c.pool.block_tables, c.pool.context_lens
    ref = oracle.decode(c.q, kb, vb, bt, cl, c.scale, oracle.BF16)
    got = oracle.decode_fp8(c.q, oracle.BF16, kc8.numpy(), vc8.numpy(), one, one, bt, cl, c.scale)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)
    got2 = oracle.decode_fp8(c.q, oracle.BF16, kc8.numpy(), vc8.numpy(), 2 * one, 2 * one, bt, cl,
                             c.scale)
    ref2 = oracle.decode((c.q.float() * 2).to(torch.bfloat16), kb, vb, bt, cl, c.scale, oracle.BF16)
    assert np.allclose(got2, 2 * ref2, rtol=0, atol=1e-12)
    got3 = oracle.decode_fp8(c.q, oracle.BF16, kc8.numpy(), vc8.numpy(), one, 4 * one, bt, cl,
                             c.scale)
    assert np.allclose(got3, 4 * ref, rtol=0, atol=1e-12)


def test_fp8_concurrency_golden():
    d = json.load(open(os.path.join(GOLDEN, "kv_bytes.json")))
    for case in d["concurrency"]:
        args = (case["weights_gb"], case["total_gb"], case["reserve_gb"])
        assert oracle.concurrency_limit(case["kv_gb_fp16"], *args) == case["fp16"]
        assert oracle.concurrency_limit(case["kv_gb_fp16"] / 2, *args) == case["fp8"]
