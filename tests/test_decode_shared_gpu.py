"""Shared-prefix decode (pd_paged_attention_decode_shared) against the oracle.

The operation is plain decode attention (nanoPD page "自定义CUDA分页注意力内
核"), so the oracle is ``oracle.decode``; the batches are forks that share a
prompt's blocks (tutorial page "LLM 推理服务引擎深度拆解", section 2.3: fork
shares every block, a written shared block is copied first).  Covers the
copy-on-write fork stress at every block size, random groups (sizes 1-32, no
sharing, empty contexts, tails of 0..several stages), every column layout
(group sizes giving 8 to 32 columns), both element types and head dims, many
small groups per CTA (the walk ring wrapping), block-permutation
bit-identity, the device check of the caller's sharing promise, and the
chained step eagerly and replayed from a CUDA graph.
"""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import assert_close, device_err, odt, u16
from tests.test_store_copy_gpu import OracleBM, fork_flow

pytestmark = pytest.mark.gpu


def _run(pd, c, groups=None, max_group=None, err=None, kc=None, vc=None, store=True):
    """Store (if any), then the shared-prefix decode; returns out on the device."""
    dev = torch.device("cuda")
    if kc is None:
        kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    if store and c.slot_mapping.numel():
        pd.pd_reshape_and_cache(c.new_key.to(dev), c.new_value.to(dev), kc, vc,
                                c.slot_mapping.to(dev))
    gs, sl = groups if groups is not None else (c.group_starts, c.shared_lens)
    if max_group is None:
        max_group = int((gs[1:] - gs[:-1]).max())
    q = c.q.to(dev)
    out = torch.full_like(q, float("nan"))
    ws = pd.decode_shared_workspace(sl.numel(), max_group, c.H, c.Hk, c.D)
    pd.pd_paged_attention_decode_shared(out, q, kc, vc, c.pool.block_tables.to(dev),
                                        c.pool.context_lens.to(dev), c.max_context_len, c.scale,
                                        gs.to(dev), sl.to(dev), max_group, ws, dev_err=err)
    return out, kc, vc


def _oracle(c, rows=None):
    kc, vc = u16(c.pool.key_cache), u16(c.pool.value_cache)
    if c.slot_mapping.numel():
        oracle.reshape_and_cache(c.new_key, c.new_value, kc, vc, c.slot_mapping, c.pool.S)
    return oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                         odt(c.dtype), rows=rows)


def _check(pd, c, what, **kw):
    err = device_err()
    out, _, _ = _run(pd, c, err=err, **kw)
    torch.cuda.synchronize()
    assert err.item() == 0, f"{what}: device error {err.item()}"
    assert_close(out.cpu(), _oracle(c), what)
    return out


@pytest.mark.parametrize("S", [8, 16, 32, 64])
def test_cow_fork_stress_shared(cuda_lib, S):
    """The copy-on-write fork stress: 32 prompts x 8 forks, copy_blocks, one
    stored token per fork, then the shared-prefix decode (groups found by
    pd_find_shared_prefixes), against the oracle and against the per-sequence
    decode."""
    pd = cuda_lib
    fc = pd_inputs.cow_fork_stress(S)
    tables, ctx, slots, pairs = fork_flow(fc, OracleBM)
    dev = torch.device("cuda")
    kg, vg = fc.key_cache.to(dev), fc.value_cache.to(dev)
    if pairs:
        pd.pd_copy_blocks([kg], [vg], torch.tensor(pairs, dtype=torch.int64, device=dev))
    pd.pd_reshape_and_cache(fc.new_key.to(dev), fc.new_value.to(dev), kg, vg,
                            torch.tensor(slots, dtype=torch.int64, device=dev))
    mb = max(len(t) for t in tables)
    bt = torch.zeros(len(tables), mb, dtype=torch.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    cl = torch.tensor(ctx, dtype=torch.int32)
    gs, sl = pd.find_shared_prefixes(bt, cl, S, max_group=8)
    assert gs.numel() == 33
    n, mcl = len(tables), max(ctx)
    q = fc.q.to(dev)
    out = torch.full_like(q, float("nan"))
    err = device_err()
    ws = pd.decode_shared_workspace(32, 8, fc.H, fc.Hk, fc.D)
    pd.pd_paged_attention_decode_shared(out, q, kg, vg, bt.to(dev), cl.to(dev), mcl, fc.scale,
                                        gs.to(dev), sl.to(dev), 8, ws, dev_err=err)
    ref_dec = torch.empty_like(q)
    pd.pd_paged_attention_decode(ref_dec, q, kg, vg, bt.to(dev), cl.to(dev), mcl, fc.scale,
                                 pd.decode_workspace(n, fc.H, fc.D, mcl), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rk, rv = u16(fc.key_cache), u16(fc.value_cache)
    if pairs:
        oracle.copy_blocks([rk], [rv], np.array(pairs, dtype=np.int64))
    oracle.reshape_and_cache(fc.new_key, fc.new_value, rk, rv, torch.tensor(slots), S)
    rows = (0, n * fc.H) if S == 16 else (0, 24 * fc.H)     # three whole groups elsewhere
    ref = oracle.decode(fc.q, rk, rv, bt, cl, fc.scale, odt(fc.dtype), rows=rows)
    got = out.cpu().reshape(-1, fc.D)[rows[0]:rows[1]]
    assert_close(got, ref.reshape(-1, fc.D)[rows[0]:rows[1]], f"cow shared S{S}")
    # both GPU paths agree with each other within the same tolerance
    d = (out.float() - ref_dec.float()).abs()
    assert bool((d <= 2e-3 + 1e-2 * ref_dec.float().abs()).all())


GROUPS = [
    (100, [101, 101, 105, 170]),        # partial prompt block, tails of 1-2 stages
    (0, [0, 5, 70]),                     # no sharing; an empty context in the group
    (64, [64]),                          # a group of one, no tail
    (130, [130, 131, 200, 131, 400, 131, 132, 135]),   # eight forks
    (1000, [1001, 1064, 1065, 1200, 1001]),
    (17, [17, 18]),
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("H,Hk,D", [(8, 2, 64), (32, 8, 128), (16, 2, 128), (12, 4, 64)])
def test_random_groups(cuda_lib, dtype, H, Hk, D):
    for S in (8, 16, 64):
        c = pd_inputs.forked_decode(f"groups S{S}", 40 + S, GROUPS, H, Hk, D, S, dtype)
        _check(cuda_lib, c, f"groups H{H} Hk{Hk} D{D} S{S} {dtype}")


@pytest.mark.parametrize("G,M", [(4, 2), (4, 3), (4, 4), (4, 5), (4, 8), (2, 16), (1, 32),
                                 (8, 4), (3, 7)])
def test_column_layouts(cuda_lib, G, M):
    """Group sizes that give 1, 2 and 4 column tiles (GH x M columns, GH the
    largest divisor of G with GH x M <= 32), including a partly empty fourth
    tile, against the oracle."""
    rng = np.random.default_rng(G * 100 + M)
    groups = []
    for gi in range(5):
        P = int(rng.integers(0, 700))
        m = int(rng.integers(1, M + 1)) if gi else M
        groups.append((P, [P + int(rng.integers(0, 90)) for _ in range(m)]))
    Hk = 2
    c = pd_inputs.forked_decode(f"layout G{G} M{M}", 7, groups, G * Hk, Hk, 128, 16,
                                torch.bfloat16)
    _check(cuda_lib, c, f"layout G{G} M{M}", max_group=M)


@pytest.mark.parametrize("members", [1, 2])
def test_many_small_groups_per_cta(cuda_lib, members):
    """400 groups of one or two short contexts (at most two 64-token stages
    each): every CTA's range spans about ten groups, so the per-CTA walk ring
    (four positions) wraps several times and most stages start a new piece."""
    rng = np.random.default_rng(400 + members)
    groups = []
    for _ in range(400):
        P = int(rng.integers(0, 48)) if members > 1 else 0
        groups.append((P, [P + int(rng.integers(1, 60)) for _ in range(members)]))
    c = pd_inputs.forked_decode(f"small groups x{members}", 11 + members, groups, 32, 8, 128,
                                16, torch.float16)
    _check(cuda_lib, c, f"400 small groups x{members}", max_group=members)


def test_bit_identical_under_block_permutation(cuda_lib):
    c = pd_inputs.forked_decode("perm", 3, GROUPS, 32, 8, 128, 16, torch.bfloat16)
    a = _check(cuda_lib, c, "perm base")
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(c.pool.NB, generator=g)
    c.pool.key_cache = c.pool.key_cache[torch.argsort(perm)].clone()
    c.pool.value_cache = c.pool.value_cache[torch.argsort(perm)].clone()
    inv = perm.to(torch.int32)            # old id i -> new id perm[i]
    c.pool.block_tables = inv[c.pool.block_tables.long()]
    c.slot_mapping = perm[c.slot_mapping // c.pool.S] * c.pool.S + c.slot_mapping % c.pool.S
    b = _check(cuda_lib, c, "perm permuted")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_repeat_runs_identical(cuda_lib):
    """Same inputs twice (the second launch over the first's workspace): the
    same bits (fixed merge order, no atomics on results)."""
    c = pd_inputs.forked_decode("repeat", 5, GROUPS, 32, 8, 128, 32, torch.float16)
    a = _check(cuda_lib, c, "repeat 1")
    b = _check(cuda_lib, c, "repeat 2")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_promise_checked_on_device(cuda_lib):
    """A member whose table differs inside the declared shared prefix, and a
    group layout that does not cover the batch, flag PD_DEVERR_SHARED_PREFIX
    (no fault: the reads stay inside the tables and the pool)."""
    pd = cuda_lib
    c = pd_inputs.forked_decode("promise", 11, GROUPS, 8, 2, 64, 16, torch.float16)
    bad = c.pool.block_tables.clone()
    r = int(c.group_starts[3]) + 2              # third fork of the eight-fork group
    bad[r, 3] = bad[r, 7]                        # inside the 128 shared tokens
    c2 = c
    c2.pool.block_tables = bad
    err = device_err()
    _run(pd, c2, err=err)
    torch.cuda.synchronize()
    assert err.item() & pd.PD_DEVERR_SHARED_PREFIX
    c = pd_inputs.forked_decode("promise2", 11, GROUPS, 8, 2, 64, 16, torch.float16)
    gs = c.group_starts.clone()
    gs[-1] -= 1                                  # the last sequence is in no group
    err = device_err()
    _run(pd, c, groups=(gs, c.shared_lens), err=err, max_group=8)
    torch.cuda.synchronize()
    assert err.item() & pd.PD_DEVERR_SHARED_PREFIX


def test_declared_prefix_longer_than_a_member(cuda_lib):
    """A declared shared length beyond the shortest member's context is cut to
    it (and to whole blocks): still the plain decode result, no flag."""
    c = pd_inputs.forked_decode("cut", 13, [(300, [300, 310, 301]), (40, [41, 90])], 8, 2, 64,
                                16, torch.bfloat16)
    sl = torch.tensor([5000, 45], dtype=torch.int32)
    _check(cuda_lib, c, "declared prefix cut", groups=(c.group_starts, sl))


@pytest.mark.parametrize("S", [8, 16, 64])
def test_step_shared_matches_separate_calls(cuda_lib, S):
    """pd_decode_step_shared (copies -> store -> decode as dependent grids)
    leaves the pools bit-exact as the oracle's copy and store do, and its
    output bit-identical to pd_copy_blocks + pd_reshape_and_cache +
    pd_paged_attention_decode_shared on the same stream; also with no copies
    and with no stored tokens."""
    pd = cuda_lib
    fc = pd_inputs.cow_fork_stress(S, n_prompts=12)
    tables, ctx, slots, pairs = fork_flow(fc, OracleBM)
    dev = torch.device("cuda")
    mb = max(len(t) for t in tables)
    bt = torch.zeros(len(tables), mb, dtype=torch.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    cl = torch.tensor(ctx, dtype=torch.int32)
    gs, sl = pd.find_shared_prefixes(bt, cl, S, max_group=8)
    n, mcl = len(tables), max(ctx)
    q = fc.q.to(dev)
    nk, nv = fc.new_key.to(dev), fc.new_value.to(dev)
    sm = torch.tensor(slots, dtype=torch.int64, device=dev)
    pr = torch.tensor(pairs, dtype=torch.int64, device=dev).view(-1, 2)
    btd, cld, gsd, sld = bt.to(dev), cl.to(dev), gs.to(dev), sl.to(dev)
    ws = pd.decode_shared_workspace(sl.numel(), 8, fc.H, fc.Hk, fc.D)
    err = device_err()
    for with_pairs, with_store in ((True, True), (False, True), (True, False)):
        k1, v1 = fc.key_cache.to(dev), fc.value_cache.to(dev)
        k2, v2 = fc.key_cache.to(dev), fc.value_cache.to(dev)
        o1, o2 = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
        if with_pairs:
            pd.pd_copy_blocks([k1], [v1], pr, dev_err=err)
        if with_store:
            pd.pd_reshape_and_cache(nk, nv, k1, v1, sm, dev_err=err)
        pd.pd_paged_attention_decode_shared(o1, q, k1, v1, btd, cld, mcl, fc.scale, gsd, sld, 8,
                                            ws, dev_err=err)
        pd.pd_decode_step_shared(o2, q, k2, v2, btd, cld, mcl, fc.scale, gsd, sld, 8,
                                 key=nk if with_store else None,
                                 value=nv if with_store else None,
                                 slot_mapping=sm if with_store else None,
                                 block_mapping=pr if with_pairs else None, workspace=ws,
                                 dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert np.array_equal(u16(k1), u16(k2))
        assert np.array_equal(u16(v1), u16(v2))
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        if with_pairs and with_store:
            rk, rv = u16(fc.key_cache), u16(fc.value_cache)
            oracle.copy_blocks([rk], [rv], np.array(pairs, dtype=np.int64))
            oracle.reshape_and_cache(fc.new_key, fc.new_value, rk, rv, torch.tensor(slots), S)
            assert np.array_equal(u16(k2), rk) and np.array_equal(u16(v2), rv)
            rows = (0, 16 * fc.H)
            ref = oracle.decode(fc.q, rk, rv, bt, cl, fc.scale, odt(fc.dtype), rows=rows)
            assert_close(o2.cpu().reshape(-1, fc.D)[rows[0]:rows[1]],
                         ref.reshape(-1, fc.D)[rows[0]:rows[1]], f"cow step S{S}")


def test_step_shared_in_a_cuda_graph(cuda_lib):
    """pd_decode_step_shared captured once in a CUDA graph and replayed over
    fresh pools (the copies and the store rewrite them each time): every
    replay gives the bits of the eager step (tensor memory is allocated and
    freed inside each launch, the arrival counters are left at zero)."""
    pd = cuda_lib
    S = 16
    fc = pd_inputs.cow_fork_stress(S, n_prompts=8)
    tables, ctx, slots, pairs = fork_flow(fc, OracleBM)
    dev = torch.device("cuda")
    mb = max(len(t) for t in tables)
    bt = torch.zeros(len(tables), mb, dtype=torch.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    cl = torch.tensor(ctx, dtype=torch.int32)
    gs, sl = pd.find_shared_prefixes(bt, cl, S, max_group=8)
    q = fc.q.to(dev)
    nk, nv = fc.new_key.to(dev), fc.new_value.to(dev)
    sm = torch.tensor(slots, dtype=torch.int64, device=dev)
    pr = torch.tensor(pairs, dtype=torch.int64, device=dev).view(-1, 2)
    btd, cld, gsd, sld = bt.to(dev), cl.to(dev), gs.to(dev), sl.to(dev)
    ws = pd.decode_shared_workspace(sl.numel(), 8, fc.H, fc.Hk, fc.D)
    err = device_err()
    kc, vc = fc.key_cache.to(dev), fc.value_cache.to(dev)
    out = torch.full_like(q, float("nan"))

    def step():
        pd.pd_decode_step_shared(out, q, kc, vc, btd, cld, max(ctx), fc.scale, gsd, sld, 8,
                                 key=nk, value=nv, slot_mapping=sm, block_mapping=pr,
                                 workspace=ws, dev_err=err)

    step()                                           # eager reference
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        kc.copy_(fc.key_cache)
        vc.copy_(fc.value_cache)
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        kc.copy_(fc.key_cache.to(dev))
        vc.copy_(fc.value_cache.to(dev))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
