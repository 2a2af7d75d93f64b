"""Host-side grouping for the shared-prefix decode (pd_find_shared_prefixes).

The rule (stated in include/pd_attn.h): consecutive sequences join the group of
the first member f while the group has room, their leading full blocks agree
with f's for at least max(min_shared_tokens, S) tokens, and no later member
shortens what the earlier ones share.  Checked against the rule written out
below on the copy-on-write fork flow (tutorial page "LLM 推理服务引擎深度拆解",
section 2.3: forks share the prompt's blocks), on random sharing patterns and
on the edge cases.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_26_gb300 as pd
import pd_inputs
from tests.test_store_copy_gpu import OracleBM, fork_flow


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pd.build.build()
    pd.load()


def rule(bt, ctx, S, max_group, min_shared):
    bt = np.asarray(bt)
    B, mb = bt.shape
    c = np.clip(np.asarray(ctx, dtype=np.int64), 0, mb * S)

    def common(i, f):
        full = min(c[i], c[f]) // S
        n = 0
        while n < full and bt[i, n] == bt[f, n]:
            n += 1
        return n * S

    need = max(min_shared, S)
    starts, shared = [0], []
    first, members, sh = 0, (1 if B else 0), 0
    for i in range(1, B):
        cc = common(i, first)
        if members < max_group and cc >= need and (members == 1 or cc >= sh):
            if members == 1:
                sh = cc
            members += 1
            continue
        shared.append(sh if members > 1 else 0)
        starts.append(i)
        first, members, sh = i, 1, 0
    if B:
        shared.append(sh if members > 1 else 0)
        starts.append(B)
    return starts, shared


def _tables(tables):
    mb = max(len(t) for t in tables)
    bt = torch.full((len(tables), mb), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    return bt


@pytest.mark.parametrize("S", [8, 16, 32, 64])
def test_fork_flow_gives_one_group_per_prompt(S):
    fc = pd_inputs.cow_fork_stress(S)
    tables, ctx, _, _ = fork_flow(fc, OracleBM)
    bt, cl = _tables(tables), torch.tensor(ctx, dtype=torch.int32)
    gs, sl = pd.find_shared_prefixes(bt, cl, S, max_group=8)
    assert gs.tolist() == list(range(0, 8 * len(fc.prompt_lens) + 1, 8))
    # the prompt's full blocks: the copy-on-write rules leave them shared,
    # while each fork writes its own copy of a partial last block
    want = [(L // S) * S for L in fc.prompt_lens.tolist()]
    assert sl.tolist() == want
    assert (gs.tolist(), sl.tolist()) == rule(bt, cl, S, 8, 0)


def test_random_sharing_patterns_follow_the_rule():
    rng = np.random.default_rng(7)
    for trial in range(200):
        S = int(rng.choice([8, 16, 32, 64]))
        B = int(rng.integers(0, 40))
        mb = int(rng.integers(1, 12))
        bt = rng.integers(0, 6, (B, mb)).astype(np.int32)     # few ids: many agreements
        # copy leading runs from the previous row to create shared prefixes
        for i in range(1, B):
            n = int(rng.integers(0, mb + 1))
            bt[i, :n] = bt[i - 1, :n]
        ctx = rng.integers(-3, mb * S + 10, B).astype(np.int32)
        max_group = int(rng.integers(1, 33))
        min_shared = int(rng.choice([0, S, 2 * S, 5 * S]))
        gs, sl = pd.find_shared_prefixes(torch.from_numpy(bt).reshape(B, mb),
                                         torch.from_numpy(ctx), S, max_group, min_shared)
        want = rule(bt.reshape(B, mb), ctx, S, max_group, min_shared)
        assert (gs.tolist(), sl.tolist()) == want, trial
        # invariants: groups tile 0..B, sizes within max_group, every member
        # agrees with the first over the group's shared tokens
        g = gs.tolist()
        assert g[0] == 0 and g[-1] == B and all(a < b for a, b in zip(g, g[1:]))
        for k in range(len(g) - 1):
            assert g[k + 1] - g[k] <= max_group
            nb = sl[k].item() // S
            for i in range(g[k], g[k + 1]):
                assert (bt[i, :nb] == bt[g[k], :nb]).all()
                assert sl[k].item() <= max(0, int(ctx[i]))


def test_edges():
    bt = torch.zeros(0, 4, dtype=torch.int32)
    gs, sl = pd.find_shared_prefixes(bt, torch.zeros(0, dtype=torch.int32), 16)
    assert gs.tolist() == [0] and sl.tolist() == []
    bt = torch.tensor([[5, 6, 7]], dtype=torch.int32)
    gs, sl = pd.find_shared_prefixes(bt, torch.tensor([40], dtype=torch.int32), 16)
    assert gs.tolist() == [0, 1] and sl.tolist() == [0]
    # identical tables, max_group 1: every sequence alone
    bt = torch.tensor([[5, 6, 7]] * 3, dtype=torch.int32)
    gs, sl = pd.find_shared_prefixes(bt, torch.tensor([40] * 3, dtype=torch.int32), 16,
                                     max_group=1)
    assert gs.tolist() == [0, 1, 2, 3] and sl.tolist() == [0, 0, 0]
    # a sequence with an empty context shares nothing, so it splits the run
    gs, sl = pd.find_shared_prefixes(bt, torch.tensor([40, 0, 40], dtype=torch.int32), 16)
    assert gs.tolist() == [0, 1, 2, 3] and sl.tolist() == [0, 0, 0]
    # the third row agrees with the first over one block only: it would
    # shorten the group's two shared blocks, so it starts a group of its own
    bt = torch.tensor([[5, 6, 7], [5, 6, 8], [5, 9, 9]], dtype=torch.int32)
    gs, sl = pd.find_shared_prefixes(bt, torch.tensor([48, 48, 48], dtype=torch.int32), 16)
    assert gs.tolist() == [0, 2, 3] and sl.tolist() == [32, 0]


def test_invalid_arguments():
    lib = pd.load()
    n = pd.ctypes.c_int(0)
    buf = (pd.ctypes.c_int32 * 8)()
    for args in [(None, 1, buf, 1, 16, 8, 0, buf, buf, pd.ctypes.byref(n)),
                 (buf, 0, buf, 1, 16, 8, 0, buf, buf, pd.ctypes.byref(n)),
                 (buf, 1, buf, -1, 16, 8, 0, buf, buf, pd.ctypes.byref(n)),
                 (buf, 1, buf, 1, 16, 33, 0, buf, buf, pd.ctypes.byref(n)),
                 (buf, 1, buf, 1, 16, 0, 0, buf, buf, pd.ctypes.byref(n)),
                 (buf, 1, buf, 1, 0, 8, 0, buf, buf, pd.ctypes.byref(n))]:
        assert lib.pd_find_shared_prefixes(*args) == 1


def test_shared_decode_validation():
    """Host checks of pd_paged_attention_decode_shared (nothing launched)."""
    lib = pd.load()
    P = 0x7f0000001000
    ws = pd.pd_decode_shared_workspace_bytes(32, 8, 32, 8, 128)
    assert ws > 0
    assert pd.pd_decode_shared_workspace_bytes(32, 33, 32, 8, 128) == 0
    assert pd.pd_decode_shared_workspace_bytes(0, 8, 32, 8, 128) == 0
    ok = [P, P, P, P, P, 16, P, 256, 32, 8, 128, 16, 4096, 2049, 0.1, P, P, 32, 8, P, ws,
          pd.PD_BF16, None, None]
    n0 = lib.pd_launch_count()
    cases = [({17: 0}, 2), ({18: 33}, 2), ({18: 0}, 2), ({15: None}, 1), ({16: None}, 1),
             ({20: ws - 1}, 5), ({19: P + 16}, 1), ({10: 96}, 2), ({8: 30}, 1)]
    for change, want in cases:
        a = list(ok)
        for i, v in change.items():
            a[i] = v
        assert lib.pd_paged_attention_decode_shared(*a) == want, change
    a = list(ok)
    a[7] = 0                               # B == 0: nothing to do
    assert lib.pd_paged_attention_decode_shared(*a) == 0
    assert lib.pd_launch_count() == n0
