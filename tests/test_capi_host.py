"""Host-side checks of the C ABI (no GPU needed): the library loads and
exports every symbol include/*.h declares, argument validation rejects bad
calls before any launch, and the C++ block manager reproduces the oracle's
block-id trace bit-exactly."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_attention_26_gb300 as pd
from paged_kv_attention_26_gb300 import build as pdbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pdbuild.build()
    return pd.load()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"PD_API[^;(]*?\b(pd_\w+)\s*\(", text, flags=re.S))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 20
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared but not exported"
    # and the binding knows the signature of each
    assert names == set(pd.SIGNATURES), names ^ set(pd.SIGNATURES)


def test_status_strings(lib):
    for code in range(7):
        assert lib.pd_status_string(code)
    assert lib.pd_launch_count() >= 0


# Fake device pointers: validation must reject these calls before launching.
P = 0x7f0000001000     # 16-byte aligned, never dereferenced


def test_store_validation(lib):
    f = lib.pd_reshape_and_cache
    ok_args = [P, P, P, P, P, 4, 2, 64, 16, 64, 128, 128, pd.PD_F16, None, None]
    bad = dict(enumerate(ok_args))
    cases = [
        ({7: 96}, 2),          # D unsupported
        ({8: 12}, 2),          # S unsupported
        ({12: 7}, 2),          # dtype
        ({5: -1}, 1),          # T < 0
        ({6: 0}, 1),           # Hk < 1
        ({2: 0}, 1),           # null cache
        ({2: P + 2}, 1),       # misaligned cache
        ({10: 100}, 1),        # token stride smaller than a token
        ({10: 132}, 1),        # token stride not a 16-byte multiple
    ]
    for change, want in cases:
        a = list(ok_args)
        for k, v in change.items():
            a[k] = v
        assert f(*a) == want, change
    a = list(ok_args)
    a[5] = 0                   # T == 0: nothing to do, no launch
    n0 = lib.pd_launch_count()
    assert f(*a) == 0
    assert lib.pd_launch_count() == n0


def test_decode_validation(lib):
    f = lib.pd_paged_attention_decode
    base = [P, P, P, P, P, 8, P, 4, 8, 2, 64, 16, 64, 100, 0.125, None, 0, pd.PD_F16, None, None]
    cases = [
        ({9: 3}, 1),           # H % Hk
        ({10: 80}, 2),         # D
        ({11: 4}, 2),          # S
        ({0: 0}, 1),           # null out
        ({1: P + 8}, 1),       # misaligned q
        ({13: -1}, 1),         # negative max_context_len
        ({5: 0}, 1),           # max_blocks_per_seq
    ]
    for change, want in cases:
        a = list(base)
        for k, v in change.items():
            a[k] = v
        assert f(*a) == want, change
    # long context needs a workspace
    need = lib.pd_decode_workspace_bytes(4, 8, 64, 5000)
    assert need > lib.pd_decode_workspace_bytes(4, 8, 64, 100) > 0
    a = list(base)
    a[13] = 5000
    assert f(*a) == 1                          # no workspace pointer
    a[15], a[16] = P, need - 1
    assert f(*a) == 5                          # too small
    a[15] = P + 16
    a[16] = need
    assert f(*a) == 1                          # not 256-byte aligned


def test_decode_step_validation(lib):
    """The fused store + decode call checks both halves before launching
    anything: an error in either leaves the launch count unchanged."""
    f = lib.pd_decode_step
    base = [P, P, P, 4, 128, 128,            # key, value, slots, T, strides
            P, P, P, P,                      # out, q, key_cache, value_cache
            P, 8, P, 4, 8, 2, 64, 16, 64,    # tables, mbps, lens, B, H, Hk, D, S, NB
            100, 0.125, None, 0, pd.PD_F16, None, None]
    cases = [
        ({3: -1}, 1),          # T < 0 (store half)
        ({4: 100}, 1),         # key stride shorter than a token
        ({0: P + 4}, 1),       # misaligned key
        ({15: 3}, 1),          # H % Hk (decode half)
        ({16: 80}, 2),         # D
        ({6: 0}, 1),           # null out
        ({19: 5000}, 1),       # long context without a workspace
        ({23: 9}, 2),          # dtype
    ]
    n0 = lib.pd_launch_count()
    for change, want in cases:
        a = list(base)
        for k, v in change.items():
            a[k] = v
        assert f(*a) == want, change
    a = list(base)
    a[3], a[13] = 0, 0         # nothing to store, nothing to decode
    assert f(*a) == 0
    assert lib.pd_launch_count() == n0
    g = lib.pd_decode_step_fp8
    a = list(base)
    a[10:10] = [None, P]       # k_scale missing
    assert g(*a) == 1
    a[10], a[11] = P, None     # v_scale missing
    assert g(*a) == 1
    assert lib.pd_launch_count() == n0
    # the one-kernel step: the same checks, then one row per sequence and a
    # kv head read by one CTA group alone
    h = lib.pd_decode_step_fused
    for change, want in cases + [({3: 3}, 1),             # T != B
                                 ({14: 40, 15: 4, 4: 256, 5: 256, 21: P, 22: 1 << 30},
                                  2)]:                    # G = 10 > 8
        a = list(base)
        for k, v in change.items():
            a[k] = v
        assert h(*a) == want, change
    a = list(base)
    a[3], a[13] = 0, 0
    assert h(*a) == 0
    assert lib.pd_launch_count() == n0


def test_verify_validation(lib):
    f = lib.pd_paged_attention_verify
    base = [P, P, P, P, P, 8, P, 4, 4, 8, 2, 64, 16, 64, 100, 0.125, None, 0, pd.PD_F16, None,
            None]
    cases = [
        ({8: 0}, 2),           # nq < 1
        ({8: 9}, 2),           # nq > 8
        ({7: 20000}, 2),       # B * nq > 65535
        ({9: 6}, 1),           # H % Hk
        ({11: 80}, 2),         # D
        ({0: 0}, 1),           # null out
    ]
    n0 = lib.pd_launch_count()
    for change, want in cases:
        a = list(base)
        for k, v in change.items():
            a[k] = v
        assert f(*a) == want, change
    # the workspace is sized for B * nq query rows
    a = list(base)
    a[14] = 5000
    need = lib.pd_decode_workspace_bytes(4 * 4, 8, 64, 5000)
    a[16], a[17] = P, lib.pd_decode_workspace_bytes(4, 8, 64, 5000)
    assert a[17] < need and f(*a) == 5          # enough for decode, not for verify
    assert lib.pd_launch_count() == n0


def test_selftest_validation(lib):
    n0 = lib.pd_launch_count()
    assert lib.pd_selftest_bounded_wait(None, 1000000, None) == 1      # dev_err required
    assert lib.pd_selftest_bounded_wait(P, 999, None) == 1             # limit too short
    assert lib.pd_selftest_bounded_wait(P, 10**10 + 1, None) == 1      # limit too long
    assert lib.pd_launch_count() == n0


def test_copy_bytes_validation(lib):
    n0 = lib.pd_launch_count()
    assert lib.pd_copy_bytes(P, P + 4096, 0, None) == 0          # nothing to copy
    assert lib.pd_copy_bytes(None, P, 64, None) == 1             # null destination
    assert lib.pd_copy_bytes(P + 8, P, 64, None) == 1            # misaligned
    assert lib.pd_copy_bytes(P, P + 4096, 40, None) == 1         # not a multiple of 16
    buf = (ctypes.c_uint8 * 256)()                               # pageable host memory
    addr = (ctypes.addressof(buf) + 15) & ~15
    assert lib.pd_copy_bytes(addr, addr + 128, 64, None) == 1    # refused: not device-visible
    assert lib.pd_launch_count() == n0


def test_verify_step_validation(lib):
    f = lib.pd_verify_step
    base = [P, P, P, 16, 128, 128,           # key, value, slots, T, strides
            P, P, P, P,                      # out, q, key_cache, value_cache
            P, 8, P, 4, 4, 8, 2, 64, 16, 64,  # tables, mbps, lens, B, nq, H, Hk, D, S, NB
            100, 0.125, None, 0, pd.PD_F16, None, None]
    n0 = lib.pd_launch_count()
    for change, want in [({14: 9}, 2), ({14: 0}, 2), ({3: -1}, 1), ({16: 3}, 1), ({17: 96}, 2)]:
        a = list(base)
        for k, v in change.items():
            a[k] = v
        assert f(*a) == want, change
    assert lib.pd_launch_count() == n0


def test_workspace_size_formula(lib):
    part = lib.pd_decode_partition_tokens(10000)
    assert part % 64 == 0
    B, H, D, ctx = 3, 8, 128, 10000
    P = -(-ctx // part) + 1            # pieces per context, at most
    need = lib.pd_decode_workspace_bytes(B, H, D, ctx)
    assert need >= B * H * (P * (D + 2) * 4 + 8)
    assert need <= B * H * (P * (D + 2) * 4 + 8) + 4 * 256


def test_copy_and_prefill_validation(lib):
    assert lib.pd_copy_blocks(P, P, 1, P, 3, 8, 128, 16, 10, 9, None, None) == 2
    assert lib.pd_copy_blocks(P, P, -1, P, 3, 8, 128, 16, 10, 1, None, None) == 1
    n0 = lib.pd_launch_count()
    assert lib.pd_copy_blocks(P, P, 1, P, 0, 8, 128, 16, 10, 1, None, None) == 0
    assert lib.pd_launch_count() == n0
    f = lib.pd_paged_prefill_chunk
    base = [P, P, 40, P, 16, P, P, P, 8, P, 2, 8, 2, 64, 16, 64, 0.125, pd.PD_BF16, None, None]
    for change, want in [({11: 3}, 1),        # H % Hk
                         ({13: 256}, 2),      # D
                         ({4: -1}, 1),        # max_q_len
                         ({2: -5}, 1),        # total_q
                         ({16: 0.0}, 1),      # scale must be positive
                         ({16: float("nan")}, 1),
                         ({1: P + 4}, 1)]:    # misaligned q
        a = list(base)
        for k, v in change.items():
            a[k] = v
        assert f(*a) == want, change


# ---- block manager: C++ against the oracle ------------------------------------

def test_bm_fork_demo_matches_golden(lib):
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "block_manager_fork_demo.json")))
    bm = pd.BlockManager(g["num_blocks"], g["block_size"])
    bm.add_seq(0)
    for _ in range(g["prompt_len"]):
        assert bm.append_slot(0)[1] is None
    assert bm.block_table(0) == g["prompt_blocks"]
    assert bm.usage == g["usage_after_prompt"]
    for c in range(1, g["n_children"] + 1):
        bm.fork(0, c)
    assert bm.usage == g["usage_after_fork"]
    res = [bm.append_slot(c) for c in range(1, g["n_children"] + 1)]
    assert [list(c) for _, c in res] == g["child_cow_copies"]
    assert [s for s, _ in res] == g["child_slots"]
    assert bm.usage == g["usage_after_child_appends"]
    for b, rc in g["ref_count_after_appends"].items():
        assert bm.ref_count(int(b)) == rc


@pytest.mark.parametrize("S,seed", [(8, 0), (16, 1), (32, 2), (64, 3)])
def test_bm_replays_oracle_trace(lib, S, seed):
    rng = np.random.default_rng(seed)
    nb = 300
    ref = oracle.BlockManager(nb, S)
    bm = pd.BlockManager(nb, S)
    seqs = {0: oracle.Sequence(ref, 0)}
    bm.add_seq(0)
    nid = 1
    for _ in range(4000):
        op = rng.integers(0, 10)
        sid = int(rng.choice(sorted(seqs)))
        if op < 7:
            try:
                want = seqs[sid].append_slot()
            except MemoryError:
                with pytest.raises(pd.PDError) as e:
                    bm.append_slot(sid)
                assert e.value.status == 4
                continue
            got = bm.append_slot(sid)
            assert got == want
        elif op < 9 and len(seqs) < 16:
            seqs[nid] = seqs[sid].fork(nid)
            bm.fork(sid, nid)
            nid += 1
        elif len(seqs) > 1:
            seqs[sid].release()
            del seqs[sid]
            bm.release(sid)
        assert bm.usage == ref.usage
    for sid, s in seqs.items():
        assert bm.block_table(sid) == s.block_table
        assert bm.seq_len(sid) == s.length
    assert [bm.ref_count(b) for b in range(nb)] == ref.ref_count
    assert bm.num_free == len(ref.free_ids)


def test_bm_errors(lib):
    bm = pd.BlockManager(2, 4)
    bm.add_seq(5)
    with pytest.raises(pd.PDError):
        bm.add_seq(5)
    with pytest.raises(pd.PDError) as e:
        bm.append_slot(6)
    assert e.value.status == 6
    for _ in range(8):
        bm.append_slot(5)
    with pytest.raises(pd.PDError) as e:
        bm.append_slot(5)
    assert e.value.status == 4
    assert bm.seq_len(5) == 8          # unchanged by the failed append
    with pytest.raises(pd.PDError):
        bm.fork(7, 8)
    assert lib.pd_bm_create(0, 16) is None
    assert lib.pd_bm_ref_count(bm._h, 99) == -1


def test_kv_pack_validation(lib):
    for f in (lib.pd_kv_pack, lib.pd_kv_unpack):
        # staging, key_caches, value_caches, L, block_ids, nblk, Hk, D, S, NB, dt
        base = [P, P, P, 4, P, 10, 8, 128, 16, 100, pd.PD_BF16, None, None]
        for change, want in [({6: 0}, 1),          # Hk
                             ({7: 96}, 2),          # D
                             ({8: 12}, 2),          # S
                             ({10: 7}, 2),          # dtype
                             ({0: None}, 1),        # staging
                             ({0: P + 8}, 1),       # misaligned staging
                             ({4: None}, 1),        # block ids
                             ({3: 70000}, 2)]:      # too many layers for the grid
            a = list(base)
            for k, v in change.items():
                a[k] = v
            assert f(*a) == want, change
        n0 = lib.pd_launch_count()
        a = list(base)
        a[5] = 0                                    # nothing to move
        assert f(*a) == 0
        a = list(base)
        a[3] = 0                                    # no layers
        assert f(*a) == 0
        assert lib.pd_launch_count() == n0
