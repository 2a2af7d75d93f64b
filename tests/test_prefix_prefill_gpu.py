"""A prefix-cache hit feeding chunked prefill (tutorial page "LLM 推理服务引擎
深度拆解", section 4: the cached part of a prompt is not recomputed): the
second request of a conversation shares the first request's cached blocks
(pd_pc_lookup -> pd_bm_add_seq_shared), stores only its new tokens and runs
pd_paged_prefill_chunk with P = hit tokens.  Its output must match the
oracle over the shared table, and the rows a no-cache prefill of the whole
prompt computes."""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import assert_close, device_err, odt, u16

pytestmark = pytest.mark.gpu

S, H, Hk, D = 16, 32, 8, 128
DT = torch.bfloat16


def _request(pd, bm, pc, seq_id, prompt, kc, vc, dev):
    """Admit a prompt: look up the cache, share the hit blocks, store the
    rest, prefill the rest.  Returns (output rows of the new tokens, block
    table, hit tokens, the q used)."""
    hit, keys, hit_blocks = pc.lookup(prompt)
    if hit:
        bm.add_seq_shared(seq_id, hit_blocks, hit)
    else:
        bm.add_seq(seq_id)
    slots = []
    for _ in range(len(prompt) - hit):
        slot, copy = bm.append_slot(seq_id)
        assert copy is None                    # the hit ends on a block boundary
        slots.append(slot)
    pos = list(range(hit, len(prompt)))
    k, v = pd_inputs.token_kv(pos, prompt[hit:], Hk, D, DT)
    err = device_err()
    pd.pd_reshape_and_cache(k.to(dev), v.to(dev), kc, vc,
                            torch.tensor(slots, dtype=torch.int64, device=dev), dev_err=err)
    table = bm.block_table(seq_id)
    evicted = pc.insert(keys, table[: len(keys)])
    for b in table[hit // S: len(keys)]:
        bm.retain(b)                           # the cache's own reference
    for b in evicted:
        bm.drop(b)
    C = len(prompt) - hit
    g = torch.Generator().manual_seed(1000 + seq_id)
    q = torch.randn(C, H, D, generator=g).to(DT)
    out = torch.empty(C, H, D, dtype=DT, device=dev)
    bt = torch.tensor([table], dtype=torch.int32, device=dev)
    cl = torch.tensor([len(prompt)], dtype=torch.int32, device=dev)
    cu = torch.tensor([0, C], dtype=torch.int32, device=dev)
    pd.pd_paged_prefill_chunk(out, q.to(dev), cu, C, kc, vc, bt, cl, D ** -0.5, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return out.cpu(), table, hit, q


def test_prefix_hit_prefill_matches_oracle_and_full_prefill(cuda_lib):
    pd = cuda_lib
    dev = torch.device("cuda")
    NB = 256
    kc = torch.zeros(NB, Hk, S, D, dtype=DT, device=dev)
    vc = torch.zeros_like(kc)
    bm, pc = pd.BlockManager(NB, S), pd.PrefixCache(128, S)
    system = list(range(600))
    p1 = system + list(range(90100, 90150))                 # 650 tokens
    out1, t1, hit1, _ = _request(pd, bm, pc, 1, p1, kc, vc, dev)
    assert hit1 == 0
    p2 = p1 + list(range(80050, 80150)) + list(range(90200, 90250))   # 800 tokens
    out2, t2, hit2, q2 = _request(pd, bm, pc, 2, p2, kc, vc, dev)
    assert hit2 == 640 and t2[:40] == t1[:40]               # 40 shared blocks
    assert all(bm.ref_count(b) == 3 for b in t1[:40])        # seq 1, seq 2, cache
    bm.release(1)                                            # cached blocks stay alive
    assert all(bm.ref_count(b) == 2 for b in t1[:40])
    # oracle over the shared table
    ref = oracle.prefill(q2, np.array([0, 160], dtype=np.int32), u16(kc.cpu()), u16(vc.cpu()),
                         np.array([t2], dtype=np.int32), np.array([800], dtype=np.int32),
                         D ** -0.5, odt(DT))
    assert_close(out2, ref, "prefix-hit prefill")
    # the same rows from a whole-prompt prefill in a fresh pool, no cache
    kf = torch.zeros_like(kc)
    vf = torch.zeros_like(kc)
    bmf, pcf = pd.BlockManager(NB, S), pd.PrefixCache(1, S)
    qf = torch.cat([torch.randn(640, H, D, generator=torch.Generator().manual_seed(7)).to(DT), q2])
    bmf.add_seq(9)
    slots = [bmf.append_slot(9)[0] for _ in range(800)]
    k, v = pd_inputs.token_kv(range(800), p2, Hk, D, DT)
    pd.pd_reshape_and_cache(k.to(dev), v.to(dev), kf, vf, torch.tensor(slots, device=dev))
    of = torch.empty(800, H, D, dtype=DT, device=dev)
    pd.pd_paged_prefill_chunk(of, qf.to(dev), torch.tensor([0, 800], dtype=torch.int32, device=dev),
                              800, kf, vf,
                              torch.tensor([bmf.block_table(9)], dtype=torch.int32, device=dev),
                              torch.tensor([800], dtype=torch.int32, device=dev), D ** -0.5)
    torch.cuda.synchronize()
    assert_close(of.cpu()[640:], ref, "whole-prompt prefill, rows of the new tokens")
