"""GPU parity of the cache-maintenance kernels: store and copy-on-write block
copy, bit-exact against the oracle, plus the full fork flow (host block
manager -> copy_blocks -> store) of the copy-on-write stress workload."""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import device_err, u16

pytestmark = pytest.mark.gpu


def _store_case(pd, key, value, kc, vc, slots, S):
    dev = torch.device("cuda")
    err = device_err()
    kcg, vcg = kc.to(dev), vc.to(dev)
    pd.pd_reshape_and_cache(key.to(dev), value.to(dev), kcg, vcg, slots.to(dev), dev_err=err)
    torch.cuda.synchronize()
    rk, rv = u16(kc), u16(vc)
    bad = oracle.reshape_and_cache(key, value, rk, rv, slots, S)
    assert np.array_equal(u16(kcg), rk) and np.array_equal(u16(vcg), rv)
    return int(err.item()), bad


def test_store_tiny(cuda_lib):
    c = pd_inputs.tiny_decode()
    err, bad = _store_case(cuda_lib, c.new_key, c.new_value, c.pool.key_cache,
                           c.pool.value_cache, c.slot_mapping, c.pool.S)
    assert err == 0 and bad == 0


def test_store_qwen3_8b_step(cuda_lib):
    c = pd_inputs.qwen3_8b_decode()
    err, _ = _store_case(cuda_lib, c.new_key, c.new_value, c.pool.key_cache,
                         c.pool.value_cache, c.slot_mapping, c.pool.S)
    assert err == 0


def test_store_chunked_prefill_mix(cuda_lib):
    m = pd_inputs.chunked_prefill_mixed()
    assert m.slot_mapping.numel() == 16 * 512 + 48
    err, _ = _store_case(cuda_lib, m.new_key, m.new_value, m.pool.key_cache,
                         m.pool.value_cache, m.slot_mapping, m.pool.S)
    assert err == 0


@pytest.mark.parametrize("D,S,dtype", [(64, 8, torch.float16), (128, 64, torch.bfloat16),
                                       (128, 32, torch.float16)])
def test_store_padding_and_bad_slots(cuda_lib, D, S, dtype):
    g = torch.Generator().manual_seed(3)
    NB, Hk, T = 9, 3, 40
    kc = torch.randn(NB, Hk, S, D, generator=g).to(dtype)
    vc = torch.randn(NB, Hk, S, D, generator=g).to(dtype)
    key = torch.randn(T, Hk, D, generator=g).to(dtype)
    value = torch.randn(T, Hk, D, generator=g).to(dtype)
    slots = torch.randperm(NB * S, generator=g)[:T].to(torch.int64)
    slots[::7] = -1                     # padding
    slots[5] = NB * S + 3               # out of range: skipped and flagged
    err, bad = _store_case(cuda_lib, key, value, kc, vc, slots, S)
    assert bad == 1
    assert err == cuda_lib.PD_DEVERR_SLOT_RANGE


def test_store_strided_tokens(cuda_lib):
    """key/value rows taken from a wider [T, 2*Hk*D] buffer (e.g. fused QKV)."""
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(4)
    NB, Hk, S, D, T = 12, 2, 16, 64, 30
    buf = torch.randn(T, 3, Hk, D, generator=g).to(torch.float16)
    key, value = buf[:, 1], buf[:, 2]
    kc = torch.zeros(NB, Hk, S, D, dtype=torch.float16)
    vc = torch.zeros_like(kc)
    slots = torch.randperm(NB * S, generator=g)[:T]
    kcg, vcg = kc.to(dev), vc.to(dev)
    bg = buf.to(dev)
    cuda_lib.pd_reshape_and_cache(bg[:, 1], bg[:, 2], kcg, vcg, slots.to(dev))
    torch.cuda.synchronize()
    rk, rv = u16(kc), u16(vc)
    oracle.reshape_and_cache(key.contiguous(), value.contiguous(), rk, rv, slots, S)
    assert np.array_equal(u16(kcg), rk) and np.array_equal(u16(vcg), rv)


@pytest.mark.parametrize("L,S,D", [(1, 16, 128), (3, 8, 64), (2, 64, 128)])
def test_copy_blocks_bit_exact(cuda_lib, L, S, D):
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(L * 100 + S)
    NB, Hk = 40, 4
    kcs = [torch.randn(NB, Hk, S, D, generator=g).to(torch.float16) for _ in range(L)]
    vcs = [torch.randn(NB, Hk, S, D, generator=g).to(torch.float16) for _ in range(L)]
    perm = torch.randperm(NB, generator=g)
    pairs = torch.stack([perm[:10], perm[10:20]], 1).to(torch.int64)
    err = device_err()
    kg = [k.to(dev) for k in kcs]
    vg = [v.to(dev) for v in vcs]
    cuda_lib.pd_copy_blocks(kg, vg, pairs.to(dev), dev_err=err)
    torch.cuda.synchronize()
    rk = [u16(k) for k in kcs]
    rv = [u16(v) for v in vcs]
    assert oracle.copy_blocks(rk, rv, pairs) == 0
    for l in range(L):
        assert np.array_equal(u16(kg[l]), rk[l]) and np.array_equal(u16(vg[l]), rv[l])
    assert err.item() == 0


def test_copy_blocks_bad_ids_flagged(cuda_lib):
    dev = torch.device("cuda")
    NB = 8
    kc = torch.arange(NB * 2 * 8 * 64, dtype=torch.int16).view(NB, 2, 8, 64).view(torch.float16)
    vc = kc.clone()
    pairs = torch.tensor([[1, 2], [NB, 3], [4, -1], [5, 6]], dtype=torch.int64)
    err = device_err()
    kg, vg = kc.to(dev), vc.to(dev)
    cuda_lib.pd_copy_blocks([kg], [vg], pairs.to(dev), dev_err=err)
    torch.cuda.synchronize()
    rk, rv = [u16(kc)], [u16(vc)]
    assert oracle.copy_blocks(rk, rv, pairs) == 2
    assert np.array_equal(u16(kg), rk[0]) and np.array_equal(u16(vg), rv[0])
    assert err.item() == cuda_lib.PD_DEVERR_BLOCK_RANGE


def fork_flow(fc, bm_cls):
    """Prompts into the pool through the block manager, fork n ways, release
    the parent, one append per child.  Returns (tables, ctx, slots, pairs)."""
    bm = bm_cls(fc.NB, fc.S)
    tables, ctx, slots, pairs = [], [], [], []
    nid = 0
    for L in fc.prompt_lens.tolist():
        parent = nid
        nid += 1
        bm.add_seq(parent)
        for _ in range(L):
            bm.append_slot(parent)
        kids = list(range(nid, nid + fc.n_fork))
        nid += fc.n_fork
        for kid in kids:
            bm.fork(parent, kid)
        bm.release(parent)
        for kid in kids:
            slot, cp = bm.append_slot(kid)
            slots.append(slot)
            if cp is not None:
                pairs.append(tuple(cp))
            tables.append(bm.block_table(kid))
            ctx.append(L + 1)
    return tables, ctx, slots, pairs


class OracleBM:
    """The oracle block manager behind the pd.BlockManager interface."""

    def __init__(self, nb, S):
        self.m = oracle.BlockManager(nb, S)
        self.seqs = {}

    def add_seq(self, sid):
        self.seqs[sid] = oracle.Sequence(self.m, sid)

    def append_slot(self, sid):
        return self.seqs[sid].append_slot()

    def fork(self, a, b):
        self.seqs[b] = self.seqs[a].fork(b)

    def release(self, sid):
        self.seqs.pop(sid).release()

    def block_table(self, sid):
        return list(self.seqs[sid].block_table)


@pytest.mark.parametrize("S", [8, 16, 32, 64])
def test_cow_fork_flow_bit_exact(cuda_lib, S):
    pd = cuda_lib
    fc = pd_inputs.cow_fork_stress(S)
    t_gpu, c_gpu, s_gpu, p_gpu = fork_flow(fc, pd.BlockManager)
    t_ref, c_ref, s_ref, p_ref = fork_flow(fc, OracleBM)
    assert (t_gpu, c_gpu, s_gpu, p_gpu) == (t_ref, c_ref, s_ref, p_ref)
    # copies: the first n_fork-1 children of a prompt with a partial last block
    n_partial = int((fc.prompt_lens % S != 0).sum())
    assert len(p_gpu) == n_partial * (fc.n_fork - 1)
    dev = torch.device("cuda")
    kg, vg = fc.key_cache.to(dev), fc.value_cache.to(dev)
    err = device_err()
    if p_gpu:
        pd.pd_copy_blocks([kg], [vg], torch.tensor(p_gpu, dtype=torch.int64, device=dev),
                          dev_err=err)
    pd.pd_reshape_and_cache(fc.new_key.to(dev), fc.new_value.to(dev), kg, vg,
                            torch.tensor(s_gpu, dtype=torch.int64, device=dev), dev_err=err)
    torch.cuda.synchronize()
    rk, rv = u16(fc.key_cache), u16(fc.value_cache)
    if p_ref:
        oracle.copy_blocks([rk], [rv], np.array(p_ref, dtype=np.int64))
    oracle.reshape_and_cache(fc.new_key, fc.new_value, rk, rv, torch.tensor(s_ref), S)
    assert np.array_equal(u16(kg), rk) and np.array_equal(u16(vg), rv)
    assert err.item() == 0
