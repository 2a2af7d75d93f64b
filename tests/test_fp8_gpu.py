"""GPU parity of the FP8 (E4M3) KV cache: the quantising store is bit-exact
against the oracle; decode over E4M3 pools matches the float64 oracle (which
widens codes exactly and applies the per-head scales) within the attention
tolerance, at small shapes, at every head grouping and at the Qwen3-8B
batch; block copies and the KV hand-over move one-byte pools bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import assert_close, device_err, odt, u16

pytestmark = pytest.mark.gpu


def _u8(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().copy()


@pytest.mark.parametrize("D,S,dtype", [(128, 16, torch.bfloat16), (64, 8, torch.float16),
                                       (128, 64, torch.float16), (64, 32, torch.bfloat16)])
def test_fp8_store_bit_exact(cuda_lib, D, S, dtype):
    pd = cuda_lib
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(D + S)
    NB, Hk, T = 11, 4, 50
    key = (torch.randn(T, Hk, D, generator=g) * 3).to(dtype)
    value = (torch.randn(T, Hk, D, generator=g) * 0.2).to(dtype)
    key[3, 1, 5] = 1e4                                      # saturates to +-448 * scale
    ks = torch.tensor([0.01, 0.02, 0.5, 1.0], dtype=torch.float32)
    vs = torch.tensor([0.001, 0.004, 0.05, 0.1], dtype=torch.float32)
    slots = torch.randperm(NB * S, generator=g)[:T].to(torch.int64)
    slots[::9] = -1
    slots[7] = NB * S + 1                                   # out of range: skipped, flagged
    kc = torch.randint(0, 256, (NB, Hk, S, D), generator=g, dtype=torch.int32).to(torch.uint8)
    vc = torch.randint(0, 256, (NB, Hk, S, D), generator=g, dtype=torch.int32).to(torch.uint8)
    rk, rv = _u8(kc), _u8(vc)
    bad = oracle.reshape_and_cache_fp8(key, value, odt(dtype), rk, rv, slots, ks, vs, S)
    kg, vg = kc.to(dev), vc.to(dev)
    err = device_err()
    pd.pd_reshape_and_cache_fp8(key.to(dev), value.to(dev), kg, vg, slots.to(dev), ks.to(dev),
                                vs.to(dev), dev_err=err)
    torch.cuda.synchronize()
    assert bad == 1 and err.item() & 0x1
    assert np.array_equal(_u8(kg), rk) and np.array_equal(_u8(vg), rv)


def _decode_fp8(pd, c, kc8, vc8, ks, vs, dev):
    out = torch.full_like(c.q, float("nan")).to(dev)
    mcl = c.max_context_len
    err = device_err()
    pd.pd_paged_attention_decode_fp8(out, c.q.to(dev), kc8.to(dev), vc8.to(dev), ks.to(dev),
                                     vs.to(dev), c.pool.block_tables.to(dev),
                                     c.pool.context_lens.to(dev), mcl, c.scale,
                                     pd.decode_workspace(c.B, c.H, c.D, mcl), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return out.cpu()


@pytest.mark.parametrize("H,Hk,D,S,dtype", [(8, 2, 64, 16, torch.float16),
                                            (32, 8, 128, 16, torch.bfloat16),
                                            (16, 16, 128, 8, torch.bfloat16),
                                            (24, 4, 64, 32, torch.float16),
                                            (32, 2, 128, 64, torch.bfloat16)])
def test_fp8_decode_matches_oracle(cuda_lib, H, Hk, D, S, dtype):
    c = pd_inputs.decode_case("fp8", H + D, [1, 5, 64, 65, 300, 1000, 0, 2049], H, Hk, D, S,
                              dtype, store_last=False)
    kc8, vc8, ks, vs = pd_inputs.fp8_pools(c.pool.key_cache, c.pool.value_cache)
    got = _decode_fp8(cuda_lib, c, kc8, vc8, ks, vs, torch.device("cuda"))
    ref = oracle.decode_fp8(c.q, odt(dtype), kc8, vc8, ks, vs, c.pool.block_tables,
                            c.pool.context_lens, c.scale)
    assert_close(got, ref, f"fp8 decode H{H} Hk{Hk} D{D} S{S}")


def test_fp8_store_then_decode_qwen3_8b_sampled(cuda_lib):
    """The Qwen3-8B batch with FP8 pools: store the step's tokens through the
    quantising store, decode, compare sampled rows with the oracle run on the
    same path."""
    pd = cuda_lib
    dev = torch.device("cuda")
    c = pd_inputs.qwen3_8b_decode()
    kc8, vc8, ks, vs = pd_inputs.fp8_pools(c.pool.key_cache, c.pool.value_cache)
    kg, vg = kc8.to(dev), vc8.to(dev)
    pd.pd_reshape_and_cache_fp8(c.new_key.to(dev), c.new_value.to(dev), kg, vg,
                                c.slot_mapping.to(dev), ks.to(dev), vs.to(dev))
    rk, rv = _u8(kc8), _u8(vc8)
    oracle.reshape_and_cache_fp8(c.new_key, c.new_value, odt(c.dtype), rk, rv, c.slot_mapping,
                                 ks, vs, c.pool.S)
    torch.cuda.synchronize()
    assert np.array_equal(_u8(kg), rk) and np.array_equal(_u8(vg), rv)
    got = _decode_fp8(pd, c, kg.cpu(), vg.cpu(), ks, vs, dev)
    rows = (96, 160)                                         # sequences 3 and 4
    ref = oracle.decode_fp8(c.q, odt(c.dtype), rk, rv, ks, vs, c.pool.block_tables,
                            c.pool.context_lens, c.scale, rows=rows)
    assert_close(got.reshape(-1, c.D)[rows[0]:rows[1]], ref, "fp8 qwen rows")
    assert torch.isfinite(got.float()).all()


def test_fp8_pools_copy_and_handover_bit_exact(cuda_lib):
    pd = cuda_lib
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(21)
    L, NB, Hk, S, D = 2, 12, 4, 16, 128
    kcs = [torch.randint(0, 256, (NB, Hk, S, D), generator=g, dtype=torch.int32).to(torch.uint8)
           for _ in range(L)]
    vcs = [torch.randint(0, 256, (NB, Hk, S, D), generator=g, dtype=torch.int32).to(torch.uint8)
           for _ in range(L)]
    kg, vg = [t.to(dev) for t in kcs], [t.to(dev) for t in vcs]
    pairs = torch.tensor([[1, 5], [3, 0], [11, 7]], dtype=torch.int64)
    pd.pd_copy_blocks(kg, vg, pairs.to(dev))
    ids = torch.tensor([4, 9, 2], dtype=torch.int32)
    st = torch.empty((L, 2, 3, Hk, S, D), dtype=torch.uint8, device=dev)
    pd.pd_kv_pack(st, kg, vg, ids.to(dev))
    torch.cuda.synchronize()
    for l in range(L):
        for s_, d_ in pairs.tolist():
            kcs[l][d_] = kcs[l][s_]
            vcs[l][d_] = vcs[l][s_]
        assert torch.equal(kg[l].cpu(), kcs[l]) and torch.equal(vg[l].cpu(), vcs[l])
        for i, b in enumerate(ids.tolist()):
            assert torch.equal(st[l, 0, i].cpu(), kcs[l][b]) and torch.equal(st[l, 1, i].cpu(), vcs[l][b])
