"""GPU parity of paged decode attention (split context, pieces merged in-kernel) against the
float64 oracle, over the five workloads and the edge cases: ragged and empty
contexts, partition boundaries, every GQA grouping, head dims, block sizes
and element types, block-permutation invariance (bit-identical), a
single-token context returning V exactly, and flagged bad inputs."""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import (assert_close, device_err, gpu_store_and_decode, odt,
                          oracle_store_and_decode, u16)
from tests.test_store_copy_gpu import OracleBM, fork_flow

pytestmark = pytest.mark.gpu


def _check(pd, c, what, rows=None):
    err = device_err()
    out, _, _ = gpu_store_and_decode(pd, c, dev_err=err)
    torch.cuda.synchronize()
    ref, _, _ = oracle_store_and_decode(c, rows=rows)
    g = out.cpu()
    if rows is not None:
        g = g.reshape(-1, c.D)[rows[0]:rows[1]].reshape(-1, c.D)
        ref = ref.reshape(-1, c.D)[rows[0]:rows[1]]
    assert_close(g, ref, what)
    assert err.item() == 0
    return out


def test_tiny_decode(cuda_lib):
    _check(cuda_lib, pd_inputs.tiny_decode(), "tiny")


def test_qwen3_8b_decode_step(cuda_lib):
    c = pd_inputs.qwen3_8b_decode()
    assert cuda_lib.pd_decode_workspace_bytes(c.B, c.H, c.D, c.max_context_len) > 0
    _check(cuda_lib, c, "qwen3_8b")


def test_single_token_context_returns_v_exactly(cuda_lib):
    c = pd_inputs.decode_case("one", 21, [1, 1, 1, 1], 32, 8, 128, 16, torch.bfloat16)
    out, _, _ = gpu_store_and_decode(cuda_lib, c)
    torch.cuda.synchronize()
    v = c.new_value                                   # [B, Hk, D]
    want = v.repeat_interleave(4, dim=1)              # head h reads kv head h // 4
    assert torch.equal(out.cpu().view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("H,Hk", [(8, 8), (8, 1), (16, 2), (6, 2), (12, 2), (32, 8), (12, 3),
                                  (20, 5)])
@pytest.mark.parametrize("D", [64, 128])
def test_gqa_groupings(cuda_lib, H, Hk, D):
    c = pd_inputs.decode_case("gqa", 30 + H + Hk + D, [1, 31, 256, 257, 700], H, Hk, D, 16,
                              torch.float16)
    _check(cuda_lib, c, f"H{H} Hk{Hk} D{D}")


@pytest.mark.parametrize("S", [8, 16, 32, 64])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_block_sizes_and_dtypes(cuda_lib, S, dtype):
    ctx = [1, S - 1, S, S + 1, 255, 256, 257, 511, 512, 513, 1500]
    c = pd_inputs.decode_case("S", 40 + S, ctx, 8, 2, 128, S, dtype, key_outlier_frac=0.05)
    _check(cuda_lib, c, f"S{S} {dtype}")


def test_empty_contexts_give_zeros(cuda_lib):
    for ctx in ([0, 5, 0], [0, 900, 0, 3]):
        c = pd_inputs.decode_case("z", 50, ctx, 8, 2, 64, 16, torch.bfloat16)
        out = _check(cuda_lib, c, f"empty {ctx}")
        for i, n in enumerate(ctx):
            if n == 0:
                assert (out[i] == 0).all()


def test_long_contexts_many_partitions(cuda_lib):
    c = pd_inputs.decode_case("long", 51, [20000, 3, 9000, 16385], 16, 4, 128, 16,
                              torch.bfloat16, key_outlier_frac=0.05)
    _check(cuda_lib, c, "long")


def test_block_permutation_gives_identical_bits(cuda_lib):
    c = pd_inputs.decode_case("perm", 52, [700, 33, 2000, 1], 32, 8, 128, 16, torch.bfloat16)
    out1, kc, vc = gpu_store_and_decode(cuda_lib, c)
    NB = kc.shape[0]
    g = torch.Generator().manual_seed(9)
    perm = torch.randperm(NB, generator=g).cuda()       # new id of old block b
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = perm[c.pool.block_tables.cuda().long()].to(torch.int32)
    out2 = torch.empty_like(out1)
    ws = cuda_lib.decode_workspace(c.B, c.H, c.D, c.max_context_len)
    cuda_lib.pd_paged_attention_decode(out2, c.q.cuda(), kc2, vc2, bt2,
                                       c.pool.context_lens.cuda(), c.max_context_len, c.scale,
                                       ws)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_repeat_runs_identical(cuda_lib):
    c = pd_inputs.qwen3_8b_decode(seed=3, B=16)
    a, kc, vc = gpu_store_and_decode(cuda_lib, c)
    b, _, _ = gpu_store_and_decode(cuda_lib, c, use_store=False, kc=kc, vc=vc)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("point", [0, 1, 2])
def test_long_context_stack_sampled_layers(cuda_lib, point):
    """Full-size layers of the 32-layer long-context stack (B, ctx) in
    {(8, 32768), (32, 8192), (128, 2048)}; layers are independent launches
    over the same table, so a sample of layers is checked in full."""
    for layer in (0, 31):
        c = pd_inputs.long_context_layer(point, layer)
        _check(cuda_lib, c, f"long_context point {point} layer {layer}")


def test_cow_fork_decode(cuda_lib):
    """Decode over the 256 forked sequences (shared prompt blocks) after the
    copy-on-write copies and stores, for block size 16; other block sizes
    on a sampled subset."""
    pd = cuda_lib
    for S in (8, 16, 32, 64):
        fc = pd_inputs.cow_fork_stress(S)
        tables, ctx, slots, pairs = fork_flow(fc, OracleBM)
        dev = torch.device("cuda")
        kg, vg = fc.key_cache.to(dev), fc.value_cache.to(dev)
        if pairs:
            pd.pd_copy_blocks([kg], [vg], torch.tensor(pairs, dtype=torch.int64, device=dev))
        pd.pd_reshape_and_cache(fc.new_key.to(dev), fc.new_value.to(dev), kg, vg,
                                torch.tensor(slots, dtype=torch.int64, device=dev))
        mb = max(len(t) for t in tables)
        bt = torch.full((len(tables), mb), 0, dtype=torch.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
        cl = torch.tensor(ctx, dtype=torch.int32)
        out = torch.empty(len(tables), fc.H, fc.D, dtype=fc.dtype, device=dev)
        ws = pd.decode_workspace(len(tables), fc.H, fc.D, max(ctx))
        pd.pd_paged_attention_decode(out, fc.q.to(dev), kg, vg, bt.to(dev), cl.to(dev),
                                     max(ctx), fc.scale, ws)
        torch.cuda.synchronize()
        rk, rv = u16(fc.key_cache), u16(fc.value_cache)
        if pairs:
            oracle.copy_blocks([rk], [rv], np.array(pairs, dtype=np.int64))
        oracle.reshape_and_cache(fc.new_key, fc.new_value, rk, rv, torch.tensor(slots), S)
        assert np.array_equal(u16(kg), rk) and np.array_equal(u16(vg), rv)
        n = len(tables)
        rows = (0, n * fc.H) if S == 16 else (0, 16 * fc.H)
        ref = oracle.decode(fc.q, rk, rv, bt, cl, fc.scale, odt(fc.dtype), rows=rows)
        assert_close(out.cpu().reshape(-1, fc.D)[rows[0]:rows[1]],
                     ref.reshape(-1, fc.D)[rows[0]:rows[1]], f"cow S{S}")


def test_bad_block_id_flagged_not_trapped(cuda_lib):
    c = pd_inputs.decode_case("bad", 60, [300, 40], 8, 2, 64, 16, torch.float16)
    c.pool.block_tables[0, 3] = c.pool.NB + 5
    c.pool.block_tables[1, 0] = -2
    err = device_err()
    gpu_store_and_decode(cuda_lib, c, use_store=False, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & cuda_lib.PD_DEVERR_BLOCK_RANGE


def test_context_beyond_table_flagged(cuda_lib):
    c = pd_inputs.decode_case("ctx", 61, [100, 40], 8, 2, 64, 16, torch.float16)
    c.pool.context_lens[1] = 10000      # longer than its table row holds
    err = device_err()
    dev = torch.device("cuda")
    out = torch.empty(c.B, c.H, c.D, dtype=c.dtype, device=dev)
    ws = cuda_lib.decode_workspace(c.B, c.H, c.D, 100)
    cuda_lib.pd_paged_attention_decode(out, c.q.to(dev), c.pool.key_cache.to(dev),
                                       c.pool.value_cache.to(dev), c.pool.block_tables.to(dev),
                                       c.pool.context_lens.to(dev), 100, c.scale, ws,
                                       dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & cuda_lib.PD_DEVERR_CTX_RANGE


def test_workspace_too_small_is_an_error(cuda_lib):
    c = pd_inputs.decode_case("ws", 62, [3000], 8, 2, 64, 16, torch.float16)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.PDError) as e:
        gpu_store_and_decode(cuda_lib, c, workspace=small)
    assert e.value.status == 5


def test_workspace_contents_do_not_matter(cuda_lib):
    """The arrival counters in the workspace carry a per-launch tag: results
    are the same bits whatever the workspace held before (fresh, random
    bytes, all ones, or the counters of an earlier launch on the same batch)."""
    pd = cuda_lib
    c = pd_inputs.qwen3_8b_decode(seed=3, B=16)
    dev = torch.device("cuda")
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    pd.pd_reshape_and_cache(c.new_key.to(dev), c.new_value.to(dev), kc, vc,
                            c.slot_mapping.to(dev))
    q = c.q.to(dev)
    bt, cl = c.pool.block_tables.to(dev), c.pool.context_lens.to(dev)
    mcl = c.max_context_len
    nbytes = pd.pd_decode_workspace_bytes(c.B, c.H, c.D, mcl)
    g = torch.Generator(device="cpu").manual_seed(5)
    fills = [None,
             torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g),
             torch.full((nbytes,), 255, dtype=torch.uint8)]
    outs = []
    for fill in fills:
        ws = pd.decode_workspace(c.B, c.H, c.D, mcl)
        if fill is not None:
            ws.view(torch.uint8)[:nbytes].copy_(fill.to(dev))
        for _ in range(2):               # the second call meets the first's counters
            out = torch.full_like(q, float("nan"))
            err = device_err()
            pd.pd_paged_attention_decode(out, q, kc, vc, bt, cl, mcl, c.scale, ws, dev_err=err)
            torch.cuda.synchronize()
            assert err.item() == 0
            outs.append(u16(out.cpu()))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    assert torch.isfinite(out.float()).all()


def test_thousands_of_short_sequences(cuda_lib):
    """3000 sequences of 0..40 tokens (a third empty): every CTA range crosses
    many streams, and the walk scans the whole batch."""
    g = torch.Generator().manual_seed(77)
    ctx = torch.randint(0, 41, (3000,), generator=g)
    ctx[::3] = 0
    c = pd_inputs.decode_case("many", 77, ctx.tolist(), 8, 2, 64, 16, torch.bfloat16)
    out = _check(cuda_lib, c, "3000 short")
    assert (out[::3] == 0).all()
