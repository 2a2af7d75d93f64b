"""GPU parity of the fused decode step (store the step's new K/V, then decode
with the decode grid launched as a programmatic dependent of the store grid):
bit-identical to the two separate calls, equal to the oracle's store then
decode, and, over many consecutive steps with every stored slot poisoned
beforehand, never reading a slot before the store grid wrote it."""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import (assert_close, device_err, gpu_store_and_decode, odt,
                          oracle_store_and_decode, u16)

pytestmark = pytest.mark.gpu


def _step(pd, c, kc, vc, dev_err=None, k_scale=None, v_scale=None):
    dev = torch.device("cuda")
    q = c.q.to(dev)
    out = torch.empty_like(q)
    ws = pd.decode_workspace(c.B, c.H, c.D, c.max_context_len)
    pd.pd_decode_step(out, q, kc, vc, c.pool.block_tables.to(dev), c.pool.context_lens.to(dev),
                      c.max_context_len, c.scale, c.new_key.to(dev), c.new_value.to(dev),
                      c.slot_mapping.to(dev), workspace=ws, k_scale=k_scale, v_scale=v_scale,
                      dev_err=dev_err)
    return out


@pytest.mark.parametrize("which", ["tiny", "qwen3_8b", "ragged"])
def test_step_equals_separate_calls_and_oracle(cuda_lib, which):
    if which == "tiny":
        c = pd_inputs.tiny_decode()
    elif which == "qwen3_8b":
        c = pd_inputs.qwen3_8b_decode()
    else:
        c = pd_inputs.decode_case("ragged", 61, [1, 0, 16, 17, 64, 65, 999, 2048, 5000], 16, 4,
                                  128, 16, torch.bfloat16, key_outlier_frac=0.05)
    dev = torch.device("cuda")
    err = device_err()
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    out = _step(cuda_lib, c, kc, vc, dev_err=err)
    sep, kc2, vc2 = gpu_store_and_decode(cuda_lib, c)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out.view(torch.int16), sep.view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc2.view(torch.int16))
    rows = (0, 64) if which == "qwen3_8b" else None     # sequences 0 and 1 of the batch
    ref, rk, rv = oracle_store_and_decode(c, rows=rows)
    g = out.cpu()
    if rows:
        g = g.reshape(-1, c.D)[rows[0]:rows[1]]
        ref = ref.reshape(-1, c.D)[rows[0]:rows[1]]
    assert_close(g, ref, f"step {which}")
    assert np.array_equal(u16(kc), rk) and np.array_equal(u16(vc), rv)


@pytest.mark.parametrize("fused", [False, True])
def test_consecutive_steps_see_their_own_tokens(cuda_lib, fused):
    """20 decode steps of 8 sequences, one new token each per step.  Every
    slot a step stores is NaN in the pool until then, so a decode that read
    it before the store grid finished (or, fused, before its own store of
    the row) would return NaN."""
    steps = 20
    ctx0 = torch.tensor([1, 15, 16, 17, 63, 64, 300, 1100])
    H, Hk, D, S = 16, 4, 128, 16
    c = pd_inputs.decode_case("steps", 62, (ctx0 + steps).tolist(), H, Hk, D, S,
                              torch.bfloat16, store_last=False)
    bt = c.pool.block_tables
    B = ctx0.shape[0]
    for i in range(steps):                      # poison every slot that a step stores
        slots = pd_inputs.slot_mapping_for(bt, torch.arange(B), ctx0 - 1 + i, S)
        c.pool.key_cache[slots // S, :, slots % S] = float("nan")
        c.pool.value_cache[slots // S, :, slots % S] = float("nan")
    dev = torch.device("cuda")
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    rk, rv = u16(c.pool.key_cache), u16(c.pool.value_cache)
    btd = bt.to(dev)
    g = torch.Generator().manual_seed(63)
    err = device_err()
    ws = cuda_lib.decode_workspace(B, H, D, int(ctx0.max()) + steps)
    outs, refs = [], []
    for i in range(steps):
        lens = (ctx0 + i).to(torch.int32)
        slots = pd_inputs.slot_mapping_for(bt, torch.arange(B), ctx0 - 1 + i, S)
        nk = torch.randn(B, Hk, D, generator=g).to(torch.bfloat16)
        nv = torch.randn(B, Hk, D, generator=g).to(torch.bfloat16)
        q = torch.randn(B, H, D, generator=g).to(torch.bfloat16)
        out = torch.empty(B, H, D, dtype=torch.bfloat16, device=dev)
        step = cuda_lib.pd_decode_step_fused if fused else cuda_lib.pd_decode_step
        step(out, q.to(dev), kc, vc, btd, lens.to(dev), int(lens.max()), c.scale, nk.to(dev),
             nv.to(dev), slots.to(dev), workspace=ws, dev_err=err)
        outs.append(out)
        oracle.reshape_and_cache(nk, nv, rk, rv, slots, S)
        refs.append(oracle.decode(q, rk, rv, bt, lens, c.scale, oracle.BF16))
    torch.cuda.synchronize()
    assert err.item() == 0
    for i in range(steps):
        assert_close(outs[i].cpu(), refs[i], f"step {i}")
    assert np.array_equal(u16(kc), rk) and np.array_equal(u16(vc), rv)


def _rows_per_sequence(c):
    """The case's new rows as one row per sequence (zeros and slot -1 for an
    empty context), the layout of the fused step."""
    ctx = c.pool.context_lens.to(torch.int64)
    B = ctx.shape[0]
    seqs = torch.nonzero(ctx > 0).flatten()
    nk = torch.zeros(B, c.Hk, c.D, dtype=c.dtype)
    nv = torch.zeros(B, c.Hk, c.D, dtype=c.dtype)
    sl = torch.full((B,), -1, dtype=torch.int64)
    nk[seqs], nv[seqs], sl[seqs] = c.new_key, c.new_value, c.slot_mapping
    return nk, nv, sl


@pytest.mark.parametrize("which", ["tiny", "qwen3_8b", "ragged", "f16_d64"])
def test_fused_step_equals_step_and_oracle(cuda_lib, which):
    """pd_decode_step_fused (the decode stores each sequence's new row right
    before copying its block) gives the bits of pd_decode_step, the same
    pools, and the oracle's store-then-decode result."""
    if which == "tiny":
        c = pd_inputs.tiny_decode()
    elif which == "qwen3_8b":
        c = pd_inputs.qwen3_8b_decode()
    elif which == "ragged":
        c = pd_inputs.decode_case("fragged", 92, [1, 0, 16, 17, 64, 65, 999, 2048, 5000], 16, 4,
                                  128, 16, torch.bfloat16, key_outlier_frac=0.05)
    else:
        c = pd_inputs.decode_case("f16d64", 93, [1, 8, 9, 63, 64, 65, 129, 700], 8, 2, 64, 8,
                                  torch.float16)
    dev = torch.device("cuda")
    nk, nv, sl = _rows_per_sequence(c)
    q, bt, cl = c.q.to(dev), c.pool.block_tables.to(dev), c.pool.context_lens.to(dev)
    ws = cuda_lib.decode_workspace(c.B, c.H, c.D, c.max_context_len)
    err = device_err()
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    out = torch.empty_like(q)
    cuda_lib.pd_decode_step_fused(out, q, kc, vc, bt, cl, c.max_context_len, c.scale,
                                  nk.to(dev), nv.to(dev), sl.to(dev), workspace=ws, dev_err=err)
    kc2, vc2 = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    ref_out = torch.empty_like(q)
    cuda_lib.pd_decode_step(ref_out, q, kc2, vc2, bt, cl, c.max_context_len, c.scale,
                            c.new_key.to(dev), c.new_value.to(dev), c.slot_mapping.to(dev),
                            workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc2.view(torch.int16))
    rows = (0, 64) if which == "qwen3_8b" else None
    ref, rk, rv = oracle_store_and_decode(c, rows=rows)
    g = out.cpu()
    if rows:
        g = g.reshape(-1, c.D)[rows[0]:rows[1]]
        ref = ref.reshape(-1, c.D)[rows[0]:rows[1]]
    assert_close(g, ref, f"fused step {which}")
    assert np.array_equal(u16(kc), rk) and np.array_equal(u16(vc), rv)


def test_fused_step_flags_a_slot_off_the_last_token(cuda_lib):
    """A slot that is not the one of the sequence's last token is not stored
    and flags PD_DEVERR_STEP_SLOT; the other sequences' rows are stored."""
    c = pd_inputs.decode_case("fbad", 94, [40, 100, 300], 8, 2, 128, 16, torch.bfloat16,
                              poison=False)
    dev = torch.device("cuda")
    nk, nv, sl = _rows_per_sequence(c)
    bad = sl.clone()
    bad[1] = pd_inputs.slot_mapping_for(c.pool.block_tables, [1], [10], 16)[0]   # token 10
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    err = device_err()
    out = torch.empty_like(c.q.to(dev))
    cuda_lib.pd_decode_step_fused(out, c.q.to(dev), kc, vc, c.pool.block_tables.to(dev),
                                  c.pool.context_lens.to(dev), c.max_context_len, c.scale,
                                  nk.to(dev), nv.to(dev), bad.to(dev),
                                  workspace=cuda_lib.decode_workspace(c.B, c.H, c.D,
                                                                      c.max_context_len),
                                  dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == cuda_lib.PD_DEVERR_STEP_SLOT
    rk, rv = u16(c.pool.key_cache), u16(c.pool.value_cache)
    keep = torch.tensor([0, 2])
    oracle.reshape_and_cache(nk[keep], nv[keep], rk, rv, sl[keep], 16)
    assert np.array_equal(u16(kc), rk) and np.array_equal(u16(vc), rv)


@pytest.mark.parametrize("T", [48, 256, 300])
def test_step_storing_early_tokens(cuda_lib, T):
    """The store writes T tokens at random positions of the sequences (early
    blocks included, several per sequence), each slot NaN in the pool until
    then: the decode grid, started while the store grid runs, must not read
    any of them before the store has written it (a read ahead would give
    NaN), and three runs of the step give the same bits."""
    B, H, Hk, D, S = 64, 32, 8, 128, 16
    g = torch.Generator().manual_seed(90 + T)
    ctx = torch.randint(64, 2049, (B,), generator=g)
    c = pd_inputs.decode_case("early", 91, ctx.tolist(), H, Hk, D, S, torch.bfloat16,
                              store_last=False, poison=False)
    bt = c.pool.block_tables
    # T distinct (sequence, position) pairs, position 0 of the first sequences included
    seqs = torch.randint(0, B, (T,), generator=g)
    pos = (torch.rand(T, generator=g) * ctx[seqs]).long()
    pos[: min(T, 16)] = 0
    seqs[: min(T, 16)] = torch.arange(min(T, 16))
    slots = pd_inputs.slot_mapping_for(bt, seqs, pos, S)
    keep = torch.ones(T, dtype=torch.bool)
    seen = set()
    for i, sl in enumerate(slots.tolist()):
        keep[i] = sl not in seen
        seen.add(sl)
    slots = torch.where(keep, slots, torch.full_like(slots, -1))
    w = slots[slots >= 0]
    c.pool.key_cache[w // S, :, w % S] = float("nan")
    c.pool.value_cache[w // S, :, w % S] = float("nan")
    nk = torch.randn(T, Hk, D, generator=g).to(torch.bfloat16)
    nv = torch.randn(T, Hk, D, generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    rk, rv = u16(c.pool.key_cache), u16(c.pool.value_cache)
    err = device_err()
    ws = cuda_lib.decode_workspace(B, H, D, c.max_context_len)
    outs = []
    for _ in range(3):           # the same step again: the store rewrites the same values
        out = torch.empty(B, H, D, dtype=torch.bfloat16, device=dev)
        cuda_lib.pd_decode_step(out, c.q.to(dev), kc, vc, bt.to(dev),
                                c.pool.context_lens.to(dev), c.max_context_len, c.scale,
                                nk.to(dev), nv.to(dev), slots.to(dev), workspace=ws, dev_err=err)
        outs.append(out)
        if len(outs) == 1:       # the next steps start from the poisoned pool again
            torch.cuda.synchronize()
            kc.copy_(c.pool.key_cache.to(dev))
            vc.copy_(c.pool.value_cache.to(dev))
    torch.cuda.synchronize()
    assert err.item() == 0
    oracle.reshape_and_cache(nk, nv, rk, rv, slots, S)
    assert np.array_equal(u16(kc), rk) and np.array_equal(u16(vc), rv)
    ref = oracle.decode(c.q, rk, rv, bt, c.pool.context_lens, c.scale, oracle.BF16,
                        rows=(0, 64))
    for i, out in enumerate(outs):
        assert not out.isnan().any()
        assert_close(out.cpu().reshape(-1, D)[0:64], ref.reshape(-1, D)[0:64],
                     f"early store T{T} #{i}")
        assert torch.equal(out.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("D", [64, 128])
def test_fp8_step_equals_separate_calls_and_oracle(cuda_lib, D):
    c = pd_inputs.decode_case("fp8step", 64 + D, [1, 17, 64, 65, 700, 2049], 32, 8, D, 16,
                              torch.bfloat16, poison=False)
    kc8, vc8, ks, vs = pd_inputs.fp8_pools(c.pool.key_cache, c.pool.value_cache)
    dev = torch.device("cuda")
    err = device_err()
    ksd, vsd = ks.to(dev), vs.to(dev)
    kg, vg = kc8.to(dev), vc8.to(dev)
    out = _step(cuda_lib, c, kg, vg, dev_err=err, k_scale=ksd, v_scale=vsd)
    kg2, vg2 = kc8.to(dev), vc8.to(dev)
    cuda_lib.pd_reshape_and_cache_fp8(c.new_key.to(dev), c.new_value.to(dev), kg2, vg2,
                                      c.slot_mapping.to(dev), ksd, vsd, dev_err=err)
    sep = torch.empty_like(out)
    cuda_lib.pd_paged_attention_decode_fp8(
        sep, c.q.to(dev), kg2, vg2, ksd, vsd, c.pool.block_tables.to(dev),
        c.pool.context_lens.to(dev), c.max_context_len, c.scale,
        cuda_lib.decode_workspace(c.B, c.H, c.D, c.max_context_len), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out.view(torch.int16), sep.view(torch.int16))
    assert torch.equal(kg, kg2) and torch.equal(vg, vg2)
    rk, rv = kc8.numpy().copy(), vc8.numpy().copy()
    oracle.reshape_and_cache_fp8(c.new_key, c.new_value, odt(c.dtype), rk, rv, c.slot_mapping,
                                 ks, vs, c.pool.S)
    assert np.array_equal(kg.cpu().numpy(), rk) and np.array_equal(vg.cpu().numpy(), rv)
    ref = oracle.decode_fp8(c.q, odt(c.dtype), rk, rv, ks, vs, c.pool.block_tables,
                            c.pool.context_lens, c.scale)
    assert_close(out, ref, f"fp8 step D{D}")


def test_step_without_new_tokens_is_plain_decode(cuda_lib):
    c = pd_inputs.decode_case("nostore", 65, [5, 80, 333], 8, 2, 64, 16, torch.float16,
                              store_last=False)
    dev = torch.device("cuda")
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    out = _step(cuda_lib, c, kc, vc)
    sep, _, _ = gpu_store_and_decode(cuda_lib, c)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), sep.view(torch.int16))


@pytest.mark.parametrize("graph,fused", [(False, False), (True, False), (True, True)])
def test_host_decode_step_replays(cuda_lib, graph, fused):
    """DecodeStep: inputs written into its pinned views, one call per step.
    Six steps with new tokens, queries and context lengths each time; with a
    CUDA graph the decode replays with its launch tag fixed at capture, so
    this also checks that the merge counters come back to zero."""
    pd = cuda_lib
    steps, B, H, Hk, D, S = 6, 8, 16, 4, 128, 16
    ctx0 = torch.tensor([1, 40, 64, 65, 300, 700, 1500, 2100])
    c = pd_inputs.decode_case("hoststep", 66, (ctx0 + steps).tolist(), H, Hk, D, S,
                              torch.bfloat16, store_last=False, poison=False)
    bt = c.pool.block_tables
    dev = torch.device("cuda")
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    rk, rv = u16(c.pool.key_cache), u16(c.pool.value_cache)
    mcl = int(ctx0.max()) + steps
    st = pd.DecodeStep(kc, vc, B, H, B, bt.shape[1], mcl, c.scale, torch.bfloat16, graph=graph,
                       fused=fused)
    assert (graph and st.graph is not None) or (not graph and st.graph is None)
    g = torch.Generator().manual_seed(67)
    for i in range(steps):
        lens = (ctx0 + i).to(torch.int32)
        slots = pd_inputs.slot_mapping_for(bt, torch.arange(B), ctx0 - 1 + i, S)
        nk = torch.randn(B, Hk, D, generator=g).to(torch.bfloat16)
        nv = torch.randn(B, Hk, D, generator=g).to(torch.bfloat16)
        q = torch.randn(B, H, D, generator=g).to(torch.bfloat16)
        h = st.host
        h["q"].copy_(q)
        h["key"].copy_(nk)
        h["value"].copy_(nv)
        h["slot_mapping"].copy_(slots)
        h["block_tables"].copy_(bt)
        h["context_lens"].copy_(lens)
        got = st().clone()
        assert st.dev_err.item() == 0
        oracle.reshape_and_cache(nk, nv, rk, rv, slots, S)
        ref = oracle.decode(q, rk, rv, bt, lens, c.scale, oracle.BF16)
        assert_close(got, ref, f"host step {i} graph={graph} fused={fused}")
    assert np.array_equal(u16(kc), rk) and np.array_equal(u16(vc), rv)
    assert st.h2d_bytes >= (B * H * D + 2 * B * Hk * D) * 2 + B * 8 + bt.numel() * 4 + B * 4
    assert st.d2h_bytes == B * H * D * 2


def test_graph_replayed_decode_matches_eager(cuda_lib):
    """pd_paged_attention_decode captured once and replayed three times gives
    the eager result every time (the tag is the same in every replay)."""
    pd = cuda_lib
    c = pd_inputs.decode_case("replay", 68, [3, 64, 65, 1000, 2500, 7000], 32, 8, 128, 16,
                              torch.bfloat16, store_last=False)
    dev = torch.device("cuda")
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    q, bt, cl = c.q.to(dev), c.pool.block_tables.to(dev), c.pool.context_lens.to(dev)
    ws = pd.decode_workspace(c.B, c.H, c.D, c.max_context_len)
    eager = torch.empty_like(q)
    pd.pd_paged_attention_decode(eager, q, kc, vc, bt, cl, c.max_context_len, c.scale, ws)
    out = torch.zeros_like(q)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pd.pd_paged_attention_decode(out, q, kc, vc, bt, cl, c.max_context_len, c.scale, ws)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_step_with_padding_slots_and_more_tokens_than_sequences(cuda_lib):
    """A step whose store carries padding slots (-1, skipped) and more rows
    than sequences (T = 2B: each sequence's last two tokens), against the
    separate calls and the oracle."""
    pd = cuda_lib
    c = pd_inputs.decode_case("pad", 69, [2, 40, 64, 65, 300], 16, 4, 128, 16, torch.float16,
                              store_last=False)
    B = c.B
    g = torch.Generator().manual_seed(70)
    seqs = torch.arange(B).repeat_interleave(2)
    pos = (c.pool.context_lens.to(torch.int64) - 2).repeat_interleave(2) + torch.tensor([0, 1] * B)
    slots = pd_inputs.slot_mapping_for(c.pool.block_tables, seqs, pos, 16)
    slots[3] = -1                                     # a padding row: skipped
    nk = torch.randn(2 * B, c.Hk, c.D, generator=g).to(torch.float16)
    nv = torch.randn(2 * B, c.Hk, c.D, generator=g).to(torch.float16)
    c.new_key, c.new_value, c.slot_mapping = nk, nv, slots
    dev = torch.device("cuda")
    err = device_err()
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    out = _step(pd, c, kc, vc, dev_err=err)
    sep, kc2, vc2 = gpu_store_and_decode(pd, c)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out.view(torch.int16), sep.view(torch.int16))
    ref, rk, rv = oracle_store_and_decode(c)
    assert_close(out.cpu(), ref, "step with padding")
    assert np.array_equal(u16(kc), rk) and np.array_equal(u16(vc), rv)


def test_copy_bytes_pinned_and_device(cuda_lib):
    """pd_copy_bytes moves bytes exactly between pinned host and device
    buffers, in both directions and device to device."""
    pd = cuda_lib
    g = torch.Generator().manual_seed(71)
    src = torch.randint(0, 256, (820 * 1024 + 48,), generator=g, dtype=torch.int32)
    src = src.to(torch.uint8).pin_memory()
    dev = torch.empty(src.shape, dtype=torch.uint8, device="cuda")
    pd.pd_copy_bytes(dev, src)
    dev2 = torch.empty_like(dev)
    pd.pd_copy_bytes(dev2, dev)
    back = torch.zeros_like(src).pin_memory()
    pd.pd_copy_bytes(back, dev2)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src) and torch.equal(back, src)


def test_host_decode_step_fp8_pools(cuda_lib):
    """DecodeStep over one-byte pools (quantising store, FP8 decode) replayed
    from a CUDA graph: pools bit-exact with the oracle's store, outputs within
    tolerance of the oracle's FP8 decode, over three steps."""
    pd = cuda_lib
    steps, B, H, Hk, D, S = 3, 6, 32, 8, 128, 16
    ctx0 = torch.tensor([1, 30, 64, 65, 500, 1300])
    c = pd_inputs.decode_case("hostfp8", 72, (ctx0 + steps).tolist(), H, Hk, D, S,
                              torch.bfloat16, store_last=False, poison=False)
    kc8, vc8, ks, vs = pd_inputs.fp8_pools(c.pool.key_cache, c.pool.value_cache)
    dev = torch.device("cuda")
    kg, vg = kc8.to(dev), vc8.to(dev)
    rk, rv = kc8.numpy().copy(), vc8.numpy().copy()
    bt = c.pool.block_tables
    mcl = int(ctx0.max()) + steps
    st = pd.DecodeStep(kg, vg, B, H, B, bt.shape[1], mcl, c.scale, torch.bfloat16,
                       k_scale=ks.to(dev), v_scale=vs.to(dev), graph=True)
    g = torch.Generator().manual_seed(73)
    for i in range(steps):
        lens = (ctx0 + i).to(torch.int32)
        slots = pd_inputs.slot_mapping_for(bt, torch.arange(B), ctx0 - 1 + i, S)
        nk = torch.randn(B, Hk, D, generator=g).to(torch.bfloat16)
        nv = torch.randn(B, Hk, D, generator=g).to(torch.bfloat16)
        q = torch.randn(B, H, D, generator=g).to(torch.bfloat16)
        h = st.host
        h["q"].copy_(q)
        h["key"].copy_(nk)
        h["value"].copy_(nv)
        h["slot_mapping"].copy_(slots)
        h["block_tables"].copy_(bt)
        h["context_lens"].copy_(lens)
        got = st().clone()
        assert st.dev_err.item() == 0
        oracle.reshape_and_cache_fp8(nk, nv, oracle.BF16, rk, rv, slots, ks, vs, S)
        ref = oracle.decode_fp8(q, oracle.BF16, rk, rv, ks, vs, bt, lens, c.scale)
        assert_close(got, ref, f"fp8 host step {i}")
    assert np.array_equal(kg.cpu().numpy(), rk) and np.array_equal(vg.cpu().numpy(), rv)
