"""GPU parity of chunked-prefill attention (tcgen05) against the float64
oracle: small mixes checked in full over shapes, GQA groupings, block sizes
and element types; the full-size 16 x 512 chunk mix on sampled rows; exact
single-key results, causality at tile edges, block-permutation invariance
and flagged bad inputs."""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import assert_close, device_err, odt, u16

pytestmark = pytest.mark.gpu


def _run(pd, m, dev_err=None, kc=None, vc=None):
    dev = torch.device("cuda")
    if kc is None:
        kc, vc = m.pool.key_cache.to(dev), m.pool.value_cache.to(dev)
        pd.pd_reshape_and_cache(m.new_key.to(dev), m.new_value.to(dev), kc, vc,
                                m.slot_mapping.to(dev))
    q = m.q_prefill.to(dev)
    out = torch.full_like(q, float("nan"))
    pd.pd_paged_prefill_chunk(out, q, m.cu_q_lens.to(dev), m.max_q_len, kc, vc,
                              m.pool.block_tables[:m.Bp].to(dev),
                              m.pool.context_lens[:m.Bp].to(dev), m.scale, dev_err=dev_err)
    torch.cuda.synchronize()
    return out, kc, vc


def _oracle(m, rows=None):
    kc, vc = u16(m.pool.key_cache), u16(m.pool.value_cache)
    oracle.reshape_and_cache(m.new_key, m.new_value, kc, vc, m.slot_mapping, m.pool.S)
    return oracle.prefill(m.q_prefill, m.cu_q_lens, kc, vc, m.pool.block_tables[:m.Bp],
                          m.pool.context_lens[:m.Bp], m.scale, odt(m.dtype), rows=rows)


def _check_full(pd, m, what):
    err = device_err()
    out, _, _ = _run(pd, m, dev_err=err)
    assert_close(out.cpu(), _oracle(m), what)
    assert err.item() == 0
    return out


def test_small_mix(cuda_lib):
    m = pd_inputs.mixed_case(70, [0, 5, 40, 300, 129], [1, 19, 33, 200, 128], [], 32, 8, 128,
                             16, torch.bfloat16)
    _check_full(cuda_lib, m, "small mix")


@pytest.mark.parametrize("H,Hk", [(8, 8), (8, 4), (8, 2), (16, 2), (6, 2), (32, 2)])
def test_gqa_groupings(cuda_lib, H, Hk):
    m = pd_inputs.mixed_case(71 + H, [0, 77, 250], [40, 70, 130], [], H, Hk, 128, 16,
                             torch.bfloat16)
    _check_full(cuda_lib, m, f"H{H} Hk{Hk}")


@pytest.mark.parametrize("S", [8, 16, 32, 64])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_block_sizes_dims_dtypes(cuda_lib, S, D, dtype):
    m = pd_inputs.mixed_case(80 + S + D, [0, 3, 127, 128, 600], [33, 1, 129, 64, 97], [], 8, 2,
                             D, S, dtype)
    _check_full(cuda_lib, m, f"S{S} D{D} {dtype}")


def test_single_key_returns_v_exactly(cuda_lib):
    m = pd_inputs.mixed_case(90, [0, 0], [1, 1], [], 32, 8, 128, 16, torch.bfloat16)
    out, _, _ = _run(cuda_lib, m)
    want = m.new_value.repeat_interleave(4, dim=1)     # [2, H, D]
    assert torch.equal(out.cpu().view(torch.int16), want.view(torch.int16))


def test_last_row_matches_decode(cuda_lib):
    pd = cuda_lib
    m = pd_inputs.mixed_case(91, [1000, 7], [300, 260], [], 32, 8, 128, 16, torch.bfloat16)
    out, kc, vc = _run(pd, m)
    dev = torch.device("cuda")
    last = (m.cu_q_lens[1:] - 1).long()
    q = m.q_prefill[last].to(dev)
    dout = torch.empty_like(q)
    cl = m.pool.context_lens[:m.Bp].to(dev)
    ws = pd.decode_workspace(m.Bp, m.H, m.D, int(cl.max()))
    pd.pd_paged_attention_decode(dout, q, kc, vc, m.pool.block_tables[:m.Bp].to(dev), cl,
                                 int(cl.max()), m.scale, ws)
    torch.cuda.synchronize()
    ref = _oracle(m)[last.numpy()]
    assert_close(out[last.to(dev)].cpu(), ref, "prefill last rows")
    assert_close(dout.cpu(), ref, "decode at ctx = P + C")


def test_block_permutation_gives_identical_bits(cuda_lib):
    pd = cuda_lib
    m = pd_inputs.mixed_case(92, [500, 0, 1234], [100, 64, 300], [], 32, 8, 128, 16,
                             torch.bfloat16)
    out1, kc, vc = _run(pd, m)
    NB = kc.shape[0]
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(5)).cuda()
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    m.pool.block_tables = perm.cpu()[m.pool.block_tables.long()].to(torch.int32)
    out2, _, _ = _run(pd, m, kc=kc2, vc=vc2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_chunked_prefill_mix_full_size_sampled(cuda_lib):
    """The 16 x 512-token chunk mix (prior lengths uniform on [0, 8192]) in the
    launch configuration the benchmark times; sampled rows vs the oracle."""
    m = pd_inputs.chunked_prefill_mixed()
    err = device_err()
    out, kc, vc = _run(cuda_lib, m, dev_err=err)
    assert err.item() == 0
    H = m.H
    rows = []
    cu = m.cu_q_lens.tolist()
    for i in range(m.Bp):
        for j in (0, 1, 31, 32, 33, 127, 128, 255, 256, 300, 480, 511):
            for h in range(0, H, 3):
                rows.append((cu[i] + j) * H + h)
    rows = np.array(rows, dtype=np.int64)
    ref = _oracle(m, rows=rows)
    got = out.cpu().reshape(-1, m.D)[torch.from_numpy(rows)]
    assert_close(got, ref, "chunked prefill mix (sampled)")
    assert torch.isfinite(out.float()).all()


def test_chunked_prefill_mix_decode_part(cuda_lib):
    """The 48 decode sequences of the same step, on the same pool."""
    pd = cuda_lib
    m = pd_inputs.chunked_prefill_mixed()
    dev = torch.device("cuda")
    kc, vc = m.pool.key_cache.to(dev), m.pool.value_cache.to(dev)
    pd.pd_reshape_and_cache(m.new_key.to(dev), m.new_value.to(dev), kc, vc,
                            m.slot_mapping.to(dev))
    bt = m.pool.block_tables[m.Bp:]
    cl = m.pool.context_lens[m.Bp:]
    q = m.q_decode.to(dev)
    out = torch.empty_like(q)
    ws = pd.decode_workspace(m.Bd, m.H, m.D, int(cl.max()))
    pd.pd_paged_attention_decode(out, q, kc, vc, bt.to(dev), cl.to(dev), int(cl.max()),
                                 m.scale, ws)
    torch.cuda.synchronize()
    rk, rv = u16(m.pool.key_cache), u16(m.pool.value_cache)
    oracle.reshape_and_cache(m.new_key, m.new_value, rk, rv, m.slot_mapping, m.pool.S)
    ref = oracle.decode(m.q_decode, rk, rv, bt, cl, m.scale, odt(m.dtype))
    assert_close(out.cpu(), ref, "mix decode part")


def test_bad_inputs_flagged(cuda_lib):
    pd = cuda_lib
    m = pd_inputs.mixed_case(93, [200, 10], [50, 20], [], 8, 2, 64, 16, torch.float16)
    m.pool.block_tables[0, 2] = m.pool.NB + 1
    err = device_err()
    _run(pd, m, dev_err=err)
    assert err.item() & pd.PD_DEVERR_BLOCK_RANGE
    m2 = pd_inputs.mixed_case(94, [20], [50], [], 8, 2, 64, 16, torch.float16)
    m2.pool.context_lens[0] = 10          # shorter than the chunk itself
    err = device_err()
    _run(pd, m2, dev_err=err)
    assert err.item() & pd.PD_DEVERR_CTX_RANGE


def test_repeat_runs_identical(cuda_lib):
    """Same inputs, same bits, run after run: catches reads of tensor memory
    that race the MMAs still accumulating into it.  Chunks end in query tiles
    with one valid token, over 1, 2 and 3 key tiles."""
    pd = cuda_lib
    m = pd_inputs.mixed_case(95, [0, 127, 300], [97, 129, 65], [], 8, 2, 128, 16, torch.bfloat16)
    first, kc, vc = _run(pd, m)
    for _ in range(8):
        again, _, _ = _run(pd, m, kc=kc, vc=vc)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))
    assert_close(first.cpu(), _oracle(m), "repeat mix")


def test_repeated_launches_and_graph_replays(cuda_lib):
    """Many launches in a row, and a launch captured in a CUDA graph and
    replayed, give the eager launch's bits every time, over a batch of many
    short chunks (more tile pairs than SMs, some tile pairs empty)."""
    pd = cuda_lib
    dev = torch.device("cuda")
    m = pd_inputs.mixed_case(96, [0, 40, 300, 900] * 12, [130, 64, 200, 65] * 12, [], 8, 2, 128,
                             16, torch.bfloat16)
    eager, kc, vc = _run(pd, m)
    assert_close(eager.cpu(), _oracle(m), "many items")
    q = m.q_prefill.to(dev)
    cu = m.cu_q_lens.to(dev)
    bt, cl = m.pool.block_tables[:m.Bp].to(dev), m.pool.context_lens[:m.Bp].to(dev)
    err = device_err()
    for _ in range(70):
        out = torch.full_like(q, float("nan"))
        pd.pd_paged_prefill_chunk(out, q, cu, m.max_q_len, kc, vc, bt, cl, m.scale, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    gout = torch.full_like(q, float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        pd.pd_paged_prefill_chunk(gout, q, cu, m.max_q_len, kc, vc, bt, cl, m.scale, dev_err=err)
    for _ in range(4):
        gout.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(gout.view(torch.int16), eager.view(torch.int16))
    assert err.item() == 0
