"""Speculative verification (multi-query decode): k + 1 query tokens per
sequence against the paged cache, causal among themselves, run through
pd_paged_prefill_chunk with every chunk length = k + 1.  Parity against the
oracle for several k, head groupings and element types; a one-token verify
equals decode; and the bench's batch (64 sequences, 4 queries each) is checked
on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import ATOL, RTOL, assert_close, device_err, odt, u16

pytestmark = pytest.mark.gpu


def _run(pd, m):
    dev = torch.device("cuda")
    kc, vc = m.pool.key_cache.to(dev), m.pool.value_cache.to(dev)
    err = device_err()
    pd.pd_reshape_and_cache(m.new_key.to(dev), m.new_value.to(dev), kc, vc,
                            m.slot_mapping.to(dev), dev_err=err)
    q = m.q_prefill.to(dev)
    out = torch.full_like(q, float("nan"))
    pd.pd_paged_prefill_chunk(out, q, m.cu_q_lens.to(dev), m.max_q_len, kc, vc,
                              m.pool.block_tables[:m.Bp].to(dev),
                              m.pool.context_lens[:m.Bp].to(dev), m.scale, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return out.cpu(), kc, vc


def _oracle(m, tokens=None):
    """Oracle output [tokens, H, D] (all tokens, or the range ``tokens``)."""
    kc, vc = u16(m.pool.key_cache), u16(m.pool.value_cache)
    oracle.reshape_and_cache(m.new_key, m.new_value, kc, vc, m.slot_mapping, m.pool.S)
    rows = None if tokens is None else np.arange(tokens[0] * m.H, tokens[1] * m.H)
    ref = oracle.prefill(m.q_prefill, m.cu_q_lens, kc, vc, m.pool.block_tables[:m.Bp],
                         m.pool.context_lens[:m.Bp], m.scale, odt(m.dtype), rows=rows)
    return ref if tokens is None else ref.reshape(tokens[1] - tokens[0], m.H, m.D)


@pytest.mark.parametrize("n_q,H,Hk,dtype", [(2, 32, 8, torch.bfloat16), (4, 32, 8, torch.bfloat16),
                                            (8, 16, 2, torch.float16), (3, 8, 8, torch.float16),
                                            (5, 32, 2, torch.bfloat16)])
def test_verify_matches_oracle(cuda_lib, n_q, H, Hk, dtype):
    m = pd_inputs.spec_verify(seed=n_q, B=6, n_q=n_q, lo=1, hi=700, H=H, Hk=Hk, D=128, S=16,
                              dtype=dtype)
    out, _, _ = _run(cuda_lib, m)
    assert_close(out, _oracle(m), f"verify n_q={n_q}")


def test_single_query_verify_equals_decode(cuda_lib):
    """n_q = 1 is a decode step: the prefill path agrees with the decode
    kernel within the tolerance (both against the same oracle)."""
    pd = cuda_lib
    m = pd_inputs.spec_verify(seed=9, B=8, n_q=1, lo=50, hi=900)
    out, kc, vc = _run(pd, m)
    dev = torch.device("cuda")
    q = m.q_prefill.to(dev)
    cl = m.pool.context_lens[:m.Bp].to(dev)
    mcl = int(m.pool.context_lens[:m.Bp].max())
    dec = torch.empty_like(q)
    pd.pd_paged_attention_decode(dec, q, kc, vc, m.pool.block_tables[:m.Bp].to(dev), cl, mcl,
                                 m.scale, pd.decode_workspace(m.Bp, m.H, m.D, mcl))
    torch.cuda.synchronize()
    ref = _oracle(m)
    assert_close(out, ref, "verify n_q=1")
    assert_close(dec.cpu(), ref, "decode")


def test_bench_batch_sampled_rows(cuda_lib):
    m = pd_inputs.spec_verify()
    out, _, _ = _run(cuda_lib, m)
    assert torch.isfinite(out.float()).all()
    tokens = (40, 72)                     # sequences 10..17
    ref = _oracle(m, tokens)
    assert_close(out[tokens[0]:tokens[1]], ref, "verify bench rows")


# ---- the dedicated verify path: the decode kernel with (head, query) columns

def _verify(pd, m, context_lens=None, dev_err=None):
    dev = torch.device("cuda")
    kc, vc = m.pool.key_cache.to(dev), m.pool.value_cache.to(dev)
    pd.pd_reshape_and_cache(m.new_key.to(dev), m.new_value.to(dev), kc, vc,
                            m.slot_mapping.to(dev))
    nq = m.max_q_len
    q = m.q_prefill.reshape(m.Bp, nq, m.H, m.D).to(dev)
    out = torch.full_like(q, float("nan"))
    cl = m.pool.context_lens[:m.Bp] if context_lens is None else context_lens
    mcl = int(cl.max())
    pd.pd_paged_attention_verify(out, q, kc, vc, m.pool.block_tables[:m.Bp].to(dev),
                                 cl.to(dev), mcl, m.scale,
                                 pd.verify_workspace(m.Bp, nq, m.H, m.D, mcl), dev_err=dev_err)
    torch.cuda.synchronize()
    return out.reshape(-1, m.H, m.D).cpu()


@pytest.mark.parametrize("n_q,H,Hk,D,dtype", [(2, 32, 8, 128, torch.bfloat16),
                                              (4, 32, 8, 128, torch.bfloat16),
                                              (8, 16, 2, 128, torch.float16),
                                              (3, 8, 8, 64, torch.float16),
                                              (5, 32, 2, 128, torch.bfloat16),
                                              (4, 16, 4, 64, torch.bfloat16),
                                              (7, 12, 4, 128, torch.float16)])
def test_verify_kernel_matches_oracle(cuda_lib, n_q, H, Hk, D, dtype):
    m = pd_inputs.spec_verify(seed=20 + n_q, B=7, n_q=n_q, lo=1, hi=1500, H=H, Hk=Hk, D=D,
                              S=16, dtype=dtype)
    err = device_err()
    out = _verify(cuda_lib, m, dev_err=err)
    assert err.item() == 0
    assert_close(out, _oracle(m), f"verify kernel n_q={n_q} H{H} Hk{Hk} D{D}")


@pytest.mark.parametrize("S", [8, 32, 64])
def test_verify_kernel_block_sizes_and_long_contexts(cuda_lib, S):
    m = pd_inputs.mixed_case(30 + S, [0, 3, S - 4, 3000, 9000], [4] * 5, [], 32, 8, 128, S,
                             torch.bfloat16)
    assert_close(_verify(cuda_lib, m), _oracle(m), f"verify S{S}")


def test_verify_one_query_equals_decode(cuda_lib):
    """nq = 1 goes through the decode path itself: bit-identical."""
    pd = cuda_lib
    m = pd_inputs.spec_verify(seed=31, B=8, n_q=1, lo=50, hi=900)
    out = _verify(pd, m)
    dev = torch.device("cuda")
    kc, vc = m.pool.key_cache.to(dev), m.pool.value_cache.to(dev)
    pd.pd_reshape_and_cache(m.new_key.to(dev), m.new_value.to(dev), kc, vc,
                            m.slot_mapping.to(dev))
    q = m.q_prefill.to(dev)
    cl = m.pool.context_lens[:m.Bp]
    mcl = int(cl.max())
    dec = torch.empty_like(q)
    pd.pd_paged_attention_decode(dec, q, kc, vc, m.pool.block_tables[:m.Bp].to(dev), cl.to(dev),
                                 mcl, m.scale, pd.decode_workspace(m.Bp, m.H, m.D, mcl))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), dec.cpu().view(torch.int16))


def test_verify_kernel_bench_batch_sampled_rows(cuda_lib):
    m = pd_inputs.spec_verify()
    out = _verify(cuda_lib, m)
    assert torch.isfinite(out.float()).all()
    tokens = (100, 140)                   # sequences 25..34
    assert_close(out[tokens[0]:tokens[1]], _oracle(m, tokens), "verify kernel bench rows")


def test_verify_empty_and_short_contexts(cuda_lib):
    """An empty context gives zero rows; a context shorter than nq is flagged
    and its queries that see no key read 0; the other sequences are exact."""
    pd = cuda_lib
    nq = 4
    m = pd_inputs.spec_verify(seed=32, B=4, n_q=nq, lo=20, hi=300)
    ref = _oracle(m).reshape(m.Bp, nq, m.H, m.D)
    cl = m.pool.context_lens[:m.Bp].clone()
    cl[1] = 0
    err = device_err()
    out = _verify(pd, m, context_lens=cl, dev_err=err).reshape(m.Bp, nq, m.H, m.D)
    assert err.item() == 0
    assert (out[1] == 0).all()
    for i in (0, 2, 3):
        assert_close(out[i], ref[i], f"seq {i} beside an empty one")
    cl[2] = 2                             # two keys for four queries: flagged
    out = _verify(pd, m, context_lens=cl, dev_err=err).reshape(m.Bp, nq, m.H, m.D)
    assert err.item() & 0x4
    assert (out[2, :2] == 0).all()        # queries at positions -2, -1
    assert torch.isfinite(out[2, 2:].float()).all()


@pytest.mark.parametrize("n_q", [1, 4])
def test_verify_step_equals_separate_calls_and_oracle(cuda_lib, n_q):
    """pd_verify_step (store the drafts, then verify as a dependent grid) is
    bit-identical to the store followed by the verify, and within tolerance
    of the oracle."""
    pd = cuda_lib
    m = pd_inputs.spec_verify(seed=40 + n_q, B=9, n_q=n_q, lo=1, hi=900)
    dev = torch.device("cuda")
    kc, vc = m.pool.key_cache.to(dev), m.pool.value_cache.to(dev)
    q = m.q_prefill.reshape(m.Bp, n_q, m.H, m.D).to(dev)
    cl = m.pool.context_lens[:m.Bp]
    mcl = int(cl.max())
    out = torch.full_like(q, float("nan"))
    err = device_err()
    pd.pd_verify_step(out, q, kc, vc, m.pool.block_tables[:m.Bp].to(dev), cl.to(dev), mcl, m.scale,
                      m.new_key.to(dev), m.new_value.to(dev), m.slot_mapping.to(dev),
                      workspace=pd.verify_workspace(m.Bp, n_q, m.H, m.D, mcl), dev_err=err)
    sep = _verify(pd, m)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = out.reshape(-1, m.H, m.D).cpu()
    assert torch.equal(got.view(torch.int16), sep.view(torch.int16))
    assert_close(got, _oracle(m), f"verify step n_q={n_q}")
