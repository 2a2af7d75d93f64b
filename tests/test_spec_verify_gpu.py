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
