"""The allocation-free decode entry point, pd_paged_attention_decode_noalloc.

It serves callers that cannot allocate device memory on the call path (for
example an engine that reserves all device memory at start-up): the library
keeps the partition scratch in its own fixed array.  These tests call it
through the C ABI twice in a row, on two different batches, and compare each
result with the regular entry point, which takes a caller-allocated
workspace.  Both run the same kernel with the same split of the work, so the
outputs must be bit-identical, not merely within the attention tolerance.
This file is collected last so that, if it fails, every other test has
already run.
"""
import pytest
import torch

import pd_inputs
from tests.parity import device_err

pytestmark = pytest.mark.gpu


def _both(pd, c):
    dev = torch.device("cuda")
    kc, vc = c.pool.key_cache.to(dev), c.pool.value_cache.to(dev)
    pd.pd_reshape_and_cache(c.new_key.to(dev), c.new_value.to(dev), kc, vc,
                            c.slot_mapping.to(dev))
    q = c.q.to(dev)
    bt, cl = c.pool.block_tables.to(dev), c.pool.context_lens.to(dev)
    mcl = c.max_context_len
    ref = torch.empty_like(q)
    ws = pd.decode_workspace(c.B, c.H, c.D, mcl)
    pd.pd_paged_attention_decode(ref, q, kc, vc, bt, cl, mcl, c.scale, ws)
    got = torch.full_like(q, float("nan"))
    err = device_err()
    pd.pd_paged_attention_decode_noalloc(got, q, kc, vc, bt, cl, mcl, c.scale, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return got, ref


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    # two calls in a row: the second batch has other shapes, so it runs over
    # the scratch the first call left behind
    cases = [pd_inputs.qwen3_8b_decode(seed=11, B=24),
             pd_inputs.decode_case("noalloc2", 12, [1, 300, 2000, 4097, 0, 17], 16, 4, 64, 8,
                                   torch.float16)]
    for c in cases:
        assert cuda_lib.pd_decode_workspace_bytes(c.B, c.H, c.D, c.max_context_len) > 0
        got, ref = _both(cuda_lib, c)
        assert torch.isfinite(got.float()).all()
        # same kernel, same work split: the 16-bit payloads match bit for bit
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_batches_beyond_its_scratch(cuda_lib):
    dev = torch.device("cuda")
    B, H, Hk, D, S = 64, 32, 8, 128, 16
    mcl = 65536                          # workspace far above 32 MiB
    assert cuda_lib.pd_decode_workspace_bytes(B, H, D, mcl) > 32 << 20
    q = torch.zeros(B, H, D, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(4, Hk, S, D, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(B, 1, dtype=torch.int32, device=dev)
    cl = torch.ones(B, dtype=torch.int32, device=dev)
    n0 = cuda_lib.launch_count()
    with pytest.raises(cuda_lib.PDError) as e:
        cuda_lib.pd_paged_attention_decode_noalloc(torch.empty_like(q), q, kc, kc, bt, cl, mcl,
                                                   0.1)
    assert e.value.status == 5            # PD_ERR_WORKSPACE_TOO_SMALL
    assert cuda_lib.launch_count() == n0  # nothing launched
