"""GPU parity of the KV hand-over kernels (pd_kv_pack / pd_kv_unpack): bit-exact
against the oracle over block sizes, head dims and element types; bad ids
flagged and skipped; and the end-to-end property the hand-over exists for:
decode attention over the receiving pool (new block ids) gives the very bits
it gave over the sending pool."""
import numpy as np
import pytest
import torch

import oracle
import pd_inputs
from tests.parity import device_err, u16

pytestmark = pytest.mark.gpu


def _gpu_lists(c, dev):
    return [k.to(dev) for k in c.key_caches], [v.to(dev) for v in c.value_caches]


@pytest.mark.parametrize("Hk,D,S,dtype", [(2, 64, 8, torch.float16), (8, 128, 16, torch.bfloat16),
                                          (4, 128, 32, torch.float16), (1, 64, 64, torch.bfloat16)])
def test_pack_unpack_bit_exact(cuda_lib, Hk, D, S, dtype):
    pd = cuda_lib
    dev = torch.device("cuda")
    c = pd_inputs.kv_transfer(seed=1, L=3, B=3, ctx=5 * S + 3, Hk=Hk, D=D, S=S, dtype=dtype)
    kg, vg = _gpu_lists(c, dev)
    send = c.block_ids(c.send_tables)
    st = pd.kv_staging(c.L, send.numel(), kg[0])
    err = device_err()
    pd.pd_kv_pack(st, kg, vg, send.to(dev), dev_err=err)
    torch.cuda.synchronize()
    ref, bad = oracle.kv_pack([u16(k) for k in c.key_caches], [u16(v) for v in c.value_caches],
                              send.numpy())
    assert bad == 0 and err.item() == 0
    assert np.array_equal(u16(st), ref)
    # unpack into a receiving pool at other ids
    recv = c.block_ids(c.recv_tables)
    g = torch.Generator().manual_seed(2)
    rk = [torch.randn(c.NB_recv, Hk, S, D, generator=g).to(dtype) for _ in range(c.L)]
    rv = [torch.randn(c.NB_recv, Hk, S, D, generator=g).to(dtype) for _ in range(c.L)]
    rkg, rvg = [t.to(dev) for t in rk], [t.to(dev) for t in rv]
    pd.pd_kv_unpack(st, rkg, rvg, recv.to(dev), dev_err=err)
    torch.cuda.synchronize()
    ok, ov = [u16(t) for t in rk], [u16(t) for t in rv]
    assert oracle.kv_unpack(ref, ok, ov, recv.numpy()) == 0
    assert err.item() == 0
    for l in range(c.L):
        assert np.array_equal(u16(rkg[l]), ok[l]) and np.array_equal(u16(rvg[l]), ov[l])


def test_bad_ids_flagged_and_skipped(cuda_lib):
    pd = cuda_lib
    dev = torch.device("cuda")
    c = pd_inputs.kv_transfer(seed=4, L=2, B=2, ctx=40, Hk=2, D=64, S=8, dtype=torch.float16)
    kg, vg = _gpu_lists(c, dev)
    ids = torch.tensor([3, -1, c.NB, 0], dtype=torch.int32)
    st = torch.full((c.L, 2, 4, c.Hk, c.S, c.D), 7.0, dtype=torch.float16, device=dev)
    err = device_err()
    pd.pd_kv_pack(st, kg, vg, ids.to(dev), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & 0x2                        # PD_DEVERR_BLOCK_RANGE
    ref = st.cpu().clone()
    for l in range(c.L):
        ref[l, 0, 0], ref[l, 1, 0] = c.key_caches[l][3], c.value_caches[l][3]
        ref[l, 0, 3], ref[l, 1, 3] = c.key_caches[l][0], c.value_caches[l][0]
    assert np.array_equal(u16(st), u16(ref))       # skipped slabs untouched


def test_decode_after_handover_is_bit_identical(cuda_lib):
    """Prefill side: pool A, tables A.  Pack the sequences' blocks, unpack them
    into pool B at the receiver's ids, decode with tables B: same bits."""
    pd = cuda_lib
    dev = torch.device("cuda")
    c = pd_inputs.kv_transfer(seed=5, L=2, B=5, ctx=700, Hk=8, D=128, S=16,
                              dtype=torch.bfloat16)
    kg, vg = _gpu_lists(c, dev)
    send, recv = c.block_ids(c.send_tables), c.block_ids(c.recv_tables)
    st = pd.kv_staging(c.L, send.numel(), kg[0])
    pd.pd_kv_pack(st, kg, vg, send.to(dev))
    rk = [torch.zeros(c.NB_recv, c.Hk, c.S, c.D, dtype=c.dtype, device=dev) for _ in range(c.L)]
    rv = [torch.zeros_like(t) for t in rk]
    pd.pd_kv_unpack(st, rk, rv, recv.to(dev))
    H = 32
    q = torch.randn(c.context_lens.numel(), H, c.D, generator=torch.Generator().manual_seed(6))
    q = q.to(c.dtype).to(dev)
    cl = c.context_lens.to(dev)
    mcl = int(c.context_lens.max())
    ws = pd.decode_workspace(q.shape[0], H, c.D, mcl)
    for l in range(c.L):
        oa, ob = torch.empty_like(q), torch.empty_like(q)
        pd.pd_paged_attention_decode(oa, q, kg[l], vg[l], c.send_tables.to(dev), cl, mcl,
                                     c.D ** -0.5, ws)
        pd.pd_paged_attention_decode(ob, q, rk[l], rv[l], c.recv_tables.to(dev), cl, mcl,
                                     c.D ** -0.5, ws)
        torch.cuda.synchronize()
        assert np.array_equal(u16(oa), u16(ob))
        assert torch.isfinite(oa.float()).all()


def test_full_size_transfer_sampled(cuda_lib):
    """The bench's hand-over (32 layers, 4 x 2048 tokens, Qwen3-8B kv shape):
    every staged slab equals its source block, checked on the device."""
    pd = cuda_lib
    dev = torch.device("cuda")
    c = pd_inputs.kv_transfer(seed=0, device=dev)
    send, recv = c.block_ids(c.send_tables).to(dev), c.block_ids(c.recv_tables).to(dev)
    st = pd.kv_staging(c.L, send.numel(), c.key_caches[0])
    err = device_err()
    pd.pd_kv_pack(st, c.key_caches, c.value_caches, send, dev_err=err)
    rk = [torch.empty(c.NB_recv, c.Hk, c.S, c.D, dtype=c.dtype, device=dev) for _ in range(c.L)]
    rv = [torch.empty_like(t) for t in rk]
    pd.pd_kv_unpack(st, rk, rv, recv, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for l in range(c.L):
        assert torch.equal(st[l, 0].view(torch.int16), c.key_caches[l][send.long()].view(torch.int16))
        assert torch.equal(st[l, 1].view(torch.int16), c.value_caches[l][send.long()].view(torch.int16))
        assert torch.equal(rk[l][recv.long()].view(torch.int16), c.key_caches[l][send.long()].view(torch.int16))
        assert torch.equal(rv[l][recv.long()].view(torch.int16), c.value_caches[l][send.long()].view(torch.int16))
