"""Helpers for GPU-vs-oracle parity tests.

Tolerance for attention outputs (fp32 accumulation, fp16/bf16 inputs and
outputs): an element passes when |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|,
the combined (allclose) reading of "max-abs 2e-3 with max-rel 1e-2".  A
literal max-abs of 2e-3 cannot hold for bf16 outputs above 0.5 in magnitude
because rounding the output alone costs up to 2^-9 of it.  Store, copy and
block bookkeeping are compared bit for bit.
"""
import numpy as np
import torch

import oracle

ATOL = 2e-3
RTOL = 1e-2


def odt(dtype) -> int:
    return oracle.BF16 if dtype == torch.bfloat16 else oracle.F16


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


# One record per comparison made in this process: (what, elements, max abs
# error, max rel error over |oracle| >= 1e-3, failing elements, largest
# err / (atol + rtol |oracle|)).  The conftest prints them at the end of a run,
# so a passing run still shows how close each case came to the bound.
RECORDS: list = []


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str, atol=ATOL, rtol=RTOL):
    g = gpu.detach().cpu().to(torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(ref).all(), f"{what}: oracle produced non-finite values"
    err = np.abs(g - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))       # NaN counts as bad
    if err.size:
        big = np.abs(ref) >= 1e-3
        RECORDS.append((what, int(err.size), float(np.nanmax(err)),
                        float(np.nanmax(err[big] / np.abs(ref[big]))) if big.any() else 0.0,
                        int(bad.sum()), float(np.nanmax(err / (atol + rtol * np.abs(ref))))))
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        rel = err / np.maximum(np.abs(ref), 1e-30)
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements out of tolerance; "
            f"max abs {np.nanmax(err):.3e}, max rel {np.nanmax(rel):.3e}; first at {idx}")
    return float(err.max()) if err.size else 0.0


def device_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def gpu_store_and_decode(pd, c, use_store=True, workspace=None, dev_err=None, kc=None, vc=None):
    """Run the case's store (if any) then decode on cuda:0; returns
    (out, key_cache, value_cache) on the device."""
    dev = torch.device("cuda")
    if kc is None:
        kc = c.pool.key_cache.to(dev)
        vc = c.pool.value_cache.to(dev)
    if use_store and c.slot_mapping.numel():
        pd.pd_reshape_and_cache(c.new_key.to(dev), c.new_value.to(dev), kc, vc,
                                c.slot_mapping.to(dev), dev_err=dev_err)
    q = c.q.to(dev)
    out = torch.empty_like(q)
    mcl = c.max_context_len
    if workspace is None:
        workspace = pd.decode_workspace(c.B, c.H, c.D, mcl)
    pd.pd_paged_attention_decode(out, q, kc, vc, c.pool.block_tables.to(dev),
                                 c.pool.context_lens.to(dev), mcl, c.scale, workspace,
                                 dev_err=dev_err)
    return out, kc, vc


def oracle_store_and_decode(c, use_store=True, rows=None):
    kc, vc = u16(c.pool.key_cache), u16(c.pool.value_cache)
    if use_store and c.slot_mapping.numel():
        oracle.reshape_and_cache(c.new_key, c.new_value, kc, vc, c.slot_mapping, c.pool.S)
    ref = oracle.decode(c.q, kc, vc, c.pool.block_tables, c.pool.context_lens, c.scale,
                        odt(c.dtype), rows=rows)
    return ref, kc, vc
