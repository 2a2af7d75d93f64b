"""Seeded synthetic workloads for paged KV-cache attention.

Shared by the tests, ``bench.py`` and the smoke check; used both by the CUDA
path and by the oracle.  It holds no attention arithmetic: it only draws
random tensors, block tables and lengths, and lays tokens out in the paged
cache format [num_blocks, num_kv_heads, block_size, head_dim] (logical token
t of a sequence sits in physical block block_table[t // S] at offset t % S).

Every generator takes an explicit seed and draws on the CPU with a
``torch.Generator`` (bit-identical data for the oracle and the GPU), except
where ``device`` names a CUDA device: that path is only for
performance-only workloads too large to draw on the host.

Poisoning: slots that no sequence may read are set to NaN, so any stray read
by a kernel shows up as NaN in its output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randint(g: torch.Generator, lo: int, hi: int, n: int) -> torch.Tensor:
    """n integers uniform on [lo, hi], both ends inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64)


@dataclass
class PagedPool:
    key_cache: torch.Tensor          # [NB, Hk, S, D]
    value_cache: torch.Tensor        # [NB, Hk, S, D]
    block_tables: torch.Tensor       # int32 [B, max_blocks]
    context_lens: torch.Tensor       # int32 [B]
    S: int
    NB: int
    pad_block: int                   # id used to pad table rows (-1 if none)
    valid: torch.Tensor = field(repr=False, default=None)  # bool [NB, S]


def blocks_needed(ctx: torch.Tensor, S: int) -> torch.Tensor:
    return (ctx + S - 1) // S


def make_block_tables(g: torch.Generator, ctx: torch.Tensor, S: int,
                      NB: int | None = None, pool_factor: float = 1.5):
    """Scatter each sequence's logical blocks over a random permutation of the
    pool.  Returns (block_tables int32 [B, max_blocks], NB, pad_block).  Rows
    are padded with an unused block id (poisoned by ``fill_pool``) when the
    pool has one, else with -1."""
    nb = blocks_needed(ctx, S)
    needed = int(nb.sum())
    if NB is None:
        NB = max(needed, int(math.ceil(pool_factor * needed)))
    assert NB >= needed
    perm = torch.randperm(NB, generator=g, dtype=torch.int64)
    max_blocks = max(1, int(nb.max()))
    pad = int(perm[needed]) if NB > needed else -1
    bt = torch.full((ctx.shape[0], max_blocks), pad, dtype=torch.int32)
    start = 0
    for i, n in enumerate(nb.tolist()):
        bt[i, :n] = perm[start:start + n].to(torch.int32)
        start += n
    return bt, NB, pad


def valid_slots(bt: torch.Tensor, ctx: torch.Tensor, S: int, NB: int) -> torch.Tensor:
    """bool [NB, S]: True where some sequence keeps a token (t < ctx)."""
    valid = torch.zeros(NB, S, dtype=torch.bool)
    for i in range(bt.shape[0]):
        c = int(ctx[i])
        if c <= 0:
            continue
        n = (c + S - 1) // S
        blocks = bt[i, :n].long()
        valid[blocks[:-1]] = True
        valid[blocks[-1], : c - (n - 1) * S] = True
    return valid


def fill_pool(g: torch.Generator, NB: int, Hk: int, S: int, D: int, dtype,
              valid: torch.Tensor | None = None, key_outlier_frac: float = 0.0,
              key_outlier_scale: float = 8.0, device="cpu"):
    """K, V ~ N(0, 1) rounded to ``dtype``.  A fraction of key vectors (each
    (block, head, offset) independently) is multiplied by ``key_outlier_scale``.
    Slots outside ``valid`` become NaN."""
    k = torch.randn(NB, Hk, S, D, generator=g, device=device)
    v = torch.randn(NB, Hk, S, D, generator=g, device=device)
    if key_outlier_frac > 0:
        sel = torch.rand(NB, Hk, S, 1, generator=g, device=device) < key_outlier_frac
        k = torch.where(sel, k * key_outlier_scale, k)
    k, v = k.to(dtype), v.to(dtype)
    if valid is not None:
        bad = (~valid.to(device)).view(NB, 1, S, 1)
        k.masked_fill_(bad, float("nan"))
        v.masked_fill_(bad, float("nan"))
    return k, v


def make_pool(g, ctx: torch.Tensor, Hk: int, D: int, S: int, dtype, NB=None,
              pool_factor=1.5, poison=True, key_outlier_frac=0.0) -> PagedPool:
    bt, NB, pad = make_block_tables(g, ctx, S, NB, pool_factor)
    valid = valid_slots(bt, ctx, S, NB)
    k, v = fill_pool(g, NB, Hk, S, D, dtype, valid if poison else None,
                     key_outlier_frac)
    return PagedPool(k, v, bt, ctx.to(torch.int32), S, NB, pad, valid)


def slot_mapping_for(bt: torch.Tensor, seq_idx, positions, S: int) -> torch.Tensor:
    """Physical slot of each (sequence, position) pair, from the block table."""
    seq_idx = torch.as_tensor(seq_idx, dtype=torch.int64)
    positions = torch.as_tensor(positions, dtype=torch.int64)
    return bt[seq_idx, positions // S].to(torch.int64) * S + positions % S


@dataclass
class DecodeCase:
    name: str
    q: torch.Tensor                  # [B, H, D]
    pool: PagedPool
    new_key: torch.Tensor            # [T, Hk, D]  stored before the attention
    new_value: torch.Tensor
    slot_mapping: torch.Tensor       # int64 [T]
    H: int
    Hk: int
    D: int
    scale: float
    dtype: torch.dtype

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def max_context_len(self):
        return int(self.pool.context_lens.max())


def decode_case(name, seed, ctx, H, Hk, D, S, dtype, NB=None, pool_factor=1.5,
                poison=True, key_outlier_frac=0.0, store_last=True) -> DecodeCase:
    """Decode workload: a paged pool holding ctx[i] tokens per sequence, one
    query token per sequence, and (``store_last``) the token at position
    ctx-1 given as a new K/V to store before the attention (its slot is
    poisoned in the pool so a missed store shows up)."""
    g = _gen(seed)
    ctx = torch.as_tensor(ctx, dtype=torch.int64)
    pool = make_pool(g, ctx, Hk, D, S, dtype, NB, pool_factor, poison, key_outlier_frac)
    B = ctx.shape[0]
    q = torch.randn(B, H, D, generator=g).to(dtype)
    if store_last:
        seqs = torch.nonzero(ctx > 0).flatten()
        pos = ctx[seqs] - 1
        slots = slot_mapping_for(pool.block_tables, seqs, pos, S)
        nk = torch.randn(seqs.shape[0], Hk, D, generator=g).to(dtype)
        nv = torch.randn(seqs.shape[0], Hk, D, generator=g).to(dtype)
        if poison:
            blk, off = slots // S, slots % S
            pool.key_cache[blk, :, off] = float("nan")
            pool.value_cache[blk, :, off] = float("nan")
    else:
        slots = torch.zeros(0, dtype=torch.int64)
        nk = torch.zeros(0, Hk, D, dtype=dtype)
        nv = torch.zeros(0, Hk, D, dtype=dtype)
    return DecodeCase(name, q, pool, nk, nv, slots, H, Hk, D, 1.0 / math.sqrt(D), dtype)


@dataclass
class ForkedDecodeCase(DecodeCase):
    """A decode batch made of groups of forks: group g is sequences
    group_starts[g] .. group_starts[g+1]-1, whose block tables hold the same
    physical blocks for the first prefix_lens[g] // S blocks."""
    group_starts: torch.Tensor = None    # int32 [n_groups + 1]
    shared_lens: torch.Tensor = None     # int32 [n_groups], tokens (the prompt length)


def forked_decode(name: str, seed: int, groups, H: int, Hk: int, D: int, S: int, dtype,
                  pool_factor: float = 1.25, poison: bool = True) -> ForkedDecodeCase:
    """groups: list of (prompt_len, [ctx of each fork]).  The prompt's full
    blocks are shared by all forks of the group (one set of physical blocks);
    from there on each fork owns its blocks, and the prompt's partial last
    block is copied into every fork's first own block (as copy-on-write leaves
    it).  Blocks are scattered over a random permutation of the pool; slots no
    fork may read are NaN.  Each fork whose last token lies in an own block
    gets that token as a new K/V to store before the attention."""
    g = _gen(seed)
    nshared = [P // S for P, _ in groups]
    own = [[max(0, (c + S - 1) // S - ns) for c in ctxs] for ns, (_, ctxs) in zip(nshared, groups)]
    needed = sum(nshared) + sum(sum(o) for o in own)
    NB = max(needed + 1, int(math.ceil(pool_factor * needed)))
    perm = torch.randperm(NB, generator=g, dtype=torch.int64).to(torch.int32)
    ctx_all = [c for _, ctxs in groups for c in ctxs]
    B = len(ctx_all)
    max_blocks = max(1, max((c + S - 1) // S for c in ctx_all) if ctx_all else 1)
    pad = int(perm[needed])
    bt = torch.full((B, max_blocks), pad, dtype=torch.int32)
    nxt, row, starts = 0, 0, [0]
    copies = []                       # (src block, dst block, tokens) of the prompt's partial block
    for (P, ctxs), ns, ow in zip(groups, nshared, own):
        shared_ids = perm[nxt:nxt + ns]
        nxt += ns
        first_own = None
        for c, n_own in zip(ctxs, ow):
            bt[row, :ns] = shared_ids[:min(ns, (c + S - 1) // S)]
            bt[row, ns:ns + n_own] = perm[nxt:nxt + n_own]
            if n_own > 0 and P % S:
                if first_own is None:
                    first_own = int(perm[nxt])
                else:
                    copies.append((first_own, int(perm[nxt]), P % S))
            nxt += n_own
            row += 1
        starts.append(row)
    ctx = torch.tensor(ctx_all, dtype=torch.int64)
    valid = valid_slots(bt, ctx, S, NB)
    k, v = fill_pool(g, NB, Hk, S, D, dtype, valid if poison else None)
    for src, dst, n in copies:
        k[dst, :, :n] = k[src, :, :n]
        v[dst, :, :n] = v[src, :, :n]
    pool = PagedPool(k, v, bt, ctx.to(torch.int32), S, NB, pad, valid)
    q = torch.randn(B, H, D, generator=g).to(dtype)
    seqs, pos = [], []
    r = 0
    for (P, ctxs), ns in zip(groups, nshared):
        for c in ctxs:
            if c > ns * S:            # the last token sits in an own block
                seqs.append(r)
                pos.append(c - 1)
            r += 1
    slots = slot_mapping_for(bt, seqs, pos, S) if seqs else torch.zeros(0, dtype=torch.int64)
    nk = torch.randn(len(seqs), Hk, D, generator=g).to(dtype)
    nv = torch.randn(len(seqs), Hk, D, generator=g).to(dtype)
    if poison and seqs:
        pool.key_cache[slots // S, :, slots % S] = float("nan")
        pool.value_cache[slots // S, :, slots % S] = float("nan")
    return ForkedDecodeCase(name, q, pool, nk, nv, slots, H, Hk, D, 1.0 / math.sqrt(D), dtype,
                            torch.tensor(starts, dtype=torch.int32),
                            torch.tensor([P for P, _ in groups], dtype=torch.int32))


# ---- the five workloads -----------------------------------------------------

def tiny_decode(seed: int = 0) -> DecodeCase:
    """4 sequences, context_lens {1,17,33,100}, 8 Q heads, 2 KV heads,
    head_dim 64, block_size 16, fp16, a 64-block pool in random order; one
    new token per sequence stored at position ctx-1."""
    c = decode_case("tiny", seed, [1, 17, 33, 100], 8, 2, 64, 16, torch.float16,
                    NB=64)
    return c


def qwen3_8b_decode(seed: int = 0, B: int = 64) -> DecodeCase:
    """Qwen3-8B-shaped single-layer decode step: 32 Q heads, 8 KV heads,
    head_dim 128, block_size 16, bf16, batch 64, context_lens uniform on
    [128, 2048], pool 1.5x the blocks needed; one store per sequence."""
    g = _gen(seed + 1000)
    ctx = randint(g, 128, 2048, B)
    return decode_case("qwen3_8b_decode", seed, ctx, 32, 8, 128, 16, torch.bfloat16)


LONG_CONTEXT_POINTS = ((8, 32768), (32, 8192), (128, 2048))


def long_context_layer(point: int, layer: int, seed: int = 0, device="cpu",
                       poison=False) -> DecodeCase:
    """One layer of the 32-layer long-context stack at batch point ``point``
    (B, ctx) in LONG_CONTEXT_POINTS: 32 Q heads, 8 KV heads, head_dim 128,
    block_size 16, bf16, pool of exactly the blocks needed in random order
    (one table shared by all layers), 5% of key vectors scaled by 8."""
    B, ctx_len = LONG_CONTEXT_POINTS[point]
    ctx = torch.full((B,), ctx_len, dtype=torch.int64)
    S, Hk, H, D = 16, 8, 32, 128
    gt = _gen(seed + 7000 + point)
    bt, NB, pad = make_block_tables(gt, ctx, S, NB=int(blocks_needed(ctx, S).sum()))
    g = _gen(seed * 1000003 + 100 * point + layer, device)
    k, v = fill_pool(g, NB, Hk, S, D, torch.bfloat16, None, key_outlier_frac=0.05,
                     device=device)
    gq = _gen(seed * 1000003 + 100 * point + layer + 50, device)
    q = torch.randn(B, H, D, generator=gq, device=device).to(torch.bfloat16)
    pool = PagedPool(k, v, bt, ctx.to(torch.int32), S, NB, pad)
    empty = torch.zeros(0, Hk, D, dtype=torch.bfloat16)
    return DecodeCase(f"long_context_{B}x{ctx_len}_L{layer}", q, pool, empty, empty,
                      torch.zeros(0, dtype=torch.int64), H, Hk, D,
                      1.0 / math.sqrt(D), torch.bfloat16)


@dataclass
class MixedCase:
    """Chunked prefill interleaved with decode in one step, one shared pool.
    Sequences 0..Bp-1 are prefill sequences (chunk of C_i tokens appended
    after P_i cached ones), Bp..Bp+Bd-1 decode sequences."""
    pool: PagedPool                  # context_lens = P_i + C_i / decode ctx
    q_prefill: torch.Tensor          # packed [sum C, H, D]
    cu_q_lens: torch.Tensor          # int32 [Bp + 1]
    prior_lens: torch.Tensor         # int64 [Bp]
    q_decode: torch.Tensor           # [Bd, H, D]
    new_key: torch.Tensor            # [sum C + Bd, Hk, D]
    new_value: torch.Tensor
    slot_mapping: torch.Tensor       # int64 [sum C + Bd]
    Bp: int
    Bd: int
    H: int
    Hk: int
    D: int
    scale: float
    dtype: torch.dtype

    @property
    def max_q_len(self):
        return int((self.cu_q_lens[1:] - self.cu_q_lens[:-1]).max())


def mixed_case(seed, prior_lens, chunk_lens, decode_ctx, H, Hk, D, S, dtype,
               pool_factor=1.5, poison=True) -> MixedCase:
    g = _gen(seed)
    P = torch.as_tensor(prior_lens, dtype=torch.int64)
    C = torch.as_tensor(chunk_lens, dtype=torch.int64)
    dctx = torch.as_tensor(decode_ctx, dtype=torch.int64)
    ctx = torch.cat([P + C, dctx])
    pool = make_pool(g, ctx, Hk, D, S, dtype, None, pool_factor, poison)
    Bp, Bd = P.shape[0], dctx.shape[0]
    cu = torch.zeros(Bp + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(C, 0).to(torch.int32)
    q_pre = torch.randn(int(C.sum()), H, D, generator=g).to(dtype)
    q_dec = torch.randn(Bd, H, D, generator=g).to(dtype)
    seqs = torch.cat([torch.repeat_interleave(torch.arange(Bp), C),
                      Bp + torch.nonzero(dctx > 0).flatten()])
    pos = torch.cat([torch.cat([torch.arange(int(P[i]), int(P[i] + C[i]))
                                for i in range(Bp)]) if Bp else
                     torch.zeros(0, dtype=torch.int64),
                     dctx[dctx > 0] - 1])
    slots = slot_mapping_for(pool.block_tables, seqs, pos, S)
    nk = torch.randn(slots.shape[0], Hk, D, generator=g).to(dtype)
    nv = torch.randn(slots.shape[0], Hk, D, generator=g).to(dtype)
    if poison:
        blk, off = slots // S, slots % S
        pool.key_cache[blk, :, off] = float("nan")
        pool.value_cache[blk, :, off] = float("nan")
    return MixedCase(pool, q_pre, cu, P, q_dec, nk, nv, slots, Bp, Bd, H, Hk, D,
                     1.0 / math.sqrt(D), dtype)


def chunked_prefill_mixed(seed: int = 0, n_prefill: int = 16, chunk: int = 512,
                          max_prior: int = 8192, n_decode: int = 48) -> MixedCase:
    """16 prefill sequences each appending a 512-token causal chunk after a
    prior length uniform on [0, 8192], plus 48 decode sequences with
    context_lens uniform on [256, 4096]; 32 Q heads, 8 KV heads, head_dim 128,
    block_size 16, bf16; pool 1.5x the blocks needed."""
    g = _gen(seed + 4000)
    P = randint(g, 0, max_prior, n_prefill)
    dctx = randint(g, 256, 4096, n_decode)
    return mixed_case(seed, P, [chunk] * n_prefill, dctx, 32, 8, 128, 16,
                      torch.bfloat16)


@dataclass
class ForkCase:
    """Parallel-sampling fork stress: prompts stored in a pool whose block ids
    come from the block manager; each prompt is forked n ways."""
    prompt_lens: torch.Tensor        # int64 [Np]
    n_fork: int
    S: int
    NB: int
    key_cache: torch.Tensor          # [NB, Hk, S, D] random contents
    value_cache: torch.Tensor
    q: torch.Tensor                  # [Np * n_fork, H, D]
    new_key: torch.Tensor            # [Np * n_fork, Hk, D]
    new_value: torch.Tensor
    H: int
    Hk: int
    D: int
    scale: float
    dtype: torch.dtype


def cow_fork_stress(S: int, seed: int = 0, n_prompts: int = 32, n_fork: int = 8,
                    lo: int = 100, hi: int = 4096, H=32, Hk=8, D=128,
                    dtype=torch.float16) -> ForkCase:
    """32 prompts with lengths uniform on [100, 4096], each forked 8 ways; pool =
    the prompts' blocks + n_fork extra blocks per prompt; fp16, 32 Q heads,
    8 KV heads, head_dim 128, block size S."""
    g = _gen(seed + 5000)
    lens = randint(g, lo, hi, n_prompts)
    NB = int(blocks_needed(lens, S).sum()) + n_fork * n_prompts
    gd = _gen(seed + 5100 + S)
    k, v = fill_pool(gd, NB, Hk, S, D, dtype)
    n = n_prompts * n_fork
    q = torch.randn(n, H, D, generator=gd).to(dtype)
    nk = torch.randn(n, Hk, D, generator=gd).to(dtype)
    nv = torch.randn(n, Hk, D, generator=gd).to(dtype)
    return ForkCase(lens, n_fork, S, NB, k, v, q, nk, nv, H, Hk, D,
                    1.0 / math.sqrt(D), dtype)


@dataclass
class TransferCase:
    """A paged cache on the sending side and the block ids the same sequences
    get on the receiving side (prefill -> decode hand-over)."""
    key_caches: list                 # L sender pools [NB, Hk, S, D]
    value_caches: list
    send_tables: torch.Tensor        # int32 [B, max_blocks], sender block ids
    recv_tables: torch.Tensor        # int32 [B, max_blocks], receiver block ids
    context_lens: torch.Tensor       # int32 [B]
    NB: int                          # sender pool size
    NB_recv: int                     # receiver pool size
    S: int
    Hk: int
    D: int
    dtype: torch.dtype

    @property
    def L(self):
        return len(self.key_caches)

    def block_ids(self, tables: torch.Tensor) -> torch.Tensor:
        """The sequences' blocks in order (sequence-major), int32 [nblk]."""
        nb = blocks_needed(self.context_lens.long(), self.S)
        return torch.cat([tables[i, :n] for i, n in enumerate(nb.tolist())])


def kv_transfer(seed: int = 0, L: int = 32, B: int = 4, ctx: int = 2048, Hk: int = 8,
                D: int = 128, S: int = 16, dtype=torch.bfloat16, pool_factor: float = 1.25,
                device="cpu") -> TransferCase:
    """L layers, B sequences of ``ctx`` tokens (Qwen3-8B kv shape by default:
    8 KV heads, head_dim 128, block size 16, bf16).  Each side scatters the
    sequences' blocks over a random permutation of its own pool (1.25x the
    blocks needed); K, V ~ N(0, 1).  One block table serves every layer."""
    g = _gen(seed + 6000)
    ctxs = torch.full((B,), ctx, dtype=torch.int64)
    send, NB, _ = make_block_tables(g, ctxs, S, None, pool_factor)
    recv, NB_recv, _ = make_block_tables(g, ctxs, S, None, pool_factor)
    gd = _gen(seed + 6100, device)
    kcs, vcs = [], []
    for _ in range(L):
        k, v = fill_pool(gd, NB, Hk, S, D, dtype, device=device)
        kcs.append(k)
        vcs.append(v)
    return TransferCase(kcs, vcs, send, recv, ctxs.to(torch.int32), NB, NB_recv, S, Hk, D,
                        dtype)


def spec_verify(seed: int = 0, B: int = 64, n_q: int = 4, lo: int = 128, hi: int = 2048,
                H: int = 32, Hk: int = 8, D: int = 128, S: int = 16,
                dtype=torch.bfloat16) -> MixedCase:
    """Speculative verification: each of B sequences with a prior context
    uniform on [lo, hi] appends n_q tokens (the last accepted token plus
    n_q - 1 drafted ones) whose queries attend causally; Qwen3-8B shape by
    default.  A prefill-chunk case with every C_i = n_q and no decode part."""
    g = _gen(seed + 7000)
    P = randint(g, lo, hi, B)
    return mixed_case(seed + 7100, P, [n_q] * B, [], H, Hk, D, S, dtype)


def token_kv(positions, token_ids, Hk: int = 8, D: int = 128, dtype=torch.bfloat16,
             seed: int = 0):
    """K and V [T, Hk, D] of tokens given by (position, token id): each pair
    draws N(0, 1) values from its own seeded generator, so equal prefixes give
    equal K/V (as a deterministic model would) whatever request they sit in."""
    ks, vs = [], []
    for p, t in zip(list(positions), list(token_ids)):
        g = _gen((seed * 1_000_003 + int(p) * 7919 + int(t)) % (2 ** 62))
        ks.append(torch.randn(Hk, D, generator=g))
        vs.append(torch.randn(Hk, D, generator=g))
    return torch.stack(ks).to(dtype), torch.stack(vs).to(dtype)


def fp8_pools(key_cache: torch.Tensor, value_cache: torch.Tensor):
    """One-byte E4M3 copies of 16-bit pools [NB, Hk, S, D] for FP8-cache tests:
    per kv head, scale = (largest finite magnitude) / 448 and code = the
    float32 value / scale cast by torch to float8_e4m3fn (NaN stays NaN).
    Returns (key codes, value codes, k_scale, v_scale), uint8 and float32 [Hk]."""
    out = []
    for pool in (key_cache, value_cache):
        x = pool.float()
        finite = torch.where(torch.isfinite(x), x.abs(), torch.zeros_like(x))
        amax = finite.amax(dim=(0, 2, 3)).clamp_min(1e-6)
        scale = (amax / 448.0).to(torch.float32)
        y = x / scale.view(1, -1, 1, 1)
        codes = y.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        codes = torch.where(torch.isnan(x), torch.full_like(codes, 0x7F), codes)
        out.append((codes.contiguous(), scale))
    return out[0][0], out[1][0], out[0][1], out[1][1]
