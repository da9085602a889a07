"""Seeded synthetic inputs for the DSA forward hot path.

This module makes inputs only: random tensors of the shapes, dtypes and value
distributions of the workloads below, and the byte encoders that turn real
values into the cache formats the path reads (bf16, fp8 e4m3 with a per-row
fp32 scale, the uniform fp8 pool with 1x64 fp32 scales, the packed 584-byte
``fp8_ds_mla`` page).  It holds none of the method's arithmetic: no index
score, no selection, no attention.  Both the CUDA path and the CPU oracle
consume what it returns; neither is imported here.

Encoders use PyTorch's own casts (``float -> bfloat16`` and
``float -> float8_e4m3fn``, both round-to-nearest-even); values are clamped to
the finite fp8 range first so that nothing saturates to NaN.

Random streams: every tensor draws from its own ``torch.Generator`` seeded
with ``seed * 1000 + n`` where ``n`` is the tensor's fixed number in the
builder (documented at each call).  A builder called with ``device="cuda"``
draws on the GPU generator, so the values differ from a CPU build of the same
case; tests always hand the oracle copies of the exact tensors the kernels
read.

Workload recipes (sizes and distributions) follow the DSA pages:
  * tokenspeed PR #627 "Add gluon kernel for DSA", Decode/Prefill tables:
    one query per request against N context tokens, 512 .. 1M.
  * aiter PR #4382 "Paged Sparse Attention Gluon Kernel", sections
    "Uniform fp8 pool - 2D" and "Packed fp8 fp8_ds_mla - 3D": the two fp8
    pool layouts, SWA window 128 + index_topk 1024, D = 448 NoPE + 64 RoPE.
  * miles PR #3608 "per-arch DSA sparse attention dispatch", section
    "Correctness": -1 padded index rows, packed sequences with 1-token
    segments.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

# Format codes shared with the C ABI (include/dsa.h).
KV_BF16 = 0
KV_FP8_UNIFORM = 1
KV_FP8_DS_MLA = 2
IDX_BF16 = 0
IDX_FP8 = 1

FP8_MAX = 448.0
PACKED_ROW_BYTES = 584  # 448 fp8 NoPE + 64 bf16 RoPE (128 B) + 8 scale bytes


def _gen(seed: int, n: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + n)
    return g


# --------------------------------------------------------------------------
# Byte encoders (input preparation, not part of the hot path)
# --------------------------------------------------------------------------

def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round float values to bf16 (RNE)."""
    return x.to(torch.bfloat16)


def to_e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    """Round float values to OCP fp8 e4m3 (RNE, clamped to +-448); uint8 view."""
    return x.float().clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def quantize_rows_e4m3(x: torch.Tensor):
    """Per-row fp8 quantisation: scale = amax(|row|) / 448, bytes = e4m3(row / scale).

    Returns (uint8 bytes with x's shape, float32 scales with x.shape[:-1]).
    An all-zero row gets scale 1.
    """
    x = x.float()
    amax = x.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    q = to_e4m3_bytes(x / scale.unsqueeze(-1))
    return q, scale.contiguous()


def pack_ds_mla_pages(nope_e4m3: torch.Tensor, exps: torch.Tensor, rope_bf16: torch.Tensor,
                      block: int) -> torch.Tensor:
    """Lay tokens out as ``fp8_ds_mla`` pages: ``[nb, block, 584]`` uint8.

    Page layout (aiter PR #4382, section "Packed fp8 fp8_ds_mla - 3D"): the
    page is block-planar, ``block x 576`` data bytes followed by
    ``block x 8`` scale bytes.  A data row is 448 fp8 NoPE bytes then the 64
    RoPE values as bf16 (128 bytes); a scale row is 7 UE8M0 exponents (one
    per 64 NoPE channels) and one zero pad byte.

    nope_e4m3: uint8 [tokens, 448]; exps: uint8 [tokens, 7];
    rope_bf16: bfloat16 [tokens, 64].  tokens must be a multiple of block.
    """
    n = nope_e4m3.shape[0]
    assert n % block == 0
    nb = n // block
    dev = nope_e4m3.device
    data = torch.empty((nb, block, 576), dtype=torch.uint8, device=dev)
    data[:, :, :448] = nope_e4m3.view(nb, block, 448)
    data[:, :, 448:] = rope_bf16.contiguous().view(torch.uint8).view(nb, block, 128)
    sc = torch.zeros((nb, block, 8), dtype=torch.uint8, device=dev)
    sc[:, :, :7] = exps.view(nb, block, 7)
    page = torch.cat([data.view(nb, block * 576), sc.view(nb, block * 8)], dim=1)
    return page.view(nb, block, PACKED_ROW_BYTES).contiguous()


# --------------------------------------------------------------------------
# KV pool description (mirrors dsa_kv_pool in include/dsa.h)
# --------------------------------------------------------------------------

@dataclass
class KVPool:
    format: int
    data: torch.Tensor                 # bf16 [rows,576] | u8 [rows,D] | u8 [nb,block,584]
    scales: Optional[torch.Tensor]     # f32 [rows, D/64] for FP8_UNIFORM
    rows: int
    block: int
    d_nope: int
    d_rope: int

    def to(self, device) -> "KVPool":
        return KVPool(self.format, self.data.to(device),
                      None if self.scales is None else self.scales.to(device),
                      self.rows, self.block, self.d_nope, self.d_rope)


def kv_bf16_pool(rows: int, seed: int, n: int, device, d_nope=512, d_rope=64) -> KVPool:
    g = _gen(seed, n, device)
    x = torch.randn((rows, d_nope + d_rope), generator=g, device=device)
    return KVPool(KV_BF16, to_bf16(x), None, rows, 1, d_nope, d_rope)


def kv_uniform_fp8_pool(rows: int, seed: int, n: int, device, d_nope=448, d_rope=64,
                        log2_lo=-4.0, log2_hi=4.0) -> KVPool:
    """Uniform fp8 pool: bytes e4m3(N(0,1)), scales 2**U[log2_lo, log2_hi] per 64 columns."""
    D = d_nope + d_rope
    g = _gen(seed, n, device)
    x = torch.randn((rows, D), generator=g, device=device)
    u = torch.rand((rows, D // 64), generator=g, device=device)
    scales = torch.exp2(log2_lo + (log2_hi - log2_lo) * u).float().contiguous()
    return KVPool(KV_FP8_UNIFORM, to_e4m3_bytes(x).contiguous(), scales, rows, 1, d_nope, d_rope)


def kv_packed_pool(tokens: int, block: int, seed: int, n: int, device,
                   exp_lo=120, exp_hi=134) -> KVPool:
    """Packed fp8_ds_mla pool: NoPE bytes e4m3(N(0,1)), UE8M0 exponents uniform in
    [exp_lo, exp_hi], RoPE bf16 N(0,1).  tokens is rounded up to whole pages;
    the pad tokens are drawn like the rest."""
    nb = (tokens + block - 1) // block
    n_tok = nb * block
    g = _gen(seed, n, device)
    nope = to_e4m3_bytes(torch.randn((n_tok, 448), generator=g, device=device))
    exps = torch.randint(exp_lo, exp_hi + 1, (n_tok, 7), generator=g, device=device).to(torch.uint8)
    rope = to_bf16(torch.randn((n_tok, 64), generator=g, device=device))
    return KVPool(KV_FP8_DS_MLA, pack_ds_mla_pages(nope, exps, rope, block), None,
                  n_tok, block, 448, 64)


# --------------------------------------------------------------------------
# Indexer inputs
# --------------------------------------------------------------------------

def indexer_grid_bf16(T: int, S: int, H_I: int, d: int, seed: int, device):
    """Integer-grid bf16 indexer inputs: q, k in {-8..8}/8, w in 2^-8 Z inside [0,1].

    Every product, partial sum and weighted head sum is a multiple of 2^-14
    below 2^9 in magnitude, so the fp32 scores are exact."""
    gq, gk, gw = _gen(seed, 1, device), _gen(seed, 2, device), _gen(seed, 3, device)
    q = torch.randint(-8, 9, (T, H_I, d), generator=gq, device=device).float() / 8
    k = torch.randint(-8, 9, (S, d), generator=gk, device=device).float() / 8
    w = torch.round(torch.rand((T, H_I), generator=gw, device=device) * 256) / 256
    return dict(idx_dtype=IDX_BF16, q_idx=to_bf16(q).contiguous(), q_scale=None,
                k_idx=to_bf16(k).contiguous(), k_scale=None, w=w.float().contiguous())


def indexer_fp8(T: int, S: int, H_I: int, d: int, seed: int, device, w_std=1.0 / 8):
    """fp8 indexer inputs: q, k ~ N(0,1) quantised per row (scale = amax/448);
    w ~ N(0,1) * w_std."""
    gq, gk, gw = _gen(seed, 1, device), _gen(seed, 2, device), _gen(seed, 3, device)
    q8, qs = quantize_rows_e4m3(torch.randn((T, H_I, d), generator=gq, device=device))
    k8, ks = quantize_rows_e4m3(torch.randn((S, d), generator=gk, device=device))
    w = torch.randn((T, H_I), generator=gw, device=device) * w_std
    return dict(idx_dtype=IDX_FP8, q_idx=q8.contiguous(), q_scale=qs, k_idx=k8.contiguous(),
                k_scale=ks, w=w.float().contiguous())


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclass
class DecodeCase:
    """One decode step: B requests, one query token each.

    Request b sees context positions [0, seq_lens[b]); its index-key rows and
    KV rows live at slots slot_base[b] + position in the index-k cache and in
    ``kv`` (the two caches share slot numbering).  ``kv_swa``/``idx_swa``
    (optional) are the separate sliding-window list of the two-loop layout."""
    name: str
    B: int
    seq_lens: torch.Tensor      # int32 [B]
    slot_base: torch.Tensor     # int32 [B]
    max_seq_len: int
    H_I: int
    d_idx: int
    indexer: dict
    k: int
    H: int
    D: int
    Dv: int
    softmax_scale: float
    q: torch.Tensor             # bf16 [B, H, D]
    kv: KVPool
    kv_swa: Optional[KVPool] = None
    idx_swa: Optional[torch.Tensor] = None   # int32 [B, k_swa]
    meta: dict = field(default_factory=dict)


def decode_case(name: str, B: int, N, H_I: int, d_idx: int, idx_kind: str, k: int, H: int,
                kv_format: int, seed: int = 0, device="cpu", softmax_scale=None,
                swa: int = 0, block: int = 256) -> DecodeCase:
    """Build a decode step.  N is one context length for all requests or a list.

    Tensor numbers: 1-3 indexer (q, k, w), 4 attention q, 5 KV pool,
    6 SWA pool."""
    lens = [int(N)] * B if isinstance(N, int) else [int(x) for x in N]
    assert len(lens) == B
    if kv_format == KV_FP8_DS_MLA:
        # the extra cache is paged; give every request whole pages
        stride = [((L + block - 1) // block) * block for L in lens]
    else:
        stride = lens
    base = [0]
    for s in stride[:-1]:
        base.append(base[-1] + s)
    S_total = base[-1] + stride[-1]
    if idx_kind == "bf16_grid":
        ind = indexer_grid_bf16(B, S_total, H_I, d_idx, seed, device)
    elif idx_kind == "fp8":
        ind = indexer_fp8(B, S_total, H_I, d_idx, seed, device)
    else:
        raise ValueError(idx_kind)
    if kv_format == KV_BF16:
        kv = kv_bf16_pool(S_total, seed, 5, device)
        D, Dv = 576, 512
    elif kv_format == KV_FP8_UNIFORM:
        kv = kv_uniform_fp8_pool(S_total, seed, 5, device)
        D, Dv = 512, 448
    else:
        kv = kv_packed_pool(S_total, block, seed, 5, device)
        D, Dv = 512, 448
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(192.0) if D == 576 else 1.0 / math.sqrt(512.0)
    gq = _gen(seed, 4, device)
    q = to_bf16(torch.randn((B, H, D), generator=gq, device=device)).contiguous()
    kv_swa = idx_swa = None
    if swa > 0:
        assert kv_format == KV_FP8_DS_MLA
        # one SWA page per request; slots 0..swa-1 of page b hold the window
        kv_swa = kv_packed_pool(B * block, block, seed, 6, device)
        idx_swa = (torch.arange(B, device=device, dtype=torch.int32)[:, None] * block
                   + torch.arange(swa, device=device, dtype=torch.int32)[None, :]).contiguous()
    return DecodeCase(name, B, torch.tensor(lens, dtype=torch.int32, device=device),
                      torch.tensor(base, dtype=torch.int32, device=device), max(lens),
                      H_I, d_idx, ind, k, H, D, Dv, float(softmax_scale), q, kv, kv_swa, idx_swa)


@dataclass
class SparseCase:
    """Sparse MLA alone: T query tokens, each with its own slot list (-1 = masked)."""
    name: str
    T: int
    H: int
    D: int
    Dv: int
    softmax_scale: float
    q: torch.Tensor            # bf16 [T, H, D]
    kv: KVPool
    idx: torch.Tensor          # int32 [T, k]
    kv_extra: Optional[KVPool] = None
    idx_extra: Optional[torch.Tensor] = None


def uniform_fp8_swa_topk_case(B=32, ctx=65536, swa=128, topk=1024, neg_frac=0.1, H=64,
                              seed=0, device="cpu") -> SparseCase:
    """Uniform fp8 pool decode (one merged SWA + top-k list per request).

    Per request b the list holds the last ``swa`` positions and ``topk``
    distinct positions drawn from the rest, as global slots b*ctx + pos, in a
    random order; round(neg_frac * len) entries, at positions drawn without
    replacement, are then set to -1.  Tensor numbers: 4 q, 5 pool, 7 lists."""
    kv = kv_uniform_fp8_pool(B * ctx, seed, 5, device)
    g = _gen(seed, 7, "cpu")
    n = swa + topk
    n_neg = int(round(neg_frac * n))
    rows = []
    for b in range(B):
        extra = torch.randperm(ctx - swa, generator=g)[:topk]
        win = torch.arange(ctx - swa, ctx)
        lst = torch.cat([win, extra]) + b * ctx
        lst = lst[torch.randperm(n, generator=g)]
        lst[torch.randperm(n, generator=g)[:n_neg]] = -1
        rows.append(lst)
    idx = torch.stack(rows).to(torch.int32).to(device).contiguous()
    gq = _gen(seed, 4, device)
    q = to_bf16(torch.randn((B, H, 512), generator=gq, device=device)).contiguous()
    return SparseCase("uniform_fp8_b%d_ctx%d" % (B, ctx), B, H, 512, 448, 1.0 / math.sqrt(512.0),
                      q, kv, idx)


@dataclass
class PrefillCase:
    """Causal prefill over packed segments.  Query t of a segment starting at
    position s0 scores keys s0..t (inclusive) of the same segment; row_start /
    row_end are those key ranges as global token rows [s0, t+1)."""
    name: str
    T: int
    seg_lens: list
    row_start: torch.Tensor    # int32 [T]
    row_end: torch.Tensor      # int32 [T]
    H_I: int
    d_idx: int
    indexer: dict
    k: int
    H: int
    softmax_scale: float
    q: torch.Tensor            # bf16 [T, H, 576]
    kv: KVPool                 # bf16 [T, 576], slot = token row


def packed_segment_lengths(total=16384, hi=8192, n_single=2, seed=0):
    """Segment lengths for a packed batch: ``n_single`` forced 1-token
    segments, then U[1, hi] draws until the total is reached, the last draw cut
    so the lengths sum to ``total`` exactly."""
    g = _gen(seed, 8, "cpu")
    lens = [1] * n_single
    while sum(lens) < total:
        x = int(torch.randint(1, hi + 1, (1,), generator=g))
        lens.append(min(x, total - sum(lens)))
    return lens


def prefill_q(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Attention queries of a prefill: bf16 N(0,1) [T, H, 576] (tensor number 4)."""
    gq = _gen(seed, 4, device)
    return to_bf16(torch.randn((T, H, 576), generator=gq, device=device)).contiguous()


def prefill_case(seg_lens, H_I=64, d_idx=128, idx_kind="fp8", k=2048, H=64, seed=0,
                 device="cpu", name=None) -> PrefillCase:
    """Tensor numbers: 1-3 indexer, 4 q, 5 KV."""
    T = int(sum(seg_lens))
    starts, ends = [], []
    s0 = 0
    for L in seg_lens:
        for t in range(L):
            starts.append(s0)
            ends.append(s0 + t + 1)
        s0 += L
    if idx_kind == "fp8":
        ind = indexer_fp8(T, T, H_I, d_idx, seed, device)
    else:
        ind = indexer_grid_bf16(T, T, H_I, d_idx, seed, device)
    kv = kv_bf16_pool(T, seed, 5, device)
    q = prefill_q(T, H, seed, device)
    return PrefillCase(name or ("prefill_T%d" % T), T, list(seg_lens),
                       torch.tensor(starts, dtype=torch.int32, device=device),
                       torch.tensor(ends, dtype=torch.int32, device=device),
                       H_I, d_idx, ind, k, H, 1.0 / math.sqrt(192.0), q, kv)


# --------------------------------------------------------------------------
# The five workloads, by name
# --------------------------------------------------------------------------

def tiny_decode(device="cpu", seed=0) -> DecodeCase:
    """Batch 1, context 512, indexer 8 heads x 64 integer-grid bf16, top-k 128,
    sparse MLA 8 heads over bf16 576-wide rows, scale 1/sqrt(192)."""
    return decode_case("tiny_decode_n512", 1, 512, 8, 64, "bf16_grid", 128, 8, KV_BF16,
                       seed=seed, device=device, softmax_scale=1.0 / math.sqrt(192.0))


def decode_sweep(B: int, N: int, device="cpu", seed=0) -> DecodeCase:
    """Batch B, context N, indexer 64 heads x 128 fp8 with per-row scales,
    w ~ N(0,1)/8, top-k 2048, sparse MLA 64 heads over bf16 576-wide rows."""
    return decode_case("decode_b%d_n%d" % (B, N), B, N, 64, 128, "fp8", 2048, 64, KV_BF16,
                       seed=seed, device=device)


def multi_token_decode(B: int, Q: int, N: int, device="cpu", seed=0, k=2048, H=64,
                       idx_kind="fp8", d_idx=128) -> DecodeCase:
    """Decode with Q query tokens per request (speculative verification):
    request b's context has N positions, the last Q of them the new tokens.
    Query row b*Q + i is new token i: it sees positions [0, N - Q + 1 + i) of
    its request (causal among the new tokens) at the request's slots.  The
    rows share their request's slot base, so the fused decode serves them as
    B*Q rows.  Indexer 64 x 128 (fp8, or the bf16 integer grid), sparse MLA
    H heads over bf16 576-wide rows; d_idx the indexer's head width."""
    assert 1 <= Q <= N
    T = B * Q
    S_total = B * N
    if idx_kind == "fp8":
        ind = indexer_fp8(T, S_total, 64, d_idx, seed, device)
    else:
        ind = indexer_grid_bf16(T, S_total, 64, d_idx, seed, device)
    kv = kv_bf16_pool(S_total, seed, 5, device)
    gq = _gen(seed, 4, device)
    q = to_bf16(torch.randn((T, H, 576), generator=gq, device=device)).contiguous()
    lens = [N - Q + 1 + i for b in range(B) for i in range(Q)]
    base = [b * N for b in range(B) for i in range(Q)]
    return DecodeCase("multi_token_b%d_q%d_n%d" % (B, Q, N), T,
                      torch.tensor(lens, dtype=torch.int32, device=device),
                      torch.tensor(base, dtype=torch.int32, device=device), N, 64, d_idx, ind,
                      k, H, 576, 512, 1.0 / math.sqrt(192.0), q, kv,
                      meta={"requests": B, "tokens_per_request": Q})


def paged_decode(B: int, N, page: int = 64, device="cpu", seed=0, k=2048, H=64,
                 idx_kind="fp8", shuffle=True) -> DecodeCase:
    """A decode step on paged caches: the index-k cache (and its scales) and
    the bf16 KV pool are cut into pages of `page` slots, and position j of
    request b lives at slot block_table[b][j // page] * page + j % page of
    both.  Built contiguous (every request a run of whole pages), then the
    pages are shuffled (the same permutation for both caches) and the block
    table follows them.  meta: block_table int32 [B, max_pages], page_size,
    and the permutation's inverse (new page -> old page) for reference."""
    lens = [int(N)] * B if isinstance(N, int) else [int(x) for x in N]
    pages = [(L + page - 1) // page for L in lens]
    npages = sum(pages)
    S_total = npages * page
    if idx_kind == "fp8":
        ind = indexer_fp8(B, S_total, 64, 128, seed, device)
    else:
        ind = indexer_grid_bf16(B, S_total, 64, 128, seed, device)
    kv = kv_bf16_pool(S_total, seed, 5, device)
    gq = _gen(seed, 4, device)
    q = to_bf16(torch.randn((B, H, 576), generator=gq, device=device)).contiguous()
    first = [0]
    for n in pages[:-1]:
        first.append(first[-1] + n)
    if shuffle:
        gp = torch.Generator().manual_seed(seed * 7919 + 17)
        perm = torch.randperm(npages, generator=gp)          # old page -> new page
    else:
        perm = torch.arange(npages)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(npages)                          # new page -> old page
    inv_d = inv.to(device)

    def by_page(x):   # rows grouped by page, reordered so that new page q holds old page inv[q]
        shp = x.shape
        return x.reshape(npages, page, *shp[1:])[inv_d].reshape(shp).contiguous()

    ind = dict(ind)
    ind["k_idx"] = by_page(ind["k_idx"])
    if ind.get("k_scale") is not None:
        ind["k_scale"] = by_page(ind["k_scale"])
    kv = KVPool(kv.format, by_page(kv.data), None, kv.rows, kv.block, kv.d_nope, kv.d_rope)
    maxp = max(pages)
    bt = torch.zeros((B, maxp), dtype=torch.int32)
    for b in range(B):
        bt[b, :pages[b]] = perm[first[b]:first[b] + pages[b]].to(torch.int32)
    return DecodeCase("paged_decode_b%d_p%d" % (B, page), B,
                      torch.tensor(lens, dtype=torch.int32, device=device),
                      torch.zeros(B, dtype=torch.int32, device=device), max(lens), 64, 128, ind,
                      k, H, 576, 512, 1.0 / math.sqrt(192.0), q, kv,
                      meta={"block_table": bt.to(device), "page_size": page,
                            "new_to_old_page": inv})


def packed_long_decode(N=1 << 20, device="cpu", seed=0, swa=128, topk=1024) -> DecodeCase:
    """Batch 1, context N on packed fp8_ds_mla pages of 256 tokens; two loops:
    the SWA window (its own packed cache) and the top-k list (indexer 64 x 128
    fp8 over all N positions)."""
    return decode_case("packed_fp8_ds_mla_n%d" % N, 1, N, 64, 128, "fp8", topk, 64,
                       KV_FP8_DS_MLA, seed=seed, device=device, swa=swa, block=256)
