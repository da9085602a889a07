"""CPU oracle for the DeepSeek Sparse Attention (DSA) forward hot path.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct
definition the CUDA library is checked against.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it.  The product path (the CUDA library and its
Python binding) never imports, links or calls anything here, and this module
imports nothing from the product package.

Everything is plain numpy in float64.  Inputs arrive as the raw bytes the
caches hold (uint16 for bf16, uint8 for fp8 and UE8M0) and are decoded here
by the format definitions, with no help from any library cast.  A library
primitive serves only as a single step (a dot product, a sort, exp/log).

What each function follows:

* Byte formats: aiter PR #4382 "Paged Sparse Attention Gluon Kernel",
  sections "fp8 flavors" (OCP float8_e4m3fn, bias 7), "Uniform fp8 pool - 2D"
  (x = fp8(byte) * kv_scales[slot, col // 64], the whole head in fp8) and
  "Packed fp8 fp8_ds_mla - 3D" (page = block x 576 data bytes then block x 8
  scale bytes; NoPE x = fp8(byte) * 2^(e - 127); RoPE read as bf16).
* Index score: the DSA lightning indexer, I[t,s] = sum_h w[t,h] *
  ReLU(q[t,h,:] . k[s,:]).  The pages call this step "scoring" (tokenspeed
  PR #627 "Add gluon kernel for DSA", Summary and Benchmark tables) without
  writing it out; the formula is the indexer's published definition.  With
  fp8 inputs the dot is taken on the decoded values times the per-row scales:
  sq[t,h] * sk[s] * (q8[t,h,:] . k8[s,:]).
* Top-k: keep the k highest scores of the valid range; -1 fills the tail
  when fewer than k are valid (miles PR #3608, "What": padded -1 indices).
  Equal scores are ordered by the lower position first.
* Sparse attention: absorbed MLA over the selected latent rows: scores
  scale * q[h,:D] . K_j, softmax over the selected j, out = sum p_j V_j[:Dv]
  with V the leading Dv dims of the same row, lse = ln sum_j exp(scores_j)
  (natural log: miles PR #3608, commit message, FlashMLA's "natural-log
  lse").  Entries equal to -1 are masked, never read (miles PR #3608, "What",
  Padding).  A row with no valid entry gives out = 0 and lse = -inf.
* Two loops: one softmax over the union of a main list into one cache and an
  extra list into another (aiter PR #4382, "Supported formats & dtypes",
  two-loop SWA main + top-k extra).
* Split combine: lse = ln sum_i exp(lse_i), out = sum_i exp(lse_i - lse) out_i
  (tokenspeed PR #664 "gfx950 Gluon bf16 MLA decode", review of the mid /
  final lse buffers; aiter PR #4382, the reduce kernel).

Every function here is pinned by tests/test_oracle_*.py against hand tables,
library routines, brute force and invariants; none says "parity unpinned".
"""

from __future__ import annotations

import numpy as np

KV_BF16 = 0
KV_FP8_UNIFORM = 1
KV_FP8_DS_MLA = 2


# --------------------------------------------------------------------------
# Byte decoders
# --------------------------------------------------------------------------

def decode_bf16(u16) -> np.ndarray:
    """bf16 bits -> float64: the bf16 pattern is the top half of an fp32."""
    u = np.asarray(u16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def decode_e4m3(u8) -> np.ndarray:
    """OCP fp8 e4m3 (bias 7) -> float64.

    sign = bit 7, exponent = bits 6..3, mantissa = bits 2..0.
    exponent 0: subnormal, m * 2^-9.  Otherwise (1 + m/8) * 2^(e-7).
    S.1111.111 is NaN; there is no infinity."""
    b = np.asarray(u8).astype(np.int64)
    s = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    out = s * mag
    return np.where((e == 0xF) & ((b & 7) == 7), np.nan, out)


def decode_ue8m0(u8) -> np.ndarray:
    """UE8M0 exponent byte -> 2^(byte - 127) as float64 (0xFF is NaN)."""
    b = np.asarray(u8).astype(np.float64)
    return np.where(b == 255, np.nan, np.exp2(b - 127.0))


# --------------------------------------------------------------------------
# KV pool rows
# --------------------------------------------------------------------------

def kv_rows(pool: dict, slots) -> np.ndarray:
    """Dequantised latent rows for the given slots, float64 [n, d_nope + d_rope].

    pool: {"format", "data" (numpy bytes / uint16), "scales", "block",
           "d_nope", "d_rope"}.
    * bf16: data uint16 [rows, D]; the row as is.
    * uniform fp8: data uint8 [rows, D], scales f32 [rows, D/64];
      x[c] = fp8(data[slot, c]) * scales[slot, c // 64] for every column
      (RoPE columns included: the whole head is fp8).
    * fp8_ds_mla: data uint8 [nb, block, 584] (any shape with that byte
      order); block_idx = slot // block, pos = slot % block.  NoPE byte c of
      the token sits at block_idx*cs0 + pos*576 + c, its exponent (group
      c // 64) at block_idx*cs0 + block*576 + pos*8 + c//64, and the RoPE
      bf16 values at bytes block_idx*cs0 + pos*576 + 448 .. +576 (cs0 =
      block * 584)."""
    slots = np.asarray(slots, dtype=np.int64)
    fmt = pool["format"]
    D = pool["d_nope"] + pool["d_rope"]
    if fmt == KV_BF16:
        data = np.asarray(pool["data"]).reshape(-1, D)
        return decode_bf16(data[slots])
    if fmt == KV_FP8_UNIFORM:
        data = np.asarray(pool["data"]).reshape(-1, D)
        sc = np.asarray(pool["scales"], dtype=np.float64).reshape(data.shape[0], D // 64)
        x = decode_e4m3(data[slots])
        cols = np.arange(D) // 64
        return x * sc[slots][:, cols]
    if fmt == KV_FP8_DS_MLA:
        assert pool["d_nope"] == 448 and pool["d_rope"] == 64
        block = int(pool["block"])
        flat = np.asarray(pool["data"]).reshape(-1)
        cs0 = block * 584
        bi, pos = slots // block, slots % block
        row0 = bi * cs0 + pos * 576
        nope_b = flat[row0[:, None] + np.arange(448)[None, :]]
        exp_b = flat[(bi * cs0 + block * 576 + pos * 8)[:, None] + np.arange(7)[None, :]]
        rope_lo = flat[row0[:, None] + 448 + 2 * np.arange(64)[None, :]].astype(np.uint16)
        rope_hi = flat[row0[:, None] + 449 + 2 * np.arange(64)[None, :]].astype(np.uint16)
        nope = decode_e4m3(nope_b) * decode_ue8m0(exp_b)[:, np.arange(448) // 64]
        rope = decode_bf16(rope_lo | (rope_hi << np.uint16(8)))
        return np.concatenate([nope, rope], axis=1)
    raise ValueError("unknown KV format %r" % (fmt,))


# --------------------------------------------------------------------------
# Index score
# --------------------------------------------------------------------------

def index_values(raw, scale, is_fp8: bool) -> np.ndarray:
    """Indexer q or k as float64: decoded bytes times the per-row scale (fp8),
    or the bf16 values (scale absent)."""
    if is_fp8:
        x = decode_e4m3(raw)
        return x * np.asarray(scale, dtype=np.float64)[..., None]
    return decode_bf16(raw)


def index_scores_one(q_t: np.ndarray, w_t: np.ndarray, k_rows: np.ndarray) -> np.ndarray:
    """I[s] = sum_h w[h] * ReLU(q[h,:] . k[s,:]) for one query token.

    q_t: [H_I, d] float64 (scales applied), w_t: [H_I], k_rows: [L, d]."""
    dots = k_rows @ q_t.T                       # [L, H_I]
    return np.maximum(dots, 0.0) @ w_t          # [L]


# --------------------------------------------------------------------------
# Top-k
# --------------------------------------------------------------------------

def canon(x: np.ndarray) -> np.ndarray:
    """-0.0 and +0.0 are the same score."""
    return np.where(x == 0, 0.0, x)


def topk_row(scores: np.ndarray, k: int) -> np.ndarray:
    """Positions of the k largest scores (ties: lower position first), then -1
    padding up to k.  Full sort by (score descending, position ascending)."""
    s = canon(np.asarray(scores, dtype=np.float64))
    assert not np.isnan(s).any(), "scores must not hold NaN"
    L = s.shape[0]
    order = np.lexsort((np.arange(L), -s))      # last key is primary
    out = np.full(k, -1, dtype=np.int64)
    n = min(L, k)
    out[:n] = order[:n]
    return out


def kth_score(scores: np.ndarray, k: int) -> float:
    """The k-th largest score of a row (the smallest one selected)."""
    s = np.sort(canon(np.asarray(scores, dtype=np.float64)))[::-1]
    return float(s[min(k, s.shape[0]) - 1])


# --------------------------------------------------------------------------
# Sparse MLA
# --------------------------------------------------------------------------

def sparse_mla_one(q_t: np.ndarray, rows: np.ndarray, softmax_scale: float, Dv: int,
                   sinks: np.ndarray | None = None):
    """Absorbed-MLA attention of one query token over already-gathered rows.

    q_t: [H, D] float64; rows: [n, D] float64 (valid rows only, duplicates
    count once per occurrence).  Returns out [H, Dv], lse [H] (natural log).

    sinks (optional, [H]): a per-head logit in the units of the scores
    s_j = softmax_scale * q . K_j that joins the softmax denominator and
    contributes no value (the "sink folded in" of the Miles sparse-attention
    pull request's forward notes): out = sum_j e^{s_j} V_j / (sum_j e^{s_j} +
    e^{sink}), lse = ln(sum_j e^{s_j} + e^{sink})."""
    H = q_t.shape[0]
    if rows.shape[0] == 0:
        lse0 = np.full(H, -np.inf) if sinks is None else np.asarray(sinks, dtype=np.float64).copy()
        return np.zeros((H, Dv)), lse0
    s = softmax_scale * (q_t @ rows.T)          # [H, n]
    if sinks is not None:
        # the sink is one more logit in every head's denominator
        s_all = np.concatenate([s, np.asarray(sinks, dtype=np.float64)[:, None]], axis=1)
    else:
        s_all = s
    m = s_all.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    lse = m[:, 0] + np.log(np.exp(s_all - m).sum(axis=1))
    p = np.exp(s - lse[:, None])                # the rows' weights (the sink carries none)
    return p @ rows[:, :Dv], lse


def sparse_mla_bwd_one(q_t: np.ndarray, rows: np.ndarray, dout_t: np.ndarray,
                       softmax_scale: float, Dv: int, sinks: np.ndarray | None = None):
    """Gradients of sparse_mla_one for one query token, given dL/dout
    (dout_t [H, Dv]); the lse output is auxiliary (no gradient flows into it).

    With s_j = scale q.K_j, p_j = e^{s_j - lse}, out = sum_j p_j V_j
    (V_j = K_j[:Dv]) and delta = dout . out (= sum_j p_j dout.V_j):
        dS_j = p_j (dout . V_j - delta)
        dq   = scale sum_j dS_j K_j
        dK_j = scale sum_h dS_hj q_h, plus sum_h p_hj dout_h on the V columns
        dsink_h = -p_sink,h delta_h,  p_sink = e^{sink - lse}
    A row's gradient is per occurrence.  Returns dq [H, D], drows [n, D],
    dsinks [H] (zeros without sinks)."""
    H, D = q_t.shape
    n = rows.shape[0]
    if n == 0:
        return np.zeros((H, D)), np.zeros((0, D)), np.zeros(H)
    out, lse = sparse_mla_one(q_t, rows, softmax_scale, Dv, sinks)
    s = softmax_scale * (q_t @ rows.T)           # [H, n]
    p = np.exp(s - lse[:, None])
    dP = dout_t @ rows[:, :Dv].T                 # [H, n]
    delta = (dout_t * out).sum(axis=1)           # [H]
    dS = p * (dP - delta[:, None])
    dq = softmax_scale * (dS @ rows)
    drows = softmax_scale * (dS.T @ q_t)
    drows[:, :Dv] += p.T @ dout_t
    dsinks = np.zeros(H)
    if sinks is not None:
        sk = np.asarray(sinks, dtype=np.float64)
        dsinks = np.where(np.isfinite(sk), -np.exp(sk - lse) * delta, 0.0)
    return dq, drows, dsinks


def sparse_mla_bwd(q: np.ndarray, pool: dict, idx: np.ndarray, dout: np.ndarray,
                   softmax_scale: float, Dv: int, sinks: np.ndarray | None = None):
    """Backward of sparse_mla (one list): dq [T, H, D], dkv [pool rows, D]
    (each selection's row gradient added to its slot; -1 entries skipped),
    dsinks [H] summed over the tokens."""
    T, H, D = q.shape
    dq = np.zeros((T, H, D))
    data = np.asarray(pool["data"])
    if pool["format"] == KV_FP8_DS_MLA:
        n_rows = data.size // 584
    else:
        n_rows = data.reshape(-1, pool["d_nope"] + pool["d_rope"]).shape[0]
    dkv = np.zeros((n_rows, D))
    dsinks = np.zeros(H)
    for t in range(T):
        sl = np.asarray(idx[t], dtype=np.int64)
        sl = sl[sl >= 0]
        rows = kv_rows(pool, sl)
        dq[t], drows, ds = sparse_mla_bwd_one(q[t], rows, dout[t], softmax_scale, Dv, sinks)
        np.add.at(dkv, sl, drows)
        dsinks += ds
    return dq, dkv, dsinks


def gather_valid(pool: dict, idx_row) -> np.ndarray:
    """Rows of the non-negative entries of one index list (-1 masked)."""
    idx_row = np.asarray(idx_row, dtype=np.int64)
    v = idx_row[idx_row >= 0]
    return kv_rows(pool, v)


def sparse_mla(q: np.ndarray, pool: dict, idx: np.ndarray, softmax_scale: float, Dv: int,
               pool_extra: dict | None = None, idx_extra: np.ndarray | None = None,
               sinks: np.ndarray | None = None):
    """Sparse MLA for T tokens.  q: [T, H, D] float64; idx: [T, k] slots into
    ``pool`` (-1 masked); optional second list idx_extra into pool_extra, in
    the same softmax; optional per-head sinks (see sparse_mla_one).  Returns
    out [T, H, Dv], lse [T, H]."""
    T, H, _ = q.shape
    out = np.zeros((T, H, Dv))
    lse = np.zeros((T, H))
    for t in range(T):
        rows = gather_valid(pool, idx[t])
        if idx_extra is not None:
            rows = np.concatenate([rows, gather_valid(pool_extra, idx_extra[t])], axis=0)
        out[t], lse[t] = sparse_mla_one(q[t], rows, softmax_scale, Dv, sinks)
    return out, lse


def combine_splits(outs: np.ndarray, lses: np.ndarray):
    """Merge split partials of one (token, head): outs [S, Dv], lses [S]."""
    lses = np.asarray(lses, dtype=np.float64)
    if np.all(np.isneginf(lses)):
        return np.zeros(outs.shape[1]), -np.inf
    m = lses.max()
    lse = m + np.log(np.exp(lses - m).sum())
    wts = np.exp(lses - lse)
    return wts @ outs, lse


# --------------------------------------------------------------------------
# Decode step: score -> top-k -> sparse MLA
# --------------------------------------------------------------------------

def decode_request(b: int, case: dict):
    """One request of a decode step.

    case (numpy): q_idx, q_scale, k_idx, k_scale, w, is_fp8, seq_lens,
    slot_base, k, q (uint16 bf16 bits [B,H,D]), kv (pool dict), softmax_scale,
    Dv, optional kv_swa / idx_swa.  The index-k cache and the KV pool share
    slot numbering: position j of request b is slot slot_base[b] + j, or,
    with a paged layout (case["block_table"] [B, pages], case["page_size"]),
    slot block_table[b][j // page] * page + j % page.
    Returns dict(scores [L], idx [k] request-local positions, out, lse)."""
    L = int(case["seq_lens"][b])
    pos = np.arange(L, dtype=np.int64)
    if case.get("block_table") is not None:
        page = int(case["page_size"])
        pos_slots = case["block_table"][b][pos // page].astype(np.int64) * page + pos % page
    else:
        pos_slots = int(case["slot_base"][b]) + pos
    fp8 = case["is_fp8"]
    qs = None if case["q_scale"] is None else case["q_scale"][b]
    ks = None if case["k_scale"] is None else case["k_scale"][pos_slots]
    q_t = index_values(case["q_idx"][b], qs, fp8)
    k_rows = index_values(case["k_idx"][pos_slots], ks, fp8)
    scores = index_scores_one(q_t, case["w"][b].astype(np.float64), k_rows)
    sel = topk_row(scores, case["k"])
    slots = np.where(sel >= 0, pos_slots[np.maximum(sel, 0)] if L > 0 else -1, -1)
    rows = gather_valid(case["kv"], slots)
    if case.get("idx_swa") is not None:
        rows = np.concatenate([gather_valid(case["kv_swa"], case["idx_swa"][b]), rows], axis=0)
    q_att = decode_bf16(case["q"][b])
    out, lse = sparse_mla_one(q_att, rows, case["softmax_scale"], case["Dv"])
    return dict(scores=scores, idx=sel, out=out, lse=lse)


def prefill_token(t: int, case: dict):
    """One query token of a causal prefill: keys row_start[t] .. row_end[t]-1.
    Returns dict(scores, idx (positions relative to row_start), out, lse)."""
    r0, r1 = int(case["row_start"][t]), int(case["row_end"][t])
    fp8 = case["is_fp8"]
    qs = None if case["q_scale"] is None else case["q_scale"][t]
    ks = None if case["k_scale"] is None else case["k_scale"][r0:r1]
    q_t = index_values(case["q_idx"][t], qs, fp8)
    k_rows = index_values(case["k_idx"][r0:r1], ks, fp8)
    scores = index_scores_one(q_t, case["w"][t].astype(np.float64), k_rows)
    sel = topk_row(scores, case["k"])
    slots = np.where(sel >= 0, sel + r0, -1)
    rows = gather_valid(case["kv"], slots)
    out, lse = sparse_mla_one(decode_bf16(case["q"][t]), rows, case["softmax_scale"], case["Dv"])
    return dict(scores=scores, idx=sel, out=out, lse=lse)
