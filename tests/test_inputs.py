"""The workload generators hold to the recipes the workloads are defined by.

The inputs module makes synthetic inputs only, but what it makes decides what
every parity test and every bench line exercises, so its recipes are pinned
here on the CPU at reduced sizes: segment lengths, causal row ranges, the
masked SWA + top-k lists of the uniform fp8 pool, the integer grid, the slot
layout of a decode batch and the named configurations."""
import math

import numpy as np
import torch

from deepseek_sparse_attention_index_gb300 import inputs as I


def test_packed_segment_lengths_recipe():
    """miles PR #3608, Correctness (packed sequences with 1-token segments):
    two 1-token segments, then U[1, 8192] draws, the last cut so the lengths
    sum to the total exactly; seeded and repeatable."""
    for total in (16384, 4096, 3):
        seg = I.packed_segment_lengths(total)
        assert sum(seg) == total
        assert seg[:2] == [1, 1][:min(2, len(seg))]
        assert all(1 <= x <= 8192 for x in seg)
    assert I.packed_segment_lengths(16384) == I.packed_segment_lengths(16384)
    assert I.packed_segment_lengths(16384, seed=1) != I.packed_segment_lengths(16384, seed=0)
    assert len(I.packed_segment_lengths(16384)) > 2   # real draws follow the two 1-token segments


def test_prefill_rows_are_causal_within_their_segment():
    """tokenspeed PR #627, Prefill table: query t of a segment that starts at
    s0 scores keys s0 .. t, inclusive of itself."""
    seg = [1, 1, 5, 3]
    case = I.prefill_case(seg, H_I=8, d_idx=64, idx_kind="bf16_grid", k=4, H=8, device="cpu")
    rs, re = case.row_start.tolist(), case.row_end.tolist()
    t = 0
    for s0, L in zip(np.cumsum([0] + seg[:-1]), seg):
        for j in range(L):
            assert rs[t] == s0 and re[t] == t + 1, t
            t += 1
    assert t == case.T == sum(seg)
    assert case.q.shape == (case.T, 8, 576) and case.kv.rows == case.T


def test_uniform_fp8_lists_recipe():
    """aiter PR #4382, Uniform fp8 pool: per request the SWA window (the last
    128 positions) plus top-k distinct positions from the rest, as global
    slots b * ctx + pos, shuffled, with round(10 %) of the entries set to -1
    (115 of 1152 at the full size)."""
    assert int(round(0.1 * (128 + 1024))) == 115
    B, ctx, swa, topk = 3, 2048, 128, 256
    case = I.uniform_fp8_swa_topk_case(B=B, ctx=ctx, swa=swa, topk=topk, H=8, device="cpu")
    idx = case.idx.numpy()
    n = swa + topk
    assert idx.shape == (B, n)
    for b in range(B):
        row = idx[b]
        valid = row[row >= 0]
        assert (row == -1).sum() == int(round(0.1 * n))
        assert len(np.unique(valid)) == len(valid)                 # distinct slots
        assert ((valid >= b * ctx) & (valid < (b + 1) * ctx)).all()  # this request's slots
        pos = valid - b * ctx
        win = pos[pos >= ctx - swa]
        assert len(win) <= swa and len(pos) - len(win) <= topk
        assert not (np.diff(row) > 0).all()                         # shuffled, not sorted


def test_integer_grid_values():
    """The integer-grid indexer (tiny decode): q, k in {-8..8}/8, w a multiple
    of 2^-8 in [0, 1], so every fp32 index score is exact."""
    ind = I.indexer_grid_bf16(5, 40, 8, 64, seed=0, device="cpu")
    for key in ("q_idx", "k_idx"):
        v = ind[key].float() * 8
        assert torch.equal(v, v.round()) and v.abs().max() <= 8
    w = ind["w"] * 256
    assert torch.equal(w, w.round()) and ind["w"].min() >= 0 and ind["w"].max() <= 1


def test_decode_batch_slot_layout():
    """A decode batch keeps each request's context at consecutive slots from
    its slot_base; packed pools start every request on a 256-slot page."""
    lens = [300, 1, 2049]
    c = I.decode_case("layout", 3, lens, 8, 64, "bf16_grid", 128, 8, I.KV_BF16, device="cpu")
    assert c.seq_lens.tolist() == lens and c.slot_base.tolist() == [0, 300, 301]
    assert c.max_seq_len == 2049
    p = I.decode_case("layout_packed", 3, lens, 8, 64, "bf16_grid", 128, 8, I.KV_FP8_DS_MLA,
                      device="cpu")
    assert p.slot_base.tolist() == [0, 512, 768]
    assert all(b % 256 == 0 for b in p.slot_base.tolist())


def test_named_configurations():
    """The fixed parameters of the named workloads: tiny decode (batch 1,
    context 512, 8 x 64 integer-grid indexer, top-k 128, 8 heads, scale
    1/sqrt(192)) and the decode sweep (64 x 128 fp8 indexer, top-k 2048,
    64 heads over 576-wide bf16 rows, Dv 512)."""
    t = I.tiny_decode(device="cpu")
    assert (t.B, t.max_seq_len, t.H_I, t.d_idx, t.k, t.H, t.D, t.Dv) == (1, 512, 8, 64, 128, 8, 576, 512)
    assert t.indexer["idx_dtype"] == I.IDX_BF16
    assert math.isclose(t.softmax_scale, 1 / math.sqrt(192))
    s = I.decode_sweep(2, 4096, device="cpu")
    assert (s.B, s.max_seq_len, s.H_I, s.d_idx, s.k, s.H, s.D, s.Dv) == (2, 4096, 64, 128, 2048, 64, 576, 512)
    assert s.indexer["idx_dtype"] == I.IDX_FP8
    # w ~ N(0, 1) / 8: 128 draws, standard deviation within a loose band
    assert 0.08 < float(s.indexer["w"].std()) < 0.17


def test_packed_pool_scale_bytes_recipe():
    """aiter PR #4382, Packed fp8_ds_mla: per page 256 x 576 data bytes, then
    256 x 8 scale bytes, 7 UE8M0 exponents in [120, 134] and one pad byte."""
    pool = I.kv_packed_pool(512, 256, seed=0, n=5, device="cpu")
    assert pool.data.shape == (2, 256, 584) and pool.rows == 512
    flat = pool.data.view(2, 256 * 584)
    sc = flat[:, 256 * 576:].view(2, 256, 8)
    assert (sc[:, :, 7] == 0).all()                              # the pad byte
    e = sc[:, :, :7]
    assert int(e.min()) >= 120 and int(e.max()) <= 134
    assert len(torch.unique(e)) == 15                            # every exponent of the range drawn


def test_uniform_pool_scales_recipe():
    """Uniform fp8 pool decode: one fp32 scale per 64 columns (D = 512: 8 per
    row), drawn log-uniform in [2^-4, 2^4]."""
    pool = I.kv_uniform_fp8_pool(4096, seed=0, n=5, device="cpu")
    assert pool.data.shape == (4096, 512) and pool.scales.shape == (4096, 8)
    l2 = torch.log2(pool.scales)
    assert float(l2.min()) >= -4 and float(l2.max()) <= 4
    # log-uniform: the log2 scales fill the interval evenly (8 bins of width 1)
    hist = torch.histc(l2, bins=8, min=-4, max=4)
    assert float(hist.min()) > 0.8 * float(hist.mean())
