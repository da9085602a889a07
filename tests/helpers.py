"""Test glue: hand torch tensors to the oracle as the raw bytes the caches hold."""
import numpy as np
import torch


def raw(t):
    """numpy view of a tensor's storage: bf16 -> uint16 bits, uint8 -> uint8,
    everything else as its own dtype."""
    if t is None:
        return None
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def pool_np(pool):
    return dict(format=pool.format, data=raw(pool.data), scales=raw(pool.scales),
                block=pool.block, d_nope=pool.d_nope, d_rope=pool.d_rope)


def decode_case_np(case):
    ind = case.indexer
    d = dict(q_idx=raw(ind["q_idx"]), q_scale=raw(ind["q_scale"]), k_idx=raw(ind["k_idx"]),
             k_scale=raw(ind["k_scale"]), w=raw(ind["w"]), is_fp8=ind["idx_dtype"] == 1,
             seq_lens=raw(case.seq_lens), slot_base=raw(case.slot_base), k=case.k,
             q=raw(case.q), kv=pool_np(case.kv), softmax_scale=case.softmax_scale, Dv=case.Dv)
    if case.kv_swa is not None:
        d["kv_swa"] = pool_np(case.kv_swa)
        d["idx_swa"] = raw(case.idx_swa)
    if case.meta.get("block_table") is not None:
        d["block_table"] = raw(case.meta["block_table"])
        d["page_size"] = case.meta["page_size"]
    return d


def prefill_case_np(case):
    ind = case.indexer
    return dict(q_idx=raw(ind["q_idx"]), q_scale=raw(ind["q_scale"]), k_idx=raw(ind["k_idx"]),
                k_scale=raw(ind["k_scale"]), w=raw(ind["w"]), is_fp8=ind["idx_dtype"] == 1,
                row_start=raw(case.row_start), row_end=raw(case.row_end), k=case.k,
                q=raw(case.q), kv=pool_np(case.kv), softmax_scale=case.softmax_scale, Dv=512)
