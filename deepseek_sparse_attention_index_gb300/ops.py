"""Thin ctypes binding of libdsa_gb300.so (C ABI: include/dsa.h).

Argument marshalling only: tensors become device pointers, shapes become the
size arguments, and the call is enqueued on torch's current CUDA stream.
Every step of the computation runs in the library's CUDA kernels.  There is
no fallback: if the library is missing or a GPU is absent, the first call
raises.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

from . import inputs as _inp

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa_gb300.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dsa.h")

DSA_OK = 0
DEVERR_INDEX_RANGE = 1
DEVERR_TIMEOUT = 2
DEVERR_FP16_RANGE = 4
MAX_TOPK = 2048

c_p = ctypes.c_void_p
c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_f32 = ctypes.c_float
c_sz = ctypes.c_size_t


class DsaKvPool(ctypes.Structure):
    _fields_ = [("data", c_p), ("scales", c_p), ("rows", c_i64), ("format", c_i32),
                ("block", c_i32), ("d_nope", c_i32), ("d_rope", c_i32)]


class DsaAttnOpts(ctypes.Structure):
    _fields_ = [("sinks", c_p), ("lse_log2", c_i32), ("rows_per_request", c_i32)]


_SIGS = {
    "dsa_status_string": (ctypes.c_char_p, [c_i32]),
    "dsa_abi_version": (c_i32, []),
    "dsa_index_score": (c_i32, [c_p, c_i32, c_p, c_p, c_p, c_i64, c_p, c_p, c_p, c_i32, c_i32,
                                c_i32, c_i64, c_p, c_i64, c_p, c_p]),
    "dsa_index_score_prefill": (c_i32, [c_p, c_i32, c_p, c_p, c_p, c_i64, c_p, c_p, c_p, c_i32,
                                        c_i32, c_i32, c_i64, c_p, c_i64, c_p, c_p]),
    "dsa_topk_workspace_size": (c_sz, [c_i32, c_i64, c_i32]),
    "dsa_topk": (c_i32, [c_p, c_i64, c_p, c_i32, c_i64, c_i32, c_p, c_p, c_p, c_p, c_sz, c_p,
                         c_p]),
    "dsa_topk_noalloc": (c_i32, [c_p, c_i64, c_p, c_i32, c_i64, c_i32, c_p, c_p, c_p, c_p, c_p]),
    "dsa_sparse_mla_workspace_size": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "dsa_sparse_mla_fwd": (c_i32, [c_p, c_i32, c_i32, c_i32, c_i32, c_f32,
                                   ctypes.POINTER(DsaKvPool), c_p, c_i32,
                                   ctypes.POINTER(DsaKvPool), c_p, c_i32,
                                   c_p, c_p, c_p, c_sz, c_p, c_p]),
    "dsa_sparse_mla_fwd_ex": (c_i32, [c_p, c_i32, c_i32, c_i32, c_i32, c_f32,
                                      ctypes.POINTER(DsaKvPool), c_p, c_i32,
                                      ctypes.POINTER(DsaKvPool), c_p, c_i32,
                                      c_p, c_p, c_p, c_sz, c_p, ctypes.POINTER(DsaAttnOpts), c_p]),
    "dsa_decode_ex": (c_i32, [c_p, c_i32, c_p, c_p, c_p, c_i64, c_p, c_i32, c_i32,
                              c_i32, c_p, c_p, c_i64, c_i32,
                              c_p, c_i32, c_i32, c_i32, c_f32, ctypes.POINTER(DsaKvPool),
                              ctypes.POINTER(DsaKvPool), c_p, c_i32,
                              c_p, c_p, c_p, c_p, c_sz, c_p, ctypes.POINTER(DsaAttnOpts), c_p]),
    "dsa_decode_paged": (c_i32, [c_p, c_i32, c_p, c_p, c_p, c_i64, c_p, c_i32, c_i32,
                                 c_i32, c_p, c_p, c_i32, c_i32, c_i64, c_i32,
                                 c_p, c_i32, c_i32, c_i32, c_f32, ctypes.POINTER(DsaKvPool),
                                 ctypes.POINTER(DsaKvPool), c_p, c_i32,
                                 c_p, c_p, c_p, c_p, c_sz, c_p, ctypes.POINTER(DsaAttnOpts), c_p]),
    "dsa_sparse_mla_bwd": (c_i32, [c_p, c_i32, c_i32, c_i32, c_i32, c_f32,
                                   ctypes.POINTER(DsaKvPool), c_p, c_i32, c_p, c_p,
                                   ctypes.POINTER(DsaAttnOpts), c_p, c_p, c_p, c_p, c_p]),
    "dsa_selftest_wait_timeout": (c_i32, [c_p, c_p, c_p]),
    "dsa_decode_workspace_size": (c_sz, [c_i32, c_i64, c_i32, c_i32, c_i32, c_i32]),
    "dsa_decode": (c_i32, [c_p, c_i32, c_p, c_p, c_p, c_i64, c_p, c_i32, c_i32,
                           c_i32, c_p, c_p, c_i64, c_i32,
                           c_p, c_i32, c_i32, c_i32, c_f32, ctypes.POINTER(DsaKvPool),
                           ctypes.POINTER(DsaKvPool), c_p, c_i32,
                           c_p, c_p, c_p, c_p, c_sz, c_p, c_p]),
    "dsa_decode_host_workspace_size": (c_sz, [c_i32, c_i64, c_i32, c_i32, c_i32, c_i32, c_i32,
                                              c_i32, c_i32, c_i32]),
    "dsa_decode_host": (c_i32, [c_p, c_i32, c_p, c_p, c_p, c_i64, c_p, c_i32, c_i32,
                                c_i32, c_p, c_p, c_i64, c_i32,
                                c_p, c_i32, c_i32, c_i32, c_f32, ctypes.POINTER(DsaKvPool),
                                ctypes.POINTER(DsaKvPool), c_p, c_i32,
                                c_p, c_p, c_p, c_p, c_sz, c_p, c_p]),
    "dsa_decode_graph_create": (c_i32, [c_p, c_i32, c_p, c_p, c_p, c_i64, c_p, c_i32, c_i32,
                                        c_i32, c_p, c_p, c_i64, c_i32,
                                        c_p, c_i32, c_i32, c_i32, c_f32,
                                        ctypes.POINTER(DsaKvPool), ctypes.POINTER(DsaKvPool), c_p,
                                        c_i32, c_p, c_p, c_p, c_p, c_sz, c_p,
                                        ctypes.POINTER(c_p)]),
    "dsa_decode_graph_launch": (c_i32, [c_p, c_p]),
    "dsa_decode_graph_destroy": (None, [c_p]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libdsa_gb300.so is missing (%s); build it with "
                               "`python -m deepseek_sparse_attention_index_gb300.build`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def header_functions() -> list:
    """Names of the functions include/dsa.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dsa_\w+)\s*\(", txt, flags=re.M)))


class DsaError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != DSA_OK:
        msg = load().dsa_status_string(status).decode()
        raise DsaError("%s failed: status %d (%s)" % (what, status, msg))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _hptr(t: Optional[torch.Tensor]):
    """Host pointer of a contiguous CPU tensor (pinned memory lets the copies overlap)."""
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("expected a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def kv_pool_struct(pool: Optional[_inp.KVPool]):
    if pool is None:
        return None
    s = DsaKvPool()
    s.data = _ptr(pool.data).value
    s.scales = None if pool.scales is None else _ptr(pool.scales).value
    s.rows = int(pool.rows)
    s.format = int(pool.format)
    s.block = int(pool.block)
    s.d_nope = int(pool.d_nope)
    s.d_rope = int(pool.d_rope)
    return s


def _ref(s):
    return None if s is None else ctypes.byref(s)


# ---------------------------------------------------------------- entry points

def _index_score(entry, q_idx, idx_dtype, q_scale, k_idx, k_scale, w, row_start, row_end,
                 max_len, scores, err_flag):
    T, H_I, d = q_idx.shape
    if scores is None:
        ld = (int(max_len) + 3) // 4 * 4
        scores = torch.full((T, max(ld, 1)), float("nan"), dtype=torch.float32, device=q_idx.device)
    st = getattr(load(), entry)(_ptr(q_idx), idx_dtype, _ptr(q_scale), _ptr(k_idx), _ptr(k_scale),
                                k_idx.shape[0], _ptr(w), _ptr(row_start), _ptr(row_end), T, H_I, d,
                                int(max_len), _ptr(scores), scores.shape[1], _ptr(err_flag),
                                _stream())
    _check(st, entry)
    return scores


def dsa_index_score(q_idx, idx_dtype, q_scale, k_idx, k_scale, w, row_start, row_end,
                    max_len: int, scores=None, err_flag=None):
    """Scores [T, ld] fp32 (see dsa_index_score in include/dsa.h)."""
    return _index_score("dsa_index_score", q_idx, idx_dtype, q_scale, k_idx, k_scale, w,
                        row_start, row_end, max_len, scores, err_flag)


def dsa_index_score_prefill(q_idx, idx_dtype, q_scale, k_idx, k_scale, w, row_start, row_end,
                            max_len: int, scores=None, err_flag=None):
    """The same scores, for causal prefill rows: four rows that start at the
    same key share each key tile (see dsa_index_score_prefill)."""
    return _index_score("dsa_index_score_prefill", q_idx, idx_dtype, q_scale, k_idx, k_scale, w,
                        row_start, row_end, max_len, scores, err_flag)


def dsa_topk_workspace_size(T: int, max_len: int, k: int) -> int:
    return int(load().dsa_topk_workspace_size(T, int(max_len), k))


def dsa_topk(scores, row_len, k: int, max_len: int, index_base=None, idx=None, lens=None,
             ws=None, err_flag=None):
    """idx [T, k] int32 (and lens [T]) from scores [T, ld] (see dsa_topk)."""
    T, ld = scores.shape
    dev = scores.device
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((T,), dtype=torch.int32, device=dev)
    need = dsa_topk_workspace_size(T, max_len, k)
    if ws is None:
        ws = workspace(need, dev)
    st = load().dsa_topk(_ptr(scores), ld, _ptr(row_len), T, int(max_len), k, _ptr(index_base),
                         _ptr(idx), _ptr(lens), _ptr(ws), ws.numel(), _ptr(err_flag), _stream())
    _check(st, "dsa_topk")
    return idx, lens


def dsa_sparse_mla_workspace_size(T, H, Dv, k, k2=0) -> int:
    return int(load().dsa_sparse_mla_workspace_size(T, H, Dv, k, k2))


def _opts(sinks, lse_log2, rows_per_request=0):
    """Attention and step options: per-head sink logits (a CUDA fp32 [H]
    tensor), the lse in log2 units, and (dsa_decode_ex) the rows a request
    contributes; None when none is asked for."""
    if sinks is None and not lse_log2 and not rows_per_request:
        return None
    o = DsaAttnOpts()
    o.sinks = None if sinks is None else _ptr(sinks).value
    o.lse_log2 = 1 if lse_log2 else 0
    o.rows_per_request = int(rows_per_request)
    return o


def dsa_sparse_mla_fwd(q, softmax_scale: float, kv: _inp.KVPool, idx, kv_extra=None,
                       idx_extra=None, out=None, lse=None, ws=None, err_flag=None,
                       sinks=None, lse_log2=False):
    """out bf16 [T, H, Dv], lse fp32 [T, H] (see dsa_sparse_mla_fwd; sinks and
    lse_log2 as dsa_attn_opts)."""
    T, H, D = q.shape
    Dv = kv.d_nope if kv.format != _inp.KV_BF16 else 512
    k = idx.shape[1]
    k2 = 0 if idx_extra is None else idx_extra.shape[1]
    dev = q.device
    if out is None:
        out = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    need = dsa_sparse_mla_workspace_size(T, H, Dv, k, k2)
    if ws is None:
        ws = workspace(need, dev)
    s1, s2 = kv_pool_struct(kv), kv_pool_struct(kv_extra)
    o = _opts(sinks, lse_log2)
    if o is None:
        st = load().dsa_sparse_mla_fwd(_ptr(q), T, H, D, Dv, float(softmax_scale), _ref(s1),
                                       _ptr(idx), k, _ref(s2), _ptr(idx_extra), k2, _ptr(out),
                                       _ptr(lse), _ptr(ws), ws.numel(), _ptr(err_flag), _stream())
    else:
        st = load().dsa_sparse_mla_fwd_ex(_ptr(q), T, H, D, Dv, float(softmax_scale), _ref(s1),
                                          _ptr(idx), k, _ref(s2), _ptr(idx_extra), k2, _ptr(out),
                                          _ptr(lse), _ptr(ws), ws.numel(), _ptr(err_flag),
                                          ctypes.byref(o), _stream())
    _check(st, "dsa_sparse_mla_fwd")
    return out, lse


def dsa_sparse_mla_bwd(q, softmax_scale: float, kv: _inp.KVPool, idx, lse, dout, sinks=None,
                       lse_log2=False, dq=None, dkv=None, dsinks=None, err_flag=None):
    """Backward of dsa_sparse_mla_fwd (see dsa_sparse_mla_bwd): returns dq fp32
    [T, H, 576], dkv fp32 [pool rows, 576] (accumulated into `dkv` when given,
    else into zeros) and dsinks fp32 [H] (with sinks)."""
    T, H, D = q.shape
    dev = q.device
    if dq is None:
        dq = torch.empty((T, H, D), dtype=torch.float32, device=dev)
    if dkv is None:
        dkv = torch.zeros((int(kv.rows), D), dtype=torch.float32, device=dev)
    if dsinks is None and sinks is not None:
        dsinks = torch.zeros((H,), dtype=torch.float32, device=dev)
    o = _opts(sinks, lse_log2)
    st = load().dsa_sparse_mla_bwd(_ptr(q), T, H, D, 512, float(softmax_scale),
                                   _ref(kv_pool_struct(kv)), _ptr(idx), idx.shape[1], _ptr(lse),
                                   _ptr(dout), None if o is None else ctypes.byref(o), _ptr(dq),
                                   _ptr(dkv), _ptr(dsinks), _ptr(err_flag), _stream())
    _check(st, "dsa_sparse_mla_bwd")
    return dq, dkv, dsinks


def dsa_decode_workspace_size(B, max_seq_len, k, H, Dv, k_swa=0) -> int:
    return int(load().dsa_decode_workspace_size(B, int(max_seq_len), k, H, Dv, k_swa))


def dsa_decode(q_idx, idx_dtype, q_scale, k_idx, k_scale, w, seq_lens, slot_base,
               max_seq_len: int, k: int, q, softmax_scale: float, kv: _inp.KVPool,
               kv_swa=None, idx_swa=None, idx_out=None, out=None, lse=None, ws=None,
               err_flag=None, sinks=None, lse_log2=False, rows_per_request=0):
    """One fused decode step (see dsa_decode; sinks, lse_log2 and
    rows_per_request as dsa_attn_opts).  Returns (idx_out, out, lse)."""
    B, H_I, d_idx = q_idx.shape
    _, H, D = q.shape
    Dv = kv.d_nope if kv.format != _inp.KV_BF16 else 512
    k_swa = 0 if idx_swa is None else idx_swa.shape[1]
    dev = q.device
    if idx_out is None:
        idx_out = torch.empty((B, k), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty((B, H, Dv), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    need = dsa_decode_workspace_size(B, max_seq_len, k, H, Dv, k_swa)
    if ws is None:
        ws = workspace(need, dev)
    s1, s2 = kv_pool_struct(kv), kv_pool_struct(kv_swa)
    args = (_ptr(q_idx), idx_dtype, _ptr(q_scale), _ptr(k_idx), _ptr(k_scale), k_idx.shape[0],
            _ptr(w), H_I, d_idx, B, _ptr(seq_lens), _ptr(slot_base), int(max_seq_len), k, _ptr(q),
            H, D, Dv, float(softmax_scale), _ref(s1), _ref(s2), _ptr(idx_swa), k_swa,
            _ptr(idx_out), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _ptr(err_flag))
    o = _opts(sinks, lse_log2, rows_per_request)
    if o is None:
        st = load().dsa_decode(*args, _stream())
    else:
        st = load().dsa_decode_ex(*args, ctypes.byref(o), _stream())
    _check(st, "dsa_decode")
    return idx_out, out, lse


def dsa_decode_host_workspace_size(B, max_seq_len, k, H_I, d_idx, idx_dtype, H, D, Dv,
                                   k_swa=0) -> int:
    return int(load().dsa_decode_host_workspace_size(B, int(max_seq_len), k, H_I, d_idx, idx_dtype,
                                                     H, D, Dv, k_swa))


def dsa_decode_host(q_idx, idx_dtype, q_scale, k_idx, k_scale, w, seq_lens, slot_base,
                    max_seq_len: int, k: int, q, softmax_scale: float, kv: _inp.KVPool,
                    kv_swa=None, idx_swa=None, idx_out=None, out=None, lse=None, ws=None,
                    err_flag=None):
    """dsa_decode with the step's inputs and outputs in host memory (see
    dsa_decode_host).  q_idx, q_scale, w, seq_lens, slot_base, q, idx_swa are
    CPU tensors (pinned for overlap); k_idx, k_scale and the pools are CUDA
    tensors.  Returns host (idx_out, out, lse), allocated pinned when not
    given; they hold the results once the current stream has passed the call."""
    B, H_I, d_idx = q_idx.shape
    _, H, D = q.shape
    Dv = kv.d_nope if kv.format != _inp.KV_BF16 else 512
    k_swa = 0 if idx_swa is None else idx_swa.shape[1]
    if idx_out is None:
        idx_out = torch.empty((B, k), dtype=torch.int32).pin_memory()
    if out is None:
        out = torch.empty((B, H, Dv), dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32).pin_memory()
    need = dsa_decode_host_workspace_size(B, max_seq_len, k, H_I, d_idx, idx_dtype, H, D, Dv,
                                          k_swa)
    if ws is None:
        ws = workspace(need, k_idx.device)
    s1, s2 = kv_pool_struct(kv), kv_pool_struct(kv_swa)
    st = load().dsa_decode_host(_hptr(q_idx), idx_dtype, _hptr(q_scale), _ptr(k_idx),
                                _ptr(k_scale), k_idx.shape[0], _hptr(w), H_I, d_idx, B,
                                _hptr(seq_lens), _hptr(slot_base), int(max_seq_len), k, _hptr(q),
                                H, D, Dv, float(softmax_scale), _ref(s1), _ref(s2),
                                _hptr(idx_swa), k_swa, _hptr(idx_out), _hptr(out), _hptr(lse),
                                _ptr(ws), ws.numel(), _ptr(err_flag), _stream())
    _check(st, "dsa_decode_host")
    return idx_out, out, lse


class DecodeGraph:
    """dsa_decode_graph: the host-buffer decode step captured once and
    replayed by launch().  Every buffer is bound at creation: the caller
    rewrites the pinned inputs in place between launches (q_idx, q_scale, w,
    seq_lens, slot_base, q, idx_swa) and reads idx_out / out / lse once a
    launch has completed on its stream.  The arguments are those of
    dsa_decode_host; host tensors must be pinned."""

    def __init__(self, q_idx, idx_dtype, q_scale, k_idx, k_scale, w, seq_lens, slot_base,
                 max_seq_len: int, k: int, q, softmax_scale: float, kv: _inp.KVPool,
                 kv_swa=None, idx_swa=None, idx_out=None, out=None, lse=None, ws=None,
                 err_flag=None):
        for t in (q_idx, q_scale, w, seq_lens, slot_base, q, idx_swa, idx_out, out, lse):
            if t is not None and (t.is_cuda or not t.is_pinned()):
                raise ValueError("DecodeGraph binds pinned host buffers")
        B, H_I, d_idx = q_idx.shape
        _, H, D = q.shape
        Dv = kv.d_nope if kv.format != _inp.KV_BF16 else 512
        k_swa = 0 if idx_swa is None else idx_swa.shape[1]
        self.idx_out = idx_out if idx_out is not None else \
            torch.empty((B, k), dtype=torch.int32).pin_memory()
        self.out = out if out is not None else \
            torch.empty((B, H, Dv), dtype=torch.bfloat16).pin_memory()
        self.lse = lse if lse is not None else torch.empty((B, H), dtype=torch.float32).pin_memory()
        need = dsa_decode_host_workspace_size(B, max_seq_len, k, H_I, d_idx, idx_dtype, H, D, Dv,
                                              k_swa)
        self.ws = ws if ws is not None else workspace(need, k_idx.device)
        # everything the graph reads or writes stays referenced as long as it
        self._keep = (q_idx, q_scale, k_idx, k_scale, w, seq_lens, slot_base, q, kv, kv_swa,
                      idx_swa, err_flag)
        self._s1, self._s2 = kv_pool_struct(kv), kv_pool_struct(kv_swa)
        h = c_p()
        st = load().dsa_decode_graph_create(
            _hptr(q_idx), idx_dtype, _hptr(q_scale), _ptr(k_idx), _ptr(k_scale), k_idx.shape[0],
            _hptr(w), H_I, d_idx, B, _hptr(seq_lens), _hptr(slot_base), int(max_seq_len), k,
            _hptr(q), H, D, Dv, float(softmax_scale), _ref(self._s1), _ref(self._s2),
            _hptr(idx_swa), k_swa, _hptr(self.idx_out), _hptr(self.out), _hptr(self.lse),
            _ptr(self.ws), self.ws.numel(), _ptr(err_flag), ctypes.byref(h))
        _check(st, "dsa_decode_graph_create")
        self._h = h

    def launch(self):
        """Enqueues one step on the current stream."""
        _check(load().dsa_decode_graph_launch(self._h, _stream()), "dsa_decode_graph_launch")
        return self.idx_out, self.out, self.lse

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load().dsa_decode_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dsa_decode_paged(q_idx, idx_dtype, q_scale, k_idx, k_scale, w, seq_lens, block_table,
                     page_size: int, max_seq_len: int, k: int, q, softmax_scale: float,
                     kv: _inp.KVPool, kv_swa=None, idx_swa=None, idx_out=None, out=None, lse=None,
                     ws=None, err_flag=None, sinks=None, lse_log2=False):
    """The fused decode step on paged caches (see dsa_decode_paged):
    block_table int32 [B, max_pages] on the device.  Returns (idx_out, out, lse);
    idx_out holds pool slots."""
    B, H_I, d_idx = q_idx.shape
    _, H, D = q.shape
    Dv = kv.d_nope if kv.format != _inp.KV_BF16 else 512
    k_swa = 0 if idx_swa is None else idx_swa.shape[1]
    dev = q.device
    if idx_out is None:
        idx_out = torch.empty((B, k), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty((B, H, Dv), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    need = dsa_decode_workspace_size(B, max_seq_len, k, H, Dv, k_swa)
    if ws is None:
        ws = workspace(need, dev)
    s1, s2 = kv_pool_struct(kv), kv_pool_struct(kv_swa)
    o = _opts(sinks, lse_log2)
    st = load().dsa_decode_paged(_ptr(q_idx), idx_dtype, _ptr(q_scale), _ptr(k_idx), _ptr(k_scale),
                                 k_idx.shape[0], _ptr(w), H_I, d_idx, B, _ptr(seq_lens),
                                 _ptr(block_table), block_table.shape[1], int(page_size),
                                 int(max_seq_len), k, _ptr(q), H, D, Dv, float(softmax_scale),
                                 _ref(s1), _ref(s2), _ptr(idx_swa), k_swa, _ptr(idx_out), _ptr(out),
                                 _ptr(lse), _ptr(ws), ws.numel(), _ptr(err_flag),
                                 None if o is None else ctypes.byref(o), _stream())
    _check(st, "dsa_decode_paged")
    return idx_out, out, lse


def decode_case(case: _inp.DecodeCase, ws=None, err_flag=None, idx_out=None, out=None, lse=None,
                rows_per_request=0):
    """dsa_decode on a generated DecodeCase."""
    ind = case.indexer
    if case.meta.get("block_table") is not None:
        return dsa_decode_paged(ind["q_idx"], ind["idx_dtype"], ind["q_scale"], ind["k_idx"],
                                ind["k_scale"], ind["w"], case.seq_lens, case.meta["block_table"],
                                case.meta["page_size"], case.max_seq_len, case.k, case.q,
                                case.softmax_scale, case.kv, case.kv_swa, case.idx_swa,
                                idx_out=idx_out, out=out, lse=lse, ws=ws, err_flag=err_flag)
    return dsa_decode(ind["q_idx"], ind["idx_dtype"], ind["q_scale"], ind["k_idx"], ind["k_scale"],
                      ind["w"], case.seq_lens, case.slot_base, case.max_seq_len, case.k, case.q,
                      case.softmax_scale, case.kv, case.kv_swa, case.idx_swa, idx_out=idx_out,
                      out=out, lse=lse, ws=ws, err_flag=err_flag,
                      rows_per_request=rows_per_request)


def selftest_wait_timeout():
    """Runs dsa_selftest_wait_timeout on the current stream and returns
    (err_flag, completed, cycles waited, limit) after synchronising."""
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    _check(load().dsa_selftest_wait_timeout(_ptr(flag), _ptr(out), _stream()),
           "dsa_selftest_wait_timeout")
    torch.cuda.synchronize()
    o = out.cpu().tolist()
    return int(flag.item()), o[0], o[1], o[2]
