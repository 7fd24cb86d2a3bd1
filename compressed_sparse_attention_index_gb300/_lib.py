"""ctypes binding of libcsa2.so: the C entry points under the same names.

Argument marshalling only: torch tensors (or raw integer device addresses)
become pointers, ``stream=None`` becomes torch's current CUDA stream, and a
non-OK status becomes a ``CSA2Error``.  Every step of the path runs in the CUDA
library; there is no other implementation to fall back to, so importing this
module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcsa2.so")

CSA2_KV_NVFP4, CSA2_IDX_MXFP4, CSA2_SWA_MXFP8 = 0, 1, 2
CSA2_OUT_BF16, CSA2_OUT_F32 = 0, 1
CSA2_OP_TOPK, CSA2_OP_SPARSE_ATTN, CSA2_OP_DECODE, CSA2_OP_DECODE_HOST, CSA2_OP_DECODE_MQ = 0, 1, 2, 3, 4
CSA2_OP_BUILD_CACHE, CSA2_OP_DECODE_REINDEX = 5, 6
STATUS = {0: "CSA2_OK", 1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED", 3: "CSA2_ERR_CUDA",
          4: "CSA2_ERR_BOUNDS", 5: "CSA2_ERR_TIMEOUT", 6: "CSA2_ERR_WORKSPACE"}

EXPORTS = ["csa2_default_params", "csa2_entry_bytes", "csa2_status_string", "csa2_fp4_pack",
           "csa2_index_score", "csa2_topk", "csa2_sparse_attn", "csa2_workspace_size",
           "csa2_get_device_status", "csa2_topk_noalloc", "csa2_decode", "csa2_decode_host",
           "csa2_index_score_mq", "csa2_decode_mq", "csa2_check_bounded_wait", "csa2_index_key_proj",
           "csa2_build_cache", "csa2_decode_reindex", "csa2_profile_events"]


class CSA2Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class csa2_params(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int), ("dim", ctypes.c_int), ("rope_dim", ctypes.c_int),
                ("rope_off", ctypes.c_int), ("rope_base", ctypes.c_double), ("sm_scale", ctypes.c_float),
                ("idx_heads", ctypes.c_int), ("idx_dim", ctypes.c_int), ("topk", ctypes.c_int),
                ("swa", ctypes.c_int), ("block", ctypes.c_int), ("pool_blocks", ctypes.c_int)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libcsa2.so (raises if it is missing) and declare the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libcsa2.so not built at {path}: run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    PP = ctypes.POINTER(csa2_params)
    sig = {
        "csa2_default_params": (i32, [PP]),
        "csa2_entry_bytes": (sz, [i32]),
        "csa2_status_string": (ctypes.c_char_p, [i32]),
        "csa2_fp4_pack": (i32, [i32, P, i64, i32, P, P, P, P]),
        "csa2_index_score": (i32, [P, P, i64, i32, P, P, P, P, P, i32, P, P, i64, PP, P]),
        "csa2_topk": (i32, [P, i64, i32, P, i64, i32, i32, P, P, P, sz, P]),
        "csa2_decode": (i32, [P, P, i64, i32, P, P, P, P, P, i32, P, P, P, i32, P, P, P, P, P, i32, PP, P, sz, P]),
        "csa2_decode_reindex": (i32, [P, P, i64, i32, P, P, P, P, P, i32, P, P, P, P, i32, P, P, P, P, P, i32, PP, P,
                                      sz, P]),
        "csa2_index_score_mq": (i32, [P, P, i64, i32, P, P, P, P, P, i32, i32, P, i64, PP, P]),
        "csa2_decode_mq": (i32, [P, P, i64, i32, P, P, P, P, P, i32, i32, P, P, P, i32, P, P, P, P, P, i32, PP, P, sz,
                                 P]),
        "csa2_decode_host": (i32, [P, P, i64, i32, P, P, i32, P, P, P, P, i32, P, P, i32, PP, P, sz, P]),
        "csa2_topk_noalloc": (i32, [P, i64, i32, P, i64, i32, i32, P, P, P]),
        "csa2_sparse_attn": (i32, [P, P, i64, i32, P, i32, P, i32, P, P, P, P, i32, P, i32, PP, P, sz, P]),
        "csa2_workspace_size": (i32, [i32, i32, i64, i32, ctypes.POINTER(sz)]),
        "csa2_get_device_status": (i32, [P, ctypes.POINTER(i32)]),
        "csa2_profile_events": (i32, [P, P]),
        "csa2_check_bounded_wait": (i32, [ctypes.c_uint, P]),
        "csa2_index_key_proj": (i32, [P, i64, P, P, P]),
        "csa2_build_cache": (i32, [P, i64, i32, P, P, P, P, P, P, sz, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, code):
    if code != 0:
        raise CSA2Error(fn, code)


def default_params() -> csa2_params:
    p = csa2_params()
    _check("csa2_default_params", load().csa2_default_params(ctypes.byref(p)))
    return p


def csa2_entry_bytes(kind: int) -> int:
    return int(load().csa2_entry_bytes(kind))


def csa2_fp4_pack(kind, src, rows, m, gate_logits, dst, dst_scales=None, stream=None):
    _check("csa2_fp4_pack", load().csa2_fp4_pack(kind, _ptr(src), int(rows), int(m), _ptr(gate_logits), _ptr(dst),
                                                 _ptr(dst_scales), _stream(stream)))


def csa2_index_score(key_nib, key_scale, n_max, n_seq, q_nib, q_scale, w, q_seq, n_vis, n_q, pool_blocks, scores,
                     score_stride, params=None, stream=None):
    pp = ctypes.byref(params) if params is not None else None
    _check("csa2_index_score", load().csa2_index_score(
        _ptr(key_nib), _ptr(key_scale), int(n_max), int(n_seq), _ptr(q_nib), _ptr(q_scale), _ptr(w), _ptr(q_seq),
        _ptr(n_vis), int(n_q), _ptr(pool_blocks), _ptr(scores), int(score_stride), pp, _stream(stream)))


def csa2_workspace_size(op, n_q, n_items, k=0) -> int:
    b = ctypes.c_size_t(0)
    _check("csa2_workspace_size", load().csa2_workspace_size(op, int(n_q), int(n_items), int(k), ctypes.byref(b)))
    return int(b.value)


def csa2_topk(scores, score_stride, n_q, n_valid, n_max, k, block, pool_blocks, out, workspace, workspace_bytes,
              stream=None):
    _check("csa2_topk", load().csa2_topk(_ptr(scores), int(score_stride), int(n_q), _ptr(n_valid), int(n_max), int(k),
                                         int(block), _ptr(pool_blocks), _ptr(out), _ptr(workspace),
                                         int(workspace_bytes), _stream(stream)))


def csa2_topk_noalloc(scores, score_stride, n_q, n_valid, n_max, k, block, pool_blocks, out, stream=None):
    """csa2_topk without a workspace argument (scratch is a fixed array inside the library)."""
    _check("csa2_topk_noalloc", load().csa2_topk_noalloc(_ptr(scores), int(score_stride), int(n_q), _ptr(n_valid),
                                                         int(n_max), int(k), int(block), _ptr(pool_blocks), _ptr(out),
                                                         _stream(stream)))


def csa2_sparse_attn(q, kv_cache, n_max, n_seq, sel, sel_stride, swa_cache, swa_cap, q_seq, pos, swa_first, swa_cnt,
                     n_q, out, out_dtype, params=None, workspace=None, workspace_bytes=0, stream=None):
    pp = ctypes.byref(params) if params is not None else None
    _check("csa2_sparse_attn", load().csa2_sparse_attn(
        _ptr(q), _ptr(kv_cache), int(n_max), int(n_seq), _ptr(sel), int(sel_stride), _ptr(swa_cache), int(swa_cap),
        _ptr(q_seq), _ptr(pos), _ptr(swa_first), _ptr(swa_cnt), int(n_q), _ptr(out), int(out_dtype), pp,
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def csa2_decode(key_nib, key_scale, n_max, n_seq, q_nib, q_scale, w, q_seq, n_vis, n_q, q, kv_cache, swa_cache,
                swa_cap, pos, swa_first, swa_cnt, sel, out, out_dtype, params=None, workspace=None,
                workspace_bytes=0, stream=None):
    pp = ctypes.byref(params) if params is not None else None
    _check("csa2_decode", load().csa2_decode(
        _ptr(key_nib), _ptr(key_scale), int(n_max), int(n_seq), _ptr(q_nib), _ptr(q_scale), _ptr(w), _ptr(q_seq),
        _ptr(n_vis), int(n_q), _ptr(q), _ptr(kv_cache), _ptr(swa_cache), int(swa_cap), _ptr(pos), _ptr(swa_first),
        _ptr(swa_cnt), _ptr(sel), _ptr(out), int(out_dtype), pp, _ptr(workspace), int(workspace_bytes),
        _stream(stream)))


def csa2_profile_events(begin=None, end=None):
    """Events (torch.cuda.Event, already recorded once so that they exist)
    that csa2_decode / csa2_decode_reindex record around their indexer launch
    on this host thread; both None: off."""
    ptr = lambda e: None if e is None else int(e.cuda_event)
    _check("csa2_profile_events", load().csa2_profile_events(ptr(begin), ptr(end)))


def csa2_decode_reindex(key_nib, key_scale, n_max, n_seq, q_nib, q_scale, w, q_seq, n_vis, n_q, pool_blocks, q,
                        kv_cache, swa_cache, swa_cap, pos, swa_first, swa_cnt, sel, out, out_dtype, params=None,
                        workspace=None, workspace_bytes=0, stream=None):
    pp = ctypes.byref(params) if params is not None else None
    _check("csa2_decode_reindex", load().csa2_decode_reindex(
        _ptr(key_nib), _ptr(key_scale), int(n_max), int(n_seq), _ptr(q_nib), _ptr(q_scale), _ptr(w), _ptr(q_seq),
        _ptr(n_vis), int(n_q), _ptr(pool_blocks), _ptr(q), _ptr(kv_cache), _ptr(swa_cache), int(swa_cap), _ptr(pos),
        _ptr(swa_first), _ptr(swa_cnt), _ptr(sel), _ptr(out), int(out_dtype), pp, _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def csa2_index_score_mq(key_nib, key_scale, n_max, n_seq, q_nib, q_scale, w, q_seq, n_vis, n_q, q_group, scores,
                        score_stride, params=None, stream=None):
    pp = ctypes.byref(params) if params is not None else None
    _check("csa2_index_score_mq", load().csa2_index_score_mq(
        _ptr(key_nib), _ptr(key_scale), int(n_max), int(n_seq), _ptr(q_nib), _ptr(q_scale), _ptr(w), _ptr(q_seq),
        _ptr(n_vis), int(n_q), int(q_group), _ptr(scores), int(score_stride), pp, _stream(stream)))


def csa2_decode_mq(key_nib, key_scale, n_max, n_seq, q_nib, q_scale, w, q_seq, n_vis, n_q, q_group, q, kv_cache,
                   swa_cache, swa_cap, pos, swa_first, swa_cnt, sel, out, out_dtype, params=None, workspace=None,
                   workspace_bytes=0, stream=None):
    pp = ctypes.byref(params) if params is not None else None
    _check("csa2_decode_mq", load().csa2_decode_mq(
        _ptr(key_nib), _ptr(key_scale), int(n_max), int(n_seq), _ptr(q_nib), _ptr(q_scale), _ptr(w), _ptr(q_seq),
        _ptr(n_vis), int(n_q), int(q_group), _ptr(q), _ptr(kv_cache), _ptr(swa_cache), int(swa_cap), _ptr(pos),
        _ptr(swa_first), _ptr(swa_cnt), _ptr(sel), _ptr(out), int(out_dtype), pp, _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def csa2_decode_host(key_nib, key_scale, n_max, n_seq, kv_cache, swa_cache, swa_cap, h_q, h_qidx, h_w, h_desc, n_q,
                     h_sel, h_out, out_dtype, params=None, workspace=None, workspace_bytes=0, stream=None):
    """csa2_decode with the step's inputs and outputs in host memory (pinned
    CPU tensors): the copies happen inside the call, on the stream."""
    pp = ctypes.byref(params) if params is not None else None
    _check("csa2_decode_host", load().csa2_decode_host(
        _ptr(key_nib), _ptr(key_scale), int(n_max), int(n_seq), _ptr(kv_cache), _ptr(swa_cache), int(swa_cap),
        _ptr(h_q), _ptr(h_qidx), _ptr(h_w), _ptr(h_desc), int(n_q), _ptr(h_sel), _ptr(h_out), int(out_dtype), pp,
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def csa2_check_bounded_wait(limit_us, stream=None):
    """Self-test of the bounded waits: a wait that cannot finish ends after
    limit_us with CSA2_ERR_TIMEOUT in the device status (read it with
    csa2_get_device_status)."""
    _check("csa2_check_bounded_wait", load().csa2_check_bounded_wait(int(limit_us), _stream(stream)))


def csa2_get_device_status(stream=None) -> int:
    v = ctypes.c_int(0)
    _check("csa2_get_device_status", load().csa2_get_device_status(_stream(stream), ctypes.byref(v)))
    return int(v.value)


def csa2_index_key_proj(latent, rows, w_idx, keys, stream=None):
    _check("csa2_index_key_proj", load().csa2_index_key_proj(_ptr(latent), int(rows), _ptr(w_idx), _ptr(keys),
                                                               _stream(stream)))


def csa2_build_cache(tokens, n_tokens, m, gate_logits, w_idx, kv, idx_nib, idx_scale, workspace, workspace_bytes,
                     stream=None):
    _check("csa2_build_cache", load().csa2_build_cache(_ptr(tokens), int(n_tokens), int(m), _ptr(gate_logits),
                                                         _ptr(w_idx), _ptr(kv), _ptr(idx_nib), _ptr(idx_scale),
                                                         _ptr(workspace), int(workspace_bytes), _stream(stream)))
