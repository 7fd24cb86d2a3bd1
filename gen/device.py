"""Device-resident synthetic workloads for the GPU tests and the benchmark.

Raw inputs (bf16 latents, keys, queries, SWA rows, fp32 weights and gate
logits) are drawn on the GPU by the CUDA twin of ``gen/inputs.py``
(``gen_cuda.cu``, same bits); the caches are then written through the
library's own cache-write entry point ``csa2_fp4_pack``, in chunks, so a
1M-entry cache never exists in bf16 all at once.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

from . import inputs as G
from .workloads import Workload, H, D, HI, DI, SWA, TOPK

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gen_cuda.cu")
LIB = os.path.join(HERE, "libcsa2gen.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "-Xcompiler", "-fPIC", "-shared", SRC, "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        P, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
        L.gen_normal_bf16.argtypes = [P, u64, i64, i64, i32, P, P]
        L.gen_zipf_keys_bf16.argtypes = [P, u64, u64, i64, i32, i64, i64, i32, P, P, P]
        L.gen_scaled_normal_f32.argtypes = [P, u64, i64, i64, i32, ctypes.c_float, P, P]
        for f in (L.gen_normal_bf16, L.gen_zipf_keys_bf16, L.gen_scaled_normal_f32):
            f.restype = i32
        _lib = L
    return _lib


class DeviceGen:
    """Device draws identical to gen.inputs (checked by a GPU test)."""

    def __init__(self, device="cuda"):
        import torch
        self.torch = torch
        self.device = device
        self.table = torch.from_numpy(G.normal_table().view(np.int16).copy()).to(device)
        self.walk_fail = torch.zeros(1, dtype=torch.int32, device=device)

    def _st(self):
        return self.torch.cuda.current_stream().cuda_stream

    def normal_bf16(self, seed, stream, sub, row0, nrows, ncols, out=None):
        t = self.torch
        if out is None:
            out = t.empty((nrows, ncols), dtype=t.bfloat16, device=self.device)
        rc = lib().gen_normal_bf16(self.table.data_ptr(), G.stream_key(seed, stream, sub), row0, nrows, ncols,
                                   out.data_ptr(), self._st())
        assert rc == 0, rc
        return out

    def zipf_keys_bf16(self, seed, sub, n_entries, row0, nrows, ncols=DI, out=None):
        t = self.torch
        if out is None:
            out = t.empty((nrows, ncols), dtype=t.bfloat16, device=self.device)
        rc = lib().gen_zipf_keys_bf16(self.table.data_ptr(), G.stream_key(seed, G.S_IDX_KEY, sub),
                                      G.stream_key(seed, G.S_ZIPF, sub), n_entries, G._bits_for(n_entries), row0,
                                      nrows, ncols, out.data_ptr(), self.walk_fail.data_ptr(), self._st())
        assert rc == 0, rc
        return out

    def weights_f32(self, seed, stream, sub, row0, nrows, ncols=HI, scale=float(G.W_STD_F32), out=None):
        t = self.torch
        if out is None:
            out = t.empty((nrows, ncols), dtype=t.float32, device=self.device)
        rc = lib().gen_scaled_normal_f32(self.table.data_ptr(), G.stream_key(seed, stream, sub), row0, nrows, ncols,
                                         scale, out.data_ptr(), self._st())
        assert rc == 0, rc
        return out


@dataclass
class DeviceWorkload:
    wl: Workload
    kv: object          # uint8 [n_seq, n_max, 288]
    key_nib: object     # uint8 [n_seq * n_max, 64]
    key_scale: object   # uint8 [n_seq * n_max, 4]
    swa: object         # uint8 [n_seq, swa_cap, 528]
    q: object           # bf16 [n_q, 64, 512]
    q_nib: object       # uint8 [n_q * 32, 64]
    q_scale: object     # uint8 [n_q * 32, 4]
    w: object           # fp32 [n_q, 32]
    q_nib_re: object = None
    q_scale_re: object = None
    w_re: object = None
    q_seq: object = None
    n_vis: object = None
    pos: object = None
    swa_first: object = None
    swa_cnt: object = None

    @property
    def n_max(self):
        return self.kv.shape[1]


def _pack(kind, src, rows, m, gate, dst, dst_scales):
    from compressed_sparse_attention_index_gb300 import csa2_fp4_pack
    csa2_fp4_pack(kind, src, rows, m, gate, dst, dst_scales)


def build_device_workload(wl: Workload, n_max: int | None = None, chunk: int = 1 << 16,
                          n_q: int | None = None) -> DeviceWorkload:
    """Draw and pack every input of a workload on the current CUDA device."""
    import torch
    from compressed_sparse_attention_index_gb300 import CSA2_KV_NVFP4, CSA2_IDX_MXFP4, CSA2_SWA_MXFP8
    dev = "cuda"
    g = DeviceGen(dev)
    N = wl.n_entries
    n_max = n_max or ((N + 127) // 128) * 128
    n_q = wl.n_q if n_q is None else n_q
    kv = torch.zeros((wl.n_seq, n_max, 288), dtype=torch.uint8, device=dev)
    key_nib = torch.zeros((wl.n_seq * n_max, 64), dtype=torch.uint8, device=dev)
    key_scale = torch.zeros((wl.n_seq * n_max, 4), dtype=torch.uint8, device=dev)
    swa = torch.zeros((wl.n_seq, wl.swa_cap, 528), dtype=torch.uint8, device=dev)
    for b in range(wl.n_seq):
        for r0 in range(0, N, chunk):
            r1 = min(N, r0 + chunk)
            n = r1 - r0
            if wl.m == 1:
                lat = g.normal_bf16(wl.seed, G.S_LATENT, b, r0, n, D)
                _pack(CSA2_KV_NVFP4, lat, n, 1, None, kv[b, r0:r1], None)
            else:
                tok = g.normal_bf16(wl.seed, G.S_LATENT, b, 2 * r0, 2 * n, D)
                gate = g.normal_bf16(wl.seed, G.S_GATE, b, 2 * r0, 2 * n, D).float()
                _pack(CSA2_KV_NVFP4, tok, 2 * n, 2, gate, kv[b, r0:r1], None)
            if wl.zipf:
                keys = g.zipf_keys_bf16(wl.seed, b, N, r0, n)
            else:
                keys = g.normal_bf16(wl.seed, G.S_IDX_KEY, b, r0, n, DI)
            base = b * n_max + r0
            _pack(CSA2_IDX_MXFP4, keys, n, 1, None, key_nib[base:base + n], key_scale[base:base + n])
        for s0 in range(0, wl.swa_cap, chunk):
            s1 = min(wl.swa_cap, s0 + chunk)
            rows = g.normal_bf16(wl.seed, G.S_SWA, b, s0, s1 - s0, D)
            _pack(CSA2_SWA_MXFP8, rows, s1 - s0, 1, None, swa[b, s0:s1], None)
    q = torch.empty((n_q, H, D), dtype=torch.bfloat16, device=dev)
    qidx = torch.empty((n_q * HI, DI), dtype=torch.bfloat16, device=dev)
    w = torch.empty((n_q, HI), dtype=torch.float32, device=dev)
    qidx_re = torch.empty_like(qidx) if wl.pool else None
    w_re = torch.empty_like(w) if wl.pool else None
    for qi in range(n_q):
        g.normal_bf16(wl.seed, G.S_Q, qi, 0, H, D, out=q[qi])
        g.normal_bf16(wl.seed, G.S_QIDX, qi, 0, HI, DI, out=qidx[qi * HI:(qi + 1) * HI])
        g.weights_f32(wl.seed, G.S_W, qi, 0, 1, out=w[qi:qi + 1])
        if wl.pool:
            g.normal_bf16(wl.seed, G.S_QIDX_RE, qi, 0, HI, DI, out=qidx_re[qi * HI:(qi + 1) * HI])
            g.weights_f32(wl.seed, G.S_W_RE, qi, 0, 1, out=w_re[qi:qi + 1])
    q_nib = torch.empty((n_q * HI, 64), dtype=torch.uint8, device=dev)
    q_scale = torch.empty((n_q * HI, 4), dtype=torch.uint8, device=dev)
    _pack(CSA2_IDX_MXFP4, qidx, n_q * HI, 1, None, q_nib, q_scale)
    dw = DeviceWorkload(wl, kv, key_nib, key_scale, swa, q, q_nib, q_scale, w)
    if wl.pool:
        dw.q_nib_re = torch.empty_like(q_nib)
        dw.q_scale_re = torch.empty_like(q_scale)
        _pack(CSA2_IDX_MXFP4, qidx_re, n_q * HI, 1, None, dw.q_nib_re, dw.q_scale_re)
        dw.w_re = w_re
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a[:n_q], dtype=np.int32)).to(dev)
    dw.q_seq, dw.n_vis, dw.pos = i32(wl.q_seq()), i32(wl.n_vis()), i32(wl.pos())
    dw.swa_first, dw.swa_cnt = i32(wl.swa_first()), i32(wl.swa_cnt())
    assert int(g.walk_fail.item()) == 0
    return dw


@dataclass
class DecoderLayers:
    """Device tensors of the decoder step's layers (see gen.workloads.DECODER_LAYERS):
    per layer an attention query and a window cache (layer 0 shares the
    workload's), per Reindex layer r an indexer query and weights."""
    q: object           # bf16 [L, n_q, 64, 512]
    swa: object         # uint8 [L, n_seq, swa_cap, 528]
    q_nib_re: dict      # r -> uint8 [n_q * 32, 64]
    q_scale_re: dict    # r -> uint8 [n_q * 32, 4]
    w_re: dict          # r -> fp32 [n_q, 32]


def build_decoder_layers(wl: Workload, dw: DeviceWorkload, layers) -> DecoderLayers:
    import torch
    from compressed_sparse_attention_index_gb300 import CSA2_IDX_MXFP4, CSA2_SWA_MXFP8
    g = DeviceGen("cuda")
    L, n_q = len(layers), dw.q.shape[0]
    q = torch.empty((L, n_q, H, D), dtype=torch.bfloat16, device="cuda")
    swa = torch.zeros((L, wl.n_seq, wl.swa_cap, 528), dtype=torch.uint8, device="cuda")
    q[0].copy_(dw.q)
    swa[0].copy_(dw.swa)
    for l in range(1, L):
        for qi in range(n_q):
            g.normal_bf16(wl.seed, G.S_LQ, l * G.LAYER_SUB + qi, 0, H, D, out=q[l, qi])
        for b in range(wl.n_seq):
            rows = g.normal_bf16(wl.seed, G.S_LSWA, l * G.LAYER_SUB + b, 0, wl.swa_cap, D)
            _pack(CSA2_SWA_MXFP8, rows, wl.swa_cap, 1, None, swa[l, b], None)
    q_nib_re, q_scale_re, w_re = {}, {}, {}
    for r in sorted({r for role, r in layers if role == "reindex"}):
        qidx = torch.empty((n_q * HI, DI), dtype=torch.bfloat16, device="cuda")
        w = torch.empty((n_q, HI), dtype=torch.float32, device="cuda")
        for qi in range(n_q):
            g.normal_bf16(wl.seed, G.S_QIDX_RE, r * G.LAYER_SUB + qi, 0, HI, DI, out=qidx[qi * HI:(qi + 1) * HI])
            g.weights_f32(wl.seed, G.S_W_RE, r * G.LAYER_SUB + qi, 0, 1, out=w[qi:qi + 1])
        q_nib_re[r] = torch.empty((n_q * HI, 64), dtype=torch.uint8, device="cuda")
        q_scale_re[r] = torch.empty((n_q * HI, 4), dtype=torch.uint8, device="cuda")
        _pack(CSA2_IDX_MXFP4, qidx, n_q * HI, 1, None, q_nib_re[r], q_scale_re[r])
        w_re[r] = w
    assert int(g.walk_fail.item()) == 0
    return DecoderLayers(q, swa, q_nib_re, q_scale_re, w_re)
