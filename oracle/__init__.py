"""CPU oracle for the CSA2 decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never calls it and
shares no code with it.  The arithmetic lives in ``csa2_oracle.c`` (fp64, one
plain loop nest per step, each step citing the page passage it restates); this
file only marshals numpy arrays and composes the steps in the order the pages
give them (score -> top-512 -> attention; pool -> reindex -> attention).

Parity status per function (the pins are the ``-m "not gpu"`` tests):
  formats, pack_*, pool_m2  pinned (closed forms, library format tables,
                            round trips, gate special cases)
  index_score               pinned (independent numpy restatement on decoded
                            values; ReLU and weight-sign cases)
  topk, pool_blocks         pinned (brute-force sort, superset invariant)
  sparse_attn               pinned (dense softmax attention, single-entry and
                            RoPE closed forms, shift invariance)
  attn_f64                  pinned (RoPE shift invariance, position 0 = no
                            rotation; sparse_attn is this on dequantised records)
  sparse_attn_lse           pinned (outputs of parts of a softmax's entries,
                            merged by their log-sum-exp, equal the whole)
DeepSeek's own numerics are not published on the pages, so parity is pinned to
the readings stated in the C source, not to DeepSeek's kernels.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

KV_BYTES, IDX_BYTES, SWA_BYTES = 288, 68, 528
H, D, HI, DI = 64, 512, 32, 128


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        sig = {
            "orc_e2m1_value": (f64, [i32]), "orc_e4m3_value": (f64, [i32]),
            "orc_e8m0_value": (f64, [i32]), "orc_e2m1_encode": (i32, [f64]),
            "orc_e4m3_encode": (i32, [f64]), "orc_bf16_from_double": (ctypes.c_uint16, [f64]),
            "orc_pack_kv": (None, [P, i64, P]), "orc_pack_idx": (None, [P, i64, P]),
            "orc_pack_swa": (None, [P, i64, P]), "orc_pool_m2": (None, [P, P, i64, P]),
            "orc_project_keys": (None, [P, i64, P, P]),
            "orc_dequant_kv": (None, [P, P]), "orc_dequant_idx": (None, [P, P]),
            "orc_dequant_swa": (None, [P, P]),
            "orc_index_score": (None, [P, i64, P, P, P]),
            "orc_topk": (i32, [P, i64, i32, P]),
            "orc_pool_blocks": (i32, [P, i64, i32, i32, P]),
            "orc_sparse_attn": (None, [P, P, i32, P, i32, i64, f64, f64, i32, i32, P]),
            "orc_sparse_attn_lse": (None, [P, P, i32, P, i32, i64, f64, f64, i32, i32, P, P]),
            "orc_attn_f64": (None, [P, P, i32, i64, f64, f64, i32, i32, P, P]),
            "orc_kv_bytes": (i32, []), "orc_idx_bytes": (i32, []), "orc_swa_bytes": (i32, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ formats
def e2m1_value(code: int) -> float: return lib().orc_e2m1_value(int(code))
def e4m3_value(b: int) -> float: return lib().orc_e4m3_value(int(b))
def e8m0_value(b: int) -> float: return lib().orc_e8m0_value(int(b))
def e2m1_encode(x: float) -> int: return lib().orc_e2m1_encode(float(x))
def e4m3_encode(x: float) -> int: return lib().orc_e4m3_encode(float(x))
def bf16_from_double(x: float) -> int: return int(lib().orc_bf16_from_double(float(x)))


def entry_bytes():
    L = lib()
    return {"kv": L.orc_kv_bytes(), "idx": L.orc_idx_bytes(), "swa": L.orc_swa_bytes()}


# ------------------------------------------------------------------ packing
def pack_kv(x_bf16: np.ndarray) -> np.ndarray:
    x = _c(x_bf16, np.uint16).reshape(-1, D)
    out = np.zeros((x.shape[0], KV_BYTES), np.uint8)
    lib().orc_pack_kv(_p(x), x.shape[0], _p(out))
    return out


def pack_idx(x_bf16: np.ndarray) -> np.ndarray:
    """Logical 68-byte records: 64 nibble bytes then 4 E8M0 bytes."""
    x = _c(x_bf16, np.uint16).reshape(-1, DI)
    out = np.zeros((x.shape[0], IDX_BYTES), np.uint8)
    lib().orc_pack_idx(_p(x), x.shape[0], _p(out))
    return out


def pack_swa(x_bf16: np.ndarray) -> np.ndarray:
    x = _c(x_bf16, np.uint16).reshape(-1, D)
    out = np.zeros((x.shape[0], SWA_BYTES), np.uint8)
    lib().orc_pack_swa(_p(x), x.shape[0], _p(out))
    return out


def pool_m2(x_bf16: np.ndarray, z: np.ndarray) -> np.ndarray:
    x = _c(x_bf16, np.uint16).reshape(-1, D)
    z = _c(z, np.float32).reshape(-1, D)
    assert x.shape == z.shape and x.shape[0] % 2 == 0
    out = np.zeros((x.shape[0] // 2, D), np.uint16)
    lib().orc_pool_m2(_p(x), _p(z), out.shape[0], _p(out))
    return out


def project_keys(x_bf16: np.ndarray, w_bf16: np.ndarray) -> np.ndarray:
    """The indexer keys of latents x ([rows][512] bf16 bits) under the 512 -> 128
    projection w ([128][512] bf16 bits): [rows][128] bf16 bits."""
    x = _c(x_bf16, np.uint16).reshape(-1, D)
    w = _c(w_bf16, np.uint16).reshape(128, D)
    out = np.zeros((x.shape[0], 128), np.uint16)
    lib().orc_project_keys(_p(x), x.shape[0], _p(w), _p(out))
    return out


def dequant_kv(rec: np.ndarray) -> np.ndarray:
    rec = _c(rec, np.uint8).reshape(-1, KV_BYTES)
    out = np.zeros((rec.shape[0], D), np.float64)
    for i in range(rec.shape[0]):
        lib().orc_dequant_kv(_p(rec[i]), _p(out[i]))
    return out


def dequant_idx(rec: np.ndarray) -> np.ndarray:
    rec = _c(rec, np.uint8).reshape(-1, IDX_BYTES)
    out = np.zeros((rec.shape[0], DI), np.float64)
    for i in range(rec.shape[0]):
        lib().orc_dequant_idx(_p(rec[i]), _p(out[i]))
    return out


def dequant_swa(rec: np.ndarray) -> np.ndarray:
    rec = _c(rec, np.uint8).reshape(-1, SWA_BYTES)
    out = np.zeros((rec.shape[0], D), np.float64)
    for i in range(rec.shape[0]):
        lib().orc_dequant_swa(_p(rec[i]), _p(out[i]))
    return out


# ------------------------------------------------------------ path steps
def index_score(keys68: np.ndarray, qidx68: np.ndarray, w: np.ndarray) -> np.ndarray:
    k = _c(keys68, np.uint8).reshape(-1, IDX_BYTES)
    q = _c(qidx68, np.uint8).reshape(HI, IDX_BYTES)
    w = _c(w, np.float32).reshape(HI)
    out = np.zeros(k.shape[0], np.float64)
    lib().orc_index_score(_p(k), k.shape[0], _p(q), _p(w), _p(out))
    return out


def topk(scores: np.ndarray, k: int = 512) -> np.ndarray:
    s = _c(scores, np.float64)
    out = np.zeros(k, np.int32)
    lib().orc_topk(_p(s), s.shape[0], k, _p(out))
    return out


def pool_blocks(scores: np.ndarray, block: int = 8, nb: int = 2048) -> np.ndarray:
    s = _c(scores, np.float64)
    out = np.zeros(nb, np.int32)
    lib().orc_pool_blocks(_p(s), s.shape[0], block, nb, _p(out))
    return out


def sparse_attn(q_bf16, kv_rows, swa_rows, pos, sm_scale=1.0 / np.sqrt(512.0), rope_base=10000.0,
                rope_off=448, rope_dim=64) -> np.ndarray:
    q = _c(q_bf16, np.uint16).reshape(H, D)
    kv = _c(kv_rows, np.uint8).reshape(-1, KV_BYTES)
    sw = _c(swa_rows, np.uint8).reshape(-1, SWA_BYTES)
    out = np.zeros((H, D), np.float64)
    lib().orc_sparse_attn(_p(q), _p(kv), kv.shape[0], _p(sw), sw.shape[0], int(pos), float(sm_scale),
                          float(rope_base), rope_off, rope_dim, _p(out))
    return out


def sparse_attn_lse(q_bf16, kv_rows, swa_rows, pos, sm_scale=1.0 / np.sqrt(512.0), rope_base=10000.0,
                    rope_off=448, rope_dim=64):
    """sparse_attn, and per head the log-sum-exp of the logits over the entries given."""
    q = _c(q_bf16, np.uint16).reshape(H, D)
    kv = _c(kv_rows, np.uint8).reshape(-1, KV_BYTES)
    sw = _c(swa_rows, np.uint8).reshape(-1, SWA_BYTES)
    out = np.zeros((H, D), np.float64)
    lse = np.zeros(H, np.float64)
    lib().orc_sparse_attn_lse(_p(q), _p(kv), kv.shape[0], _p(sw), sw.shape[0], int(pos), float(sm_scale),
                              float(rope_base), rope_off, rope_dim, _p(out), _p(lse))
    return out, lse


def attn_f64(q, k, pos, sm_scale=1.0 / np.sqrt(512.0), rope_base=10000.0, rope_off=448, rope_dim=64,
             with_lse=False):
    """The attention arithmetic of sparse_attn on fp64 inputs (no cache
    records): q [64][512], k [n][512] (keys = values).  Returns out [64][512]
    (and the per-head log-sum-exp when with_lse)."""
    q = _c(q, np.float64).reshape(H, D)
    k = _c(k, np.float64).reshape(-1, D)
    out = np.zeros((H, D), np.float64)
    lse = np.zeros(H, np.float64)
    lib().orc_attn_f64(_p(q), _p(k), k.shape[0], int(pos), float(sm_scale), float(rope_base), rope_off, rope_dim,
                       _p(out), _p(lse))
    return (out, lse) if with_lse else out


from .compose import *  # noqa: E402,F401,F403  (workload-level compositions)
