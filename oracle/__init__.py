"""fp64 CPU oracle for unified paged varlen attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The product path never
imports this package.

The arithmetic lives in ``ua_oracle.c`` (plain C, fp64, see its header for the
definition it writes out); this module compiles it with gcc on first use and
wraps it with ctypes.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against a library routine (torch fp64 scaled_dot_product_attention on dense
per-sequence K/V with an explicit bottom-right mask), closed forms (a single
visible key, identical keys, zero scale, a hand-derived two-key example under
``tests/golden/``), exact mask-boundary counts, and invariances (physical
placement, aliasing, decode vs prefill, chunking, split-KV merge).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ua_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libua_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {1: "bad shape", 2: "bad sequence lengths", 3: "block id out of range", 4: "out of memory"}


class OracleError(ValueError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, fp64, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.ua_oracle_attention.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i,
                                                ctypes.c_double, i, i, i, P, P, i]
            lib.ua_oracle_attention.restype = i
            lib.ua_oracle_attention_fp8kv.argtypes = [P, P, P, ctypes.c_double, ctypes.c_double,
                                                      P, P, P, i, i, i, i, i, i, i,
                                                      ctypes.c_double, i, P, P, i]
            lib.ua_oracle_attention_fp8kv.restype = i
            lib.ua_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.ua_oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.ua_oracle_merge.argtypes = [i, P, P, ctypes.c_int64, i, P, P]
            lib.ua_oracle_merge.restype = i
            lib.ua_oracle_max_threads.restype = i
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().ua_oracle_max_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table, softmax_scale,
              causal, num_kv_heads=None, key_window=None, nthreads=0):
    """fp64 attention over a paged varlen batch.

    q: uint16 (bf16 bits) [total_q, Hq, D]; k_cache / v_cache: uint16
    [num_blocks, block_size, Hkv, D]; cu_seqlens_q int32 [N+1]; seqused_k int32
    [N]; block_table int32 [N, stride].  Returns (out fp64 [total_q, Hq, D],
    lse fp64 [total_q, Hq]) with lse the natural-log normaliser.
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    sk = np.ascontiguousarray(seqused_k, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    if bt.ndim == 1:
        bt = bt.reshape(len(sk), -1)
    total_q, hq, d = q.shape
    nb, bs, hk, d2 = k_cache.shape
    if num_kv_heads is not None and num_kv_heads != hk:
        raise OracleError("num_kv_heads disagrees with the cache shape")
    if d2 != d or v_cache.shape != k_cache.shape:
        raise OracleError("q / cache shapes disagree")
    if len(cu) != len(sk) + 1 or (len(sk) and cu[-1] != total_q):
        raise OracleError("cu_seqlens_q does not match q")
    lo, hi = (0, 2**31 - 1) if key_window is None else key_window
    out = np.zeros((total_q, hq, d), dtype=np.float64)
    lse = np.full((total_q, hq), -np.inf, dtype=np.float64)
    rc = _load().ua_oracle_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu), _ptr(sk),
                                     _ptr(bt), len(sk), hq, hk, d, bs, nb, bt.shape[1],
                                     float(softmax_scale), int(bool(causal)), int(lo), int(hi),
                                     _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"oracle error {rc}"))
    return out, lse


def attention_batch(batch, key_window=None, nthreads=0):
    """``attention`` on a ``workloads.Batch``."""
    s = batch.spec
    return attention(batch.q, batch.k_cache, batch.v_cache, batch.cu_seqlens_q, batch.seqused_k,
                     batch.block_table, s.softmax_scale, s.causal, key_window=key_window,
                     nthreads=nthreads)


def merge(outs, lses):
    """Log-sum-exp merge of partials over disjoint key sets (same shapes as ``attention``)."""
    outs = [np.ascontiguousarray(o, dtype=np.float64) for o in outs]
    lses = [np.ascontiguousarray(l, dtype=np.float64) for l in lses]
    shape = outs[0].shape
    d = shape[-1]
    rows = int(np.prod(shape[:-1]))
    out = np.zeros(shape, dtype=np.float64)
    lse = np.zeros(shape[:-1], dtype=np.float64)
    op = (ctypes.c_void_p * len(outs))(*[o.ctypes.data for o in outs])
    lp = (ctypes.c_void_p * len(lses))(*[l.ctypes.data for l in lses])
    _load().ua_oracle_merge(len(outs), ctypes.cast(op, ctypes.c_void_p),
                            ctypes.cast(lp, ctypes.c_void_p), rows, d, _ptr(out), _ptr(lse))
    return out, lse


def kv_append(k_cache, v_cache, k_new, v_new, cu_seqlens_q, seqused_k, block_table):
    """Write each new token's K and V rows into its page slot; returns new caches.

    The reading (the pages say only that seqused_k counts the whole context and
    that the cache is paged): the Lq new tokens of sequence s are the LAST Lq
    positions of its context of Lk = seqused_k[s] tokens, so token i of the
    sequence goes to position p = Lk - Lq + i, page block_table[s][p // bs],
    slot p % bs.  Every other cache entry is left as it was.  Plain loops; the
    caches are copied, not modified.  k_new / v_new: uint16 (bf16 bits)
    [total_q, Hkv, D]; caches [num_blocks, bs, Hkv, D].
    """
    k_out = np.array(k_cache, dtype=np.uint16, copy=True)
    v_out = np.array(v_cache, dtype=np.uint16, copy=True)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    sk = np.asarray(seqused_k, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    bs = k_out.shape[1]
    for s in range(len(sk)):
        lq = int(cu[s + 1] - cu[s])
        lk = int(sk[s])
        if lq > lk:
            raise OracleError("a sequence has more new tokens than context")
        for i in range(lq):
            t = int(cu[s]) + i
            pos = lk - lq + i
            page = int(bt[s, pos // bs])
            if not 0 <= page < k_out.shape[0]:
                raise OracleError("block id out of range")
            k_out[page, pos % bs] = k_new[t]
            v_out[page, pos % bs] = v_new[t]
    return k_out, v_out


def e4m3_to_f64(code: int) -> float:
    """Value of one FP8 E4M3 byte (see ua_oracle_e4m3_to_f64)."""
    return float(_load().ua_oracle_e4m3_to_f64(int(code) & 0xff))


def attention_fp8kv(q, k_cache, v_cache, k_scale, v_scale, cu_seqlens_q, seqused_k, block_table,
                    softmax_scale, causal, nthreads=0):
    """fp64 attention over a paged cache of E4M3 bytes (k = k_scale * e4m3(byte), v likewise).

    q: uint16 (bf16 bits) [total_q, Hq, D]; k_cache / v_cache: uint8
    [num_blocks, block_size, Hkv, D].  Returns (out fp64, lse fp64) as ``attention``.
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint8)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint8)
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    sk = np.ascontiguousarray(seqused_k, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    if bt.ndim == 1:
        bt = bt.reshape(len(sk), -1)
    total_q, hq, d = q.shape
    nb, bs, hk, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise OracleError("q / cache shapes disagree")
    if len(cu) != len(sk) + 1 or (len(sk) and cu[-1] != total_q):
        raise OracleError("cu_seqlens_q does not match q")
    out = np.zeros((total_q, hq, d), dtype=np.float64)
    lse = np.full((total_q, hq), -np.inf, dtype=np.float64)
    rc = _load().ua_oracle_attention_fp8kv(_ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale),
                                           float(v_scale), _ptr(cu), _ptr(sk), _ptr(bt), len(sk),
                                           hq, hk, d, bs, nb, bt.shape[1], float(softmax_scale),
                                           int(bool(causal)), _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"oracle error {rc}"))
    return out, lse
