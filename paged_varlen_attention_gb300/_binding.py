"""ctypes binding of ``libua_gb300.so`` (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels.  This
module checks tensor types, reads the host copies of the varlen metadata the
planner needs, keeps a per-device workspace (PyTorch is used for device
memory and streams only), and calls the C ABI declared in
``include/unified_attention.h``.  There is no fallback: if the library is not
built, every call raises ``UAError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libua_gb300.so")

STATUS = {0: "UA_OK", 1: "UA_ERR_INVALID_ARG", 2: "UA_ERR_UNSUPPORTED", 3: "UA_ERR_WORKSPACE",
          4: "UA_ERR_CUDA", 5: "UA_ERR_DEVICE_CHECK"}
DEVICE_BAD_BLOCK_ID = 0x1
DEVICE_WAIT_TIMEOUT = 0x2
DEVICE_BAD_METADATA = 0x4

SYMBOLS = ("unified_attention", "unified_attention_lse", "ua_merge_attn_states", "ua_kv_append",
           "unified_attention_append", "unified_attention_fp8kv", "ua_workspace_size_fp8kv",
           "ua_workspace_size", "ua_status_string", "ua_device_status", "ua_plan_inspect",
           "ua_profile_enable", "ua_profile_read", "unified_attention_device_plan",
           "ua_workspace_size_device_plan", "ua_device_plan_build", "ua_device_plan_layout",
           "unified_attention_device_planned", "ua_test_set_wait_limit")


class UAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the CUDA library; raise if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise UAError(4, f"CUDA library missing at {_LIB_PATH}; build it with "
                             "`python -m paged_varlen_attention_gb300.build_lib`")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.unified_attention.argtypes = [P, P, P, P, P, P, ctypes.c_float, I32, P, P, P,
                                          I32, I32, I32, I32, I32, I32, I32, P, ctypes.c_size_t, P]
        lib.unified_attention.restype = ctypes.c_int
        lib.unified_attention_lse.argtypes = [P, P, P, P, P, P, ctypes.c_float, I32, P, P, P, P,
                                              I32, I32, I32, I32, I32, I32, I32, P,
                                              ctypes.c_size_t, P]
        lib.unified_attention_lse.restype = ctypes.c_int
        lib.ua_merge_attn_states.argtypes = [P, P, P, P, P, P, I64, I32, P]
        lib.ua_merge_attn_states.restype = ctypes.c_int
        lib.unified_attention_fp8kv.argtypes = [P, P, P, ctypes.c_float, ctypes.c_float, P, P, P,
                                                ctypes.c_float, I32, P, P, P, P, I32, I32, I32,
                                                I32, I32, I32, I32, P, ctypes.c_size_t, P]
        lib.unified_attention_fp8kv.restype = ctypes.c_int
        lib.ua_workspace_size_fp8kv.argtypes = [P, P, I32, I32, I32, I32, I32, I32, I32,
                                                ctypes.POINTER(ctypes.c_size_t)]
        lib.ua_workspace_size_fp8kv.restype = ctypes.c_int
        lib.ua_kv_append.argtypes = [P, P, P, P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, P]
        lib.ua_kv_append.restype = ctypes.c_int
        lib.unified_attention_append.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_float, I32, P, P,
                                                 P, I32, I32, I32, I32, I32, I32, I32, P,
                                                 ctypes.c_size_t, P]
        lib.unified_attention_append.restype = ctypes.c_int
        lib.ua_workspace_size.argtypes = [P, P, I32, I32, I32, I32, I32, I32, I32,
                                          ctypes.POINTER(ctypes.c_size_t)]
        lib.ua_workspace_size.restype = ctypes.c_int
        lib.ua_status_string.argtypes = [ctypes.c_int]
        lib.ua_status_string.restype = ctypes.c_char_p
        lib.ua_device_status.argtypes = [ctypes.POINTER(I32)]
        lib.ua_device_status.restype = ctypes.c_int
        lib.ua_plan_inspect.argtypes = [P, P, I32, I32, I32, I32, I32, I32, I32, I32, P, P, I64,
                                        ctypes.POINTER(I64)]
        lib.ua_plan_inspect.restype = ctypes.c_int
        lib.ua_test_set_wait_limit.argtypes = [ctypes.c_uint64]
        lib.ua_test_set_wait_limit.restype = ctypes.c_int
        lib.ua_profile_enable.argtypes = [I32]
        lib.ua_profile_enable.restype = ctypes.c_int
        lib.ua_profile_read.argtypes = [I32, P, P]
        lib.ua_profile_read.restype = ctypes.c_int
        lib.unified_attention_device_plan.argtypes = [P, P, P, P, P, P, ctypes.c_float, I32, P, P,
                                                      I32, I32, I32, I32, I32, I32, I32, I32, I32,
                                                      I32, ctypes.c_float, ctypes.c_float, P,
                                                      ctypes.c_size_t, P]
        lib.unified_attention_device_plan.restype = ctypes.c_int
        lib.unified_attention_device_planned.argtypes = lib.unified_attention_device_plan.argtypes
        lib.unified_attention_device_planned.restype = ctypes.c_int
        lib.ua_workspace_size_device_plan.argtypes = [I32, I32, I32, I32, I32, I32, I32, I32, I32,
                                                      ctypes.POINTER(ctypes.c_size_t)]
        lib.ua_workspace_size_device_plan.restype = ctypes.c_int
        lib.ua_device_plan_build.argtypes = [P, P, I32, I32, I32, I32, I32, I32, I32, I32, I32, I32,
                                             P, ctypes.c_size_t, P]
        lib.ua_device_plan_build.restype = ctypes.c_int
        lib.ua_device_plan_layout.argtypes = [I32, I32, I32, I32, I32, I32, I32, I32, I32, I32, P, P]
        lib.ua_device_plan_layout.restype = ctypes.c_int
        _lib = lib
        return lib


def _host_i32(x) -> np.ndarray:
    """Host int32 copy of metadata (numpy array, list or tensor; a CUDA tensor is read back)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise UAError(rc, what)


def workspace_size(cu_seqlens_q_host, seqused_k_host, num_q_heads, num_kv_heads, head_size,
                   block_table_stride, causal=True, block_size=16) -> int:
    lib = load_library()
    cu = _host_i32(cu_seqlens_q_host)
    sk = _host_i32(seqused_k_host)
    out = ctypes.c_size_t(0)
    _check(lib.ua_workspace_size(_np_ptr(cu), _np_ptr(sk), len(sk), num_q_heads, num_kv_heads,
                                 head_size, block_size, block_table_stride, int(bool(causal)),
                                 ctypes.byref(out)), "ua_workspace_size")
    return int(out.value)


_workspaces = {}


def _workspace(torch, device, nbytes):
    """Grow-only per-device workspace (allocated through PyTorch)."""
    key = device.index if device.index is not None else torch.cuda.current_device()
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    return buf


def unified_attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table, softmax_scale,
                      causal=True, out=None, *, cu_seqlens_q_host=None, seqused_k_host=None,
                      workspace=None, stream=None, lse=None, k_new=None, v_new=None):
    """Attention over a paged varlen batch (see ``include/unified_attention.h``).

    q: bf16 [total_q, Hq, D]; k_cache / v_cache: bf16 [num_blocks, block_size, Hkv, D]
    (block_size a multiple of 16, at most 256); cu_seqlens_q int32 [N+1], seqused_k int32 [N], block_table int32 [N, stride],
    all CUDA tensors.  Host copies of cu_seqlens_q / seqused_k may be passed to
    avoid a device-to-host read.  Returns ``out`` (bf16 [total_q, Hq, D]).
    lse: an fp32 CUDA tensor [total_q, Hq] to also receive each row's natural-log
    softmax normaliser (calls ``unified_attention_lse``).
    k_new, v_new: the new tokens' K / V rows (bf16 [total_q, Hkv, D]) to write into
    their pages first (calls ``unified_attention_append``; see ``kv_append``).
    """
    import torch

    lib = load_library()
    for name, t, dt in (("q", q, torch.bfloat16), ("k_cache", k_cache, torch.bfloat16),
                        ("v_cache", v_cache, torch.bfloat16),
                        ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                        ("seqused_k", seqused_k, torch.int32),
                        ("block_table", block_table, torch.int32)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise UAError(1, f"{name} must be a contiguous CUDA {dt} tensor")
    total_q, hq, d = q.shape
    nb, bs, hk, d2 = k_cache.shape
    if v_cache.shape != k_cache.shape or d2 != d:
        raise UAError(1, "q / k_cache / v_cache shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() \
            or not out.is_cuda:
        raise UAError(1, "out must be a contiguous CUDA bf16 tensor shaped like q")
    cu_h = _host_i32(cu_seqlens_q if cu_seqlens_q_host is None else cu_seqlens_q_host)
    sk_h = _host_i32(seqused_k if seqused_k_host is None else seqused_k_host)
    num_seqs = int(sk_h.shape[0])
    stride = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    if workspace is None:
        need = workspace_size(cu_h, sk_h, hq, hk, d, stride, causal, bs)
        workspace = _workspace(torch, q.device, need)
    ws_ptr = workspace.data_ptr() if workspace.numel() else None
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    if k_new is not None:
        if v_new is None:
            raise UAError(1, "k_new and v_new go together")
        if lse is not None:
            kv_append(k_new, v_new, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
                      cu_seqlens_q_host=cu_h, seqused_k_host=sk_h, stream=stream)
        else:
            for name, t in (("k_new", k_new), ("v_new", v_new)):
                if (not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous()
                        or tuple(t.shape) != (total_q, hk, d)):
                    raise UAError(1, f"{name} must be a contiguous CUDA bf16 tensor [total_q, Hkv, D]")
            rc = lib.unified_attention_append(
                q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                v_cache.data_ptr(), cu_seqlens_q.data_ptr(), seqused_k.data_ptr(),
                block_table.data_ptr(), float(softmax_scale), int(bool(causal)), out.data_ptr(),
                _np_ptr(cu_h), _np_ptr(sk_h), num_seqs, hq, hk, d, bs, nb, stride, ws_ptr,
                workspace.numel(), stream)
            _check(rc, "unified_attention_append")
            return out
    if lse is None:
        rc = lib.unified_attention(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   cu_seqlens_q.data_ptr(), seqused_k.data_ptr(),
                                   block_table.data_ptr(), float(softmax_scale), int(bool(causal)),
                                   out.data_ptr(), _np_ptr(cu_h), _np_ptr(sk_h), num_seqs, hq, hk,
                                   d, bs, nb, stride, ws_ptr, workspace.numel(), stream)
        _check(rc, "unified_attention")
        return out
    if (not lse.is_cuda or lse.dtype != torch.float32 or not lse.is_contiguous()
            or tuple(lse.shape) != (total_q, hq)):
        raise UAError(1, "lse must be a contiguous CUDA float32 tensor [total_q, Hq]")
    rc = lib.unified_attention_lse(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   cu_seqlens_q.data_ptr(), seqused_k.data_ptr(),
                                   block_table.data_ptr(), float(softmax_scale), int(bool(causal)),
                                   out.data_ptr(), lse.data_ptr(), _np_ptr(cu_h), _np_ptr(sk_h),
                                   num_seqs, hq, hk, d, bs, nb, stride, ws_ptr, workspace.numel(),
                                   stream)
    _check(rc, "unified_attention_lse")
    return out


def merge_attn_states(out_a, lse_a, out_b, lse_b, out=None, lse_out=None, stream=None):
    """Combine two results of the same rows over disjoint key sets (``ua_merge_attn_states``).

    out_a / out_b: bf16 CUDA [..., D]; lse_a / lse_b: fp32 CUDA [...] (one per row).
    Returns ``(out, lse_out)``; lse_out is None unless given.
    """
    import torch

    lib = load_library()
    for name, t, dt in (("out_a", out_a, torch.bfloat16), ("out_b", out_b, torch.bfloat16),
                        ("lse_a", lse_a, torch.float32), ("lse_b", lse_b, torch.float32)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise UAError(1, f"{name} must be a contiguous CUDA {dt} tensor")
    if out_b.shape != out_a.shape or lse_a.shape != out_a.shape[:-1] or lse_b.shape != lse_a.shape:
        raise UAError(1, "merge inputs disagree in shape")
    if out is None:
        out = torch.empty_like(out_a)
    d = int(out_a.shape[-1])
    rows = int(lse_a.numel())
    if stream is None:
        stream = torch.cuda.current_stream(out_a.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = lib.ua_merge_attn_states(out_a.data_ptr(), lse_a.data_ptr(), out_b.data_ptr(),
                                  lse_b.data_ptr(), out.data_ptr(),
                                  None if lse_out is None else lse_out.data_ptr(), rows, d, stream)
    _check(rc, "ua_merge_attn_states")
    return out, lse_out


def device_status() -> int:
    """Synchronise, then read and clear the kernels' device status word."""
    lib = load_library()
    code = ctypes.c_int32(0)
    rc = lib.ua_device_status(ctypes.byref(code))
    if rc not in (0, 5):
        _check(rc, "ua_device_status")
    return int(code.value)


def plan_inspect(cu_seqlens_q_host, seqused_k_host, num_q_heads, num_kv_heads, head_size,
                 block_table_stride, causal=True, num_sms=152, block_size=16):
    """Host-only view of the work partition (no CUDA call).  Returns (counts, items)."""
    lib = load_library()
    cu = _host_i32(cu_seqlens_q_host)
    sk = _host_i32(seqused_k_host)
    counts = np.zeros(9, dtype=np.int32)
    n = ctypes.c_int64(0)
    args = (_np_ptr(cu), _np_ptr(sk), len(sk), num_q_heads, num_kv_heads, head_size, block_size,
            block_table_stride, int(bool(causal)), num_sms)
    _check(lib.ua_plan_inspect(*args, _np_ptr(counts), None, 0, ctypes.byref(n)),
           "ua_plan_inspect")
    items = np.zeros((max(int(n.value), 1), 8), dtype=np.int32)
    _check(lib.ua_plan_inspect(*args, _np_ptr(counts), _np_ptr(items), int(n.value),
                               ctypes.byref(n)), "ua_plan_inspect")
    keys = ("dec_ctas", "pieces", "split_units", "slots", "prefill_tiles", "prefill_ctas",
            "dec_pages", "workspace_bytes", "prefill_sms_side_by_side")
    return dict(zip(keys, (int(c) for c in counts))), items[:int(n.value)]


def set_test_wait_limit(limit_ns: int = 0):
    """Test hook (``ua_test_set_wait_limit``): the decode kernel's main-loop waits of
    later calls give up after limit_ns nanoseconds (0: the library's 4 s)."""
    _check(load_library().ua_test_set_wait_limit(int(limit_ns)), "ua_test_set_wait_limit")


def profile_enable(on: bool = True):
    _check(load_library().ua_profile_enable(int(bool(on))), "ua_profile_enable")


def profile_read(calls_back: int = 0):
    """(ms[decode, prefill, combine, plan_copy], launches[...]) of a profiled call
    (0 = the latest, up to 63 back); -1 = that step did not run."""
    ms = np.zeros(4, dtype=np.float32)
    ln = np.zeros(4, dtype=np.int32)
    _check(load_library().ua_profile_read(int(calls_back), _np_ptr(ms), _np_ptr(ln)),
           "ua_profile_read")
    return ms.tolist(), ln.tolist()


def kv_append(k_new, v_new, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table, *,
              cu_seqlens_q_host=None, seqused_k_host=None, stream=None):
    """Write the new tokens' K / V rows ([total_q, Hkv, D] bf16 CUDA tensors) into
    their pages of k_cache / v_cache (``ua_kv_append``): token i of sequence s goes to
    context position seqused_k[s] - Lq + i."""
    import torch

    lib = load_library()
    for name, t, dt in (("k_new", k_new, torch.bfloat16), ("v_new", v_new, torch.bfloat16),
                        ("k_cache", k_cache, torch.bfloat16), ("v_cache", v_cache, torch.bfloat16),
                        ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                        ("seqused_k", seqused_k, torch.int32),
                        ("block_table", block_table, torch.int32)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise UAError(1, f"{name} must be a contiguous CUDA {dt} tensor")
    nb, bs, hk, d = k_cache.shape
    if v_cache.shape != k_cache.shape or k_new.shape[1:] != (hk, d) or v_new.shape != k_new.shape:
        raise UAError(1, "k_new / v_new / cache shapes disagree")
    cu_h = _host_i32(cu_seqlens_q if cu_seqlens_q_host is None else cu_seqlens_q_host)
    sk_h = _host_i32(seqused_k if seqused_k_host is None else seqused_k_host)
    if len(cu_h) and int(cu_h[-1]) != k_new.shape[0]:
        raise UAError(1, "cu_seqlens_q does not match k_new")
    stride = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    if stream is None:
        stream = torch.cuda.current_stream(k_new.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = lib.ua_kv_append(k_new.data_ptr(), v_new.data_ptr(), cu_seqlens_q.data_ptr(),
                          seqused_k.data_ptr(), block_table.data_ptr(), k_cache.data_ptr(),
                          v_cache.data_ptr(), _np_ptr(cu_h), _np_ptr(sk_h), int(sk_h.shape[0]), hk,
                          d, bs, nb, stride, stream)
    _check(rc, "ua_kv_append")


def unified_attention_fp8kv(q, k_cache, v_cache, k_scale, v_scale, cu_seqlens_q, seqused_k,
                            block_table, softmax_scale, causal=True, out=None, *,
                            cu_seqlens_q_host=None, seqused_k_host=None, workspace=None,
                            stream=None, lse=None):
    """Attention over a paged cache of FP8 E4M3 bytes (``unified_attention_fp8kv``).

    k_cache / v_cache: uint8 CUDA tensors [num_blocks, block_size, Hkv, 128] of E4M3 codes
    with k = k_scale * e4m3(byte), v = v_scale * e4m3(byte); the rest as
    ``unified_attention``.  Returns ``out``.
    """
    import torch

    lib = load_library()
    for name, t, dt in (("q", q, torch.bfloat16), ("k_cache", k_cache, torch.uint8),
                        ("v_cache", v_cache, torch.uint8),
                        ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                        ("seqused_k", seqused_k, torch.int32),
                        ("block_table", block_table, torch.int32)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise UAError(1, f"{name} must be a contiguous CUDA {dt} tensor")
    total_q, hq, d = q.shape
    nb, bs, hk, d2 = k_cache.shape
    if v_cache.shape != k_cache.shape or d2 != d:
        raise UAError(1, "q / k_cache / v_cache shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    if lse is not None and (not lse.is_cuda or lse.dtype != torch.float32
                            or tuple(lse.shape) != (total_q, hq) or not lse.is_contiguous()):
        raise UAError(1, "lse must be a contiguous CUDA float32 tensor [total_q, Hq]")
    cu_h = _host_i32(cu_seqlens_q if cu_seqlens_q_host is None else cu_seqlens_q_host)
    sk_h = _host_i32(seqused_k if seqused_k_host is None else seqused_k_host)
    num_seqs = int(sk_h.shape[0])
    stride = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    if workspace is None:
        need = ctypes.c_size_t(0)
        _check(lib.ua_workspace_size_fp8kv(_np_ptr(cu_h), _np_ptr(sk_h), num_seqs, hq, hk, d, bs,
                                           stride, int(bool(causal)), ctypes.byref(need)),
               "ua_workspace_size_fp8kv")
        workspace = _workspace(torch, q.device, int(need.value))
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = lib.unified_attention_fp8kv(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     float(k_scale), float(v_scale), cu_seqlens_q.data_ptr(),
                                     seqused_k.data_ptr(), block_table.data_ptr(),
                                     float(softmax_scale), int(bool(causal)), out.data_ptr(),
                                     None if lse is None else lse.data_ptr(), _np_ptr(cu_h),
                                     _np_ptr(sk_h), num_seqs, hq, hk, d, bs, nb, stride,
                                     workspace.data_ptr() if workspace.numel() else None,
                                     workspace.numel(), stream)
    _check(rc, "unified_attention_fp8kv")
    return out


def _stream_handle(torch, device, stream):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def workspace_size_device_plan(num_seqs, max_total_q, num_q_heads, num_kv_heads, head_size,
                               block_table_stride, kv_fp8=False, block_size=16, max_seq_q=0):
    """Bytes of workspace ``unified_attention_device_plan`` needs for these capacities."""
    lib = load_library()
    need = ctypes.c_size_t(0)
    _check(lib.ua_workspace_size_device_plan(int(num_seqs), int(max_total_q), int(max_seq_q),
                                             int(num_q_heads),
                                             int(num_kv_heads), int(head_size), int(block_size),
                                             int(block_table_stride), int(bool(kv_fp8)),
                                             ctypes.byref(need)),
           "ua_workspace_size_device_plan")
    return int(need.value)


def unified_attention_device_plan(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
                                  softmax_scale, causal=True, out=None, *, workspace, lse=None,
                                  num_seqs=None, max_seq_q=0, kv_fp8=False, k_scale=1.0,
                                  v_scale=1.0, stream=None, reuse_plan=False):
    """Attention planned on the GPU (``unified_attention_device_plan``): no host copies of
    the metadata, so the call can be captured in a CUDA graph and replayed after
    ``cu_seqlens_q`` / ``seqused_k`` / ``block_table`` / ``q`` are rewritten in place.

    q / out: bf16 [max_total_q, Hq, D] buffers (their first dimension is the token
    capacity); k_cache / v_cache: bf16, or uint8 E4M3 codes with ``kv_fp8``; lse:
    optional float32 [max_total_q, Hq].  ``workspace``: a uint8 CUDA tensor of at least
    ``workspace_size_device_plan`` bytes, owned by the caller (a captured graph keeps
    using it; size it with the same ``max_seq_q``).  ``num_seqs`` defaults to
    ``seqused_k.shape[0]``; ``max_seq_q`` bounds one sequence's query tokens (0: the
    capacity) -- with ``max_seq_q * Hq / Hkv <= 16`` the prefill kernel is not launched.
    ``reuse_plan``: skip the planner and use the plan an earlier call left in
    ``workspace`` for the same metadata (``unified_attention_device_planned``; e.g.
    every layer after the first in one model step).  Returns ``out``.
    """
    import torch

    lib = load_library()
    cache_dt = torch.uint8 if kv_fp8 else torch.bfloat16
    for name, t, dt in (("q", q, torch.bfloat16), ("k_cache", k_cache, cache_dt),
                        ("v_cache", v_cache, cache_dt),
                        ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                        ("seqused_k", seqused_k, torch.int32),
                        ("block_table", block_table, torch.int32),
                        ("workspace", workspace, torch.uint8)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise UAError(1, f"{name} must be a contiguous CUDA {dt} tensor")
    max_total_q, hq, d = q.shape
    nb, bs, hk, d2 = k_cache.shape
    if v_cache.shape != k_cache.shape or d2 != d:
        raise UAError(1, "q / k_cache / v_cache shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise UAError(1, "out must be a contiguous bf16 tensor shaped like q")
    if lse is not None and (not lse.is_cuda or lse.dtype != torch.float32
                            or tuple(lse.shape) != (max_total_q, hq) or not lse.is_contiguous()):
        raise UAError(1, "lse must be a contiguous CUDA float32 tensor [max_total_q, Hq]")
    ns = int(seqused_k.shape[0]) if num_seqs is None else int(num_seqs)
    stride = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    fn = lib.unified_attention_device_planned if reuse_plan else lib.unified_attention_device_plan
    rc = fn(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), cu_seqlens_q.data_ptr(),
        seqused_k.data_ptr(), block_table.data_ptr(), float(softmax_scale), int(bool(causal)),
        out.data_ptr(), None if lse is None else lse.data_ptr(), ns, max_total_q, int(max_seq_q),
        hq, hk, d, bs,
        nb, stride, int(bool(kv_fp8)), float(k_scale), float(v_scale), workspace.data_ptr(),
        workspace.numel(), _stream_handle(torch, q.device, stream))
    _check(rc, "unified_attention_device_plan")
    return out


def device_plan(cu_seqlens_q, seqused_k, causal, num_q_heads, num_kv_heads, head_size,
                block_table_stride, max_total_q, kv_fp8=False, max_seq_q=0):
    """Run only the device planner on CUDA int32 metadata and read the plan back (synchronises).

    Returns a dict of numpy arrays: ``header`` (int64 dec_ctas, n_pieces, n_comb,
    n_slots, pre_ctas, n_tiles, dec_pages, error), ``cta_begin`` [dec_ctas + 1],
    ``pieces`` [n_pieces, 8] (seq, kvh, row0, nrows, page_begin, page_end, slot, unit),
    ``comb`` [n_comb, 8], ``tiles`` [n_tiles, 8] (seq, kvh, row0, nrows, kv_tiles, q0,
    lq, lk) and ``pre_begin`` [pre_ctas + 1].
    """
    import torch

    lib = load_library()
    dev = cu_seqlens_q.device
    ns = int(seqused_k.shape[0])
    nbytes = workspace_size_device_plan(ns, max_total_q, num_q_heads, num_kv_heads, head_size,
                                        block_table_stride, kv_fp8, max_seq_q=max_seq_q)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
    props = torch.cuda.get_device_properties(dev)
    offs = np.zeros(8, np.int64)
    caps = np.zeros(8, np.int32)
    _check(lib.ua_device_plan_layout(ns, int(max_total_q), int(max_seq_q), int(num_q_heads),
                                     int(num_kv_heads),
                                     int(head_size), 16, int(block_table_stride),
                                     int(bool(kv_fp8)), props.multi_processor_count,
                                     _np_ptr(offs), _np_ptr(caps)), "ua_device_plan_layout")
    _check(lib.ua_device_plan_build(cu_seqlens_q.data_ptr(), seqused_k.data_ptr(),
                                    int(bool(causal)), ns, int(max_total_q), int(max_seq_q),
                                    int(num_q_heads),
                                    int(num_kv_heads), int(head_size), 16,
                                    int(block_table_stride), int(bool(kv_fp8)), ws.data_ptr(),
                                    ws.numel(), torch.cuda.current_stream(dev).cuda_stream),
           "ua_device_plan_build")
    torch.cuda.synchronize(dev)
    raw = ws.cpu().numpy()

    def i32(off, n, cols=1):
        a = raw[off:off + 4 * n * cols].view(np.int32)
        return a.reshape(n, cols) if cols > 1 else a

    hdr = raw[offs[0]:offs[0] + 64].view(np.int64).copy()
    dec_ctas, n_pieces, n_comb, _, pre_ctas, n_tiles = (int(x) for x in hdr[:6])
    return {
        "header": hdr,
        "cta_begin": i32(offs[1], dec_ctas + 1).copy(),
        "pieces": i32(offs[2], n_pieces, 8).copy(),
        "comb": i32(offs[3], n_comb, 8).copy(),
        "tiles": i32(offs[5], n_tiles, 8).copy(),
        "pre_begin": i32(offs[6], pre_ctas + 1).copy(),
        "caps": caps,
    }
