"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

from paged_varlen_attention_gb300 import _binding as B
from paged_varlen_attention_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return B.load_library()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                            text, flags=re.M)
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("unified_attention", "ua_workspace_size", "ua_status_string", "ua_device_status",
              "ua_plan_inspect", "ua_profile_enable", "ua_profile_read"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code, name in B.STATUS.items():
        assert lib.ua_status_string(code).decode() == name


def _call(lib, cu, sk, hq=4, hk=2, d=64, bs=16, nb=8, stride=4, causal=1, scale=0.125,
          ptr=16, out=16, ws=None, ws_bytes=0):
    cu = np.asarray(cu, np.int32)
    sk = np.asarray(sk, np.int32)
    p = ctypes.c_void_p(ptr) if ptr else None
    o = ctypes.c_void_p(out) if out else None
    return lib.unified_attention(p, p, p, p, p, p, scale, causal, o,
                                 cu.ctypes.data_as(ctypes.c_void_p),
                                 sk.ctypes.data_as(ctypes.c_void_p), len(sk), hq, hk, d, bs, nb,
                                 stride, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(cu=[0, 1, 6], sk=[17, 4]), 1),          # Lk < Lq with causal
    (dict(cu=[0, 1, 6], sk=[0, 40]), 1),          # Lq > 0, Lk = 0
    (dict(cu=[1, 1, 6], sk=[17, 40]), 1),         # cu[0] != 0
    (dict(cu=[0, 3, 2], sk=[17, 40]), 1),         # decreasing cu
    (dict(cu=[0, 1, 6], sk=[17, 90]), 1),         # needs more pages than the table holds
    (dict(cu=[0, 1, 6], sk=[17, 40], hq=6, hk=4), 2),   # Hq not a multiple of Hkv
    (dict(cu=[0, 1, 6], sk=[17, 40], d=72), 2),   # unsupported head sizes
    (dict(cu=[0, 1, 6], sk=[17, 40], d=512), 2),
    (dict(cu=[0, 1, 6], sk=[17, 40], bs=24), 2),  # pages not a multiple of 16 tokens
    (dict(cu=[0, 1, 6], sk=[17, 40], bs=512), 2), # pages above 256 tokens
    (dict(cu=[0, 1, 6], sk=[17, 40], bs=32, stride=2), 3),   # 32-token pages: no workspace for the table
    (dict(cu=[0, 1, 6], sk=[17, 40], ptr=0), 1),  # null device pointers
    (dict(cu=[0, 1, 6], sk=[17, 40], ptr=8), 1),  # misaligned buffers
    (dict(cu=[0, 1, 6], sk=[17, 40], scale=float("nan")), 1),
    (dict(cu=[0, 1, 6], sk=[17, 40], nb=0), 1),
])
def test_invalid_arguments_rejected_before_any_launch(lib, kw, code):
    assert _call(lib, **kw) == code


def test_empty_batch_is_a_no_op(lib):
    assert _call(lib, cu=[0], sk=[]) == 0
    assert _call(lib, cu=[0, 0, 0], sk=[5, 9]) == 0      # two sequences, no new tokens


def test_noncausal_allows_more_queries_than_keys(lib):
    # passes validation; stops only when it needs the device (no GPU here)
    cu = np.asarray([0, 5], np.int32)
    sk = np.asarray([3], np.int32)
    counts, _ = B.plan_inspect(cu, sk, 4, 2, 64, 1, causal=False)
    assert counts["dec_pages"] > 0 or counts["prefill_tiles"] > 0
    with pytest.raises(B.UAError):
        B.plan_inspect(cu, sk, 4, 2, 64, 1, causal=True)


def test_kv_append_rejects_more_new_tokens_than_context(lib):
    import ctypes
    cu = np.array([0, 5], np.int32)
    sk = np.array([3], np.int32)          # Lq = 5 > Lk = 3
    p = ctypes.c_void_p(16)
    rc = lib.ua_kv_append(p, p, p, p, p, p, p, cu.ctypes.data_as(ctypes.c_void_p),
                          sk.ctypes.data_as(ctypes.c_void_p), 1, 2, 64, 16, 8, 1, None)
    assert rc == 1                        # UA_ERR_INVALID_ARG, nothing launched


def test_missing_library_raises_no_fallback(monkeypatch, tmp_path):
    """Without the built CUDA library every entry point raises: nothing falls
    back to another implementation."""
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "_LIB_PATH", str(tmp_path / "libua_gb300.so"))
    with pytest.raises(B.UAError) as e:
        B.load_library()
    assert e.value.status == 4
    with pytest.raises(B.UAError):
        B.workspace_size(np.array([0, 1], np.int32), np.array([5], np.int32), 4, 2, 64, 1)
    with pytest.raises(B.UAError):
        B.plan_inspect(np.array([0, 1], np.int32), np.array([5], np.int32), 4, 2, 64, 1)


def test_binding_rejects_host_tensors_before_any_cuda_call(lib):
    """The Python binding only marshals: tensors that are not contiguous CUDA
    tensors of the right dtype are refused with UA_ERR_INVALID_ARG (1)."""
    import torch
    import paged_varlen_attention_gb300 as ua

    q = torch.zeros(5, 4, 64, dtype=torch.bfloat16)
    kc = torch.zeros(3, 16, 2, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 1, 5], dtype=torch.int32)
    sk = torch.tensor([17, 40], dtype=torch.int32)
    bt = torch.zeros(2, 3, dtype=torch.int32)
    lse = torch.zeros(5, 4, dtype=torch.float32)
    calls = [
        lambda: ua.unified_attention(q, kc, kc, cu, sk, bt, 0.125, True,
                                     cu_seqlens_q_host=cu.numpy(), seqused_k_host=sk.numpy()),
        lambda: ua.kv_append(q[:, :2], q[:, :2], kc, kc, cu, sk, bt,
                             cu_seqlens_q_host=cu.numpy(), seqused_k_host=sk.numpy()),
        lambda: ua.merge_attn_states(q, lse, q, lse),
        lambda: ua.unified_attention_fp8kv(q, kc.view(torch.uint8), kc.view(torch.uint8), 1.0, 1.0,
                                           cu, sk, bt, 0.125, True, cu_seqlens_q_host=cu.numpy(),
                                           seqused_k_host=sk.numpy()),
        lambda: ua.unified_attention_device_plan(q, kc, kc, cu, sk, bt, 0.125, True,
                                                 workspace=torch.zeros(256, dtype=torch.uint8)),
    ]
    for call in calls:
        with pytest.raises(B.UAError) as e:
            call()
        assert e.value.status == 1


def test_header_is_plain_c_and_the_library_links_from_c(lib, tmp_path):
    """The boundary is a C ABI: a C99 program includes the header, links the
    library and makes a host-only call (shape check, no CUDA call)."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "abi.c"
    src.write_text(
        '#include <stdio.h>\n#include "unified_attention.h"\n'
        "int main(void) {\n"
        "    int32_t cu[3] = {0, 1, 6}, sk[2] = {17, 40};\n"
        "    size_t bytes = 0;\n"
        "    ua_status st = ua_workspace_size(cu, sk, 2, 4, 2, 72, 16, 3, 1, &bytes);\n"
        '    printf("%s\\n", ua_status_string(st));\n'
        "    return st == UA_ERR_UNSUPPORTED ? 0 : 1;\n}\n")
    libdir = os.path.dirname(B._LIB_PATH)
    exe = tmp_path / "abi"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                        str(src), "-L", libdir, "-lua_gb300", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "UA_ERR_UNSUPPORTED", r.stdout + r.stderr
