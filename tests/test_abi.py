"""The C-ABI library loads and exports every function include/*.h declares;
host-only checks of the device entry points' argument validation (no GPU work
is launched: every call here fails its checks before any CUDA call)."""
from __future__ import annotations

import ctypes as C
import glob
import os
import re
import subprocess

import radixattention_prefix_shared_tree_gb300 as ra

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:rc_status|void|const char\s*\*)\s*(\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("rc_create", "rc_destroy", "rc_match_prefix", "rc_insert", "rc_release", "rc_evict", "rc_alloc",
              "rc_free", "sched_order", "rc_stats", "rc_dump", "kv_store", "attn_decode", "attn_extend",
              "attn_decode_workspace", "attn_extend_workspace", "rc_sync", "rc_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(built):
    lib = C.CDLL(ra.library_path())
    out = subprocess.run(["nm", "-D", "--defined-only", ra.library_path()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None
    assert set(ra.SIGNATURES) <= declared_functions()


def test_strerror_and_argument_checks(built):
    assert ra.rc_strerror(ra.RC_OK) == "ok"
    assert "free slots" in ra.rc_strerror(ra.RC_ERR_NOMEM)
    L = ra.lib()
    # null descriptors are rejected on the host, before any CUDA call
    assert L.kv_store(None, None, None, None, 0, None, None, None) == ra.RC_ERR_ARG
    assert L.attn_decode(None, None, None, 0, None, None, None, None, 0, None) == ra.RC_ERR_ARG
    assert L.attn_extend(None, None, None, None, 0, 0, None, None, None, 0, None) == ra.RC_ERR_ARG
    n = C.c_size_t(0)
    assert L.attn_decode_workspace(None, 1, 1, None, C.byref(n)) == ra.RC_ERR_ARG
    assert L.rc_probe_wait_timeout(None, None) == ra.RC_ERR_ARG
    h = C.c_void_p()
    assert L.rc_create(-1, C.byref(h)) == ra.RC_ERR_ARG
    assert L.rc_create(10, None) == ra.RC_ERR_ARG


def test_host_calls_reject_bad_arguments(built):
    c = ra.RadixCache(16)
    L = ra.lib()
    m, node = C.c_int64(), C.c_int64()
    assert L.rc_match_prefix(c.handle, None, -1, 0, C.byref(m), None, C.byref(node)) == ra.RC_ERR_ARG
    assert c.alloc(17)[0] == ra.RC_ERR_NOMEM
    assert c.release(999) == ra.RC_ERR_STATE
    assert c.free([16]) == ra.RC_ERR_ARG
    assert c.sched_order(7, [[1]])[0] == ra.RC_ERR_ARG
    assert c.evict(-3)[0] == ra.RC_ERR_ARG


def test_pool_descriptor_rejects_non_contiguous_tensors():
    import pytest
    import torch
    k = torch.zeros(64, 8, 128, dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    d = ra.make_pool_desc(k, v)
    assert (d.n_slots, d.kv_heads, d.head_dim_k, d.head_dim_v) == (64, 8, 128, 128)
    head_major = torch.zeros(8, 64, 128, dtype=torch.bfloat16).permute(1, 0, 2)   # [n_slots, H, d] view
    with pytest.raises(ValueError):
        ra.make_pool_desc(head_major, v)
    with pytest.raises(ValueError):
        ra.make_pool_desc(k, head_major)
    codes = torch.zeros(64, 8, 128, dtype=torch.uint8)
    with pytest.raises(ValueError):
        ra.make_pool_desc(codes, codes, k_scale=torch.zeros(8, 64).t(), v_scale=torch.zeros(64, 8))


def test_device_calls_refuse_strided_views(built):
    import pytest
    import torch
    q = torch.zeros(4, 32, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ra._tp(q[:, :8])
    with pytest.raises(ValueError):
        ra._tp(q.transpose(0, 1))
    assert ra._tp(None) is None
    assert ra._tp(q[1]).value == q[1].data_ptr()


def test_binding_structs_match_the_header(tmp_path):
    """Every struct the binding passes by pointer has the header's size and
    field offsets (a C program compiled against include/radixattn.h prints
    them; the ctypes mirrors must agree field by field)."""
    structs = {"rc_request": ra.rc_request, "rc_stats_t": ra.rc_stats_t, "rc_pool_desc": ra.rc_pool_desc,
               "rc_attn_desc": ra.rc_attn_desc, "rc_kv_table": ra.rc_kv_table, "rc_cascade": ra.rc_cascade,
               "rc_decode_step": ra.rc_decode_step}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "radixattn.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'    printf("{name} size %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'    printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = {}
    for ln in subprocess.check_output([str(exe)], text=True).splitlines():
        name, field, val = ln.split()
        got[(name, field)] = int(val)
    for name, cls in structs.items():
        assert got[(name, "size")] == C.sizeof(cls), name
        for f, _ in cls._fields_:
            assert got[(name, f)] == getattr(cls, f).offset, (name, f)
