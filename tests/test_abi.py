"""CPU tests of the boundary: the library builds, loads, exports every symbol
the header declares, and its host-side argument validation rejects bad
inputs before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "etc_moe.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(etc_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from moe_layer_scheduling_gb300 import binding
    return binding.load()


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("etc_moe_plan", "etc_moe_forward", "etc_splitk_rowsum", "etc_chain_forward",
                     "etc_moe_forward_unfused", "etc_plan_destroy", "etc_last_error",
                     "etc_mlp_plan", "etc_mlp_forward", "etc_mlp_forward_unfused",
                     "etc_chain_plan"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in etc_moe.h but not exported"


def test_binding_names_match_the_header():
    from moe_layer_scheduling_gb300 import binding
    assert sorted(binding.EXPORTED) == _declared()
    for name in _declared():
        assert callable(getattr(binding, name)), name


def test_library_is_built_for_sm103a():
    from moe_layer_scheduling_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


def _opts(**kw):
    from moe_layer_scheduling_gb300 import binding
    base = dict(hidden=2048, n_experts=128, top_k=8, inter=768, t_max=64, sched=0, n_blocks=1,
                rms_eps=1e-6, router_bias=None, wait_timeout_ns=0, debug_flags=0, debug_arg=0)
    base.update(kw)
    return binding.etc_moe_opts(**base)


@pytest.mark.parametrize("bad", [
    dict(hidden=100), dict(hidden=0), dict(hidden=12416), dict(n_experts=7), dict(n_experts=136), dict(n_experts=512),
    dict(top_k=0),
    dict(top_k=17), dict(inter=100), dict(t_max=0), dict(sched=5), dict(sched=3),
    dict(sched=2, n_blocks=2), dict(n_blocks=0),
    dict(n_blocks=9), dict(router_bias=8),
])
def test_plan_rejects_bad_options_on_the_host(lib, bad):
    from moe_layer_scheduling_gb300 import binding
    h = ctypes.c_void_p()
    o = _opts(**bad)
    rc = lib.etc_moe_plan(ctypes.byref(h), ctypes.byref(o))
    assert rc == binding.ETC_ERR_INVALID
    assert h.value is None
    assert lib.etc_last_error().decode() != ""


@pytest.mark.parametrize("bad", [
    dict(hidden=100), dict(hidden=0), dict(hidden=16512), dict(inter=32), dict(inter=0),
    dict(inter=65600), dict(t_max=0), dict(t_max=65537), dict(sched=2), dict(sched=7),
    dict(out_dtype=2),
])
def test_mlp_plan_rejects_bad_options_on_the_host(lib, bad):
    from moe_layer_scheduling_gb300 import binding
    base = dict(hidden=4096, inter=12288, t_max=8192, sched=0, wait_timeout_ns=0, debug_flags=0,
                out_dtype=0)
    base.update(bad)
    o = binding.etc_mlp_opts(**base)
    h = ctypes.c_void_p()
    assert lib.etc_mlp_plan(ctypes.byref(h), ctypes.byref(o)) == binding.ETC_ERR_INVALID
    assert h.value is None
    assert lib.etc_last_error().decode() != ""


@pytest.mark.parametrize("n_blocks", [0, 5, -1])
def test_chain_plan_rejects_bad_block_counts_on_the_host(lib, n_blocks):
    from moe_layer_scheduling_gb300 import binding
    h = ctypes.c_void_p()
    o = _opts()
    assert lib.etc_chain_plan(ctypes.byref(h), ctypes.byref(o), n_blocks) == binding.ETC_ERR_INVALID
    assert h.value is None
    assert o.n_blocks == 1  # the caller's options are not modified
    assert lib.etc_chain_plan(ctypes.byref(h), None, 2) == binding.ETC_ERR_INVALID


def test_mlp_null_plan_is_rejected(lib):
    from moe_layer_scheduling_gb300 import binding
    assert lib.etc_mlp_forward(None, None, None, None, None, 1, None) == binding.ETC_ERR_INVALID
    assert lib.etc_mlp_forward_unfused(None, None, None, None, None, 1, None) == binding.ETC_ERR_INVALID
    assert lib.etc_mlp_plan(None, None) == binding.ETC_ERR_INVALID


def test_null_plan_is_rejected(lib):
    from moe_layer_scheduling_gb300 import binding
    assert lib.etc_moe_forward(None, None, None, None, None, None, 1, None) == binding.ETC_ERR_INVALID
    assert lib.etc_plan_check(None) == binding.ETC_ERR_INVALID
    assert lib.etc_moe_plan(None, None) == binding.ETC_ERR_INVALID


@pytest.mark.parametrize("n_rows,n_cols,n_split,sched", [
    (-1, 64, 4, 0), (8, 0, 4, 0), (8, 64, 0, 0), (8, 64, 65, 0), (8, 60, 4, 0),
    (8, 24, 4, 0), (8, 4 * 16388, 4, 0), (8, 64, 4, 7),
])
def test_splitk_rejects_bad_sizes_on_the_host(lib, n_rows, n_cols, n_split, sched):
    from moe_layer_scheduling_gb300 import binding
    rc = lib.etc_splitk_rowsum(None, None, n_rows, n_cols, n_split, None, sched)
    assert rc == binding.ETC_ERR_INVALID


def test_splitk_fault_injection_needs_static(lib):
    from moe_layer_scheduling_gb300 import binding
    rc = lib.etc_splitk_rowsum_ex(None, None, 8, 64, 4, None, binding.ETC_SCHED_DYNAMIC, 0,
                                  binding.ETC_DEBUG_FAULT_EXTRA_WAIT, 0)
    assert rc == binding.ETC_ERR_UNIMPLEMENTED


def test_splitk_zero_rows_is_a_noop(lib):
    from moe_layer_scheduling_gb300 import binding
    before = lib.etc_launch_count()
    assert lib.etc_splitk_rowsum(None, None, 0, 64, 4, None, 0) == binding.ETC_OK
    assert lib.etc_launch_count() == before


def test_task_descriptor_fields_round_trip():
    # The 32-bit descriptor layout the dynamic queue stores (type, block, a, b).
    src = open(os.path.join(ROOT, "moe_layer_scheduling_gb300", "csrc", "etc_internal.h")).read()
    assert "type[31:28] blk[27:25] a[24:8] b[7:0]" in src

    def enc(t, blk, a, b):
        return (t << 28) | (blk << 25) | (a << 8) | b

    for t, blk, a, b in [(6, 0, 383, 11), (7, 3, 131071, 255), (2, 1, 0, 31)]:
        d = enc(t, blk, a, b)
        assert (d >> 28, (d >> 25) & 7, (d >> 8) & 0x1FFFF, d & 0xFF) == (t, blk, a, b)


def _header_struct_fields(name):
    """(field, C type) pairs of `typedef struct { ... } name;` in the header, in order."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"typedef struct \{([^{}]*)\}\s*" + name + r"\s*;", src)
    assert m, name
    fields = []
    for decl in m.group(1).split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        ctype, _, rest = decl.rpartition(" ")
        for f in rest.split(","):
            f = f.strip()
            stars = len(f) - len(f.lstrip("*"))
            fields.append((f.lstrip("*"), ctype + "*" * stars))
    return fields


@pytest.mark.parametrize("struct", ["etc_moe_opts", "etc_mlp_opts"])
def test_binding_structs_match_the_header(struct):
    import ctypes as C

    from moe_layer_scheduling_gb300 import binding
    ctype_of = {"int": C.c_int, "unsigned": C.c_uint, "float": C.c_float,
                "unsigned long long": C.c_ulonglong, "const float*": C.c_void_p}
    hdr = _header_struct_fields(struct)
    py = getattr(binding, struct)._fields_
    assert [f for f, _ in hdr] == [f for f, _ in py], struct
    for (f, ct), (_, pt) in zip(hdr, py):
        assert ctype_of[ct] is pt, (struct, f, ct, pt)
