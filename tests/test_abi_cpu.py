"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/moe.h declares, and validates arguments before it
launches anything (invalid calls return an error without touching CUDA)."""
import ctypes
import re

import pytest

import __graft_entry__
import expert_ffn_layer_gb300 as moe

ROOT = __graft_entry__.ROOT


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return moe.load()


def _declared_functions():
    text = (ROOT / "include" / "moe.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(moe.EXPORTS) == declared


def test_status_strings(lib):
    for code, name in moe.STATUS.items():
        assert moe.status_string(code).startswith(name)


def _hy3(T=8):
    return moe.dims(T, 4096, 192, 1536, 8)


def test_check_dims(lib):
    assert moe.moe_check_dims(_hy3()) == 0
    assert moe.moe_check_dims(moe.dims(0, 4096, 192, 1536, 8)) == 0          # empty batch is valid
    assert moe.moe_check_dims(moe.dims(8, 4000, 192, 1536, 8)) == 2          # H % 64
    assert moe.moe_check_dims(moe.dims(8, 4096, 192, 1500, 8)) == 2          # I % 64
    assert moe.moe_check_dims(moe.dims(8, 4096, 300, 1536, 8)) == 2          # E > 256
    assert moe.moe_check_dims(moe.dims(8, 4096, 8, 1536, 9)) == 2           # k > E
    assert moe.moe_check_dims(moe.dims(8, 4096, 64, 1536, 17)) == 2         # k > 16
    assert moe.moe_check_dims(moe.dims(-1, 4096, 64, 1536, 8)) == 1
    assert moe.moe_check_dims(moe.dims(8, 4096, 64, 1536, 0)) == 1
    assert moe.moe_check_dims(moe.dims(8, 4096, 64, 1536, 8, score_mode="softmax", route_scale=2.0)) == 1
    assert moe.moe_check_dims(moe.dims(8, 4096, 64, 1536, 8, renorm_eps=-1.0)) == 1
    assert moe.moe_check_dims(moe.dims(8, 4096, 64, 1536, 8, I_shared=100)) == 2
    assert moe.moe_check_dims(moe.dims(8, 4096, 64, 1536, 8, I_shared=100, has_shared=False)) == 0


def test_workspace_bytes(lib):
    d = _hy3(4096)
    n = moe.moe_workspace_bytes(d)
    S = 4096 * 8
    # dominated by y_sorted [S,H], y_shared [T,H], A_act [S,I], A_shared [T,I]
    # (bf16) and the W8A8 path's activation codes [S,I], [T,I] (one byte each);
    # the rest (routing tables, the router's bf16 weight halves and its split-K
    # partial logits, the W8A8 path's quantised hidden state, activation row
    # maxima and row scales) is a few tens of MB
    core = 2 * (S * 4096 + 4096 * 4096 + S * 1536 + 4096 * 1536) + (S * 1536 + 4096 * 1536)
    assert core <= n <= core + (64 << 20)
    assert n % 256 == 0
    assert moe.moe_workspace_bytes(_hy3(8)) < n
    assert lib.moe_workspace_bytes(ctypes.byref(moe.dims(8, 4000, 192, 1536, 8))) == 0


def test_invalid_arguments_are_rejected_before_launch(lib):
    d = _hy3()
    byref = ctypes.byref
    # null pointers
    assert lib.moe_route(byref(d), None, None, None, None, None, None, None, 0, None) == 1
    assert lib.moe_permute(byref(d), None, None, None, None, None, None, 0, None) == 1
    assert lib.moe_expert_ffn(byref(d), *([None] * 12), 0, None) == 1
    assert lib.moe_combine(byref(d), None, None, None, None, None, None) == 1
    assert lib.moe_layer_forward(byref(d), *([None] * 11), 0, None) == 1
    assert lib.moe_fused_moe(byref(d), *([None] * 9), 0, None) == 1
    assert lib.moe_expert_ffn_fp8(byref(d), None, None, None, None, None, None, None, 0, None) == 1
    assert lib.moe_layer_forward_fp8(byref(d), None, None, None, None, None, None, 0, None) == 1
    assert lib.moe_expert_ffn_w8a8(byref(d), None, None, None, None, None, None, None, 0, None) == 1
    assert lib.moe_layer_forward_w8a8(byref(d), None, None, None, None, None, None, 0, None) == 1
    # W8A8 needs H, I and I_shared multiples of 128 (checked before any pointer)
    assert lib.moe_expert_ffn_w8a8(byref(moe.dims(8, 192, 4, 64, 2)), None, None, None, None, None, None, None, 0,
                                   None) == 2
    assert lib.moe_quantize_fp8_rows(None, 4, 12, None, None, None) == 1      # cols % 8
    assert lib.moe_quantize_fp8_rows(None, 0, 16, None, None, None) == 0      # nothing to do
    # an FP8 weight struct with a missing scale array is rejected before launch
    fp8 = moe.MoeFp8Experts(gate=0x100000, up=0x100000, down=0x100000, gate_scale=0x100000, up_scale=None,
                            down_scale=0x100000, s_gate=0x100000, s_up=0x100000, s_down=0x100000,
                            s_gate_scale=0x100000, s_up_scale=0x100000, s_down_scale=0x100000)
    g = 0x100000
    assert lib.moe_expert_ffn_fp8(byref(d), g, g, g, byref(fp8), g, g, g, 1 << 40, None) == 1
    # misaligned pointer (never dereferenced: validation fails first)
    bad = 0x1003
    assert lib.moe_combine(byref(d), bad, bad, bad, bad, bad, None) == 1
    # a short workspace is reported as such (pointers aligned, never dereferenced)
    good = 0x100000
    args = [good] * 10  # hidden, router_w, bias, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, out
    assert lib.moe_layer_forward(byref(d), *args, good, 16, None) == 3
    # unsupported shapes win over pointer checks
    assert lib.moe_route(byref(moe.dims(8, 4000, 192, 1536, 8)), good, good, None, None, good, good, None, 0,
                         None) == 2
    assert lib.moe_ws_init(None, 0, None) == 1
    bits = ctypes.c_uint32()
    assert lib.moe_ws_read_error(None, 0, 0, None, byref(bits)) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib

    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "_LIB_PATH", tmp_path / "missing.so")
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        moe.load()
    importlib.reload(moe)


def _c_struct_fields(typedef_name):
    """(name, C type) of each field of `typedef struct { ... } typedef_name;` in
    moe.h, in declaration order (comments stripped; 'T, H, E' style lists split)."""
    text = re.sub(r"/\*.*?\*/", "", (ROOT / "include" / "moe.h").read_text(), flags=re.S)
    m = re.search(r"typedef struct \{([^{}]*)\}\s*" + typedef_name + r"\s*;", text)
    assert m, typedef_name
    fields = []
    for decl in m.group(1).split(";"):
        decl = decl.strip()
        if not decl:
            continue
        ctype, names = re.match(r"((?:const\s+)?[a-z0-9_]+\s*\**)\s*(.*)", decl).groups()
        for n in names.split(","):
            n = n.strip()
            stars = n.count("*")
            fields.append((n.lstrip("*").strip(), ctype.replace(" ", "") + "*" * stars))
    return fields


def test_binding_structs_match_the_header():
    """The ctypes mirrors of moe_dims and moe_fp8_experts have the header's
    fields in the header's order, with matching scalar kinds (a reordered or
    retyped field would silently pass the wrong value)."""
    dims = _c_struct_fields("moe_dims")
    assert [n for n, _ in dims] == [n for n, _ in moe.MoeDims._fields_]
    kinds = {"int": ctypes.c_int, "float": ctypes.c_float}
    for (n, t), (bn, bt) in zip(dims, moe.MoeDims._fields_):
        assert kinds[t] is bt, (n, t, bt)
    fp8 = _c_struct_fields("moe_fp8_experts")
    assert [n for n, _ in fp8] == [n for n, _ in moe.MoeFp8Experts._fields_]
    assert all(t.endswith("*") for _, t in fp8)                 # every field a pointer
    assert all(bt is ctypes.c_void_p for _, bt in moe.MoeFp8Experts._fields_)
    assert ctypes.sizeof(moe.MoeFp8Experts) == len(fp8) * ctypes.sizeof(ctypes.c_void_p)
