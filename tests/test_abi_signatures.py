"""The binding's ctypes signatures match include/lq.h: every declared entry
point has a binding entry with the same number of parameters (a mismatch
would pass garbage through the C ABI without any error)."""
import os
import re

import lattice_vq_weight_gb300 as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_declarations():
    text = open(os.path.join(ROOT, "include", "lq.h")).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)          # comments
    decls = {}
    for m in re.finditer(r"\b(lq_\w+)\s*\(([^;{]*?)\)\s*;", text):
        name, params = m.group(1), m.group(2).strip()
        if params in ("", "void"):
            n = 0
        else:
            n = len([p for p in params.split(",") if p.strip()])
        decls[name] = n
    return decls


def test_every_declaration_is_bound_with_the_same_arity():
    decls = header_declarations()
    assert len(decls) >= 30
    missing = sorted(set(decls) - set(L.SIGNATURES))
    assert not missing, f"declared but not bound: {missing}"
    wrong = {name: (decls[name], len(L.SIGNATURES[name][1])) for name in decls
             if len(L.SIGNATURES[name][1]) != decls[name]}
    assert not wrong, f"arity (header, binding) differs: {wrong}"


def test_binding_declares_nothing_extra():
    extra = sorted(set(L.SIGNATURES) - set(header_declarations()))
    assert not extra, f"bound but not declared: {extra}"


def _ctype_of(c_decl: str):
    """ctypes type of one C parameter or return declaration."""
    import ctypes
    d = " ".join(c_decl.replace("const", " ").split())
    if "*" in d:
        return ctypes.c_void_p
    base = d.split()[0] if d else d
    return {"int": ctypes.c_int32, "int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64,
            "uint64_t": ctypes.c_uint64, "float": ctypes.c_float, "double": ctypes.c_double,
            "size_t": ctypes.c_size_t, "lq_status": ctypes.c_int32}.get(base)


def test_every_parameter_and_return_type_matches():
    import ctypes
    text = open(os.path.join(ROOT, "include", "lq.h")).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    bad = []
    for m in re.finditer(r"(\b[\w ]+?\**)\s*\b(lq_\w+)\s*\(([^;{]*?)\)\s*;", text):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        if name not in L.SIGNATURES:
            continue
        want_ret, want_args = L.SIGNATURES[name]
        ret_t = _ctype_of(ret.split("\n")[-1])
        if "char" in ret and "*" in ret:
            ret_t = ctypes.c_char_p
        if ret_t is not None and ctypes.sizeof(ret_t) != ctypes.sizeof(want_ret):
            bad.append((name, "return", ret))
        if params in ("", "void"):
            continue
        for i, (c, b) in enumerate(zip(params.split(","), want_args)):
            t = _ctype_of(c.strip().rsplit(" ", 1)[0] if "*" not in c else c)
            if t is None:
                bad.append((name, i, c.strip()))
            elif t is ctypes.c_void_p:
                if b not in (ctypes.c_void_p, ctypes.c_char_p):
                    bad.append((name, i, c.strip()))
            elif ctypes.sizeof(t) != ctypes.sizeof(b) or (t in (ctypes.c_float, ctypes.c_double)) != (
                    b in (ctypes.c_float, ctypes.c_double)):
                bad.append((name, i, c.strip()))
    assert not bad, f"type mismatches: {bad}"
