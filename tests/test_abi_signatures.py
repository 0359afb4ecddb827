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
