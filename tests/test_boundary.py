"""The C-ABI boundary without a GPU: the library builds for sm_103a, loads,
and exports every entry point include/minfer.h declares; the Python binding
marshals exactly those names; error codes agree between header and binding."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "minfer.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(minfer_\w+)\s*\(", text)))


def _defines():
    out = {}
    for m in re.finditer(r"#define\s+(MINFER_\w+)\s+\(?(-?\d+)\)?", open(HEADER).read()):
        out[m.group(1)] = int(m.group(2))
    return out


@pytest.fixture(scope="module")
def libpath():
    from quantized_transformer_prefill_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("minfer_load_weights", "minfer_kv_create", "minfer_prefill", "minfer_free",
                     "minfer_prefill_device", "minfer_kv_read", "minfer_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(minfer_\w+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(libpath)  # loads without a GPU
    for n in _declared():
        assert getattr(lib, n) is not None


def test_binding_matches_header(libpath):
    import quantized_transformer_prefill_gb300 as qp
    assert sorted(qp.SIGNATURES) == _declared()
    d = _defines()
    for code, name in qp.ERR_NAMES.items():
        assert d["MINFER_" + name] == code
    for code, name in qp.DEV_NAMES.items():
        assert d["MINFER_" + name] == code
    assert sorted(k for k in d if k.startswith("MINFER_DEV_")) == \
        sorted("MINFER_" + n for n in qp.DEV_NAMES.values())
    assert d["MINFER_F32"] == qp.MINFER_F32 and d["MINFER_Q8_0"] == qp.MINFER_Q8_0


def test_strerror_without_gpu(libpath):
    import quantized_transformer_prefill_gb300 as qp
    assert qp.lib().minfer_strerror(-2).decode().startswith("position out of range")
    assert qp.lib().minfer_strerror(0).decode() == "ok"


def test_create_without_gpu_fails_cleanly(libpath):
    """With no CUDA device the library returns an error code instead of
    falling back to anything."""
    import quantized_transformer_prefill_gb300 as qp
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    import synth
    ptr = ctypes.c_void_p()
    hp = qp.hparams_of(synth.TINY)
    rc = qp.lib().minfer_model_create(ctypes.byref(hp), ctypes.byref(ptr))
    assert rc == -6 and not ptr.value


_CITATION = re.compile(r'"09 · Prefill"|"05 · Graph build"|walkthrough index')


def test_every_declaration_cites_its_passage():
    """Each entry point of the header is preceded by a comment that names the
    passage of the pages defining it (page title and section), or says that
    the pages have no counterpart.  Declarations that follow one another with
    no comment between them share the comment above the first."""
    text = open(HEADER).read()
    last_comment = ""
    missing = []
    seen = []
    for m in re.finditer(r"/\*.*?\*/|\b(minfer_\w+)\s*\(", text, flags=re.S):
        if m.group(0).startswith("/*"):
            last_comment = m.group(0)
            continue
        # a declaration: the name follows its return type at the start of a line
        line = text[text.rfind("\n", 0, m.start()) + 1:m.start()]
        if not re.fullmatch(r"(int|void|const char\*)\s+", line):
            continue
        seen.append(m.group(1))
        # the comment's text with its line-leading '*' markers removed
        squashed = " ".join(re.sub(r"\n\s*\*(?!/)", " ", last_comment).split())
        if not (_CITATION.search(squashed) or "no counterpart" in squashed):
            missing.append(m.group(1))
    assert sorted(set(seen)) == _declared()
    assert not missing, f"declarations without a page citation: {missing}"
