"""The C ABI library, on the CPU: it loads, exports every symbol include/bep.h
declares, and rejects bad configurations before touching a device."""
import ctypes
import os
import re

import pytest

import moe_expert_dispatch_online_gb300 as bep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libbep():
    from moe_expert_dispatch_online_gb300 import _build
    _build.build()
    return bep.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "bep.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bep_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_symbols() == sorted(bep.SYMBOLS)


def test_library_exports_every_declared_symbol(libbep):
    for name in declared_symbols():
        assert hasattr(libbep, name), name
        assert getattr(libbep, name) is not None


def test_no_oracle_in_product_path():
    """The package never imports the oracle (oracle/ is test infrastructure)."""
    pkg = os.path.join(ROOT, "moe_expert_dispatch_online_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                with open(os.path.join(dirpath, fn)) as f:
                    src = f.read()
                assert "import oracle" not in src and "from oracle" not in src, fn
                assert "liboracle" not in src, fn


def _create(lib, **kw):
    base = dict(R=8, E=64, B=8, K=4, S=1024, H=1024, Hp=512, mode=bep.BEP_TRAIN)
    base.update(kw)
    c = bep._Config(*[base[n] for n in ("R", "E", "B", "K", "S", "H", "Hp", "mode")])
    h = ctypes.c_void_p()
    rc = lib.bep_create(ctypes.byref(c), ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("kw,code", [
    (dict(E=63), bep.BEP_ERR_SIZE),            # E % R != 0
    (dict(B=7), bep.BEP_ERR_MODE),             # training needs B == E/R
    (dict(mode=1, B=8), bep.BEP_ERR_MODE),     # inference needs B < E/R
    (dict(mode=1, B=0), bep.BEP_ERR_MODE),
    (dict(mode=2), bep.BEP_ERR_ARG),
    (dict(K=0), bep.BEP_ERR_ARG),
    (dict(K=33), bep.BEP_ERR_SIZE),
    (dict(K=65, E=64), bep.BEP_ERR_SIZE),
    (dict(R=65, E=130, B=2), bep.BEP_ERR_SIZE),
    (dict(E=4096, B=512), bep.BEP_ERR_SIZE),
    (dict(H=100), bep.BEP_ERR_SIZE),
    (dict(Hp=96), bep.BEP_ERR_SIZE),
    (dict(S=1 << 26, K=8), bep.BEP_ERR_SIZE),  # R*S*K >= 2^31
    (dict(S=-1), bep.BEP_ERR_ARG),
])
def test_create_rejects_bad_configs(libbep, kw, code):
    rc, h = _create(libbep, **kw)
    assert rc == code
    assert not h.value


def test_null_arguments(libbep):
    assert libbep.bep_create(None, None) == bep.BEP_ERR_ARG
    assert libbep.bep_plan(None, None, None, None, None, None, None) == bep.BEP_ERR_ARG
    assert libbep.bep_dispatch(None, None, None, None, None) == bep.BEP_ERR_ARG
    assert libbep.bep_combine(None, None, None, None, 8, None, None) == bep.BEP_ERR_ARG
    assert libbep.bep_status(None, None, None) == bep.BEP_ERR_ARG
    libbep.bep_destroy(None)


def test_strerror(libbep):
    for code in (0, -1, -2, -3, -4, -5, 1, 2, 4, 8, 16):
        assert libbep.bep_strerror(code)
